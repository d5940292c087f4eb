"""Pins for the backward oracle of the scan (the gradients of
ℓ = Σ dout·out + Σ dhT·h_L with respect to every input).

Each pin is a function of an oracle callable ``fn(u, delta, A, B, C, dout, D, z, bias,
h0, dhT) -> dict of gradients``.  Both oracles (the C loop and the NumPy restatement)
pass every pin; every planted mistake (a mutated copy built here on the CPU) fails one.
The pins do not use either oracle's derivation: central finite differences of the
forward oracle, and torch.autograd through a forward written here with torch ops.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from oracle import numpy_oracle

GRADS = ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "dbias", "dh0")


def c_bwd(u, delta, A, B, C, dout, D=None, z=None, bias=None, h0=None, dhT=None):
    return oracle.scan_bwd(u, delta, A, B, C, dout, D=D, z=z, bias=bias, h0=h0, dhT=dhT)


def np_bwd(u, delta, A, B, C, dout, D=None, z=None, bias=None, h0=None, dhT=None):
    return numpy_oracle.scan_bwd(u, delta, A, B, C, dout, D=D, z=z, bias=bias, h0=h0, dhT=dhT)


def problem(rng, batch=2, d=2, N=3, L=6, zero_a=True):
    p = dict(u=rng.standard_normal((batch, d, L)),
             delta=rng.standard_normal((batch, d, L)) * 0.7 - 1.5,
             A=-np.exp(rng.uniform(np.log(0.2), np.log(6.0), (d, N))),
             B=rng.standard_normal((batch, L, N)), C=rng.standard_normal((batch, L, N)),
             D=rng.standard_normal(d), z=rng.standard_normal((batch, d, L)), bias=0.3 * rng.standard_normal(d),
             h0=rng.standard_normal((batch, d, N)))
    if zero_a:
        p["A"][0, 1] = 0.0  # a state with A = 0 (Ā = 1, B̄ = ΔB)
    return p


def loss(p, dout, dhT):
    out, hT = oracle.scan(p["u"], p["delta"], p["A"], p["B"], p["C"], D=p["D"], z=p["z"], bias=p["bias"], h0=p["h0"])
    return float((out * dout).sum() + (hT * dhT).sum())


NAMES = dict(du="u", ddelta="delta", dA="A", dB="B", dC="C", dD="D", dz="z", dbias="bias", dh0="h0")


def pin_finite_differences(fn):
    """Every entry of every gradient against a central difference of the forward oracle."""
    rng = np.random.default_rng(11)
    p = problem(rng)
    dout = rng.standard_normal(p["u"].shape)
    dhT = rng.standard_normal(p["h0"].shape)
    g = fn(p["u"], p["delta"], p["A"], p["B"], p["C"], dout, D=p["D"], z=p["z"], bias=p["bias"], h0=p["h0"], dhT=dhT)
    eps = 1e-6
    for gk, name in NAMES.items():
        arr = p[name]
        fd = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + eps
            lp = loss(p, dout, dhT)
            arr[idx] = keep - eps
            lm = loss(p, dout, dhT)
            arr[idx] = keep
            fd[idx] = (lp - lm) / (2 * eps)
        scale = max(1.0, float(np.abs(fd).max()))
        np.testing.assert_allclose(g[gk], fd, rtol=0, atol=2e-6 * scale, err_msg=gk)


def _torch_forward(p):
    """The scan written with torch ops (float64) for autograd."""
    u, delta, A, B, C, D, z, bias, h0 = (p[k] for k in ("u", "delta", "A", "B", "C", "D", "z", "bias", "h0"))
    dt = torch.nn.functional.softplus(delta + bias[None, :, None])
    h = h0
    ys = []
    for t in range(u.shape[2]):
        dA = dt[:, :, t, None] * A[None]
        h = torch.exp(dA) * h + torch.expm1(dA) / A[None] * B[:, None, t, :] * u[:, :, t, None]
        y = (h * C[:, None, t, :]).sum(-1) + D[None] * u[:, :, t]
        ys.append(y * torch.nn.functional.silu(z[:, :, t]))
    return torch.stack(ys, dim=2), h


def pin_autograd(fn):
    """Against torch.autograd through a forward written with torch ops (A != 0)."""
    rng = np.random.default_rng(12)
    p = problem(rng, batch=2, d=3, N=4, L=9, zero_a=False)
    dout = rng.standard_normal(p["u"].shape)
    dhT = rng.standard_normal(p["h0"].shape)
    tp = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    out, hT = _torch_forward(tp)
    ell = (out * torch.tensor(dout)).sum() + (hT * torch.tensor(dhT)).sum()
    ell.backward()
    g = fn(p["u"], p["delta"], p["A"], p["B"], p["C"], dout, D=p["D"], z=p["z"], bias=p["bias"], h0=p["h0"], dhT=dhT)
    for gk, name in NAMES.items():
        np.testing.assert_allclose(g[gk], tp[name].grad.numpy(), rtol=1e-9, atol=1e-11, err_msg=gk)


def pin_linear_in_upstream(fn):
    """The gradients are linear in (dout, dhT)."""
    rng = np.random.default_rng(13)
    p = problem(rng)
    g1o, g2o = rng.standard_normal(p["u"].shape), rng.standard_normal(p["u"].shape)
    g1h, g2h = rng.standard_normal(p["h0"].shape), rng.standard_normal(p["h0"].shape)
    kw = dict(D=p["D"], z=p["z"], bias=p["bias"], h0=p["h0"])
    a = fn(p["u"], p["delta"], p["A"], p["B"], p["C"], g1o, dhT=g1h, **kw)
    b = fn(p["u"], p["delta"], p["A"], p["B"], p["C"], g2o, dhT=g2h, **kw)
    s = fn(p["u"], p["delta"], p["A"], p["B"], p["C"], 2.0 * g1o - g2o, dhT=2.0 * g1h - g2h, **kw)
    for k in GRADS:
        np.testing.assert_allclose(s[k], 2.0 * a[k] - b[k], rtol=1e-9, atol=1e-12, err_msg=k)


PINS = [pin_finite_differences, pin_autograd, pin_linear_in_upstream]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
@pytest.mark.parametrize("impl", [c_bwd, np_bwd], ids=["c", "numpy"])
def test_pin(impl, pin):
    pin(impl)


def test_two_backward_oracles_agree():
    rng = np.random.default_rng(14)
    for shape in [(2, 3, 4, 9), (1, 5, 16, 40), (3, 1, 1, 3)]:
        p = problem(rng, *shape, zero_a=shape[2] > 1)
        dout = rng.standard_normal(p["u"].shape)
        dhT = rng.standard_normal(p["h0"].shape)
        gc = c_bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], dout, D=p["D"], z=p["z"], bias=p["bias"],
                   h0=p["h0"], dhT=dhT)
        gn = np_bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], dout, D=p["D"], z=p["z"], bias=p["bias"],
                    h0=p["h0"], dhT=dhT)
        for k in GRADS:
            np.testing.assert_allclose(gc[k], gn[k], rtol=1e-11, atol=1e-13, err_msg=k)


# ---------------------------------------------------- planted mistakes ----

def _mutant(kind):
    """A copy of the NumPy backward with one plausible mistake planted."""
    def fn(u, delta, A, B, C, dout, D=None, z=None, bias=None, h0=None, dhT=None):
        batch, d, L = u.shape
        N = A.shape[1]
        r = delta + bias[None, :, None]
        dt = np.logaddexp(0.0, r)
        a = A[None]
        safe_a = np.where(a == 0.0, 1.0, a)
        hs = np.zeros((L + 1, batch, d, N))
        hs[0] = h0
        for t in range(L):
            abar, phi = numpy_oracle.discretize(dt[:, :, t, None], a)
            hs[t + 1] = abar * hs[t] + phi * B[:, None, t, :] * u[:, :, t, None]
        g = dict(du=np.empty_like(u), ddelta=np.empty_like(u), dz=np.empty_like(u), dA=np.zeros_like(A),
                 dB=np.zeros_like(B), dC=np.zeros_like(C), dD=np.zeros(d), dbias=np.zeros(d))
        dh = dhT.copy()
        for t in range(L - 1, -1, -1):
            x = u[:, :, t]
            hc = hs[t] if kind == "dC_prev_state" else hs[t + 1]
            y = np.einsum("bdn,bn->bd", hs[t + 1], C[:, t]) + D[None] * x
            s = expit(z[:, :, t])
            dsil = s if kind == "no_dsilu" else s * (1.0 + z[:, :, t] * (1.0 - s))
            g["dz"][:, :, t] = dout[:, :, t] * y * dsil
            dy = dout[:, :, t] * z[:, :, t] * s
            g["dD"] += (dy * x).sum(axis=0)
            dx = np.zeros_like(x) if kind == "dx_no_D" else dy * D[None]
            dh = dh + dy[:, :, None] * C[:, None, t, :]
            g["dC"][:, t] += np.einsum("bd,bdn->bn", dy, hc)
            abar, phi = numpy_oracle.discretize(dt[:, :, t, None], a)
            bx = B[:, None, t, :] * x[:, :, None]
            g["dB"][:, t] += np.einsum("bdn,bdn,bd->bn", dh, np.ones_like(phi) if kind == "dB_no_phi" else phi, x)
            dx = dx + np.einsum("bdn,bdn,bn->bd", dh, phi, B[:, t])
            dtn = dt[:, :, t, None]
            g["ddelta"][:, :, t] = (dh * abar * (a * hs[t] + bx)).sum(axis=2) * (
                1.0 if kind == "no_softplus_grad" else expit(r[:, :, t]))
            g["dbias"] += g["ddelta"][:, :, t].sum(axis=0)
            second = 0.0 if kind == "dA_one_term" else 1.0
            da = np.where(a == 0.0, dh * (dtn * hs[t] + second * bx * dtn * dtn / 2.0),
                          dh * (dtn * abar * hs[t] + second * bx * (dtn * abar - phi) / safe_a))
            g["dA"] += da.sum(axis=0)
            g["du"][:, :, t] = dx
            dh = dh if kind == "no_decay" else dh * abar
        g["dh0"] = dh
        return g
    return fn


MUTANTS = ["no_dsilu", "no_decay", "no_softplus_grad", "dB_no_phi", "dA_one_term", "dx_no_D", "dC_prev_state"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistake(kind):
    fn = _mutant(kind)
    failed = []
    for pin in PINS:
        try:
            pin(fn)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {kind}"


def test_unmutated_copy_passes():
    fn = _mutant("none")
    for pin in PINS:
        pin(fn)

"""Pins for the CPU oracle: facts fixed by the pages and by mathematics, not by
the oracle itself.

Each pin is a function of an oracle callable
``fn(u, delta, A, B, C, D=None, z=None, bias=None, h0=None) -> (out, hT)``.
Both oracles (the C loop and the NumPy restatement) must pass every pin, and
every planted mistake (a mutated copy of the NumPy oracle, built here on the
CPU) must fail at least one of them.
"""
import json
import os

import numpy as np
import pytest
from scipy.integrate import solve_ivp
from scipy.special import expit

import oracle
from oracle import numpy_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def inv_softplus(dt):
    """Δraw such that softplus(Δraw) = dt."""
    return np.log(np.expm1(dt))


def c_oracle(u, delta, A, B, C, D=None, z=None, bias=None, h0=None):
    return oracle.scan(u, delta, A, B, C, D=D, z=z, bias=bias, h0=h0, threads=2)


def np_oracle(u, delta, A, B, C, D=None, z=None, bias=None, h0=None):
    return numpy_oracle.scan(u, delta, A, B, C, D=D, z=z, bias=bias, h0=h0)


def rand_problem(rng, batch=2, d=3, N=4, L=17, gate=True, skip=True, with_bias=True):
    u = rng.standard_normal((batch, d, L))
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(0.5), (batch, d, L)))
    bias = 0.3 * rng.standard_normal(d) if with_bias else None
    delta = inv_softplus(dt) - (bias[None, :, None] if with_bias else 0.0)
    A = -np.exp(rng.uniform(np.log(0.2), np.log(8.0), (d, N)))
    B = rng.standard_normal((batch, L, N))
    C = rng.standard_normal((batch, L, N))
    D = rng.standard_normal(d) if skip else None
    z = rng.standard_normal((batch, d, L)) if gate else None
    return dict(u=u, delta=delta, A=A, B=B, C=C, D=D, z=z, bias=bias)


# ---------------------------------------------------------------- pins ----

def pin_worked_example(fn):
    """Page 'Mambaとは？…', scalar例: A=-1, B=C=1, D=0, Δ=0.5 → Ā≈0.607, B̄≈0.393,
    impulse weights 0.393, 0.239, 0.145, 0.088."""
    g = _golden("scalar_worked_example.json")
    p = g["inputs"]
    L = p["impulse_length"]
    x = np.zeros((1, 1, L)); x[0, 0, 0] = 1.0
    out, _ = fn(x, np.full((1, 1, L), inv_softplus(p["delta"])), np.array([[p["A"]]]),
                np.full((1, L, 1), p["B"]), np.full((1, L, 1), p["C"]), D=np.array([p["D"]]))
    y = out[0, 0]
    dec = g["decimals"]
    pr = g["printed"]
    assert np.round(y, dec).tolist() == pr["impulse_weights"]
    assert round(y[0], dec) == pr["Bbar"]              # first weight is B̄ (C = 1)
    assert round(y[1] / y[0], dec) == pr["Abar"]       # each step back multiplies by Ā


def pin_retention(fn):
    """Page 'Mambaとは？…', Mambaの核心: A=-1, Δ=0.1 keeps 0.905 of the state, Δ=2.0 keeps 0.135."""
    g = _golden("retention_examples.json")
    for case in g["cases"]:
        x = np.array([[[1.0, 0.0, 0.0]]])
        out, _ = fn(x, np.full((1, 1, 3), inv_softplus(case["delta"])), np.array([[g["A"]]]),
                    np.ones((1, 3, 1)), np.ones((1, 3, 1)))
        y = out[0, 0]
        assert round(y[1] / y[0], g["decimals"]) == case["Abar"]
        assert round(y[2] / y[1], g["decimals"]) == case["Abar"]


def pin_impulse_decay(fn):
    """Page 'Mamba / SSMと拡散LM', ① 線形スキャン: an impulse decaying at 0.8 per step is
    almost gone after 50 steps."""
    g = _golden("impulse_decay.json")
    steps = g["steps"]
    dt = -np.log(g["decay"])                        # A = -1 so that Ā = 0.8
    x = np.zeros((1, 1, steps + 1)); x[0, 0, 0] = 1.0
    out, _ = fn(x, np.full((1, 1, steps + 1), inv_softplus(dt)), np.array([[-1.0]]),
                np.ones((1, steps + 1, 1)), np.ones((1, steps + 1, 1)))
    y = out[0, 0]
    assert np.all(np.diff(y) < 0)
    assert y[steps] / y[0] < g["vanished_below"]
    assert y[steps] / y[0] == pytest.approx(g["decay"] ** steps, rel=1e-9)


def pin_running_sum(fn):
    """A → 0: Ā = 1 and B̄ = ΔB, so the state is the running sum Σ Δ_s B_s x_s
    (page 'Mamba / SSMと拡散LM': with decay 1 the inputs accumulate)."""
    rng = np.random.default_rng(11)
    L, N = 40, 3
    u = rng.standard_normal((1, 1, L))
    dt = rng.uniform(0.01, 0.3, (1, 1, L))
    B = rng.standard_normal((1, L, N))
    for k in range(N):
        Cs = np.zeros((1, L, N)); Cs[0, :, k] = 1.0
        out, hT = fn(u, inv_softplus(dt), np.zeros((1, N)), B, Cs)
        expect = np.cumsum(dt[0, 0] * B[0, :, k] * u[0, 0])
        np.testing.assert_allclose(out[0, 0], expect, rtol=1e-12, atol=1e-12)
    # continuity of the limit: a tiny negative A gives the same result to O(|A|)
    out0, _ = fn(u, inv_softplus(dt), np.zeros((1, N)), B, np.ones((1, L, N)))
    out1, _ = fn(u, inv_softplus(dt), np.full((1, N), -1e-9), B, np.ones((1, L, N)))
    np.testing.assert_allclose(out1, out0, rtol=1e-6, atol=1e-8)


def pin_zoh_ode(fn):
    """ZOH is the exact solution of dh/dt = A h + B x with x (and B) held
    constant over each step ('State Space Models（SSM）とMamba' §2.1–2.2).
    Integrate the continuous system numerically and read out y_k = C_k h_k + D x_k."""
    rng = np.random.default_rng(5)
    batch, d, N, L = 1, 2, 3, 6
    p = rand_problem(rng, batch, d, N, L, gate=False, with_bias=False)
    dt = np.logaddexp(0.0, p["delta"])  # step sizes the oracle will see
    out, hT = fn(**p)
    for c in range(d):
        h = np.zeros(N)
        for t in range(L):
            a, b, x = p["A"][c], p["B"][0, t], p["u"][0, c, t]
            sol = solve_ivp(lambda s, hh: a * hh + b * x, (0.0, dt[0, c, t]), h,
                            method="DOP853", rtol=1e-12, atol=1e-14)
            h = sol.y[:, -1]
            y = p["C"][0, t] @ h + p["D"][c] * x
            assert out[0, c, t] == pytest.approx(y, rel=1e-8, abs=1e-10)
        np.testing.assert_allclose(hT[0, c], h, rtol=1e-8, atol=1e-10)


def pin_lti_convolution(fn):
    """Time-invariant case: y = x * K̄ with K̄ = (CB̄, CĀB̄, CĀ²B̄, …)
    ('State Space Models（SSM）とMamba' §2.3; 'Mambaとは？…' 固定SSMには…二つの顔).
    K̄ is built by brute-force powers; B̄ by numerical quadrature of ∫exp(Aτ)dτ B."""
    rng = np.random.default_rng(7)
    d, N, L = 3, 4, 24
    A = -np.exp(rng.uniform(np.log(0.3), np.log(5.0), (d, N)))
    dtc = rng.uniform(0.05, 0.6, d)
    Bv, Cv = rng.standard_normal(N), rng.standard_normal(N)
    u = rng.standard_normal((1, d, L))
    delta = np.broadcast_to(inv_softplus(dtc)[None, :, None], (1, d, L)).copy()
    out, _ = fn(u, delta, A, np.broadcast_to(Bv, (1, L, N)).copy(),
                np.broadcast_to(Cv, (1, L, N)).copy())
    from scipy.integrate import quad
    for c in range(d):
        abar = np.exp(dtc[c] * A[c])
        bbar = np.array([quad(lambda s, a=A[c, n]: np.exp(a * s), 0.0, dtc[c], epsabs=1e-15, epsrel=1e-13)[0]
                         for n in range(N)]) * Bv
        K = np.array([sum(Cv[n] * abar[n] ** k * bbar[n] for n in range(N)) for k in range(L)])
        y = np.convolve(u[0, c], K)[:L]
        np.testing.assert_allclose(out[0, c], y, rtol=1e-9, atol=1e-12)


def pin_affine_composition(fn):
    """Each token is an affine map h ↦ Ā h + B̄x; composing the maps in any
    bracketing gives the sequential result ('Mambaとは？…', Selective Scanは
    選択機構そのものではない: (A₂,b₂)∘(A₁,b₁) = (A₂A₁, A₂b₁+b₂) is associative)."""
    rng = np.random.default_rng(3)
    p = rand_problem(rng, 1, 2, 3, 12, gate=False)
    L, N = 12, 3
    # per-token maps read off the oracle itself on one-token problems
    maps = []
    for t in range(L):
        sl = dict(u=p["u"][:, :, t:t + 1], delta=p["delta"][:, :, t:t + 1], A=p["A"],
                  B=p["B"][:, t:t + 1], C=p["C"][:, t:t + 1], bias=p["bias"])
        _, b_t = fn(**sl)                                   # h0 = 0 → b
        _, one = fn(**{**sl, "u": np.zeros_like(sl["u"])}, h0=np.ones((1, 2, N)))  # x = 0, h0 = 1 → Ā
        maps.append((one[0], b_t[0]))

    def compose(m2, m1):
        return (m2[0] * m1[0], m2[0] * m1[1] + m2[1])

    def tree(lo, hi, split_rng):
        if hi - lo == 1:
            return maps[lo]
        mid = split_rng.integers(lo + 1, hi)
        return compose(tree(mid, hi, split_rng), tree(lo, mid, split_rng))

    _, hT = fn(**p)
    for seed in range(5):
        _, b = tree(0, L, np.random.default_rng(seed))
        np.testing.assert_allclose(hT[0], b, rtol=1e-12, atol=1e-14)


def pin_skip_and_gate(fn):
    """D is a skip path that bypasses the state; the gate multiplies the whole
    SSM output by silu(z) ('Mambaとは？…', 状態空間モデル… (D) and Mamba block step 4)."""
    rng = np.random.default_rng(9)
    p = rand_problem(rng, 2, 3, 4, 9)
    zeroC = {**p, "C": np.zeros_like(p["C"])}
    out, _ = fn(**{**zeroC, "z": None})
    np.testing.assert_allclose(out, p["D"][None, :, None] * p["u"], rtol=1e-14, atol=1e-14)
    out, _ = fn(**zeroC)
    silu = p["z"] * expit(p["z"])
    np.testing.assert_allclose(out, p["D"][None, :, None] * p["u"] * silu, rtol=1e-13, atol=1e-14)
    # gate identities: silu(0) = 0 and silu(z) - silu(-z) = z
    y, _ = fn(**{**p, "z": None})
    o0, _ = fn(**{**p, "z": np.zeros_like(p["z"])})
    np.testing.assert_allclose(o0, 0.0, atol=1e-15)
    op, _ = fn(**p)
    om, _ = fn(**{**p, "z": -p["z"]})
    np.testing.assert_allclose(op - om, y * p["z"], rtol=1e-11, atol=1e-12)


def pin_locality_and_causality(fn):
    """y_t uses only inputs at times ≤ t, and reads the state through C_t only."""
    rng = np.random.default_rng(13)
    p = rand_problem(rng, 1, 2, 3, 15)
    base, _ = fn(**p)
    s = 7
    for key in ("u", "delta", "z"):
        q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
        q[key][:, :, s] += 1.0
        o, _ = fn(**q)
        np.testing.assert_array_equal(o[:, :, :s], base[:, :, :s])
        assert np.all(o[:, :, s] != base[:, :, s])
    for key in ("B", "C"):
        q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
        q[key][:, s, :] += 1.0
        o, _ = fn(**q)
        np.testing.assert_array_equal(o[:, :, :s], base[:, :, :s])
        if key == "C":   # the readout at t uses C_t and nothing else
            np.testing.assert_array_equal(o[:, :, s + 1:], base[:, :, s + 1:])
        else:            # B_s enters the state and so every later output
            assert np.all(o[:, :, s + 1:] != base[:, :, s + 1:])


def pin_linearity(fn):
    """With Δ, B, C fixed and no gate, the map u → y is linear."""
    rng = np.random.default_rng(17)
    p = rand_problem(rng, 1, 2, 4, 11, gate=False)
    u2 = rng.standard_normal(p["u"].shape)
    o1, h1 = fn(**p)
    o2, h2 = fn(**{**p, "u": u2})
    o3, h3 = fn(**{**p, "u": 2.5 * p["u"] - 0.75 * u2})
    np.testing.assert_allclose(o3, 2.5 * o1 - 0.75 * o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(h3, 2.5 * h1 - 0.75 * h2, rtol=1e-11, atol=1e-12)


def pin_split_continue(fn):
    """Running the first part, then continuing from its final state, equals one
    run ('Mambaとは？…', training、prefill、decode: decode carries the state on)."""
    rng = np.random.default_rng(19)
    p = rand_problem(rng, 2, 3, 4, 20)
    full, hT = fn(**p)
    k = 8
    def part(lo, hi):
        return dict(u=p["u"][:, :, lo:hi], delta=p["delta"][:, :, lo:hi], A=p["A"],
                    B=p["B"][:, lo:hi], C=p["C"][:, lo:hi], D=p["D"], z=p["z"][:, :, lo:hi],
                    bias=p["bias"])
    o1, h1 = fn(**part(0, k))
    o2, h2 = fn(**part(k, 20), h0=h1)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=2), full, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(h2, hT, rtol=1e-12, atol=1e-14)


def pin_step_size_limits(fn):
    """Δ → 0 keeps the state and ignores the input; large Δ forgets the state and
    writes x·B/|A| ('State Space Models（SSM）とMamba' §4.2 直感; 'Mamba / SSMと拡散LM'
    ② 選択的 SSM: a closed gate leaves only the decay).  softplus(Δraw + bias) is
    unchanged by moving a constant between Δraw and the bias."""
    rng = np.random.default_rng(23)
    N = 3
    h0 = rng.standard_normal((1, 1, N))
    A = -np.array([[1.0, 2.0, 4.0]])
    B = rng.standard_normal((1, 1, N))
    _, h = fn(np.array([[[5.0]]]), np.array([[[-60.0]]]), A, B, np.ones((1, 1, N)), h0=h0)
    np.testing.assert_allclose(h, h0, rtol=1e-20, atol=1e-20)
    _, h = fn(np.array([[[5.0]]]), np.array([[[60.0]]]), A, B, np.ones((1, 1, N)), h0=h0)
    np.testing.assert_allclose(h[0, 0], 5.0 * B[0, 0] / np.abs(A[0]), rtol=1e-14)
    p = rand_problem(rng, 1, 3, 2, 8)
    o1, _ = fn(**p)
    o2, _ = fn(**{**p, "delta": p["delta"] + 0.7, "bias": p["bias"] - 0.7})
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    o3, _ = fn(**{**p, "delta": p["delta"] + p["bias"][None, :, None], "bias": None})
    np.testing.assert_allclose(o3, o1, rtol=1e-12, atol=1e-13)


PINS = [pin_worked_example, pin_retention, pin_impulse_decay, pin_running_sum, pin_zoh_ode,
        pin_lti_convolution, pin_affine_composition, pin_skip_and_gate,
        pin_locality_and_causality, pin_linearity, pin_split_continue, pin_step_size_limits]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
@pytest.mark.parametrize("impl", [c_oracle, np_oracle], ids=["c", "numpy"])
def test_pin(impl, pin):
    pin(impl)


def test_two_oracles_agree():
    """The C loop and the NumPy restatement agree on a ragged random problem."""
    rng = np.random.default_rng(29)
    for shape in [(2, 5, 7, 33), (1, 16, 4, 64), (3, 2, 1, 5)]:
        p = rand_problem(rng, *shape)
        oc, hc = c_oracle(**p)
        on, hn = np_oracle(**p)
        np.testing.assert_allclose(oc, on, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(hc, hn, rtol=1e-12, atol=1e-13)


def test_step_equals_scan():
    """L recurrent steps reproduce the parallel-mode scan exactly (same arithmetic)."""
    rng = np.random.default_rng(31)
    p = rand_problem(rng, 2, 3, 4, 10)
    out, hT = oracle.scan(**p)
    state = np.zeros((2, 3, 4))
    for t in range(10):
        y, state = oracle.step(state, p["u"][:, :, t], p["delta"][:, :, t], p["A"], p["B"][:, t],
                               p["C"][:, t], D=p["D"], z=p["z"][:, :, t], bias=p["bias"])
        np.testing.assert_array_equal(y, out[:, :, t])
    np.testing.assert_array_equal(state, hT)
    yn, sn = numpy_oracle.step(np.zeros((2, 3, 4)), p["u"][:, :, 0], p["delta"][:, :, 0], p["A"],
                               p["B"][:, 0], p["C"][:, 0], D=p["D"], z=p["z"][:, :, 0], bias=p["bias"])
    np.testing.assert_allclose(yn, out[:, :, 0], rtol=1e-13)


# ---------------------------------------------------- planted mistakes ----

def _mutant(kind):
    """A copy of the NumPy oracle with one plausible mistake planted."""
    def fn(u, delta, A, B, C, D=None, z=None, bias=None, h0=None):
        u, delta, A, B, C = (np.asarray(x, np.float64) for x in (u, delta, A, B, C))
        batch, d, L = u.shape
        N = A.shape[1]
        r = delta + (0.0 if (bias is None or kind == "bias_ignored") else bias[None, :, None])
        dt = r if kind == "no_softplus" else np.logaddexp(0.0, r)
        h = np.zeros((batch, d, N)) if h0 is None else np.array(h0, np.float64)
        out = np.empty((batch, d, L))
        for t in range(L):
            dA = dt[:, :, t, None] * A[None]
            abar = np.exp(-dA if kind == "sign_A" else dA)
            safe = np.where(A == 0, 1.0, A)[None]
            if kind == "euler_B":
                phi = np.broadcast_to(dt[:, :, t, None], dA.shape)
            elif kind == "no_div_A":
                phi = np.expm1(dA)
            else:
                phi = np.where(A[None] == 0, dt[:, :, t, None], np.expm1(dA) / safe)
            Bt = C[:, None, t, :] if kind == "swap_BC" else B[:, None, t, :]
            Ct = B[:, t, :] if kind == "swap_BC" else C[:, t, :]
            if kind == "B_reversed":
                Bt = B[:, None, L - 1 - t, :]
            h_prev = h
            h = abar * h + phi * Bt * u[:, :, t, None]
            hr = h_prev if kind == "stale_readout" else h
            y = np.einsum("bdn,bn->bd", hr, Ct)
            if z is not None and kind == "gate_before_D":
                y = y * (z[:, :, t] * expit(z[:, :, t]))
            if D is not None and kind != "drop_D":
                y = y + D[None, :] * u[:, :, t]
            if z is not None and kind != "gate_before_D":
                g = expit(z[:, :, t]) if kind == "sigmoid_gate" else z[:, :, t] * expit(z[:, :, t])
                y = y * g
            out[:, :, t] = y
        return out, h
    return fn


MUTANTS = ["no_softplus", "bias_ignored", "sign_A", "euler_B", "no_div_A", "swap_BC",
           "B_reversed", "stale_readout", "gate_before_D", "drop_D", "sigmoid_gate"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistake(kind):
    fn = _mutant(kind)
    failed = []
    for pin in PINS:
        try:
            pin(fn)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {kind!r}"


def test_unmutated_copy_passes():
    """The mutation harness itself is sound: with no mistake planted it passes every pin."""
    fn = _mutant("none")
    for pin in PINS:
        pin(fn)

"""Pins of the Mamba-2 (SSD) layer-scan oracle, none of which uses the oracle's own
arithmetic: the pages' duality statement (the scalar-A SSM equals masked linear
attention, "Mambaとは？Transformer以外の系列モデル", section Mamba-2とTransformerとの関係性;
"State Space Models（SSM）とMamba" §4.6 Mamba-2) computed as a quadratic form,
plain causal linear attention when A = 0, the single-token closed form, the impulse
response, the chunked evaluation and the head-to-group mapping."""
import numpy as np
import pytest

import oracle
import oracle.numpy_oracle as no
import workloads as W

KEYS = ("x", "dt", "A", "B", "C", "D", "z", "dt_bias")


def _np(inp):
    return {k: (None if inp[k] is None else inp[k].double().numpy()) for k in KEYS}


def _rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


@pytest.mark.parametrize("shape", [(2, 37, 4, 3, 2, 5), (1, 64, 3, 8, 1, 16), (2, 1, 6, 2, 3, 4), (1, 50, 2, 1, 2, 1)])
@pytest.mark.parametrize("opts", [dict(), dict(gate=False), dict(skip=False, with_bias=False)])
def test_ssd_recurrence_equals_quadratic_form(shape, opts):
    inp = _np(W.random_ssd_inputs(*shape, seed=sum(shape), **opts))
    out, hT = oracle.ssd_scan(**inp)
    out2, hT2 = no.ssd_dual(**inp)
    assert _rel(out, out2) < 1e-12
    assert _rel(hT, hT2) < 1e-12


def test_ssd_is_causal_linear_attention_when_A_is_zero():
    """A = 0 and one step size: y_t = Δ C_t Σ_{s≤t} B_s x_sᵀ (a running key-value sum)."""
    rng = np.random.default_rng(3)
    b, L, H, P, G, N = 2, 20, 2, 3, 1, 4
    x = rng.standard_normal((b, L, H, P))
    B = rng.standard_normal((b, L, G, N))
    C = rng.standard_normal((b, L, G, N))
    step = 0.07
    dt = np.full((b, L, H), np.log(np.expm1(step)))
    out, hT = oracle.ssd_scan(x, dt, np.zeros(H), B, C)
    kv = np.cumsum(np.einsum("bsn,bshp->bshpn", B[:, :, 0], x), axis=1)      # Σ_{s≤t} x_s B_sᵀ
    expect = step * np.einsum("btn,bthpn->bthp", C[:, :, 0], kv)
    assert _rel(out, expect) < 1e-12
    assert _rel(hT, step * kv[:, -1]) < 1e-12


def test_ssd_single_token():
    """L = 1: y = φ (C·B) x + D x, gated, with φ = expm1(Δa)/a."""
    inp = _np(W.random_ssd_inputs(2, 1, 4, 3, 2, 5, seed=7))
    out, _ = oracle.ssd_scan(**inp)
    delta = np.log1p(np.exp(inp["dt"][:, 0] + inp["dt_bias"]))                # [b, H]
    a = inp["A"]
    phi = np.expm1(delta * a) / a
    g = np.arange(4) // 2
    cb = np.einsum("bhn,bhn->bh", inp["C"][:, 0, g], inp["B"][:, 0, g])
    x, z = inp["x"][:, 0], inp["z"][:, 0]
    y = (phi * cb)[:, :, None] * x + inp["D"][None, :, None] * x
    expect = y * z / (1.0 + np.exp(-z))
    assert _rel(out[:, 0], expect) < 1e-13


def test_ssd_impulse_response():
    """x = unit impulse at t = 0, B = C = e_0: y_t = φ_0 exp(a Σ_{0<k≤t} Δ_k)."""
    b, L, H, P, G, N = 1, 30, 2, 2, 1, 3
    rng = np.random.default_rng(5)
    x = np.zeros((b, L, H, P))
    x[0, 0, 1, 1] = 1.0
    B = np.zeros((b, L, G, N))
    C = np.zeros((b, L, G, N))
    B[..., 0] = 1.0
    C[..., 0] = 1.0
    dt = rng.uniform(-3.0, 0.0, (b, L, H))
    A = np.array([-0.5, -2.5])
    out, _ = oracle.ssd_scan(x, dt, A, B, C)
    delta = np.log1p(np.exp(dt[0, :, 1]))
    phi0 = np.expm1(delta[0] * A[1]) / A[1]
    expect = phi0 * np.exp(A[1] * (np.cumsum(delta) - delta[0]))
    assert _rel(out[0, :, 1, 1], expect) < 1e-13
    assert np.all(out[0, :, 0] == 0.0) and np.all(out[0, :, 1, 0] == 0.0)


@pytest.mark.parametrize("chunk", [1, 4, 7, 64])
def test_ssd_chunked_evaluation(chunk):
    """Quadratic form inside chunks plus the carried state between them equals the
    recurrence (the decomposition that makes the chunk work matrix products)."""
    inp = _np(W.random_ssd_inputs(2, 45, 4, 3, 2, 6, seed=chunk))
    out, hT = oracle.ssd_scan(**inp)
    out2, hT2 = no.ssd_chunked(**inp, chunk=chunk)
    assert _rel(out, out2) < 1e-12
    assert _rel(hT, hT2) < 1e-12


def test_ssd_heads_read_their_own_group():
    """Changing group 1's B and C changes heads 2, 3 (group 1) and leaves heads 0, 1."""
    inp = _np(W.random_ssd_inputs(1, 25, 4, 3, 2, 5, seed=11))
    out, _ = oracle.ssd_scan(**inp)
    inp2 = dict(inp)
    inp2["B"] = inp["B"].copy()
    inp2["C"] = inp["C"].copy()
    inp2["B"][:, :, 1] *= -1.7
    inp2["C"][:, :, 1] += 0.3
    out2, _ = oracle.ssd_scan(**inp2)
    assert np.array_equal(out[:, :, :2], out2[:, :, :2])
    assert not np.allclose(out[:, :, 2:], out2[:, :, 2:])


def test_ssd_initial_state_continues_a_split_sequence():
    """Running the first part, then the rest from its final state, equals one run."""
    inp = _np(W.random_ssd_inputs(2, 40, 4, 3, 2, 5, seed=13))
    out, hT = oracle.ssd_scan(**inp)
    first = {k: (v if k in ("A", "D", "dt_bias") or v is None else v[:, :17]) for k, v in inp.items()}
    rest = {k: (v if k in ("A", "D", "dt_bias") or v is None else v[:, 17:]) for k, v in inp.items()}
    o1, h1 = oracle.ssd_scan(**first)
    o2, h2 = oracle.ssd_scan(**rest, h0=h1)
    assert _rel(np.concatenate([o1, o2], axis=1), out) < 1e-13
    assert _rel(h2, hT) < 1e-13

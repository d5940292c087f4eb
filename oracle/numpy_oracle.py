"""Second, independent restatement of the oracle in NumPy float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).  It is written
separately from ``ssm_oracle.c`` so that the two can be checked against each
other: vectorised over (batch, channel, state), sequential over t.  softplus
is evaluated with ``np.logaddexp`` and the gate with ``scipy.special.expit``
rather than the C file's hand-written forms.

Definitions followed: zero-order hold Ā = exp(ΔA), B̄ = (ΔA)^-1(exp(ΔA) - I)ΔB
("State Space Models（SSM）とMamba" §2.2 離散化), recurrence h_t = Ā h_{t-1} + B̄ x_t
and readout y_t = C_t h_t + D x_t ("Mambaとは？Transformer以外の系列モデル",
section 状態空間モデルを一つの式から理解する), gate y · silu(z) (same page,
section Mamba blockのarchitecture).
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit


def _arr(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def discretize(dt, a):
    """ZOH for diagonal A: returns (Ā, B̄/B) elementwise; B̄/B = Δ at a == 0."""
    dA = dt * a
    abar = np.exp(dA)
    safe_a = np.where(a == 0.0, 1.0, a)
    phi = np.where(a == 0.0, dt, np.expm1(dA) / safe_a)
    return abar, phi


def scan(u, delta, A, B, C, D=None, z=None, bias=None, h0=None):
    u, delta, A, B, C = (_arr(x) for x in (u, delta, A, B, C))
    D, z, bias, h0 = (_arr(x) for x in (D, z, bias, h0))
    batch, d_inner, L = u.shape
    N = A.shape[1]
    r = delta + (bias[None, :, None] if bias is not None else 0.0)
    dt = np.logaddexp(0.0, r)                      # softplus
    h = np.zeros((batch, d_inner, N)) if h0 is None else h0.copy()
    out = np.empty((batch, d_inner, L))
    for t in range(L):
        abar, phi = discretize(dt[:, :, t, None], A[None, :, :])
        bbar = phi * B[:, None, t, :]
        h = abar * h + bbar * u[:, :, t, None]
        y = np.einsum("bdn,bn->bd", h, C[:, t, :])
        if D is not None:
            y = y + D[None, :] * u[:, :, t]
        if z is not None:
            y = y * (z[:, :, t] * expit(z[:, :, t]))
        out[:, :, t] = y
    return out, h


def step(state, x, delta, A, B, C, D=None, z=None, bias=None):
    """One recurrent-mode token: returns (out [batch, d_inner], new_state)."""
    out, h = scan(_arr(x)[:, :, None], _arr(delta)[:, :, None], A, _arr(B)[:, None, :],
                  _arr(C)[:, None, :], D, None if z is None else _arr(z)[:, :, None], bias,
                  _arr(state))
    return out[:, :, 0], h


def conv1d(x, w, bias=None, state0=None):
    """Causal depthwise Conv1D + SiLU, vectorised over (batch, channel) and over
    the W taps: the sequence is prefixed with the W-1 carried inputs (zeros when
    state0 is None) and tap k multiplies the window shifted by W-1-k
    ("Mambaとは？Transformer以外の系列モデル", section Mamba blockのarchitecture,
    steps 2-3)."""
    x, w, bias, state0 = (_arr(v) for v in (x, w, bias, state0))
    batch, d, L = x.shape
    W = w.shape[1]
    pre_pad = np.zeros((batch, d, W - 1)) if state0 is None else state0
    xt = np.concatenate([pre_pad, x], axis=2)  # x̃, length L + W - 1
    pre = np.zeros((batch, d, L)) if bias is None else np.broadcast_to(bias[None, :, None], (batch, d, L)).copy()
    for k in range(W):
        pre += w[None, :, k, None] * xt[:, :, k:k + L]
    out = pre * expit(pre)
    return out, xt[:, :, L:].copy()


def scan_bwd(u, delta, A, B, C, dout, D=None, z=None, bias=None, h0=None, dhT=None):
    """Gradients of sum(dout * out) + sum(dhT * h_L) of ``scan``, written
    independently of the C oracle: vectorised over (batch, channel, state),
    sequential over t, with the step-size and A derivatives in factored form
        dℓ/dΔ_t = Σ_n dh_t Ā_t (a h_{t-1} + B_t x_t)
        dℓ/da   = Σ_t dh_t (Δ_t Ā_t h_{t-1} + B_t x_t (Δ_t Ā_t − φ_t)/a)   (a → 0: Δ h_{t-1} + B x Δ²/2)
    (the chain rule on the zero-order hold of "State Space Models（SSM）とMamba" §2.2)."""
    u, delta, A, B, C, dout = (_arr(x) for x in (u, delta, A, B, C, dout))
    D, z, bias, h0, dhT = (_arr(x) for x in (D, z, bias, h0, dhT))
    batch, d, L = u.shape
    N = A.shape[1]
    r = delta + (0.0 if bias is None else bias[None, :, None])
    dt = np.logaddexp(0.0, r)                                     # [b, d, L]
    a = A[None]                                                   # [1, d, N]
    hs = np.zeros((L + 1, batch, d, N))
    if h0 is not None:
        hs[0] = h0
    abar_all = np.empty((L, batch, d, N))
    phi_all = np.empty((L, batch, d, N))
    for t in range(L):
        abar, phi = discretize(dt[:, :, t, None], a)
        abar_all[t], phi_all[t] = abar, phi
        hs[t + 1] = abar * hs[t] + phi * B[:, None, t, :] * u[:, :, t, None]
    g = {k: None for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "dbias", "dh0")}
    g["du"] = np.empty_like(u)
    g["ddelta"] = np.empty_like(u)
    g["dB"] = np.zeros_like(B)
    g["dC"] = np.zeros_like(C)
    g["dA"] = np.zeros_like(A)
    if D is not None:
        g["dD"] = np.zeros(d)
    if z is not None:
        g["dz"] = np.empty_like(u)
    dbias = np.zeros(d)
    dh = np.zeros((batch, d, N)) if dhT is None else dhT.copy()
    safe_a = np.where(a == 0.0, 1.0, a)
    for t in range(L - 1, -1, -1):
        x = u[:, :, t]
        y = np.einsum("bdn,bn->bd", hs[t + 1], C[:, t])
        if D is not None:
            y = y + D[None] * x
        dy = dout[:, :, t]
        if z is not None:
            s = expit(z[:, :, t])
            g["dz"][:, :, t] = dout[:, :, t] * y * s * (1.0 + z[:, :, t] * (1.0 - s))
            dy = dy * z[:, :, t] * s
        dx = np.zeros_like(x) if D is None else dy * D[None]
        if D is not None:
            g["dD"] += (dy * x).sum(axis=0)
        dh = dh + dy[:, :, None] * C[:, None, t, :]
        g["dC"][:, t] += np.einsum("bd,bdn->bn", dy, hs[t + 1])
        abar, phi = abar_all[t], phi_all[t]
        bx = B[:, None, t, :] * x[:, :, None]                     # B x, [b, d, N]
        g["dB"][:, t] += np.einsum("bdn,bdn,bd->bn", dh, phi, x)
        dx = dx + np.einsum("bdn,bdn,bn->bd", dh, phi, B[:, t])
        dtn = dt[:, :, t, None]
        ddt = (dh * abar * (a * hs[t] + bx)).sum(axis=2)
        da = np.where(a == 0.0, dh * (dtn * hs[t] + bx * dtn * dtn / 2.0),
                      dh * (dtn * abar * hs[t] + bx * (dtn * abar - phi) / safe_a))
        g["dA"] += da.sum(axis=0)
        g["du"][:, :, t] = dx
        dr = ddt * expit(r[:, :, t])
        g["ddelta"][:, :, t] = dr
        dbias += dr.sum(axis=0)
        dh = dh * abar
    g["dbias"] = dbias
    g["dh0"] = dh
    return g


def _ssd_prep(x, dt, A, B, C, D, z, dt_bias):
    x, dt, A, B, C = (_arr(v) for v in (x, dt, A, B, C))
    D, z, dt_bias = (_arr(v) for v in (D, z, dt_bias))
    H, G = x.shape[2], B.shape[2]
    r = dt + (dt_bias[None, None, :] if dt_bias is not None else 0.0)
    delta = np.logaddexp(0.0, r)                           # [batch, L, H]
    la = delta * A[None, None, :]                          # log Ā_t
    safe = np.where(A == 0.0, 1.0, A)[None, None, :]
    phi = np.where(A[None, None, :] == 0.0, delta, np.expm1(la) / safe)
    head_group = np.arange(H) // (H // G)
    Bh, Ch = B[:, :, head_group, :], C[:, :, head_group, :]   # [batch, L, H, N]
    return x, D, z, la, phi, Bh, Ch


def _gate(y, x, D, z):
    if D is not None:
        y = y + D[None, None, :, None] * x
    if z is not None:
        y = y * (z * expit(z))
    return y


def ssd_dual(x, dt, A, B, C, D=None, z=None, dt_bias=None):
    """The quadratic ("attention") form of the Mamba-2 layer scan, with no
    recurrence: y_t = Σ_{s≤t} (Π_{s<k≤t} Ā_k) φ_s (C_t·B_s) x_s + D x_t, i.e. causal
    linear attention with queries C, keys B, values φ x and a decay mask
    ("Mambaとは？Transformer以外の系列モデル", section Mamba-2とTransformerとの関係性).
    Returns (out [batch, L, H, P], hT [batch, H, P, N])."""
    x, D, z, la, phi, Bh, Ch = _ssd_prep(x, dt, A, B, C, D, z, dt_bias)
    L = x.shape[1]
    cum = np.cumsum(la, axis=1)                            # Σ_{k≤t} log Ā_k
    diff = cum[:, :, None, :] - cum[:, None, :, :]         # [batch, t, s, H]
    causal = np.tril(np.ones((L, L), bool))[None, :, :, None]
    decay = np.where(causal, np.exp(np.where(causal, diff, 0.0)), 0.0)
    cb = np.einsum("bthn,bshn->btsh", Ch, Bh)
    M = decay * cb * phi[:, None, :, :]
    y = np.einsum("btsh,bshp->bthp", M, x)
    w = np.exp(cum[:, -1:, :] - cum) * phi                 # weight of token s in the final state
    hT = np.einsum("bsh,bshp,bshn->bhpn", w, x, Bh)
    return _gate(y, x, D, z), hT


def ssd_chunked(x, dt, A, B, C, D=None, z=None, dt_bias=None, chunk=64):
    """The chunked evaluation of the same map: inside each chunk the quadratic form,
    between chunks the state, carried as h ← e^{Σ log Ā over the chunk} h + (the
    chunk's own contribution), and read by every token as C_t e^{Σ log Ā since the
    chunk's start} h.  Returns (out, hT) as ``ssd_dual``."""
    x, D, z, la, phi, Bh, Ch = _ssd_prep(x, dt, A, B, C, D, z, dt_bias)
    batch, L, H, P = x.shape
    N = Bh.shape[-1]
    y = np.zeros((batch, L, H, P))
    h = np.zeros((batch, H, P, N))
    for c0 in range(0, L, chunk):
        sl = slice(c0, min(L, c0 + chunk))
        q = sl.stop - sl.start
        cum = np.cumsum(la[:, sl], axis=1)                 # since the chunk's start, inclusive
        diff = cum[:, :, None, :] - cum[:, None, :, :]
        causal = np.tril(np.ones((q, q), bool))[None, :, :, None]
        decay = np.where(causal, np.exp(np.where(causal, diff, 0.0)), 0.0)
        cb = np.einsum("bthn,bshn->btsh", Ch[:, sl], Bh[:, sl])
        y[:, sl] = np.einsum("btsh,bshp->bthp", decay * cb * phi[:, None, sl, :], x[:, sl])
        y[:, sl] += np.einsum("bth,bthn,bhpn->bthp", np.exp(cum), Ch[:, sl], h)
        w = np.exp(cum[:, -1:, :] - cum) * phi[:, sl]
        h = np.exp(cum[:, -1, :])[:, :, None, None] * h + np.einsum("bsh,bshp,bshn->bhpn", w, x[:, sl], Bh[:, sl])
    return _gate(y, x, D, z), h

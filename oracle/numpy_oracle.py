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

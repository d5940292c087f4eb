"""Double-precision CPU oracle for the selective state-space scan (S6).

TEST INFRASTRUCTURE ONLY.  The library never imports this package.  The tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` are its only
users.  It shares no code with the CUDA path: the arithmetic lives in
``ssm_oracle.c`` (compiled with plain gcc, no fast-math) and, as an independent
second restatement, in ``numpy_oracle.py``.

What it computes (the plain definition, sequential over t, in float64):

    Δ_t   = softplus(Δraw_t + bias)
    Ā     = exp(Δ_t A),  B̄ = (Δ_t A)^-1 (exp(Δ_t A) - I) Δ_t B_t
    h_t   = Ā h_{t-1} + B̄ x_t            (h_0 = 0 unless h0 is given)
    y_t   = C_t h_t + D x_t
    out_t = y_t · silu(z_t)

Sources: "State Space Models（SSM）とMamba" §2.2 離散化 and §4.2 Selective SSM;
"Mambaとは？Transformer以外の系列モデル", sections 状態空間モデルを一つの式から理解する,
固定SSMには「再帰」と「畳み込み」の二つの顔がある and Mamba blockのarchitecture.

Parity pinned: every function here is checked against the pages' worked
example, closed forms, brute-force convolution and invariants in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libssm_oracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into a shared library (plain gcc, IEEE math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_scan.argtypes = [i64, i64, i64, i64] + [dp] * 11 + [i64, i64]
            lib.oracle_scan.restype = None
            lib.oracle_step.argtypes = [i64, i64, i64] + [dp] * 10 + [i64, i64]
            lib.oracle_step.restype = None
            lib.oracle_scan_bwd.argtypes = [i64, i64, i64, i64] + [dp] * 21
            lib.oracle_scan_bwd.restype = None
            lib.oracle_conv1d.argtypes = [i64, i64, i64, i64] + [dp] * 6 + [i64, i64]
            lib.oracle_conv1d.restype = None
            lib.oracle_conv1d_step.argtypes = [i64, i64, i64] + [dp] * 5 + [i64, i64]
            lib.oracle_conv1d_step.restype = None
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _row_ranges(rows: int, threads: int):
    threads = max(1, min(threads, rows))
    step = (rows + threads - 1) // threads
    return [(s, min(rows, s + step)) for s in range(0, rows, step)]


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def scan(u, delta, A, B, C, D=None, z=None, bias=None, h0=None, threads: int | None = None):
    """Parallel-mode selective scan, sequential loop in float64.

    u, delta, z: [batch, d_inner, L]; B, C: [batch, L, N]; A: [d_inner, N];
    D, bias: [d_inner]; h0: [batch, d_inner, N] or None (zero state).
    Returns (out [batch, d_inner, L], hT [batch, d_inner, N]) as float64 arrays.
    Rows (batch, channel) are independent, so they are split between threads;
    each row is one plain sequential loop.
    """
    u, delta, A, B, C = (_f64(x) for x in (u, delta, A, B, C))
    D, z, bias, h0 = (_f64(x) for x in (D, z, bias, h0))
    batch, d_inner, L = u.shape
    N = A.shape[1]
    assert delta.shape == u.shape and A.shape == (d_inner, N)
    assert B.shape == (batch, L, N) and C.shape == (batch, L, N)
    assert z is None or z.shape == u.shape
    assert D is None or D.shape == (d_inner,)
    assert bias is None or bias.shape == (d_inner,)
    assert h0 is None or h0.shape == (batch, d_inner, N)
    out = np.empty((batch, d_inner, L), np.float64)
    hT = np.empty((batch, d_inner, N), np.float64)
    lib = _load()
    args = [batch, d_inner, N, L] + [_ptr(x) for x in (u, delta, A, B, C, D, z, bias, h0, out, hT)]
    ranges = _row_ranges(batch * d_inner, threads or default_threads())
    if len(ranges) == 1:
        lib.oracle_scan(*args, *ranges[0])
    else:
        with ThreadPoolExecutor(len(ranges)) as ex:
            list(ex.map(lambda rg: lib.oracle_scan(*args, *rg), ranges))
    return out, hT


def scan_bwd(u, delta, A, B, C, dout, D=None, z=None, bias=None, h0=None, dhT=None):
    """Gradients of sum(dout * out) + sum(dhT * h_L) of ``scan`` with respect to
    its inputs (plain reverse-mode loop, float64, one thread).

    Returns a dict with du, ddelta, dz [batch, d_inner, L]; dA [d_inner, N];
    dB, dC [batch, L, N]; dD, dbias [d_inner]; dh0 [batch, d_inner, N]
    (entries for absent optional inputs are None).
    """
    u, delta, A, B, C, dout = (_f64(x) for x in (u, delta, A, B, C, dout))
    D, z, bias, h0, dhT = (_f64(x) for x in (D, z, bias, h0, dhT))
    batch, d_inner, L = u.shape
    N = A.shape[1]
    assert dout.shape == u.shape and delta.shape == u.shape and A.shape == (d_inner, N)
    assert B.shape == (batch, L, N) and C.shape == (batch, L, N)
    out = dict(du=np.empty_like(u), ddelta=np.empty_like(u), dA=np.zeros((d_inner, N)),
               dB=np.zeros((batch, L, N)), dC=np.zeros((batch, L, N)),
               dD=np.zeros(d_inner) if D is not None else None,
               dz=np.empty_like(u) if z is not None else None,
               dbias=np.zeros(d_inner), dh0=np.empty((batch, d_inner, N)))
    work = np.empty((L + 1) * N)
    lib = _load()
    lib.oracle_scan_bwd(batch, d_inner, N, L, *(_ptr(v) for v in (u, delta, A, B, C, D, z, bias, h0, dout, dhT)),
                        *(_ptr(out[k]) for k in ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "dbias", "dh0")),
                        _ptr(work))
    return out


def step(state, x, delta, A, B, C, D=None, z=None, bias=None, threads: int | None = None):
    """Recurrent-mode single token for every (batch, channel) row.

    state: [batch, d_inner, N] (not modified; the new state is returned);
    x, delta, z: [batch, d_inner]; B, C: [batch, N]; A: [d_inner, N].
    Returns (out [batch, d_inner], new_state [batch, d_inner, N]).
    """
    st = _f64(state).copy()
    x, delta, A, B, C = (_f64(v) for v in (x, delta, A, B, C))
    D, z, bias = (_f64(v) for v in (D, z, bias))
    batch, d_inner, N = st.shape
    assert x.shape == (batch, d_inner) and delta.shape == (batch, d_inner)
    assert A.shape == (d_inner, N) and B.shape == (batch, N) and C.shape == (batch, N)
    out = np.empty((batch, d_inner), np.float64)
    lib = _load()
    args = [batch, d_inner, N] + [_ptr(v) for v in (st, x, delta, A, B, C, D, z, bias, out)]
    ranges = _row_ranges(batch * d_inner, threads or 1)
    if len(ranges) == 1:
        lib.oracle_step(*args, *ranges[0])
    else:
        with ThreadPoolExecutor(len(ranges)) as ex:
            list(ex.map(lambda rg: lib.oracle_step(*args, *rg), ranges))
    return out, st


def conv1d(x, w, bias=None, state0=None, threads: int | None = None):
    """Causal depthwise Conv1D + SiLU over whole sequences.

    x: [batch, d_inner, L]; w: [d_inner, W]; bias: [d_inner] or None;
    state0: [batch, d_inner, W-1] (the W-1 inputs before x, oldest first) or None (zeros).
    Returns (out [batch, d_inner, L], stateT [batch, d_inner, W-1]) as float64 arrays.
    """
    x, w, bias, state0 = (_f64(v) for v in (x, w, bias, state0))
    batch, d_inner, L = x.shape
    W = w.shape[1]
    assert w.shape == (d_inner, W) and 1 <= W <= 64
    assert bias is None or bias.shape == (d_inner,)
    assert state0 is None or state0.shape == (batch, d_inner, W - 1)
    out = np.empty((batch, d_inner, L), np.float64)
    stateT = np.empty((batch, d_inner, W - 1), np.float64)
    lib = _load()
    args = [batch, d_inner, L, W] + [_ptr(v) for v in (x, w, bias, state0, out, stateT)]
    ranges = _row_ranges(batch * d_inner, threads or default_threads())
    if len(ranges) == 1:
        lib.oracle_conv1d(*args, *ranges[0])
    else:
        with ThreadPoolExecutor(len(ranges)) as ex:
            list(ex.map(lambda rg: lib.oracle_conv1d(*args, *rg), ranges))
    return out, stateT


def conv1d_step(state, x, w, bias=None):
    """One decode token of the causal Conv1D + SiLU.

    state: [batch, d_inner, W-1] (not modified; the new state is returned);
    x: [batch, d_inner]; w: [d_inner, W].  Returns (out [batch, d_inner], new_state).
    """
    st = _f64(state).copy()
    x, w, bias = (_f64(v) for v in (x, w, bias))
    batch, d_inner = x.shape
    W = w.shape[1]
    assert st.shape == (batch, d_inner, W - 1) and w.shape == (d_inner, W)
    out = np.empty((batch, d_inner), np.float64)
    lib = _load()
    lib.oracle_conv1d_step(batch, d_inner, W, *(_ptr(v) for v in (st, x, w, bias, out)), 0, batch * d_inner)
    return out, st


def ssd_scan(x, dt, A, B, C, D=None, z=None, dt_bias=None, h0=None, threads: int | None = None):
    """The Mamba-2 layer scan (state space duality form of the selective SSM):
    the state matrix of each head is a scalar times the identity, so each head's
    headdim channels share their step size, their A and the B, C of their group.

    x, z: [batch, L, H, P]; dt (Δraw): [batch, L, H]; A, D, dt_bias: [H];
    B, C: [batch, L, G, N], head h reading group h // (H // G);
    h0: [batch, H, P, N] or None.  Returns (out [batch, L, H, P], hT [batch, H, P, N]).

    Channel (h, p) is the selective scan above on one row with A[c, n] = A[h] for
    every n and Δraw = dt[..., h], so the result is ``scan`` applied group by group
    ("Mambaとは？Transformer以外の系列モデル", section Mamba-2とTransformerとの関係性;
    "State Space Models（SSM）とMamba" §4.6 Mamba-2: the SSM with this structure is
    the one that coincides with masked linear attention).  Discretisation is the
    zero-order hold of the scan, as the pages define no other.
    """
    x, dt, A, B, C = (_f64(v) for v in (x, dt, A, B, C))
    D, z, dt_bias, h0 = (_f64(v) for v in (D, z, dt_bias, h0))
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert H % G == 0 and dt.shape == (batch, L, H) and A.shape == (H,)
    assert B.shape == (batch, L, G, N) and C.shape == (batch, L, G, N)
    assert z is None or z.shape == x.shape
    assert h0 is None or h0.shape == (batch, H, P, N)
    hpg = H // G

    def rows(t):  # [batch, L, hpg, P] -> [batch, hpg * P, L]
        return np.ascontiguousarray(t.transpose(0, 2, 3, 1).reshape(batch, hpg * P, L))

    out = np.empty((batch, L, H, P))
    hT = np.empty((batch, H, P, N))
    for g in range(G):
        hs = slice(g * hpg, (g + 1) * hpg)
        u = rows(x[:, :, hs, :])
        delta = rows(np.broadcast_to(dt[:, :, hs, None], (batch, L, hpg, P)))
        Af = np.repeat(np.repeat(A[hs], P)[:, None], N, axis=1)
        o, hg = scan(u, delta, Af, B[:, :, g, :], C[:, :, g, :],
                     D=None if D is None else np.repeat(D[hs], P),
                     z=None if z is None else rows(z[:, :, hs, :]),
                     bias=None if dt_bias is None else np.repeat(dt_bias[hs], P),
                     h0=None if h0 is None else np.ascontiguousarray(h0[:, hs].reshape(batch, hpg * P, N)),
                     threads=threads)
        out[:, :, hs, :] = o.reshape(batch, hpg, P, L).transpose(0, 3, 1, 2)
        hT[:, hs] = hg.reshape(batch, hpg, P, N)
    return out, hT

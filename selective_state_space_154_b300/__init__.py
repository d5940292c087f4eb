"""B300-native selective state-space scan (S6): Python binding of the C ABI.

The compute path is entirely in ``_lib/libssm_b300.so`` (CUDA, sm_103a); this
module only marshals torch tensors into pointers, sizes and the current CUDA
stream.  The functions named like the C entry points take the same arguments
(see ``include/ssm_scan.h``) and raise ``SsmError`` on a non-OK status.
``scan_fwd`` / ``step`` are conveniences that allocate outputs with torch.

There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "SsmError", "ssm_scan_workspace_bytes", "ssm_scan_fwd", "ssm_step", "ssm_scan_check",
    "ssm_status_string", "scan_fwd", "step", "library_path", "load_library", "ssm_scan_fwd_noalloc",
    "SSM_NOALLOC_SCRATCH_BYTES", "ssm_step_check", "ssm_scan_fwd_from_state",
    "ssm_conv1d_fwd", "ssm_conv1d_step", "conv1d", "conv1d_step",
    "ssm_scan_fwd_host", "ssm_scan_fwd_host_staging_bytes", "reload_test_hooks",
    "ssm_scan_bwd_workspace_bytes", "ssm_scan_bwd", "scan_bwd",
    "ssm_scan_bwd_deterministic_workspace_bytes",
    "ssd_scan_workspace_bytes", "ssd_scan_fwd", "ssd_scan", "ssd_step",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libssm_b300.so")

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_ALIGNMENT, SSM_ERR_WORKSPACE, \
    SSM_ERR_CUDA, SSM_ERR_TIMEOUT = range(7)
SSM_DTYPE_F32, SSM_DTYPE_BF16 = 0, 1
def __getattr__(name):
    # SSM_NOALLOC_SCRATCH_BYTES: the size of the library's static scratch, read from the library
    if name == "SSM_NOALLOC_SCRATCH_BYTES":
        return int(load_library().ssm_noalloc_scratch_bytes())
    raise AttributeError(name)
_DTYPES = {torch.float32: SSM_DTYPE_F32, torch.bfloat16: SSM_DTYPE_BF16}


class SsmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {ssm_status_string(status)}"
        if status == SSM_ERR_CUDA:
            code = int(load_library().ssm_last_cuda_error())
            msg += (f" (driver error {code - 10000})" if code >= 10000 else f" (CUDA error {code})")
        super().__init__(msg)


class ssm_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("d_inner", ctypes.c_int64), ("d_state", ctypes.c_int64),
                ("seqlen", ctypes.c_int64), ("act", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class ssd_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("ngroups", ctypes.c_int64), ("d_state", ctypes.c_int64),
                ("act", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with `python -m selective_state_space_154_b300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            dp = ctypes.POINTER(ssm_dims)
            lib.ssm_scan_workspace_bytes.argtypes = [dp]
            lib.ssm_scan_workspace_bytes.restype = sz
            lib.ssm_scan_fwd.argtypes = [vp] * 10 + [dp, vp, sz, vp]
            lib.ssm_scan_fwd.restype = i32
            lib.ssm_scan_fwd_from_state.argtypes = [vp] * 11 + [dp, vp, sz, vp]
            lib.ssm_scan_fwd_from_state.restype = i32
            lib.ssm_step.argtypes = [vp] * 10 + [dp, vp]
            lib.ssm_step.restype = i32
            lib.ssm_scan_check.argtypes = [vp, sz]
            lib.ssm_scan_check.restype = i32
            lib.ssm_step_check.argtypes = [vp]
            lib.ssm_step_check.restype = i32
            lib.ssm_scan_fwd_noalloc.argtypes = [vp] * 10 + [dp, vp]
            lib.ssm_scan_fwd_noalloc.restype = i32
            lib.ssm_scan_bwd_workspace_bytes.argtypes = [dp]
            lib.ssm_scan_bwd_workspace_bytes.restype = sz
            lib.ssm_scan_bwd.argtypes = [vp] * 17 + [dp, vp, sz, vp]
            lib.ssm_scan_bwd.restype = i32
            lib.ssm_scan_bwd_deterministic_workspace_bytes.argtypes = [dp]
            lib.ssm_scan_bwd_deterministic_workspace_bytes.restype = sz
            lib.ssm_scan_bwd_deterministic.argtypes = [vp] * 17 + [dp, vp, sz, vp]
            lib.ssm_scan_bwd_deterministic.restype = i32
            lib.ssm_conv1d_fwd.argtypes = [vp] * 6 + [dp, i32, vp]
            lib.ssm_conv1d_fwd.restype = i32
            lib.ssm_conv1d_step.argtypes = [vp] * 5 + [dp, i32, vp]
            lib.ssm_conv1d_step.restype = i32
            sdp = ctypes.POINTER(ssd_dims)
            lib.ssd_scan_workspace_bytes.argtypes = [sdp]
            lib.ssd_scan_workspace_bytes.restype = sz
            lib.ssd_scan_fwd.argtypes = [vp] * 11 + [sdp, vp, sz, vp]
            lib.ssd_scan_fwd.restype = i32
            lib.ssd_step.argtypes = [vp] * 10 + [sdp, vp]
            lib.ssd_step.restype = i32
            lib.ssm_status_string.argtypes = [i32]
            lib.ssm_status_string.restype = ctypes.c_char_p
            lib.ssm_test_hooks_reload.argtypes = []
            lib.ssm_test_hooks_reload.restype = None
            lib.ssm_scan_fwd_host_staging_bytes.argtypes = [dp, ctypes.c_int64]
            lib.ssm_scan_fwd_host_staging_bytes.restype = sz
            lib.ssm_scan_fwd_host.argtypes = [vp] * 11 + [dp, ctypes.c_int64, vp, sz, vp, vp, vp]
            lib.ssm_scan_fwd_host.restype = i32
            lib.ssm_last_cuda_error.argtypes = []
            lib.ssm_last_cuda_error.restype = i32
            lib.ssm_noalloc_scratch_bytes.argtypes = []
            lib.ssm_noalloc_scratch_bytes.restype = sz
            _lib = lib
    return _lib


def ssm_status_string(status: int) -> str:
    return load_library().ssm_status_string(int(status)).decode()


def reload_test_hooks() -> None:
    """Make the library read its SSM_* test-hook environment variables again (it reads
    them once otherwise)."""
    load_library().ssm_test_hooks_reload()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, shape, device, required=True):
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(batch, d_inner, d_state, seqlen, dtype):
    if dtype not in _DTYPES:
        raise TypeError(f"activation dtype must be float32 or bfloat16, got {dtype}")
    return ssm_dims(int(batch), int(d_inner), int(d_state), int(seqlen), _DTYPES[dtype], 0)


def ssm_scan_workspace_bytes(batch, d_inner, d_state, seqlen, dtype=torch.bfloat16) -> int:
    d = _dims(batch, d_inner, d_state, seqlen, dtype)
    return int(load_library().ssm_scan_workspace_bytes(ctypes.byref(d)))


def ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, out, final_state, workspace=None, stream=None,
                 initial_state=None):
    """Parallel-mode scan into caller-provided ``out`` (and ``final_state``),
    from h = 0, or from ``initial_state`` (ssm_scan_fwd_from_state) when given."""
    lib = load_library()
    if not isinstance(u, torch.Tensor) or u.dim() != 3:
        raise ValueError("u must be a [batch, d_inner, seqlen] tensor")
    batch, d_inner, L = u.shape
    if not isinstance(A, torch.Tensor) or A.dim() != 2:
        raise ValueError("A must be a [d_inner, d_state] tensor")
    N = A.shape[1]
    act, dev = u.dtype, u.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    _check(u, "u", act, (batch, d_inner, L), dev)
    _check(delta, "delta", act, (batch, d_inner, L), dev)
    _check(A, "A", torch.float32, (d_inner, N), dev)
    _check(B, "B", act, (batch, L, N), dev)
    _check(C, "C", act, (batch, L, N), dev)
    _check(D, "D", torch.float32, (d_inner,), dev, required=False)
    _check(z, "z", act, (batch, d_inner, L), dev, required=False)
    _check(delta_bias, "delta_bias", torch.float32, (d_inner,), dev, required=False)
    _check(out, "out", act, (batch, d_inner, L), dev)
    _check(final_state, "final_state", torch.float32, (batch, d_inner, N), dev, required=False)
    _check(initial_state, "initial_state", torch.float32, (batch, d_inner, N), dev, required=False)
    dims = _dims(batch, d_inner, N, L, act)
    with torch.cuda.device(dev):
        need = int(lib.ssm_scan_workspace_bytes(ctypes.byref(dims)))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        tail = (ctypes.byref(dims), _ptr(workspace), ws_bytes, _stream_handle(stream, dev))
        if initial_state is None:
            st = lib.ssm_scan_fwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                  _ptr(delta_bias), _ptr(out), _ptr(final_state), *tail)
        else:
            st = lib.ssm_scan_fwd_from_state(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                             _ptr(delta_bias), _ptr(initial_state), _ptr(out), _ptr(final_state),
                                             *tail)
    if st != SSM_OK:
        raise SsmError(st, "ssm_scan_fwd" if initial_state is None else "ssm_scan_fwd_from_state")
    return workspace


def ssm_scan_fwd_host_staging_bytes(batch, d_inner, d_state, seqlen, piece_len, dtype=torch.bfloat16) -> int:
    d = _dims(batch, d_inner, d_state, seqlen, dtype)
    return int(load_library().ssm_scan_fwd_host_staging_bytes(ctypes.byref(d), int(piece_len)))


def ssm_scan_fwd_host(u, delta, A, B, C, D, z, delta_bias, out, final_state=None, initial_state=None,
                      piece_len=1 << 16, staging=None, stream=None, h2d_stream=None, d2h_stream=None):
    """ssm_scan_fwd over host tensors (u, delta, z, B, C, out; page-locked for overlap),
    A, D, delta_bias, initial_state and final_state on the device: the C call pipelines
    the copies with the scan in pieces of ``piece_len`` tokens.  Allocates the device
    staging memory when it is not given.  Returns the staging tensor."""
    lib = load_library()
    if not isinstance(u, torch.Tensor) or u.dim() != 3:
        raise ValueError("u must be a [batch, d_inner, seqlen] tensor")
    batch, d_inner, L = u.shape
    if not isinstance(A, torch.Tensor) or A.dim() != 2:
        raise ValueError("A must be a [d_inner, d_state] tensor")
    N = A.shape[1]
    act, dev, host = u.dtype, A.device, torch.device("cpu")
    if dev.type != "cuda":
        raise ValueError("A must be on a CUDA device")
    _check(u, "u", act, (batch, d_inner, L), host)
    _check(delta, "delta", act, (batch, d_inner, L), host)
    _check(B, "B", act, (batch, L, N), host)
    _check(C, "C", act, (batch, L, N), host)
    _check(z, "z", act, (batch, d_inner, L), host, required=False)
    _check(out, "out", act, (batch, d_inner, L), host)
    _check(A, "A", torch.float32, (d_inner, N), dev)
    _check(D, "D", torch.float32, (d_inner,), dev, required=False)
    _check(delta_bias, "delta_bias", torch.float32, (d_inner,), dev, required=False)
    _check(final_state, "final_state", torch.float32, (batch, d_inner, N), dev, required=False)
    _check(initial_state, "initial_state", torch.float32, (batch, d_inner, N), dev, required=False)
    dims = _dims(batch, d_inner, N, L, act)
    with torch.cuda.device(dev):
        need = int(lib.ssm_scan_fwd_host_staging_bytes(ctypes.byref(dims), int(piece_len)))
        if staging is None:
            staging = torch.empty(need, dtype=torch.uint8, device=dev)
        sbytes = staging.numel() * staging.element_size()
        main = _stream_handle(stream, dev)
        h2d = main if h2d_stream is None else ctypes.c_void_p(h2d_stream.cuda_stream)
        d2h = main if d2h_stream is None else ctypes.c_void_p(d2h_stream.cuda_stream)
        st = lib.ssm_scan_fwd_host(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                   _ptr(delta_bias), _ptr(initial_state), _ptr(out), _ptr(final_state),
                                   ctypes.byref(dims), int(piece_len), _ptr(staging), sbytes, main, h2d, d2h)
    if st != SSM_OK:
        raise SsmError(st, "ssm_scan_fwd_host")
    return staging


def ssm_scan_fwd_from_state(u, delta, A, B, C, D, z, delta_bias, initial_state, out, final_state,
                            workspace=None, stream=None):
    """The scan starting from ``initial_state`` (same arguments as the C call)."""
    if initial_state is None:
        raise ValueError("initial_state is required")
    return ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, out, final_state, workspace=workspace,
                        stream=stream, initial_state=initial_state)


def ssm_scan_fwd_noalloc(u, delta, A, B, C, D, z, delta_bias, out, final_state, stream=None):
    """ssm_scan_fwd using the library's static device scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/ssm_scan.h)."""
    lib = load_library()
    batch, d_inner, L = u.shape
    N = A.shape[1]
    act, dev = u.dtype, u.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    _check(u, "u", act, (batch, d_inner, L), dev)
    _check(delta, "delta", act, (batch, d_inner, L), dev)
    _check(A, "A", torch.float32, (d_inner, N), dev)
    _check(B, "B", act, (batch, L, N), dev)
    _check(C, "C", act, (batch, L, N), dev)
    _check(D, "D", torch.float32, (d_inner,), dev, required=False)
    _check(z, "z", act, (batch, d_inner, L), dev, required=False)
    _check(delta_bias, "delta_bias", torch.float32, (d_inner,), dev, required=False)
    _check(out, "out", act, (batch, d_inner, L), dev)
    _check(final_state, "final_state", torch.float32, (batch, d_inner, N), dev, required=False)
    dims = _dims(batch, d_inner, N, L, act)
    with torch.cuda.device(dev):
        st = lib.ssm_scan_fwd_noalloc(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                      _ptr(delta_bias), _ptr(out), _ptr(final_state), ctypes.byref(dims),
                                      _stream_handle(stream, dev))
    if st != SSM_OK:
        raise SsmError(st, "ssm_scan_fwd_noalloc")


def ssm_step(state, x, delta, A, B, C, D, z, delta_bias, out, stream=None):
    """Recurrent-mode single token; ``state`` is updated in place."""
    lib = load_library()
    if not isinstance(state, torch.Tensor) or state.dim() != 3:
        raise ValueError("state must be a [batch, d_inner, d_state] tensor")
    batch, d_inner, N = state.shape
    act, dev = x.dtype, state.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    _check(state, "state", torch.float32, (batch, d_inner, N), dev)
    _check(x, "x", act, (batch, d_inner), dev)
    _check(delta, "delta", act, (batch, d_inner), dev)
    _check(A, "A", torch.float32, (d_inner, N), dev)
    _check(B, "B", act, (batch, N), dev)
    _check(C, "C", act, (batch, N), dev)
    _check(D, "D", torch.float32, (d_inner,), dev, required=False)
    _check(z, "z", act, (batch, d_inner), dev, required=False)
    _check(delta_bias, "delta_bias", torch.float32, (d_inner,), dev, required=False)
    _check(out, "out", act, (batch, d_inner), dev)
    dims = _dims(batch, d_inner, N, 1, act)
    with torch.cuda.device(dev):
        st = lib.ssm_step(_ptr(state), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                          _ptr(delta_bias), _ptr(out), ctypes.byref(dims), _stream_handle(stream, dev))
    if st != SSM_OK:
        raise SsmError(st, "ssm_step")


def ssm_scan_bwd_workspace_bytes(batch, d_inner, d_state, seqlen, dtype=torch.bfloat16) -> int:
    d = _dims(batch, d_inner, d_state, seqlen, dtype)
    return int(load_library().ssm_scan_bwd_workspace_bytes(ctypes.byref(d)))


def ssm_scan_bwd_deterministic_workspace_bytes(batch, d_inner, d_state, seqlen, dtype=torch.bfloat16) -> int:
    d = _dims(batch, d_inner, d_state, seqlen, dtype)
    return int(load_library().ssm_scan_bwd_deterministic_workspace_bytes(ctypes.byref(d)))


def ssm_scan_bwd(u, delta, A, B, C, D, z, delta_bias, dout, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias,
                 workspace=None, stream=None, deterministic=False):
    """Backward of the scan into caller-provided gradient tensors (see include/ssm_scan.h);
    ``deterministic`` selects ssm_scan_bwd_deterministic (bitwise reproducible sums)."""
    lib = load_library()
    batch, d_inner, L = u.shape
    N = A.shape[1]
    act, dev = u.dtype, u.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    for name, t in (("u", u), ("delta", delta), ("dout", dout), ("du", du), ("ddelta", ddelta)):
        _check(t, name, act, (batch, d_inner, L), dev)
    _check(z, "z", act, (batch, d_inner, L), dev, required=False)
    _check(dz, "dz", act, (batch, d_inner, L), dev, required=z is not None)
    _check(A, "A", torch.float32, (d_inner, N), dev)
    _check(dA, "dA", torch.float32, (d_inner, N), dev)
    for name, t in (("B", B), ("C", C)):
        _check(t, name, act, (batch, L, N), dev)
    for name, t in (("dB", dB), ("dC", dC)):
        _check(t, name, torch.float32, (batch, L, N), dev)
    _check(D, "D", torch.float32, (d_inner,), dev, required=False)
    _check(dD, "dD", torch.float32, (d_inner,), dev, required=D is not None)
    _check(delta_bias, "delta_bias", torch.float32, (d_inner,), dev, required=False)
    _check(ddelta_bias, "ddelta_bias", torch.float32, (d_inner,), dev, required=False)
    dims = _dims(batch, d_inner, N, L, act)
    with torch.cuda.device(dev):
        size_fn = lib.ssm_scan_bwd_deterministic_workspace_bytes if deterministic else lib.ssm_scan_bwd_workspace_bytes
        need = int(size_fn(ctypes.byref(dims)))
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        ws_bytes = workspace.numel() * workspace.element_size()
        fn = lib.ssm_scan_bwd_deterministic if deterministic else lib.ssm_scan_bwd
        st = fn(*(_ptr(t) for t in (u, delta, A, B, C, D, z, delta_bias, dout, du, ddelta, dA, dB, dC, dD, dz,
                                    ddelta_bias)),
                ctypes.byref(dims), _ptr(workspace), ws_bytes, _stream_handle(stream, dev))
    if st != SSM_OK:
        raise SsmError(st, "ssm_scan_bwd_deterministic" if deterministic else "ssm_scan_bwd")
    return workspace


def scan_bwd(u, delta, A, B, C, dout, D=None, z=None, delta_bias=None, stream=None, deterministic=False):
    """Allocate the gradients and run ``ssm_scan_bwd``; returns a dict like the oracle's."""
    g = dict(du=torch.empty_like(u), ddelta=torch.empty_like(u),
             dA=torch.empty(A.shape, dtype=torch.float32, device=u.device),
             dB=torch.empty(B.shape, dtype=torch.float32, device=u.device),
             dC=torch.empty(C.shape, dtype=torch.float32, device=u.device),
             dD=torch.empty_like(D) if D is not None else None,
             dz=torch.empty_like(u) if z is not None else None,
             dbias=torch.empty((u.shape[1],), dtype=torch.float32, device=u.device))
    ssm_scan_bwd(u, delta, A, B, C, D, z, delta_bias, dout, g["du"], g["ddelta"], g["dA"], g["dB"], g["dC"], g["dD"],
                 g["dz"], g["dbias"], stream=stream, deterministic=deterministic)
    return g


def _conv_dims(x, batch, d_inner, seqlen):
    return _dims(batch, d_inner, 1, seqlen, x.dtype)


def ssm_conv1d_fwd(x, weight, bias, initial_conv_state, out, final_conv_state, stream=None):
    """Causal depthwise Conv1D + SiLU over [batch, d_inner, L] (see include/ssm_scan.h)."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 3:
        raise ValueError("x must be a [batch, d_inner, seqlen] tensor")
    if not isinstance(weight, torch.Tensor) or weight.dim() != 2:
        raise ValueError("weight must be a [d_inner, width] tensor")
    batch, d_inner, L = x.shape
    width = weight.shape[1]
    act, dev = x.dtype, x.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    _check(x, "x", act, (batch, d_inner, L), dev)
    _check(weight, "weight", torch.float32, (d_inner, width), dev)
    _check(bias, "bias", torch.float32, (d_inner,), dev, required=False)
    _check(out, "out", act, (batch, d_inner, L), dev)
    for name, t in (("initial_conv_state", initial_conv_state), ("final_conv_state", final_conv_state)):
        if t is not None and width > 1:
            _check(t, name, act, (batch, d_inner, width - 1), dev)
    dims = _conv_dims(x, batch, d_inner, L)
    with torch.cuda.device(dev):
        st = lib.ssm_conv1d_fwd(_ptr(x), _ptr(weight), _ptr(bias), _ptr(initial_conv_state), _ptr(out),
                                _ptr(final_conv_state), ctypes.byref(dims), int(width), _stream_handle(stream, dev))
    if st != SSM_OK:
        raise SsmError(st, "ssm_conv1d_fwd")


def ssm_conv1d_step(conv_state, x, weight, bias, out, stream=None):
    """One decode token of the causal Conv1D + SiLU; ``conv_state`` is updated in place."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a [batch, d_inner] tensor")
    batch, d_inner = x.shape
    width = weight.shape[1]
    act, dev = x.dtype, x.device
    _check(x, "x", act, (batch, d_inner), dev)
    _check(weight, "weight", torch.float32, (d_inner, width), dev)
    _check(bias, "bias", torch.float32, (d_inner,), dev, required=False)
    _check(out, "out", act, (batch, d_inner), dev)
    if width > 1:
        _check(conv_state, "conv_state", act, (batch, d_inner, width - 1), dev)
    dims = _conv_dims(x, batch, d_inner, 1)
    with torch.cuda.device(dev):
        st = lib.ssm_conv1d_step(_ptr(conv_state), _ptr(x), _ptr(weight), _ptr(bias), _ptr(out),
                                 ctypes.byref(dims), int(width), _stream_handle(stream, dev))
    if st != SSM_OK:
        raise SsmError(st, "ssm_conv1d_step")


def conv1d(x, weight, bias=None, initial_conv_state=None, return_final_state=False, stream=None):
    """Allocate ``out`` (and the final conv state) and run ``ssm_conv1d_fwd``."""
    out = torch.empty_like(x)
    fs = None
    if return_final_state:
        fs = torch.empty((x.shape[0], x.shape[1], max(weight.shape[1] - 1, 0)), dtype=x.dtype, device=x.device)
    ssm_conv1d_fwd(x, weight, bias, initial_conv_state, out, fs, stream=stream)
    return (out, fs) if return_final_state else out


def conv1d_step(conv_state, x, weight, bias=None, out=None, stream=None):
    """Run ``ssm_conv1d_step`` (state updated in place) and return the output."""
    if out is None:
        out = torch.empty_like(x)
    ssm_conv1d_step(conv_state, x, weight, bias, out, stream=stream)
    return out


def ssm_scan_check(workspace) -> int:
    """Status of the device error word after the scan's stream was synchronised."""
    if workspace is None:
        return SSM_OK
    return int(load_library().ssm_scan_check(_ptr(workspace), workspace.numel() * workspace.element_size()))


def ssm_step_check(stream=None, device=None) -> int:
    """Synchronise the stream, then read and clear the device's step error word."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(load_library().ssm_step_check(_stream_handle(stream, dev)))


def scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, return_final_state=False,
             workspace=None, stream=None, initial_state=None):
    """Allocate ``out`` (and ``final_state``) and run ``ssm_scan_fwd`` (from
    ``initial_state`` when given)."""
    out = torch.empty_like(u)
    fs = None
    if return_final_state:
        fs = torch.empty((u.shape[0], u.shape[1], A.shape[1]), dtype=torch.float32, device=u.device)
    ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, out, fs, workspace=workspace, stream=stream,
                 initial_state=initial_state)
    return (out, fs) if return_final_state else out


def step(state, x, delta, A, B, C, D=None, z=None, delta_bias=None, out=None, stream=None):
    """Run ``ssm_step`` (state updated in place) and return the output."""
    if out is None:
        out = torch.empty_like(x)
    ssm_step(state, x, delta, A, B, C, D, z, delta_bias, out, stream=stream)
    return out


def _ssd_dims(batch, seqlen, nheads, headdim, ngroups, d_state, dtype):
    if dtype not in _DTYPES:
        raise TypeError(f"activation dtype must be float32 or bfloat16, got {dtype}")
    return ssd_dims(int(batch), int(seqlen), int(nheads), int(headdim), int(ngroups), int(d_state), _DTYPES[dtype], 0)


def ssd_scan_workspace_bytes(batch, seqlen, nheads, headdim, ngroups, d_state, dtype=torch.bfloat16) -> int:
    d = _ssd_dims(batch, seqlen, nheads, headdim, ngroups, d_state, dtype)
    return int(load_library().ssd_scan_workspace_bytes(ctypes.byref(d)))


def ssd_scan_fwd(x, dt, A, B, C, D, z, dt_bias, initial_state, out, final_state, workspace=None, stream=None):
    """Mamba-2 (SSD) layer scan into caller-provided ``out`` (and ``final_state``);
    see include/ssm_scan.h.  x, z, out: [batch, L, H, P]; dt: [batch, L, H];
    B, C: [batch, L, G, N]; A, D, dt_bias: [H]; states [batch, H, P, N] (fp32)."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 4:
        raise ValueError("x must be a [batch, seqlen, nheads, headdim] tensor")
    if not isinstance(B, torch.Tensor) or B.dim() != 4:
        raise ValueError("B must be a [batch, seqlen, ngroups, d_state] tensor")
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    act, dev = x.dtype, x.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    _check(x, "x", act, (batch, L, H, P), dev)
    _check(dt, "dt", act, (batch, L, H), dev)
    _check(A, "A", torch.float32, (H,), dev)
    _check(B, "B", act, (batch, L, G, N), dev)
    _check(C, "C", act, (batch, L, G, N), dev)
    _check(D, "D", torch.float32, (H,), dev, required=False)
    _check(z, "z", act, (batch, L, H, P), dev, required=False)
    _check(dt_bias, "dt_bias", torch.float32, (H,), dev, required=False)
    _check(initial_state, "initial_state", torch.float32, (batch, H, P, N), dev, required=False)
    _check(out, "out", act, (batch, L, H, P), dev)
    _check(final_state, "final_state", torch.float32, (batch, H, P, N), dev, required=False)
    dims = _ssd_dims(batch, L, H, P, G, N, act)
    with torch.cuda.device(dev):
        need = int(lib.ssd_scan_workspace_bytes(ctypes.byref(dims)))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = lib.ssd_scan_fwd(*(_ptr(t) for t in (x, dt, A, B, C, D, z, dt_bias, initial_state, out, final_state)),
                              ctypes.byref(dims), _ptr(workspace), ws_bytes, _stream_handle(stream, dev))
    if st != SSM_OK:
        raise SsmError(st, "ssd_scan_fwd")
    return workspace


def ssd_scan(x, dt, A, B, C, D=None, z=None, dt_bias=None, initial_state=None, return_final_state=False,
             workspace=None, stream=None):
    """Allocate ``out`` (and the final state) and run ``ssd_scan_fwd``."""
    out = torch.empty_like(x)
    fs = None
    if return_final_state:
        fs = torch.empty((x.shape[0], x.shape[2], x.shape[3], B.shape[3]), dtype=torch.float32, device=x.device)
    ssd_scan_fwd(x, dt, A, B, C, D, z, dt_bias, initial_state, out, fs, workspace=workspace, stream=stream)
    return (out, fs) if return_final_state else out


def ssd_step(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, out=None, stream=None):
    """One decode token of the Mamba-2 layer (``state`` [batch, H, P, N] fp32 updated in
    place); x, z: [batch, H, P]; dt: [batch, H]; B, C: [batch, G, N].  Returns ``out``."""
    lib = load_library()
    if not isinstance(state, torch.Tensor) or state.dim() != 4:
        raise ValueError("state must be a [batch, nheads, headdim, d_state] tensor")
    if not isinstance(B, torch.Tensor) or B.dim() != 3:
        raise ValueError("B must be a [batch, ngroups, d_state] tensor")
    batch, H, P, N = state.shape
    G = B.shape[1]
    act, dev = x.dtype, state.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    if out is None:
        out = torch.empty_like(x)
    _check(state, "state", torch.float32, (batch, H, P, N), dev)
    _check(x, "x", act, (batch, H, P), dev)
    _check(dt, "dt", act, (batch, H), dev)
    _check(A, "A", torch.float32, (H,), dev)
    _check(B, "B", act, (batch, G, N), dev)
    _check(C, "C", act, (batch, G, N), dev)
    _check(D, "D", torch.float32, (H,), dev, required=False)
    _check(z, "z", act, (batch, H, P), dev, required=False)
    _check(dt_bias, "dt_bias", torch.float32, (H,), dev, required=False)
    _check(out, "out", act, (batch, H, P), dev)
    dims = _ssd_dims(batch, 1, H, P, G, N, act)
    with torch.cuda.device(dev):
        st = lib.ssd_step(*(_ptr(t) for t in (state, x, dt, A, B, C, D, z, dt_bias, out)), ctypes.byref(dims),
                          _stream_handle(stream, dev))
    if st != SSM_OK:
        raise SsmError(st, "ssd_step")
    return out

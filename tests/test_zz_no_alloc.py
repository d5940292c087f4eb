"""ssm_scan_fwd_noalloc: the scan for callers that cannot allocate device memory.

It must give what ssm_scan_fwd gives with a caller-provided workspace, also on
the second of two calls in a row (the static scratch keeps the previous call's
contents and each call must reset what has to start at zero), and refuse
problems whose scratch would not fit in the static array.
Runs last (file name) so that a stop at the first failure has run every other test.
"""
import ctypes

import pytest
import torch

import selective_state_space_154_b300 as ssm
import workloads as W
from parity import TOL, rel_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, inp, out, fs):
    b, d, L = inp["u"].shape
    dims = ssm.ssm_dims(b, d, inp["A"].shape[1], L, ssm.SSM_DTYPE_BF16 if inp["u"].dtype == torch.bfloat16
                        else ssm.SSM_DTYPE_F32, 0)
    return lib.ssm_scan_fwd_noalloc(_ptr(inp["u"]), _ptr(inp["delta"]), _ptr(inp["A"]), _ptr(inp["B"]),
                                    _ptr(inp["C"]), _ptr(inp.get("D")), _ptr(inp.get("z")), _ptr(inp.get("bias")),
                                    _ptr(out), _ptr(fs), ctypes.byref(dims),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("shape", [(1, 256, 16, 1 << 17), (2, 300, 16, 20000), (3, 40, 16, 700)],
                         ids=["chunked", "chunked_ragged", "no_scratch"])
def test_noalloc_matches_workspace_call_twice(shape):
    lib = ssm.load_library()
    b, d, N, L = shape
    inp = W.random_scan_inputs(b, d, N, L, dtype=torch.bfloat16, device=DEV, seed=sum(shape), a_kind="random")
    ref_out, ref_fs = ssm.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                   inp["bias"], return_final_state=True)
    torch.cuda.synchronize()
    tol = TOL[torch.bfloat16]
    for call in range(2):
        out = torch.full_like(inp["u"], float("nan"))
        fs = torch.full((b, d, N), float("nan"), device=DEV)
        assert _noalloc(lib, inp, out, fs) == ssm.SSM_OK
        torch.cuda.synchronize()
        assert rel_err(to_np(out), to_np(ref_out)) <= tol, f"call {call}"
        assert rel_err(to_np(fs), to_np(ref_fs)) <= tol, f"call {call}"


def test_noalloc_refuses_scratch_beyond_the_static_array(hooks):
    """A forced split into many chunks needs more scratch than the static array holds."""
    hooks.set("SSM_FORCE_CHUNKS", "4096")
    b, d, N, L = 1, 1024, 16, 1 << 17
    need = ssm.ssm_scan_workspace_bytes(b, d, N, L, torch.bfloat16)
    assert need > ssm.SSM_NOALLOC_SCRATCH_BYTES
    inp = W.random_scan_inputs(b, d, N, L, dtype=torch.bfloat16, device=DEV, seed=3)
    out = torch.zeros_like(inp["u"])
    assert _noalloc(ssm.load_library(), inp, out, None) == ssm.SSM_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0  # nothing was launched

"""ssm_scan_fwd_host: a sequence in host memory, copied and scanned in pieces.

The pieces continue from one another's state, so the result must equal one
ssm_scan_fwd of the whole sequence on the device (outputs to two bf16 ulps: a
piece boundary only re-associates the state's float32 sums; final state to 1e-5),
for ragged last pieces, with and without z, from an initial state, on three
separate streams or on one.
"""
import pytest
import torch

import selective_state_space_154_b300 as ssm
import workloads as W
from parity import rel_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _host(t):
    return None if t is None else t.to("cpu").pin_memory()


@pytest.mark.parametrize("piece", [3000, 4096, 10008], ids=["ragged_pieces", "aligned_pieces", "one_piece"])
@pytest.mark.parametrize("streams", ["three", "one"])
def test_host_pieces_equal_one_device_scan(piece, streams):
    b, d, N, L = 2, 300, 16, 10008
    inp = W.random_scan_inputs(b, d, N, L, dtype=torch.bfloat16, device=DEV, seed=piece, a_kind="random")
    ref, ref_fs = ssm.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                               inp["bias"], return_final_state=True)
    hu, hd, hz, hB, hC = (_host(inp[k]) for k in ("u", "delta", "z", "B", "C"))
    out = torch.full(hu.shape, float("nan"), dtype=hu.dtype).pin_memory()
    fs = torch.full((b, d, N), float("nan"), device=DEV)
    kw = {}
    if streams == "three":
        kw = dict(h2d_stream=torch.cuda.Stream(), d2h_stream=torch.cuda.Stream())
    ssm.ssm_scan_fwd_host(hu, hd, inp["A"], hB, hC, inp["D"], hz, inp["bias"], out, final_state=fs,
                          piece_len=piece, **kw)
    torch.cuda.current_stream().synchronize()
    assert rel_err(to_np(out), to_np(ref)) <= 2 * 2.0 ** -8
    assert rel_err(to_np(fs), to_np(ref_fs)) <= 1e-5


def test_host_from_initial_state_without_gate():
    b, d, N, L = 1, 130, 16, 5000
    inp = W.random_scan_inputs(b, d, N, L, dtype=torch.bfloat16, device=DEV, seed=7, a_kind="random", gate=False)
    h0 = torch.randn((b, d, N), generator=torch.Generator(device=DEV).manual_seed(8), device=DEV)
    ref, ref_fs = ssm.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], None, inp["bias"],
                               return_final_state=True, initial_state=h0)
    hu, hd, hB, hC = (_host(inp[k]) for k in ("u", "delta", "B", "C"))
    out = torch.empty(hu.shape, dtype=hu.dtype).pin_memory()
    fs = torch.empty((b, d, N), device=DEV)
    ssm.ssm_scan_fwd_host(hu, hd, inp["A"], hB, hC, inp["D"], None, inp["bias"], out, final_state=fs,
                          initial_state=h0, piece_len=1024, h2d_stream=torch.cuda.Stream(),
                          d2h_stream=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    assert rel_err(to_np(out), to_np(ref)) <= 2 * 2.0 ** -8
    assert rel_err(to_np(fs), to_np(ref_fs)) <= 1e-5

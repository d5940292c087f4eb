"""GPU parity of the streamed row kernel (bf16, d_state 16) against the CPU oracle.

The planner takes this kernel for bf16 activations with 16 states, 16-byte
aligned tensors and a length that is a multiple of 8; these tests force it
(SSM_FORCE_KERNEL=stream) and cover both CTA sizes (512 and 128 rows), rows and
tokens that do not fill a CTA or a 32-token stage, the carry between chunks, the exact branch for A = 0, the optional
inputs, the initial state, bitwise repeatability and the reported timeout.
Tolerance: 2e-2 (bf16 activations, fp32 state) against the oracle fed the same
rounded inputs, as for every scan kernel.
"""
import pytest
import torch

import oracle
import selective_state_space_154_b300 as ssm
import workloads as W
from parity import TOL, rel_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_BF16 = TOL[torch.bfloat16]


@pytest.fixture(params=[512, 128], ids=["rb512", "rb128"])
def stream(request, hooks):
    hooks.set("SSM_FORCE_KERNEL", "stream")
    hooks.set("SSM_STREAM_ROWS", request.param)
    return hooks


def compare(inp, h0=None):
    b, d, L = inp["u"].shape
    out = torch.full_like(inp["u"], float("nan"))
    fs = torch.full((b, d, 16), float("nan"), device=DEV)
    if h0 is None:
        ws = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp.get("D"), inp.get("z"),
                              inp.get("bias"), out, fs)
    else:
        ws = ssm.ssm_scan_fwd_from_state(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp.get("D"),
                                         inp.get("z"), inp.get("bias"), h0, out, fs)
    torch.cuda.synchronize()
    assert ssm.ssm_scan_check(ws) == ssm.SSM_OK
    ref, href = oracle.scan(*(to_np(inp[k]) for k in ("u", "delta", "A", "B", "C")), D=to_np(inp.get("D")),
                            z=to_np(inp.get("z")), bias=to_np(inp.get("bias")),
                            h0=None if h0 is None else to_np(h0))
    e, eh = rel_err(to_np(out), ref), rel_err(to_np(fs), href)
    assert e <= TOL_BF16, f"out rel err {e:.3e}"
    assert eh <= TOL_BF16, f"final_state rel err {eh:.3e}"
    return out, fs


@pytest.mark.parametrize("L", [8, 16, 24, 40, 264, 1000])
def test_ragged_tokens(stream, L):
    """Lengths that end inside a stage, inside the first stage, and several stages."""
    inp = W.random_scan_inputs(2, 40, 16, L, dtype=torch.bfloat16, device=DEV, seed=L, a_kind="random")
    compare(inp)


@pytest.mark.parametrize("d", [1, 127, 129, 600])
def test_ragged_rows(stream, d):
    """Channel counts that leave a CTA's rows partly empty (rows past d_inner are zero-filled)."""
    inp = W.random_scan_inputs(2, d, 16, 200, dtype=torch.bfloat16, device=DEV, seed=d, a_kind="random")
    compare(inp)


@pytest.mark.parametrize("chunks", [2, 3, 7])
def test_chunk_carry(stream, chunks):
    """The sequence split into chunks combined through the published aggregates."""
    stream.set("SSM_FORCE_CHUNKS", chunks)
    inp = W.random_scan_inputs(2, 130, 16, 64 * 23 + 8, dtype=torch.bfloat16, device=DEV, seed=chunks,
                               a_kind="random")
    compare(inp)


def test_chunk_carry_slow_decay(stream):
    """Small |A|·Δ: the carry hardly decays inside a chunk, so pass two covers whole chunks.
    (|A| is kept at 0.01 and above: the bf16 path forms Ā - 1 from Ā as the hardware ex2
    returns it, about 2^-22 relative, so Ā - 1 is off by ~2^-22 / |Δ A| relative.)"""
    stream.set("SSM_FORCE_CHUNKS", 4)
    inp = W.random_scan_inputs(1, 70, 16, 2048, dtype=torch.bfloat16, device=DEV, seed=8, a_kind="random")
    inp["A"] = inp["A"] * 0.05
    compare(inp)


@pytest.mark.parametrize("chunks", [1, 5])
def test_zero_and_tiny_A(stream, chunks):
    """A = 0 and |A| < 2^-60 (the exact branch, taken by the warps holding such rows)."""
    stream.set("SSM_FORCE_CHUNKS", chunks)
    inp = W.random_scan_inputs(1, 200, 16, 1200, dtype=torch.bfloat16, device=DEV, seed=3, a_kind="random")
    A = inp["A"].clone()
    A[::3, 0] = 0.0
    A[1::5, 5] = -1e-30
    A[2::7, :] = 0.0
    inp["A"] = A
    compare(inp)


@pytest.mark.parametrize("opt", ["no_D", "no_z", "no_bias", "all_off"])
def test_optional_inputs(stream, opt):
    inp = W.random_scan_inputs(2, 70, 16, 96, dtype=torch.bfloat16, device=DEV, seed=5, a_kind="random",
                               gate=opt not in ("no_z", "all_off"), skip=opt not in ("no_D", "all_off"),
                               with_bias=opt not in ("no_bias", "all_off"))
    compare(inp)


@pytest.mark.parametrize("chunks", [1, 3])
def test_initial_state(stream, chunks):
    stream.set("SSM_FORCE_CHUNKS", chunks)
    inp = W.random_scan_inputs(2, 70, 16, 704, dtype=torch.bfloat16, device=DEV, seed=31, a_kind="random")
    h0 = 2.0 * torch.randn((2, 70, 16), generator=torch.Generator(device=DEV).manual_seed(32), device=DEV)
    compare(inp, h0=h0)


@pytest.mark.parametrize("ctas", [3, 5, 7, 11])
def test_work_items_across_tiles(stream, ctas):
    """Item counts that are not a multiple of the row tiles: ranges end one tile's
    sequence and start the next's, so segments differ in length and a CTA runs two (the
    next tile's first segment, then the end of its own)."""
    stream.set("SSM_STREAM_CTAS", ctas)
    inp = W.random_scan_inputs(2, 130, 16, 32 * 37 + 8, dtype=torch.bfloat16, device=DEV, seed=80 + ctas,
                               a_kind="random")
    compare(inp)
    h0 = torch.randn((2, 130, 16), generator=torch.Generator(device=DEV).manual_seed(ctas), device=DEV)
    compare(inp, h0=h0)


def test_item_count_does_not_change_results(stream):
    """The same scan cut into 1, 5 and 9 work items per tile-sequence agrees to the output
    rounding, and so do its final states."""
    inp = W.random_scan_inputs(3, 200, 16, 3000, dtype=torch.bfloat16, device=DEV, seed=90)
    res = []
    for ctas in (1, 5, 9):
        stream.set("SSM_STREAM_CTAS", ctas * 3)
        res.append(ssm.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                inp["bias"], return_final_state=True))
    torch.cuda.synchronize()
    for out, fs in res[1:]:
        assert rel_err(to_np(out), to_np(res[0][0])) <= 2 * 2.0 ** -8
        assert rel_err(to_np(fs), to_np(res[0][1])) <= 1e-5


def test_chunking_does_not_change_results(stream):
    """Every output is computed from its true state and rounded once, chunked or not."""
    inp = W.random_scan_inputs(2, 256, 16, 4000, dtype=torch.bfloat16, device=DEV, seed=51)
    stream.set("SSM_FORCE_CHUNKS", 1)
    one = ssm.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["bias"])
    stream.set("SSM_FORCE_CHUNKS", 6)
    six = ssm.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["bias"])
    torch.cuda.synchronize()
    e = rel_err(to_np(six), to_np(one))
    assert e <= 2 * 2.0 ** -8, f"chunked vs unchunked: {e:.3e}"


def test_repeat_calls_are_identical(stream):
    """The carry combines the chunks' aggregates in a fixed order: bitwise repeatable."""
    stream.set("SSM_FORCE_CHUNKS", 9)
    inp = W.random_scan_inputs(1, 600, 16, 1 << 14, dtype=torch.bfloat16, device=DEV, seed=2)
    r1 = ssm.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["bias"],
                      return_final_state=True)
    r2 = ssm.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["bias"],
                      return_final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])


def test_lookback_timeout_is_reported_and_context_survives(stream):
    """Test hook: the carry waits on a flag nothing sets; the bounded wait gives up, the
    error word reads SSM_ERR_TIMEOUT and the device stays usable."""
    stream.set("SSM_FORCE_CHUNKS", 2)
    stream.set("SSM_FAULT", "lookback")
    stream.set("SSM_LOOKBACK_TIMEOUT_MS", 200)
    inp = W.random_scan_inputs(1, 64, 16, 1024, dtype=torch.bfloat16, device=DEV, seed=1)
    out = torch.empty_like(inp["u"])
    ws = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                          inp["bias"], out, None)
    torch.cuda.synchronize()
    assert ssm.ssm_scan_check(ws) == ssm.SSM_ERR_TIMEOUT
    stream.unset("SSM_FAULT")
    compare(inp)

"""GPU parity of the causal depthwise Conv1D + SiLU (ssm_conv1d_fwd / ssm_conv1d_step)
against the oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_154_b300 as ssm
import workloads as W
from parity import TOL, rel_err, spread_rows, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ref(inp, state=True):
    return oracle.conv1d(to_np(inp["x"]), to_np(inp["w"]), bias=to_np(inp["bias"]),
                         state0=to_np(inp["state"]) if state else None)


def _check(got, ref, dtype):
    e = rel_err(to_np(got), ref)
    assert e <= TOL[dtype], f"rel err {e:.3e}"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("width", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("L", [1, 3, 7, 8, 9, 255, 256, 257, 1000])
def test_conv_fwd_matches_oracle(dtype, width, L):
    inp = W.conv_inputs(2, 37, L, width, dtype=dtype, device=DEV, seed=L * 10 + width)
    out, sT = ssm.conv1d(inp["x"], inp["w"], inp["bias"], inp["state"], return_final_state=True)
    torch.cuda.synchronize()
    ref, rs = _ref(inp, state=width > 1)
    _check(out, ref, dtype)
    if width > 1:
        np.testing.assert_array_equal(to_np(sT), rs)  # the raw inputs, exactly


@pytest.mark.parametrize("opt", ["no_bias", "no_state", "neither"])
def test_conv_optional_inputs(opt):
    inp = W.conv_inputs(3, 20, 300, 4, device=DEV, seed=5, with_bias=opt == "no_state",
                        with_state=opt == "no_bias")
    out = ssm.conv1d(inp["x"], inp["w"], inp["bias"], inp["state"])
    torch.cuda.synchronize()
    ref, _ = _ref(inp, state=inp["state"] is not None)
    _check(out, ref, torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_conv_unaligned_views(dtype):
    """Rows that are not 16-byte aligned take the element path."""
    src = W.conv_inputs(2, 9, 123, 4, dtype=dtype, device=DEV, seed=8)
    big = torch.zeros((2 * 9 * 123 + 1,), dtype=dtype, device=DEV)
    x = big[1:].view(2, 9, 123)
    x.copy_(src["x"])
    out_big = torch.zeros_like(big)
    out = out_big[1:].view(2, 9, 123)
    ssm.ssm_conv1d_fwd(x, src["w"], src["bias"], src["state"], out, None)
    torch.cuda.synchronize()
    ref, _ = _ref(src)
    _check(out, ref, dtype)
    assert out_big[0].item() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("width", [1, 2, 4, 8])
@pytest.mark.parametrize("d_inner", [50, 1028])
def test_conv_step_matches_oracle_and_fwd(dtype, width, d_inner):
    """d_inner 1028 with bf16 and width 4 takes the four-channels-per-thread vector kernel,
    the other cases the per-channel one; both match the oracle and the sequence form bit
    for bit."""
    inp = W.conv_inputs(3, d_inner, 12, width, dtype=dtype, device=DEV, seed=width)
    state = inp["state"].clone() if width > 1 else None
    ref_state = to_np(inp["state"]) if width > 1 else np.zeros((3, d_inner, 0))
    outs = []
    for t in range(12):
        x = inp["x"][:, :, t].contiguous()
        y = ssm.conv1d_step(state, x, inp["w"], inp["bias"])
        ry, ref_state = oracle.conv1d_step(ref_state, to_np(x), to_np(inp["w"]), to_np(inp["bias"]))
        torch.cuda.synchronize()
        _check(y, ry, dtype)
        outs.append(y)
    if width > 1:
        np.testing.assert_array_equal(to_np(state), ref_state)
    full = ssm.conv1d(inp["x"], inp["w"], inp["bias"], inp["state"])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(torch.stack(outs, dim=2)), to_np(full))  # same arithmetic


def test_prefill_then_decode_conv_state():
    """Prefill a prompt, keep its final conv state, then decode token by token:
    equals one conv over prompt + generated tokens."""
    inp = W.conv_inputs(2, 64, 310, 4, device=DEV, seed=13, with_state=False)
    whole = ssm.conv1d(inp["x"], inp["w"], inp["bias"])
    _, state = ssm.conv1d(inp["x"][:, :, :300].contiguous(), inp["w"], inp["bias"], return_final_state=True)
    for t in range(300, 310):
        y = ssm.conv1d_step(state, inp["x"][:, :, t].contiguous(), inp["w"], inp["bias"])
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_np(y), to_np(whole[:, :, t]))


def test_conv_on_the_2p8b_layer_shape():
    """x of the 2.8B-shaped layer (4 x 5120 x 4096), sampled rows against the oracle."""
    shape = W.SCAN_SHAPES["mamba2p8b_layer"]
    inp = W.conv_inputs(shape.batch, shape.d_inner, shape.seqlen, device=DEV, seed=3)
    out, sT = ssm.conv1d(inp["x"], inp["w"], inp["bias"], inp["state"], return_final_state=True)
    torch.cuda.synchronize()
    rows = spread_rows(shape.batch, shape.d_inner, 24, seed=2)
    ib = torch.tensor([r[0] for r in rows], device=DEV)
    ic = torch.tensor([r[1] for r in rows], device=DEV)
    sub = dict(x=inp["x"][ib, ic][None], w=inp["w"][ic], bias=inp["bias"][ic], state=inp["state"][ib, ic][None])
    ref, rs = _ref(sub)
    _check(out[ib, ic][None], ref, torch.bfloat16)
    np.testing.assert_array_equal(to_np(sT[ib, ic][None]), rs)

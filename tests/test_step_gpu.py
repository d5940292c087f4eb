"""GPU parity of ssm_step (recurrent decode mode) against the oracle, and
ssm_step iterated L times against ssm_scan_fwd on the same sequences."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_154_b300 as ssm
import workloads as W
from parity import TOL, oracle_rows, rel_err, spread_rows, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rand_step_inputs(batch, d, N, steps, dtype, seed):
    shape = W.DecodeShape("t", batch, d, N, steps, dtype)
    inp = W.decode_inputs(shape, device=DEV, seed=seed)
    g = torch.Generator(device=DEV).manual_seed(seed + 77)
    r = torch.rand((d, N), generator=g, device=DEV)
    inp["A"] = -torch.exp(np.log(0.2) + r * (np.log(8.0) - np.log(0.2)))
    return inp


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("batch,d,N", [(1, 1, 1), (3, 37, 3), (2, 64, 4), (2, 33, 16), (1, 70, 17),
                                       (2, 16, 64), (4, 40, 13)])
def test_step_small(dtype, batch, d, N):
    steps = 6
    inp = _rand_step_inputs(batch, d, N, steps, dtype, seed=batch * 100 + d + N)
    g = torch.Generator(device=DEV).manual_seed(3)
    state = torch.randn((batch, d, N), generator=g, device=DEV)
    ref_state = to_np(state)
    for s in range(steps):
        out = ssm.step(state, inp["x"][s], inp["delta"][s], inp["A"], inp["B"][s], inp["C"][s],
                       D=inp["D"], z=inp["z"][s], delta_bias=inp["bias"])
        ref_out, ref_state = oracle.step(ref_state, inp["x"][s], inp["delta"][s], inp["A"], inp["B"][s],
                                         inp["C"][s], D=inp["D"], z=inp["z"][s], bias=inp["bias"])
        torch.cuda.synchronize()
        assert rel_err(to_np(out), ref_out) <= TOL[dtype]
        assert rel_err(to_np(state), ref_state) <= TOL[dtype]


@pytest.fixture(params=["pipe", "plain"])
def step_kernel(request, hooks):
    """Run a test with the pipelined step kernel where the shape allows it, or with
    the generic one (SSM_FORCE_STEP=plain)."""
    if request.param == "plain":
        hooks.set("SSM_FORCE_STEP", "plain")
    return request.param


# shapes the pipelined kernel takes: d_inner a multiple of 512 / (d_state / 4) rows;
# (64, 4096, 16) gives each CTA more tiles than it has pipeline stages
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("batch,d,N", [(1, 128, 16), (3, 256, 16), (2, 512, 4), (1, 256, 8), (2, 64, 32),
                                       (2, 64, 64), (64, 4096, 16)])
def test_step_tiled_shapes(step_kernel, dtype, batch, d, N):
    steps = 3
    inp = _rand_step_inputs(batch, d, N, steps, dtype, seed=batch * 7 + d + N)
    g = torch.Generator(device=DEV).manual_seed(5)
    state = torch.randn((batch, d, N), generator=g, device=DEV)
    ref_state = to_np(state)
    for s in range(steps):
        z = inp["z"][s] if s != 1 else None  # one step without the gate
        out = ssm.step(state, inp["x"][s], inp["delta"][s], inp["A"], inp["B"][s], inp["C"][s],
                       D=inp["D"], z=z, delta_bias=inp["bias"])
        ref_out, ref_state = oracle.step(ref_state, inp["x"][s], inp["delta"][s], inp["A"], inp["B"][s],
                                         inp["C"][s], D=inp["D"], z=z, bias=inp["bias"])
        torch.cuda.synchronize()
        assert rel_err(to_np(out), ref_out) <= TOL[dtype]
        assert rel_err(to_np(state), ref_state) <= TOL[dtype]
    assert ssm.ssm_step_check() == ssm.SSM_OK


def test_step_wait_timeout_is_reported_and_state_kept(hooks):
    """Test hook: the pipelined kernel's first wait is on a barrier nothing
    completes; the bounded wait gives up, every tile is left unchanged,
    ssm_step_check reports SSM_ERR_TIMEOUT once, and the next step is clean."""
    batch, d, N = 4, 1024, 16
    inp = _rand_step_inputs(batch, d, N, 1, torch.bfloat16, seed=21)
    state = torch.randn((batch, d, N), device=DEV)
    before = state.clone()
    hooks.set("SSM_FAULT", "step")
    hooks.set("SSM_LOOKBACK_TIMEOUT_MS", "100")
    ssm.step(state, inp["x"][0], inp["delta"][0], inp["A"], inp["B"][0], inp["C"][0], D=inp["D"], z=inp["z"][0],
             delta_bias=inp["bias"])
    assert ssm.ssm_step_check() == ssm.SSM_ERR_TIMEOUT
    assert torch.equal(state, before)
    assert ssm.ssm_step_check() == ssm.SSM_OK  # the check cleared the word
    hooks.unset("SSM_FAULT")
    out = ssm.step(state, inp["x"][0], inp["delta"][0], inp["A"], inp["B"][0], inp["C"][0], D=inp["D"],
                   z=inp["z"][0], delta_bias=inp["bias"])
    ref_out, ref_state = oracle.step(to_np(before), inp["x"][0], inp["delta"][0], inp["A"], inp["B"][0],
                                     inp["C"][0], D=inp["D"], z=inp["z"][0], bias=inp["bias"])
    assert ssm.ssm_step_check() == ssm.SSM_OK
    assert rel_err(to_np(out), ref_out) <= TOL[torch.bfloat16]
    assert rel_err(to_np(state), ref_state) <= TOL[torch.bfloat16]


def test_step_optional_and_zero_A():
    inp = _rand_step_inputs(2, 40, 16, 3, torch.bfloat16, seed=9)
    inp["A"][::4, 2] = 0.0
    state = torch.zeros((2, 40, 16), device=DEV)
    ref_state = np.zeros((2, 40, 16))
    for s in range(3):
        out = ssm.step(state, inp["x"][s], inp["delta"][s], inp["A"], inp["B"][s], inp["C"][s])
        ref_out, ref_state = oracle.step(ref_state, inp["x"][s], inp["delta"][s], inp["A"], inp["B"][s],
                                         inp["C"][s])
        torch.cuda.synchronize()
        assert rel_err(to_np(out), ref_out) <= TOL[torch.bfloat16]
        assert rel_err(to_np(state), ref_state) <= TOL[torch.bfloat16]


def _as_scan(inp):
    """Step inputs [steps, batch, ...] as one scan problem [batch, d, L] / [batch, L, N]."""
    return dict(u=inp["x"].permute(1, 2, 0).contiguous(), delta=inp["delta"].permute(1, 2, 0).contiguous(),
                z=inp["z"].permute(1, 2, 0).contiguous(), B=inp["B"].permute(1, 0, 2).contiguous(),
                C=inp["C"].permute(1, 0, 2).contiguous(), A=inp["A"], D=inp["D"], bias=inp["bias"])


def test_decode_workload_matches_oracle_and_scan(step_kernel):
    """256 x 5120 x 16, 1000 steps from a zero state: sampled rows against the
    oracle; every output and the final state against ssm_scan_fwd on the same
    1000-token sequences."""
    shape = W.DECODE_SHAPE
    inp = W.decode_inputs(shape, device=DEV, seed=0)
    b, d, N, S = shape.batch, shape.d_inner, shape.d_state, shape.steps
    state = torch.zeros((b, d, N), device=DEV)
    outs = torch.empty((S, b, d), dtype=shape.dtype, device=DEV)
    for s in range(S):
        ssm.ssm_step(state, inp["x"][s], inp["delta"][s], inp["A"], inp["B"][s], inp["C"][s], inp["D"],
                     inp["z"][s], inp["bias"], outs[s])
    torch.cuda.synchronize()
    scan_in = _as_scan(inp)
    rows = spread_rows(b, d, 40, seed=4)
    ref, href = oracle_rows(scan_in, rows)
    ib = torch.tensor([r[0] for r in rows], device=DEV)
    ic = torch.tensor([r[1] for r in rows], device=DEV)
    got = to_np(outs[:, ib, ic].transpose(0, 1))
    assert rel_err(got, ref) <= TOL[shape.dtype]
    assert rel_err(to_np(state[ib, ic]), href) <= TOL[shape.dtype]
    # iterated steps vs the parallel-mode scan, everywhere
    out_scan, fs_scan = ssm.scan_fwd(scan_in["u"], scan_in["delta"], scan_in["A"], scan_in["B"], scan_in["C"],
                                     scan_in["D"], scan_in["z"], scan_in["bias"], return_final_state=True)
    torch.cuda.synchronize()
    o_step = outs.permute(1, 2, 0).float()
    rms = o_step.pow(2).mean().sqrt()
    err = ((out_scan.float() - o_step).abs() / torch.maximum(o_step.abs(), rms)).max().item()
    assert err <= TOL[shape.dtype]
    rms_h = fs_scan.pow(2).mean().sqrt()
    err_h = ((fs_scan - state).abs() / torch.maximum(fs_scan.abs(), rms_h)).max().item()
    assert err_h <= TOL[shape.dtype]
    assert ssm.ssm_step_check() == ssm.SSM_OK


def test_prefill_then_decode_continues_the_state():
    """Scan a prompt, then decode from its final state: equals one scan over
    prompt + generated tokens (prefill → decode hand-off)."""
    batch, d, N, L0, S = 2, 48, 16, 300, 20
    full = W.random_scan_inputs(batch, d, N, L0 + S, dtype=torch.bfloat16, device=DEV, seed=12)
    ref, _ = ssm.scan_fwd(full["u"], full["delta"], full["A"], full["B"], full["C"], full["D"], full["z"],
                          full["bias"], return_final_state=True)
    pre = {k: v for k, v in full.items()}
    for k in ("u", "delta", "z"):
        pre[k] = full[k][:, :, :L0].contiguous()
    for k in ("B", "C"):
        pre[k] = full[k][:, :L0].contiguous()
    _, state = ssm.scan_fwd(pre["u"], pre["delta"], pre["A"], pre["B"], pre["C"], pre["D"], pre["z"],
                            pre["bias"], return_final_state=True)
    for s in range(S):
        t = L0 + s
        y = ssm.step(state, full["u"][:, :, t].contiguous(), full["delta"][:, :, t].contiguous(), full["A"],
                     full["B"][:, t].contiguous(), full["C"][:, t].contiguous(), full["D"],
                     full["z"][:, :, t].contiguous(), full["bias"])
        torch.cuda.synchronize()
        assert rel_err(to_np(y), to_np(ref[:, :, t]), rms_ref=float(ref.float().pow(2).mean().sqrt())) <= 2e-2

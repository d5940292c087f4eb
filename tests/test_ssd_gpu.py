"""GPU parity of ssd_scan_fwd (the Mamba-2 layer scan on the tensor cores) with the
float64 oracle on the same bf16-rounded inputs: whole outputs at small sizes that
still span several 128-token chunks and a ragged tail, and sampled heads over the
full Mamba-2-2.7B-shaped layer."""
import pytest
import torch

import oracle
import selective_state_space_154_b300 as ssm
import workloads as W
from parity import TOL, rel_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = TOL[torch.bfloat16]


@pytest.fixture(params=["ssd_walk", "ssd_chunks"], ids=["walk", "chunks"])
def form(request, hooks):
    """Both forms of the layer scan: one CTA walking the sequence of each (batch, head),
    and the chunk-parallel launches."""
    hooks.set("SSM_FORCE_KERNEL", request.param)
    return hooks


def _oracle(inp, h0=None):
    return oracle.ssd_scan(*(to_np(inp[k]) for k in ("x", "dt", "A", "B", "C")), D=to_np(inp["D"]),
                           z=to_np(inp["z"]), dt_bias=to_np(inp["dt_bias"]), h0=to_np(h0))


def _gpu(inp, h0=None):
    out, fs = ssm.ssd_scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"], z=inp["z"],
                           dt_bias=inp["dt_bias"], initial_state=h0, return_final_state=True)
    torch.cuda.synchronize()
    return out, fs


def _compare(inp, h0=None):
    out, fs = _gpu(inp, h0)
    ref, href = _oracle(inp, h0)
    assert rel_err(to_np(out), ref) <= BF16
    assert rel_err(to_np(fs), href) <= BF16


@pytest.mark.parametrize("shape", [(1, 128, 2, 64, 1, 128), (2, 300, 4, 64, 2, 128), (1, 1, 2, 64, 1, 128),
                                   (1, 129, 3, 64, 3, 128), (2, 700, 2, 64, 1, 128), (1, 2048, 4, 64, 2, 128)],
                         ids=["one_chunk", "ragged_groups", "one_token", "chunk_plus_one", "six_chunks",
                              "sixteen_chunks"])
def test_ssd_matches_oracle(shape, form):
    _compare(W.random_ssd_inputs(*shape, device=DEV, seed=sum(shape)))


@pytest.mark.parametrize("opts", [dict(gate=False), dict(skip=False), dict(with_bias=False),
                                  dict(gate=False, skip=False, with_bias=False)],
                         ids=["no_z", "no_D", "no_bias", "all_off"])
def test_ssd_optional_inputs(opts, form):
    _compare(W.random_ssd_inputs(1, 260, 2, 64, 1, 128, device=DEV, seed=5, **opts))


def test_ssd_initial_state_continues_a_split_sequence(form):
    inp = W.random_ssd_inputs(2, 400, 2, 64, 1, 128, device=DEV, seed=8)
    g = torch.Generator(device=DEV).manual_seed(3)
    h0 = torch.randn((2, 2, 64, 128), generator=g, device=DEV)
    _compare(inp, h0)
    ref, href = _oracle(inp, h0)
    # the first 250 tokens, then the rest from the device's final state
    first = {k: (v if k in ("A", "D", "dt_bias") or v is None else v[:, :250].contiguous()) for k, v in inp.items()}
    rest = {k: (v if k in ("A", "D", "dt_bias") or v is None else v[:, 250:].contiguous()) for k, v in inp.items()}
    o1, f1 = _gpu(first, h0)
    o2, f2 = _gpu(rest, f1)
    assert rel_err(to_np(torch.cat([o1, o2], dim=1)), ref) <= BF16
    assert rel_err(to_np(f2), href) <= BF16


def test_ssd_zero_A_is_linear_attention(form):
    inp = W.random_ssd_inputs(1, 300, 2, 64, 1, 128, device=DEV, seed=12)
    inp["A"].zero_()
    _compare(inp)


def test_ssd_empty_sequence_passes_the_state_through(form):
    inp = W.random_ssd_inputs(1, 0, 2, 64, 1, 128, device=DEV, seed=2)
    h0 = torch.randn((1, 2, 64, 128), device=DEV)
    out, fs = _gpu(inp, h0)
    assert out.numel() == 0
    assert torch.equal(fs, h0)


def test_ssd_mamba2_2p7b_layer_sampled_heads():
    """The full 4 × 4096 × 80 × 64 (N = 128) layer on the device; the oracle recomputes
    heads 0, 37 and 79 of every batch over the whole sequence."""
    shape = W.SSD_SHAPES["mamba2_2p7b_layer"]
    inp = W.ssd_inputs(shape, device=DEV, seed=0)
    ws = torch.empty(ssm.ssd_scan_workspace_bytes(shape.batch, shape.seqlen, shape.nheads, shape.headdim,
                                                  shape.ngroups, shape.d_state), dtype=torch.uint8, device=DEV)
    out, fs = ssm.ssd_scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], D=inp["D"], z=inp["z"],
                           dt_bias=inp["dt_bias"], return_final_state=True, workspace=ws)
    torch.cuda.synchronize()
    assert ssm.ssm_scan_check(ws) == ssm.SSM_OK
    for h in (0, 37, 79):
        sub = {k: (None if v is None else v[..., h:h + 1] if k in ("A", "D", "dt_bias", "dt") else v)
               for k, v in inp.items()}
        sub["x"] = inp["x"][:, :, h:h + 1]
        sub["z"] = inp["z"][:, :, h:h + 1]
        ref, href = _oracle(sub)
        assert rel_err(to_np(out[:, :, h:h + 1]), ref) <= BF16, h
        assert rel_err(to_np(fs[:, h:h + 1]), href) <= BF16, h


@pytest.mark.parametrize("shape", [(1, 300, 5, 64, 1, 128), (1, 260, 12, 64, 2, 128), (2, 150, 14, 64, 2, 128),
                                   (1, 400, 16, 64, 1, 128)],
                         ids=["5_heads_per_cta", "6_heads_per_cta", "7_heads_per_cta", "8_heads_per_cta_x2"])
def test_ssd_heads_per_cta(shape, hooks):
    """Chunk-parallel form: a CTA takes up to 8 heads of one group (the largest divisor
    of heads per group): odd and even counts, several head blocks per group."""
    hooks.set("SSM_FORCE_KERNEL", "ssd_chunks")
    _compare(W.random_ssd_inputs(*shape, device=DEV, seed=shape[2]))


def test_ssd_walk_is_chosen_for_many_heads_and_matches():
    """2 × 40 heads reach the planner's threshold for the walking form (its workspace is
    the error words alone); four groups, a ragged last chunk, an initial state."""
    assert ssm.ssd_scan_workspace_bytes(2, 333, 40, 64, 4, 128) == 256
    inp = W.random_ssd_inputs(2, 333, 40, 64, 4, 128, device=DEV, seed=77)
    h0 = torch.randn((2, 40, 64, 128), generator=torch.Generator(device=DEV).manual_seed(78), device=DEV)
    _compare(inp, h0)


def test_ssd_wait_timeout_is_reported_and_the_context_recovers(form):
    """Test hook: the first tensor-core wait (of the output kernel, or of the walking
    kernel) is on an mbarrier that nothing arrives on.  The wait gives up after 200 ms, lets its issued products finish, frees its
    tensor memory and sets the workspace's error word; the next clean call is correct."""
    inp = W.random_ssd_inputs(1, 300, 2, 64, 1, 128, device=DEV, seed=4)
    ws = torch.empty(ssm.ssd_scan_workspace_bytes(1, 300, 2, 64, 1, 128), dtype=torch.uint8, device=DEV)
    args = (inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"])
    kw = dict(D=inp["D"], z=inp["z"], dt_bias=inp["dt_bias"], return_final_state=True, workspace=ws)
    form.set("SSM_FAULT", "ssd")
    form.set("SSM_LOOKBACK_TIMEOUT_MS", "200")
    ssm.ssd_scan(*args, **kw)
    torch.cuda.synchronize()
    assert ssm.ssm_scan_check(ws) == ssm.SSM_ERR_TIMEOUT
    form.unset("SSM_FAULT")
    form.unset("SSM_LOOKBACK_TIMEOUT_MS")
    out, fs = ssm.ssd_scan(*args, **kw)
    torch.cuda.synchronize()
    assert ssm.ssm_scan_check(ws) == ssm.SSM_OK
    ref, href = _oracle(inp)
    assert rel_err(to_np(out), ref) <= BF16
    assert rel_err(to_np(fs), href) <= BF16


def _step_inputs(inp, t):
    """Token t of a sequence's inputs, in the decode layout."""
    return dict(x=inp["x"][:, t].contiguous(), dt=inp["dt"][:, t].contiguous(), B=inp["B"][:, t].contiguous(),
                C=inp["C"][:, t].contiguous(), z=None if inp["z"] is None else inp["z"][:, t].contiguous())


@pytest.mark.parametrize("opts", [dict(), dict(gate=False, skip=False, with_bias=False)], ids=["all", "none"])
def test_ssd_step_matches_oracle(opts):
    """One decode token from a random state: the oracle's scan of one token from that state."""
    inp = W.random_ssd_inputs(2, 1, 4, 64, 2, 128, device=DEV, seed=14, **opts)
    g = torch.Generator(device=DEV).manual_seed(15)
    state = torch.randn((2, 4, 64, 128), generator=g, device=DEV)
    ref, href = _oracle(inp, state)
    tok = _step_inputs(inp, 0)
    y = ssm.ssd_step(state, tok["x"], tok["dt"], inp["A"], tok["B"], tok["C"], D=inp["D"], z=tok["z"],
                     dt_bias=inp["dt_bias"])
    torch.cuda.synchronize()
    assert rel_err(to_np(y), ref[:, 0]) <= BF16
    assert rel_err(to_np(state), href) <= 1e-5  # fp32 state: one update's rounding


def test_ssd_prefill_then_decode():
    """ssd_scan_fwd over the first 300 tokens, then 20 ssd_step calls from its final state:
    the outputs and the final state match the oracle over all 320 tokens, and the device's
    own scan of all 320."""
    L0, L = 300, 320
    inp = W.random_ssd_inputs(2, L, 4, 64, 2, 128, device=DEV, seed=16)
    ref, href = _oracle(inp)
    pre = {k: (v if k in ("A", "D", "dt_bias") or v is None else v[:, :L0].contiguous()) for k, v in inp.items()}
    _, state = _gpu(pre)
    ys = []
    for t in range(L0, L):
        tok = _step_inputs(inp, t)
        ys.append(ssm.ssd_step(state, tok["x"], tok["dt"], inp["A"], tok["B"], tok["C"], D=inp["D"], z=tok["z"],
                               dt_bias=inp["dt_bias"]))
    torch.cuda.synchronize()
    dec = torch.stack(ys, dim=1)
    assert rel_err(to_np(dec), ref[:, L0:]) <= BF16
    assert rel_err(to_np(state), href) <= BF16
    full, _ = _gpu(inp)
    assert rel_err(to_np(dec), to_np(full[:, L0:])) <= BF16


def test_ssd_step_mamba2_2p7b_decode_sampled_heads():
    """A 2.7B-shaped decode batch (64 × 80 heads × 64 × 128 state): heads 0, 41, 79 against the oracle."""
    shape = W.SsdShape("decode", 64, 1, 80, 64, 1, 128, torch.bfloat16)
    inp = W.ssd_inputs(shape, device=DEV, seed=3)
    g = torch.Generator(device=DEV).manual_seed(4)
    state = torch.randn((64, 80, 64, 128), generator=g, device=DEV)
    state0 = state.clone()
    tok = _step_inputs(inp, 0)
    y = ssm.ssd_step(state, tok["x"], tok["dt"], inp["A"], tok["B"], tok["C"], D=inp["D"], z=tok["z"],
                     dt_bias=inp["dt_bias"])
    torch.cuda.synchronize()
    for h in (0, 41, 79):
        sub = {k: (None if v is None else v[..., h:h + 1] if k in ("A", "D", "dt_bias", "dt") else v)
               for k, v in inp.items()}
        sub["x"] = inp["x"][:, :, h:h + 1]
        sub["z"] = inp["z"][:, :, h:h + 1]
        ref, href = _oracle(sub, state0[:, h:h + 1])
        assert rel_err(to_np(y[:, h:h + 1]), ref[:, 0]) <= BF16, h
        assert rel_err(to_np(state[:, h:h + 1]), href) <= 1e-5, h


@pytest.mark.parametrize("split", [2, 3, 5])
def test_ssd_walk_segments_from_a_state_only_prefix(hooks, split):
    """Every (batch, head) cut into `split` segments of chunks: each segment's CTA walks the
    chunks before it for the state alone, then its own in full; outputs and the final
    state (written by the last segment) match the oracle, from a nonzero initial state."""
    hooks.set("SSM_FORCE_KERNEL", "ssd_walk")
    hooks.set("SSM_SSD_SPLIT", split)
    inp = W.random_ssd_inputs(2, 700, 3, 64, 1, 128, device=DEV, seed=60 + split)
    h0 = torch.randn((2, 3, 64, 128), generator=torch.Generator(device=DEV).manual_seed(split), device=DEV)
    _compare(inp, h0)


def test_ssd_walk_remainder_units_split_across_the_gpu():
    """2 × 80 heads: one full round of CTAs, and the units left over cut into segments
    (the default split); sampled heads of both kinds against the oracle."""
    inp = W.random_ssd_inputs(2, 1000, 80, 64, 4, 128, device=DEV, seed=71)
    out, fs = _gpu(inp)
    for b_, h_ in ((0, 3), (1, 60), (1, 68), (1, 79)):
        # head h_ of batch b_, with its group's B and C (20 heads per group)
        sub = {k: (None if v is None else v[b_:b_ + 1, :, h_:h_ + 1] if k in ("x", "z", "dt")
                   else v[h_:h_ + 1] if k in ("A", "D", "dt_bias") else v[b_:b_ + 1, :, (h_ // 20):(h_ // 20) + 1])
               for k, v in inp.items()}
        ref, href = _oracle(sub)
        assert rel_err(to_np(out[b_:b_ + 1, :, h_:h_ + 1]), ref) <= BF16, (b_, h_)
        assert rel_err(to_np(fs[b_:b_ + 1, h_:h_ + 1]), href) <= BF16, (b_, h_)

"""GPU parity of ssm_scan_bwd (the backward of the scan with recomputed states)
against the float64 backward oracle on the same rounded inputs."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_154_b300 as ssm
import workloads as W
from parity import TOL, rel_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
GRADS = ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "dbias")


def _run(inp, dout):
    g = ssm.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dout, D=inp.get("D"), z=inp.get("z"),
                     delta_bias=inp.get("bias"))
    torch.cuda.synchronize()
    return g


def _ref(inp, dout):
    return oracle.scan_bwd(*(to_np(inp[k]) for k in ("u", "delta", "A", "B", "C")), to_np(dout),
                           D=to_np(inp.get("D")), z=to_np(inp.get("z")), bias=to_np(inp.get("bias")))


def _compare(inp, dout, tol):
    g, r = _run(inp, dout), _ref(inp, dout)
    for k in GRADS:
        if r[k] is None or g[k] is None:
            continue
        e = rel_err(to_np(g[k]), r[k])
        assert e <= tol, f"{k}: rel err {e:.3e}"


def _dout(inp, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(inp["u"].shape, generator=gen, device=DEV).to(inp["u"].dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("L", [1, 7, 8, 9, 100])
def test_bwd_ragged_lengths(dtype, L):
    inp = W.random_scan_inputs(2, 37, 16, L, dtype=dtype, device=DEV, seed=L + 5, a_kind="random")
    _compare(inp, _dout(inp, L), TOL[dtype])


@pytest.mark.parametrize("N", [1, 4, 13, 16])
def test_bwd_state_sizes(N):
    inp = W.random_scan_inputs(2, 130, N, 64, dtype=torch.bfloat16, device=DEV, seed=N, a_kind="random")
    _compare(inp, _dout(inp, N), TOL[torch.bfloat16])


@pytest.mark.parametrize("opt", ["no_D", "no_z", "no_bias", "all_off"])
def test_bwd_optional_inputs(opt):
    inp = W.random_scan_inputs(2, 40, 16, 50, dtype=torch.bfloat16, device=DEV, seed=3, a_kind="random",
                               gate=opt not in ("no_z", "all_off"), skip=opt not in ("no_D", "all_off"),
                               with_bias=opt not in ("no_bias", "all_off"))
    _compare(inp, _dout(inp, 4), TOL[torch.bfloat16])


def test_bwd_zero_A():
    inp = W.random_scan_inputs(2, 40, 16, 60, dtype=torch.float32, device=DEV, seed=6, a_kind="random")
    inp["A"][::3, 2] = 0.0
    _compare(inp, _dout(inp, 7), TOL[torch.float32])


def test_bwd_mamba130m_shaped_rows():
    """The 130M-shaped layer's shape with fewer channels (the oracle runs on one core):
    2 x 256 x 16 x 2048, bf16."""
    inp = W.random_scan_inputs(2, 256, 16, 2048, dtype=torch.bfloat16, device=DEV, seed=11)
    _compare(inp, _dout(inp, 12), TOL[torch.bfloat16])


def test_bwd_rejects_large_d_state():
    inp = W.random_scan_inputs(1, 8, 32, 16, dtype=torch.bfloat16, device=DEV, seed=1)
    with pytest.raises(ssm.SsmError):
        _run(inp, _dout(inp, 1))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("chunks", [1, 2, 5, 19])
def test_bwd_sequence_chunks(hooks, dtype, chunks):
    """The sequence split into chunks (38 blocks of 8 tokens, the last ragged, over
    1, 2, 5 or 19 chunks) gives the oracle's gradients."""
    hooks.set("SSM_BWD_CHUNKS", str(chunks))
    inp = W.random_scan_inputs(2, 70, 16, 300, dtype=dtype, device=DEV, seed=chunks, a_kind="random")
    _compare(inp, _dout(inp, chunks + 1), TOL[dtype])


def test_bwd_sequence_chunks_zero_A(hooks):
    """Chunk summaries with A = 0 states (no decay across chunks) on the scalar path."""
    hooks.set("SSM_BWD_CHUNKS", "4")
    inp = W.random_scan_inputs(1, 40, 16, 200, dtype=torch.float32, device=DEV, seed=9, a_kind="random")
    inp["A"][::2, 5] = 0.0
    _compare(inp, _dout(inp, 10), TOL[torch.float32])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_bwd_few_rows_long_sequence(dtype):
    """One row tile over 6000 tokens: the planner splits the sequence into many chunks."""
    inp = W.random_scan_inputs(1, 64, 16, 6000, dtype=dtype, device=DEV, seed=21)
    _compare(inp, _dout(inp, 22), TOL[dtype])


def test_bwd_chunk_counts_agree(hooks):
    """fp32 gradients with 1 and 7 chunks agree to rounding (the chunk combine is exact
    algebra; only the order of additions differs)."""
    inp = W.random_scan_inputs(2, 50, 16, 500, dtype=torch.float32, device=DEV, seed=31, a_kind="random")
    dout = _dout(inp, 32)
    hooks.set("SSM_BWD_CHUNKS", "1")
    g1 = _run(inp, dout)
    hooks.set("SSM_BWD_CHUNKS", "7")
    g7 = _run(inp, dout)
    for k in GRADS:
        if g1[k] is None:
            continue
        a, b = to_np(g1[k]), to_np(g7[k])
        assert rel_err(b, a) <= 2e-5, k


@pytest.mark.parametrize("chunks", [0, 3])
def test_bwd_deterministic_bitwise_and_parity(hooks, chunks):
    """ssm_scan_bwd_deterministic: two calls return the same bits for every gradient, they
    match the oracle like the atomic mode, and the two modes agree to rounding."""
    if chunks:
        hooks.set("SSM_BWD_CHUNKS", chunks)
    inp = W.random_scan_inputs(3, 150, 16, 300, dtype=torch.bfloat16, device=DEV, seed=21, a_kind="random")
    dout = _dout(inp, 22)
    kw = dict(D=inp["D"], z=inp["z"], delta_bias=inp["bias"])
    g1 = ssm.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dout, deterministic=True, **kw)
    g2 = ssm.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dout, deterministic=True, **kw)
    ga = ssm.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dout, **kw)
    torch.cuda.synchronize()
    r = _ref(inp, dout)
    for k in GRADS:
        assert torch.equal(g1[k], g2[k]), f"{k}: deterministic mode differs between calls"
        e = rel_err(to_np(g1[k]), r[k])
        assert e <= TOL[torch.bfloat16], f"{k}: rel err {e:.3e}"
        e2 = rel_err(to_np(g1[k]), to_np(ga[k]).astype(np.float64))
        assert e2 <= 1e-3, f"{k}: deterministic vs atomic {e2:.3e}"


def test_bwd_deterministic_fp32_no_optional():
    inp = W.random_scan_inputs(2, 70, 13, 90, dtype=torch.float32, device=DEV, seed=23, a_kind="random",
                               gate=False, skip=False, with_bias=False)
    dout = _dout(inp, 24)
    g = ssm.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dout, deterministic=True)
    torch.cuda.synchronize()
    r = _ref(inp, dout)
    for k in GRADS:
        if r[k] is None or g[k] is None:
            continue
        e = rel_err(to_np(g[k]), r[k])
        assert e <= TOL[torch.float32], f"{k}: rel err {e:.3e}"


@pytest.mark.parametrize("form", ["lane", "quad"])
@pytest.mark.parametrize("chunks", [1, 3, 7])
@pytest.mark.parametrize("gate", [True, False], ids=["z", "no_z"])
def test_bwd_prefetched_blocks(hooks, chunks, gate, form):
    """bf16 with d_state 16 and L a multiple of 8: both kernels copy the next block's raw
    inputs (and the gradient kernel its checkpoint) by cp.async while the current block
    computes; across chunk counts, with and without the gate, in both modes, with the
    gradient pass at one thread per row (the default here) and at four."""
    hooks.set("SSM_BWD_CHUNKS", str(chunks))
    if form == "quad":
        hooks.set("SSM_BWD_FORM", "quad")
    inp = W.random_scan_inputs(2, 150, 16, 512, dtype=torch.bfloat16, device=DEV, seed=40 + chunks, a_kind="random",
                               gate=gate)
    dout = _dout(inp, 41)
    _compare(inp, dout, TOL[torch.bfloat16])
    g = ssm.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dout, D=inp.get("D"), z=inp.get("z"),
                     delta_bias=inp.get("bias"), deterministic=True)
    torch.cuda.synchronize()
    r = _ref(inp, dout)
    for k in GRADS:
        if r[k] is None or g[k] is None:
            continue
        e = rel_err(to_np(g[k]), r[k])
        assert e <= TOL[torch.bfloat16], f"{k}: rel err {e:.3e}"


@pytest.mark.parametrize("chunks", [1, 4])
def test_bwd_lane_zero_A_and_padding_rows(hooks, chunks):
    """The one-thread-per-row gradient pass with A = 0 states in some rows (the tile that
    holds them takes the general per-state form, the others the fused one) and a last tile
    of 36 rows past d_inner (100 channels in 64-row tiles)."""
    hooks.set("SSM_BWD_CHUNKS", str(chunks))
    inp = W.random_scan_inputs(2, 100, 16, 96, dtype=torch.bfloat16, device=DEV, seed=50 + chunks,
                               a_kind="random")
    inp["A"][70::5, 3] = 0.0
    inp["A"][80, :] = 0.0
    _compare(inp, _dout(inp, 51), TOL[torch.bfloat16])


def test_bwd_lane_and_quad_forms_agree(hooks):
    """The two gradient passes give the same gradients to rounding on the same inputs
    (the 130M-shaped layer's rows over a shorter sequence, five chunks)."""
    hooks.set("SSM_BWD_CHUNKS", "5")
    inp = W.random_scan_inputs(2, 192, 16, 800, dtype=torch.bfloat16, device=DEV, seed=61)
    dout = _dout(inp, 62)
    gl = _run(inp, dout)
    hooks.set("SSM_BWD_FORM", "quad")
    gq = _run(inp, dout)
    r = _ref(inp, dout)
    for k in GRADS:
        if gl[k] is None:
            continue
        el, eq = rel_err(to_np(gl[k]), r[k]), rel_err(to_np(gq[k]), r[k])
        assert el <= TOL[torch.bfloat16] and eq <= TOL[torch.bfloat16], f"{k}: {el:.3e} / {eq:.3e}"


def test_bwd_unaligned_gradient_views():
    """bf16, d_state 16, L a multiple of 8, with du, the Δraw gradient and dz 2-byte aligned
    only (the gradient passes store them one element at a time): the result matches the
    oracle like the aligned call's."""
    b, d, N, L = 2, 70, 16, 96
    inp = W.random_scan_inputs(b, d, N, L, dtype=torch.bfloat16, device=DEV, seed=71, a_kind="random")
    dout = _dout(inp, 72)

    def off_view(shape, dtype):
        n = int(np.prod(shape))
        return torch.empty(n + 1, dtype=dtype, device=DEV)[1:].view(shape)

    g = dict(du=off_view(inp["u"].shape, torch.bfloat16), ddelta=off_view(inp["u"].shape, torch.bfloat16),
             dz=off_view(inp["u"].shape, torch.bfloat16),
             dA=torch.empty(inp["A"].shape, dtype=torch.float32, device=DEV),
             dB=torch.empty(inp["B"].shape, dtype=torch.float32, device=DEV),
             dC=torch.empty(inp["C"].shape, dtype=torch.float32, device=DEV),
             dD=torch.empty_like(inp["D"]), dbias=torch.empty((d,), dtype=torch.float32, device=DEV))
    assert g["du"].data_ptr() % 16 != 0
    ssm.ssm_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["bias"], dout,
                     g["du"], g["ddelta"], g["dA"], g["dB"], g["dC"], g["dD"], g["dz"], g["dbias"])
    torch.cuda.synchronize()
    r = _ref(inp, dout)
    for k in GRADS:
        e = rel_err(to_np(g[k]), r[k])
        assert e <= TOL[torch.bfloat16], f"{k}: rel err {e:.3e}"


@pytest.mark.parametrize("name", ["mamba130m_layer", "mamba2p8b_layer"])
def test_bwd_layer_full_size_sampled(name):
    """The Mamba-shaped layers at full size (8 × 1536 × 16 × 2048 and 4 × 5120 × 16 × 4096,
    bf16), with the benchmark's inputs and launch (the planner's chunk count, one thread per
    row): du, the Δraw gradient and dz of six channels in every batch row, and those
    channels' dA, dD and dbias (sums over the batch), against the oracle run on those
    channels alone; on the 130M-shaped layer also dB and dC of batch row 0 (sums over all
    1536 channels) against the oracle run on that batch row (the 2.8B-shaped layer's would
    take the single-threaded oracle about a minute)."""
    shape = W.SCAN_SHAPES[name]
    inp = W.scan_inputs(shape, device=DEV, seed=0)
    gen = torch.Generator(device=DEV).manual_seed(1)
    dout = torch.randn(inp["u"].shape, generator=gen, device=DEV).to(shape.dtype)
    g = _run(inp, dout)
    tol = TOL[torch.bfloat16]
    d = shape.d_inner
    chans = [0, 1, d // 3, d // 2, d - 2, d - 1]
    pick = lambda t: to_np(t[:, chans])
    r = oracle.scan_bwd(pick(inp["u"]), pick(inp["delta"]), to_np(inp["A"][chans]), to_np(inp["B"]),
                        to_np(inp["C"]), pick(dout), D=to_np(inp["D"][chans]), z=pick(inp["z"]),
                        bias=to_np(inp["bias"][chans]))
    for k in ("du", "ddelta", "dz"):
        e = rel_err(to_np(g[k][:, chans]), r[k])
        assert e <= tol, f"{k}: rel err {e:.3e}"
    for k in ("dA", "dD", "dbias"):
        e = rel_err(to_np(g[k][chans]), r[k])
        assert e <= tol, f"{k}: rel err {e:.3e}"
    if name != "mamba130m_layer":
        return
    row0 = lambda t: to_np(t[:1])
    r0 = oracle.scan_bwd(row0(inp["u"]), row0(inp["delta"]), to_np(inp["A"]), row0(inp["B"]), row0(inp["C"]),
                         row0(dout), D=to_np(inp["D"]), z=row0(inp["z"]), bias=to_np(inp["bias"]))
    for k in ("dB", "dC"):
        e = rel_err(to_np(g[k][:1]), r0[k])
        assert e <= tol, f"{k}: rel err {e:.3e}"

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

"""Seeded synthetic inputs for the selective state-space scan.

This module only draws random numbers in the shapes, dtypes and distributions
of the workloads; it holds none of the method's arithmetic.  Both the CUDA path
(through the tests and the benchmark) and the oracle consume what it produces.

Every tensor has its own generator, seeded from (seed, tensor id), so any one
tensor can be redrawn without the others.  Activations are drawn in float32 and
rounded to the activation dtype (round-to-nearest-even for bf16); the oracle is
fed exactly those rounded values.

Workloads (Mamba-shaped layers; batch, d_inner, d_state N, length L):

    tiny_fp32        1 ×   16 × 4  × 64         fp32
    mamba130m_layer  8 × 1536 × 16 × 2048       bf16
    mamba2p8b_layer  4 × 5120 × 16 × 4096       bf16
    long_1m          1 × 2048 × 16 × 1,048,576  bf16
    decode           256 × 5120 × 16, 1000 recurrent steps, bf16 I/O, fp32 state

Distributions: A[c, n] = -(n + 1); u, z, B, C, D ~ N(0, 1); for the scans the
step dt ~ log-uniform[1e-3, 0.1] per element, passed as Δraw = log(expm1(dt))
with bias = 0; for decode Δraw ~ N(0, 1) and bias[c] = log(expm1(dt_c)) with
dt_c ~ log-uniform[1e-3, 0.1] per channel.

Mamba-2 (SSD) layer workloads (batch, L, heads × headdim, groups, d_state N):

    mamba2_130m_layer  8 × 2048, 24 × 64, 1 group, N 128   bf16
    mamba2_2p7b_layer  4 × 4096, 80 × 64, 1 group, N 128   bf16

with x, z, B, C ~ N(0, 1) (layout [batch][L][heads][headdim] and
[batch][L][groups][N]), A[h] ~ -U(1, 16) per head, D ~ N(0, 1) per head and the
step dt ~ log-uniform[1e-3, 0.1] per (batch, token, head), passed as
Δraw = log(expm1(dt)) with dt_bias = 0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class ScanShape:
    name: str
    batch: int
    d_inner: int
    d_state: int
    seqlen: int
    dtype: torch.dtype

    @property
    def rows(self) -> int:
        return self.batch * self.d_inner

    @property
    def channel_tokens(self) -> int:
        return self.batch * self.d_inner * self.seqlen


@dataclass(frozen=True)
class DecodeShape:
    name: str
    batch: int
    d_inner: int
    d_state: int
    steps: int
    dtype: torch.dtype


SCAN_SHAPES = {
    "tiny_fp32": ScanShape("tiny_fp32", 1, 16, 4, 64, torch.float32),
    "mamba130m_layer": ScanShape("mamba130m_layer", 8, 1536, 16, 2048, torch.bfloat16),
    "mamba2p8b_layer": ScanShape("mamba2p8b_layer", 4, 5120, 16, 4096, torch.bfloat16),
    "long_1m": ScanShape("long_1m", 1, 2048, 16, 1 << 20, torch.bfloat16),
}
DECODE_SHAPE = DecodeShape("decode", 256, 5120, 16, 1000, torch.bfloat16)


@dataclass(frozen=True)
class SsdShape:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    ngroups: int
    d_state: int
    dtype: torch.dtype

    @property
    def channel_tokens(self) -> int:
        return self.batch * self.seqlen * self.nheads * self.headdim


SSD_SHAPES = {
    "mamba2_130m_layer": SsdShape("mamba2_130m_layer", 8, 2048, 24, 64, 1, 128, torch.bfloat16),
    "mamba2_2p7b_layer": SsdShape("mamba2_2p7b_layer", 4, 4096, 80, 64, 1, 128, torch.bfloat16),
}

# tensor ids: each tensor is drawn from its own stream
_IDS = dict(u=1, delta=2, z=3, B=4, C=5, D=6, A=7, bias=8, x=9, dt=10)


def _gen(device, seed: int, tid: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + tid)
    return g


def _normal(shape, device, seed, name, dtype):
    g = _gen(device, seed, _IDS[name])
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def _log_uniform(shape, device, seed, name, lo=1e-3, hi=0.1):
    g = _gen(device, seed, _IDS[name])
    r = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return torch.exp(math.log(lo) + r * (math.log(hi) - math.log(lo)))


def a_matrix(d_inner: int, d_state: int, device) -> torch.Tensor:
    """A[c, n] = -(n + 1), fp32."""
    n = torch.arange(1, d_state + 1, device=device, dtype=torch.float32)
    return (-n).expand(d_inner, d_state).contiguous()


def scan_inputs(shape: ScanShape, device="cpu", seed: int = 0, gate: bool = True,
                skip: bool = True, with_bias: bool = True):
    """Inputs of one scan call as a dict of tensors on ``device``.

    u, delta, z: [batch, d_inner, L] (act dtype); B, C: [batch, L, N] (act dtype);
    A: [d_inner, N], D, bias: [d_inner] (fp32).
    """
    b, d, N, L, dt_ = shape.batch, shape.d_inner, shape.d_state, shape.seqlen, shape.dtype
    dt = _log_uniform((b, d, L), device, seed, "dt")
    delta = torch.log(torch.expm1(dt)).to(dt_)
    del dt
    out = dict(
        u=_normal((b, d, L), device, seed, "u", dt_),
        delta=delta,
        A=a_matrix(d, N, device),
        B=_normal((b, L, N), device, seed, "B", dt_),
        C=_normal((b, L, N), device, seed, "C", dt_),
        D=_normal((d,), device, seed, "D", torch.float32) if skip else None,
        z=_normal((b, d, L), device, seed, "z", dt_) if gate else None,
        bias=torch.zeros(d, device=device, dtype=torch.float32) if with_bias else None,
    )
    return out


def decode_inputs(shape: DecodeShape, device="cpu", seed: int = 0, steps: int | None = None):
    """Inputs of ``steps`` recurrent steps.

    x, delta, z: [steps, batch, d_inner] (act dtype); B, C: [steps, batch, N];
    A: [d_inner, N], D, bias: [d_inner] (fp32).
    """
    s = shape.steps if steps is None else steps
    b, d, N, dt_ = shape.batch, shape.d_inner, shape.d_state, shape.dtype
    dtc = _log_uniform((d,), device, seed, "dt")
    return dict(
        x=_normal((s, b, d), device, seed, "x", dt_),
        delta=_normal((s, b, d), device, seed, "delta", dt_),
        z=_normal((s, b, d), device, seed, "z", dt_),
        B=_normal((s, b, N), device, seed, "B", dt_),
        C=_normal((s, b, N), device, seed, "C", dt_),
        A=a_matrix(d, N, device),
        D=_normal((d,), device, seed, "D", torch.float32),
        bias=torch.log(torch.expm1(dtc)),
    )


def random_scan_inputs(batch, d_inner, d_state, seqlen, dtype=torch.bfloat16, device="cpu",
                       seed: int = 0, gate=True, skip=True, with_bias=True, a_kind="s4d"):
    """Arbitrary-shape inputs for edge-case tests, same distributions as the
    workloads; ``a_kind='random'`` draws A = -exp(U[log 0.2, log 8]) instead of
    -(n+1), and a nonzero bias ~ 0.5·N(0,1) is used."""
    shape = ScanShape("custom", batch, d_inner, d_state, seqlen, dtype)
    inp = scan_inputs(shape, device, seed, gate, skip, with_bias=False)
    if a_kind == "random":
        g = _gen(device, seed, 101)
        r = torch.rand((d_inner, d_state), generator=g, device=device)
        inp["A"] = -torch.exp(math.log(0.2) + r * (math.log(8.0) - math.log(0.2)))
    if with_bias:
        g = _gen(device, seed, 102)
        inp["bias"] = 0.5 * torch.randn(d_inner, generator=g, device=device)
    return inp


# Causal Conv1D in front of the scan: width 4 as in Mamba; x, and the carried
# state, ~ N(0, 1) in the activation dtype; weight and bias ~ U(-1/sqrt(W), 1/sqrt(W))
# in fp32 (the usual initial range of a depthwise convolution with W taps).
CONV_WIDTH = 4


def conv_inputs(batch, d_inner, seqlen, width=CONV_WIDTH, dtype=torch.bfloat16, device="cpu", seed: int = 0,
                with_bias=True, with_state=True):
    bound = 1.0 / math.sqrt(width)
    g = _gen(device, seed, 201)
    w = (2.0 * torch.rand((d_inner, width), generator=g, device=device) - 1.0) * bound
    g = _gen(device, seed, 202)
    bias = (2.0 * torch.rand((d_inner,), generator=g, device=device) - 1.0) * bound if with_bias else None
    g = _gen(device, seed, 203)
    x = torch.randn((batch, d_inner, seqlen), generator=g, device=device).to(dtype)
    state = None
    if with_state and width > 1:
        g = _gen(device, seed, 204)
        state = torch.randn((batch, d_inner, width - 1), generator=g, device=device).to(dtype)
    return dict(x=x, w=w, bias=bias, state=state)


def ssd_inputs(shape: SsdShape, device="cpu", seed: int = 0, gate: bool = True, skip: bool = True,
               with_bias: bool = True, bias_scale: float = 0.0):
    """Inputs of one Mamba-2 layer scan: x, z [batch, L, H, P] and B, C [batch, L, G, N]
    (act dtype); dt (Δraw) [batch, L, H] (act dtype); A, D, dt_bias [H] (fp32).
    bias_scale > 0 draws dt_bias ~ bias_scale·N(0, 1) instead of zeros."""
    b, L, H, P, G, N, dt_ = (shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.ngroups,
                             shape.d_state, shape.dtype)
    step = _log_uniform((b, L, H), device, seed, "dt")
    dt = torch.log(torch.expm1(step)).to(dt_)
    del step
    ga = _gen(device, seed, _IDS["A"])
    A = -(1.0 + 15.0 * torch.rand((H,), generator=ga, device=device, dtype=torch.float32))
    bias = None
    if with_bias:
        bias = (bias_scale * _normal((H,), device, seed, "bias", torch.float32) if bias_scale > 0
                else torch.zeros(H, device=device, dtype=torch.float32))
    return dict(
        x=_normal((b, L, H, P), device, seed, "x", dt_),
        dt=dt,
        A=A,
        B=_normal((b, L, G, N), device, seed, "B", dt_),
        C=_normal((b, L, G, N), device, seed, "C", dt_),
        D=_normal((H,), device, seed, "D", torch.float32) if skip else None,
        z=_normal((b, L, H, P), device, seed, "z", dt_) if gate else None,
        dt_bias=bias,
    )


def random_ssd_inputs(batch, seqlen, nheads, headdim, ngroups, d_state, dtype=torch.bfloat16, device="cpu",
                      seed: int = 0, gate=True, skip=True, with_bias=True):
    """ssd_inputs for an arbitrary shape, with dt_bias ~ 0.5·N(0, 1) when present."""
    shape = SsdShape("custom", batch, seqlen, nheads, headdim, ngroups, d_state, dtype)
    return ssd_inputs(shape, device, seed, gate, skip, with_bias, bias_scale=0.5 if with_bias else 0.0)

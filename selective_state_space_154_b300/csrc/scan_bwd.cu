// Backward of the selective scan (d_state ≤ 16) for sm_103a: the gradients of
// ℓ = Σ dout·out with respect to u, Δraw, A, B, C, D, z and the Δ bias, with
// the states recomputed rather than stored (the pages' third hardware-aware
// ingredient: "Mambaとは？Transformer以外の系列モデル", section Selective Scanは
// 選択機構そのものではない).  The chain rule applied is that of the scan's
// definition ("State Space Models（SSM）とMamba" §2.2 離散化; "Mambaとは？…",
// sections 状態空間モデルを一つの式から理解する and Mamba blockのarchitecture):
// per token, with Ā = exp(Δa), φ = expm1(Δa)/a (Δ when a = 0), q = φ B x,
//   dy = dout·silu(z), dz = dout·y·silu'(z), dD += dy x, dx = dy D
//   dh_t += dy C_t, dC_t += dy h_t
//   dB_t += dh_t φ x, dx += dh_t φ B, dΔ += dh_t Ā (a h_{t-1} + B x)
//   da += dh_t (Δ Ā h_{t-1} + B x (Δ Ā − φ)/a), dh_{t-1} = Ā dh_t
//   dΔraw = dΔ·sigmoid(Δraw + bias), dbias += dΔraw.
//
// Organisation: one thread per (batch, channel) row holding its 16 states, a
// CTA of kBwdRows rows of one batch.  Pass one runs the scan forward and saves
// the state every kBwdTok tokens to the workspace.  Pass two walks the
// kBwdTok-token blocks backwards: it reloads the block's starting state,
// recomputes the block's states into shared memory, and runs the adjoint
// recurrence over the block in reverse.  Per-row sums over the states stay in
// the thread; the sums of dB and dC over channels are reduced across the warp
// (reduce-scatter by shuffles), across the CTA's warps in shared memory, and
// added to global memory once per CTA; dA, dD and dbias are accumulated in
// registers over the whole sequence and added once per row.
#include <cstdint>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kBwdRows = 128;  // rows (threads) per CTA
constexpr int kBwdTok = 8;     // tokens per block = checkpoint interval
constexpr int kBwdN = 16;      // states per row held by a thread
constexpr int kWarps = kBwdRows / 32;

struct BwdSmem {
  float a[kBwdRows][kBwdN];                  // A (0 for |A| < 2^-60 and padded states)
  float ia[kBwdRows][kBwdN];                 // 1/A (0 where a is 0)
  float4 hs[kBwdTok + 1][kBwdN / 4][kBwdRows];  // h_{t0-1} .. h_{t0+7}, [step][quad][row]
  float bc[kBwdTok][2][kBwdN];               // B | C of the block's tokens, fp32
  float red[kWarps][kBwdTok][32];            // per-warp sums of the 32 (B|C, n) slots
};

template <typename T>
__device__ __forceinline__ float ldf(const void* base, int64_t i) {
  return Act<T>::to_f(static_cast<const T*>(base)[i]);
}
template <typename T>
__device__ __forceinline__ void stf(void* base, int64_t i, float v) {
  static_cast<T*>(base)[i] = Act<T>::from_f(v);
}

// Stage B and C of tokens [t0, t0 + nv) of batch b into shared memory as fp32.
template <typename T>
__device__ __forceinline__ void stage_bc(BwdSmem& sm, const BwdArgs& p, int64_t b, int64_t t0, int nv) {
  const int N = (int)p.N;
  for (int i = threadIdx.x; i < kBwdTok * 2 * kBwdN; i += kBwdRows) {
    const int v = i / (2 * kBwdN), w = (i / kBwdN) & 1, n = i % kBwdN;
    float val = 0.f;
    if (v < nv && n < N) val = ldf<T>(w ? p.C : p.B, (b * p.L + t0 + v) * N + n);
    sm.bc[v][w][n] = val;
  }
}

// Warp reduce-scatter of 32 values per lane: afterwards v[0] of lane l holds the
// sum over the warp's lanes of slot l (at each step a lane keeps the half of its
// slots named by its own bit and adds the partner's copy of that half).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32]) {
  const unsigned lane = threadIdx.x & 31u;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = up ? v[i] : v[i + off];
      const float keep = up ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

template <typename T>
__global__ void __launch_bounds__(kBwdRows, 2) scan_bwd_kernel(const BwdArgs p) {
  using AT = Act<T>;
  constexpr bool FAST = AT::kFast;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int N = (int)p.N;
  const int64_t L = p.L;
  const int64_t b = blockIdx.x / p.ctiles;
  const int64_t c0 = (int64_t)(blockIdx.x % p.ctiles) * kBwdRows;
  const int nrows = (int)((p.d_inner - c0) < kBwdRows ? (p.d_inner - c0) : kBwdRows);
  const int r = threadIdx.x;
  const bool row_ok = r < nrows;
  const int64_t c = c0 + (row_ok ? r : 0);
  const int64_t row = b * p.d_inner + c;
  const int warp = r >> 5, lane = r & 31;

#pragma unroll
  for (int n = 0; n < kBwdN; ++n) {
    const float av = (row_ok && n < N) ? p.A[c * N + n] : 0.f;
    const bool zero = fabsf(av) < 8.673617e-19f;  // |A| < 2^-60 counts as A = 0
    sm.a[r][n] = zero ? 0.f : av;
    sm.ia[r][n] = zero ? 0.f : 1.f / av;
  }
  const float Dc = (row_ok && p.D) ? p.D[c] : 0.f;
  const float biasc = (row_ok && p.bias) ? p.bias[c] : 0.f;
  const int64_t nblk = p.nblk;
  float* ck = p.ckpt + (size_t)(blockIdx.x * (int64_t)kBwdRows + r) * nblk * kBwdN;  // this row's checkpoints
  __syncthreads();

  // ---------------- pass one: forward, checkpoint every kBwdTok tokens ----------------
  float h[kBwdN];
#pragma unroll
  for (int n = 0; n < kBwdN; ++n) h[n] = 0.f;
  for (int64_t blk = 0; blk < nblk; ++blk) {
    const int64_t t0 = blk * kBwdTok;
    const int nv = (int)(L - t0 < kBwdTok ? L - t0 : kBwdTok);
#pragma unroll
    for (int q = 0; q < kBwdN / 4; ++q)
      reinterpret_cast<float4*>(ck + blk * kBwdN)[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    __syncthreads();  // the previous block's bc is no longer read
    stage_bc<T>(sm, p, b, t0, nv);
    __syncthreads();
    for (int v = 0; v < nv; ++v) {
      const int64_t i = row * L + t0 + v;
      const float x = row_ok ? ldf<T>(p.u, i) : 0.f;
      const float rr = (row_ok ? ldf<T>(p.delta, i) : 0.f) + biasc;
      const float dt = FAST ? softplus_fast(rr) : softplus_precise(rr);
#pragma unroll
      for (int n = 0; n < kBwdN; ++n) {
        const float a = sm.a[r][n], iav = sm.ia[r][n];
        float abar, phi;
        if (a != 0.f) {
          abar = FAST ? ex2_approx(dt * a * kLog2e) : expf(dt * a);
          phi = (FAST ? abar - 1.f : expm1f(dt * a)) * iav;
        } else {
          abar = 1.f;
          phi = dt;
        }
        h[n] = fmaf(abar, h[n], phi * sm.bc[v][0][n] * x);
      }
    }
  }

  // ---------------- pass two: blocks in reverse, adjoint recurrence ----------------
  float dh[kBwdN], dA_acc[kBwdN];
#pragma unroll
  for (int n = 0; n < kBwdN; ++n) dh[n] = dA_acc[n] = 0.f;
  float dD_acc = 0.f, db_acc = 0.f;
  for (int64_t blk = nblk - 1; blk >= 0; --blk) {
    const int64_t t0 = blk * kBwdTok;
    const int nv = (int)(L - t0 < kBwdTok ? L - t0 : kBwdTok);
    __syncthreads();  // bc, hs and red of the previous block are no longer read
    stage_bc<T>(sm, p, b, t0, nv);
    // recompute the block's states from its checkpoint
#pragma unroll
    for (int q = 0; q < kBwdN / 4; ++q) {
      const float4 hv = reinterpret_cast<const float4*>(ck + blk * kBwdN)[q];
      h[4 * q] = hv.x; h[4 * q + 1] = hv.y; h[4 * q + 2] = hv.z; h[4 * q + 3] = hv.w;
      sm.hs[0][q][r] = hv;
    }
    __syncthreads();  // bc staged
    for (int v = 0; v < nv; ++v) {
      const int64_t i = row * L + t0 + v;
      const float x = row_ok ? ldf<T>(p.u, i) : 0.f;
      const float rr = (row_ok ? ldf<T>(p.delta, i) : 0.f) + biasc;
      const float dt = FAST ? softplus_fast(rr) : softplus_precise(rr);
#pragma unroll
      for (int n = 0; n < kBwdN; ++n) {
        const float a = sm.a[r][n], iav = sm.ia[r][n];
        float abar, phi;
        if (a != 0.f) {
          abar = FAST ? ex2_approx(dt * a * kLog2e) : expf(dt * a);
          phi = (FAST ? abar - 1.f : expm1f(dt * a)) * iav;
        } else {
          abar = 1.f;
          phi = dt;
        }
        h[n] = fmaf(abar, h[n], phi * sm.bc[v][0][n] * x);
      }
#pragma unroll
      for (int q = 0; q < kBwdN / 4; ++q)
        sm.hs[v + 1][q][r] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    }
    // adjoint over the block, last token first
    for (int v = nv - 1; v >= 0; --v) {
      const int64_t i = row * L + t0 + v;
      const float x = row_ok ? ldf<T>(p.u, i) : 0.f;
      const float rr = (row_ok ? ldf<T>(p.delta, i) : 0.f) + biasc;
      const float go = row_ok ? ldf<T>(p.dout, i) : 0.f;
      const float dt = FAST ? softplus_fast(rr) : softplus_precise(rr);
      float hv[kBwdN], hp[kBwdN];
#pragma unroll
      for (int q = 0; q < kBwdN / 4; ++q) {
        const float4 a4 = sm.hs[v + 1][q][r], p4 = sm.hs[v][q][r];
        hv[4 * q] = a4.x; hv[4 * q + 1] = a4.y; hv[4 * q + 2] = a4.z; hv[4 * q + 3] = a4.w;
        hp[4 * q] = p4.x; hp[4 * q + 1] = p4.y; hp[4 * q + 2] = p4.z; hp[4 * q + 3] = p4.w;
      }
      float y = Dc * x;
#pragma unroll
      for (int n = 0; n < kBwdN; ++n) y = fmaf(sm.bc[v][1][n], hv[n], y);
      float dy = go;
      if (p.z) {
        const float zv = row_ok ? ldf<T>(p.z, i) : 0.f;
        const float s = FAST ? rcp_approx(1.f + ex2_approx(-zv * kLog2e)) : 1.f / (1.f + expf(-zv));
        dy = go * zv * s;
        if (row_ok) stf<T>(p.dz, i, go * y * s * (1.f + zv * (1.f - s)));
      }
      float dx = dy * Dc;
      dD_acc = fmaf(dy, x, dD_acc);
      float ddt = 0.f;
      float slots[32];  // [0..15] dB, [16..31] dC of this row and token
#pragma unroll
      for (int n = 0; n < kBwdN; ++n) {
        const float a = sm.a[r][n], iav = sm.ia[r][n];
        const float Bn = sm.bc[v][0][n], Cn = sm.bc[v][1][n];
        dh[n] = fmaf(dy, Cn, dh[n]);
        slots[16 + n] = dy * hv[n];
        float abar, phi;
        if (a != 0.f) {
          abar = FAST ? ex2_approx(dt * a * kLog2e) : expf(dt * a);
          phi = (FAST ? abar - 1.f : expm1f(dt * a)) * iav;
        } else {
          abar = 1.f;
          phi = dt;
        }
        const float bx = Bn * x;
        const float g = dh[n];
        slots[n] = g * phi * x;
        dx = fmaf(g * phi, Bn, dx);
        if (a != 0.f) {
          ddt = fmaf(g * abar, fmaf(a, hp[n], bx), ddt);
          dA_acc[n] = fmaf(g, fmaf(dt * abar, hp[n], bx * (dt * abar - phi) * iav), dA_acc[n]);
        } else {
          ddt = fmaf(g, bx, ddt);
          dA_acc[n] = fmaf(g, fmaf(dt, hp[n], 0.5f * bx * dt * dt), dA_acc[n]);
        }
        dh[n] = g * abar;
      }
      const float sig = FAST ? rcp_approx(1.f + ex2_approx(-rr * kLog2e)) : 1.f / (1.f + expf(-rr));
      const float dr = ddt * sig;
      db_acc += dr;
      if (row_ok) {
        stf<T>(p.du, i, dx);
        stf<T>(p.ddelta, i, dr);
      }
      // Σ over the CTA's rows of the 32 (B|C, n) slots: warp reduce-scatter, then shared memory
      sm.red[warp][v][lane] = warp_reduce_scatter32(slots);
    }
    __syncthreads();  // red complete
    for (int s = threadIdx.x; s < nv * 32; s += kBwdRows) {
      const int v = s >> 5, slot = s & 31, n = slot & 15;
      if (n >= N) continue;
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) sum += sm.red[w][v][slot];
      atomicAdd((slot < 16 ? p.dB : p.dC) + (b * L + t0 + v) * N + n, sum);
    }
  }
  if (row_ok) {
#pragma unroll
    for (int n = 0; n < kBwdN; ++n)
      if (n < N) atomicAdd(p.dA + c * N + n, dA_acc[n]);
    if (p.dD) atomicAdd(p.dD + c, dD_acc);
    if (p.dbias) atomicAdd(p.dbias + c, db_acc);
  }
}

template <typename T>
cudaError_t bwd_launch_t(const BwdArgs& p, cudaStream_t s) {
  const cudaError_t e =
      cudaFuncSetAttribute(scan_bwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(BwdSmem));
  if (e != cudaSuccess) return e;
  scan_bwd_kernel<T><<<(unsigned)(p.batch * p.ctiles), kBwdRows, sizeof(BwdSmem), s>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t scan_bwd_workspace_bytes(int64_t batch, int64_t d_inner, int64_t L) {
  const int64_t ctiles = (d_inner + kBwdRows - 1) / kBwdRows;
  const int64_t nblk = (L + kBwdTok - 1) / kBwdTok;
  return (size_t)(batch * ctiles * kBwdRows) * (size_t)nblk * kBwdN * sizeof(float);
}

cudaError_t scan_bwd_launch(BwdArgs p, cudaStream_t stream) {
  p.ctiles = (int)((p.d_inner + kBwdRows - 1) / kBwdRows);
  p.nblk = (p.L + kBwdTok - 1) / kBwdTok;
  return p.act == 1 ? bwd_launch_t<__nv_bfloat16>(p, stream) : bwd_launch_t<float>(p, stream);
}

}  // namespace ssm

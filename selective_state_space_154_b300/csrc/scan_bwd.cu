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
// Organisation: four threads per (batch, channel) row, four states each; a CTA
// holds kBwdRows rows of one batch.  Pass one runs the scan forward and saves
// the state every kBwdTok tokens to the workspace.  Pass two walks the
// kBwdTok-token blocks backwards: it reloads the block's starting state,
// recomputes the block's states into shared memory, and runs the adjoint
// recurrence over the block in reverse.  Per (row, token) scalars (Δ, x, the
// gate terms) are evaluated once per row into shared memory; sums over a row's
// states take two shuffles; the sums of dB and dC over channels are reduced
// across the warp's rows (reduce-scatter by shuffles), across the CTA's warps in
// shared memory, and added to global memory once per CTA; dA, dD and dbias are
// accumulated in registers over the whole sequence and added once per row.
#include <cstdint>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kBwdRows = 64;                    // rows per CTA
constexpr int kBwdTpr = 4;                      // threads per row
constexpr int kBwdG = 4;                        // states per thread
constexpr int kBwdThreads = kBwdRows * kBwdTpr; // 256
constexpr int kBwdTok = 8;                      // tokens per block = checkpoint interval
constexpr int kBwdN = kBwdTpr * kBwdG;          // 16 states per row
constexpr int kWarps = kBwdThreads / 32;

// per (row, token) scalars of a block
struct TokScalars {
  float x;      // u
  float dt;     // Δ = softplus(Δraw + bias)
  float sig;    // sigmoid(Δraw + bias) = dΔ/dΔraw
  float dy;     // dout·silu(z) (dout without a gate)
  float dzf;    // dout·silu'(z): dz = dzf·y
};

struct BwdSmem {
  float4 hs[kBwdTok + 1][kBwdRows][kBwdTpr];  // h_{t0-1} .. h_{t0+7}, [step][row][quad]
  TokScalars ts[kBwdTok][kBwdRows];
  float bc[kBwdTok][2][kBwdN];                // B | C of the block's tokens, fp32
  float red[kWarps][kBwdTok][32];             // per-warp sums of the 32 (B|C, n) slots
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
  for (int i = threadIdx.x; i < kBwdTok * 2 * kBwdN; i += kBwdThreads) {
    const int v = i / (2 * kBwdN), w = (i / kBwdN) & 1, n = i % kBwdN;
    float val = 0.f;
    if (v < nv && n < N) val = ldf<T>(w ? p.C : p.B, (b * p.L + t0 + v) * N + n);
    sm.bc[v][w][n] = val;
  }
}

// The per-token scalars of the block's tokens for this thread's row: thread g of
// the row takes tokens g and g + 4.  Visible to the row's four threads after __syncwarp.
template <typename T>
__device__ __forceinline__ void row_scalars(BwdSmem& sm, const BwdArgs& p, int r, int g, bool row_ok, int64_t row,
                                            int64_t t0, int nv, float biasc, bool with_grad) {
  constexpr bool FAST = Act<T>::kFast;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int v = g + 4 * k;
    if (v >= nv) continue;
    const int64_t i = row * p.L + t0 + v;
    TokScalars s{};
    if (row_ok) {
      s.x = ldf<T>(p.u, i);
      const float rr = ldf<T>(p.delta, i) + biasc;
      s.dt = FAST ? softplus_fast(rr) : softplus_precise(rr);
      if (with_grad) {
        s.sig = FAST ? rcp_approx(1.f + ex2_approx(-rr * kLog2e)) : 1.f / (1.f + expf(-rr));
        const float go = ldf<T>(p.dout, i);
        if (p.z) {
          const float zv = ldf<T>(p.z, i);
          const float sz = FAST ? rcp_approx(1.f + ex2_approx(-zv * kLog2e)) : 1.f / (1.f + expf(-zv));
          s.dy = go * zv * sz;
          s.dzf = go * sz * (1.f + zv * (1.f - sz));
        } else {
          s.dy = go;
          s.dzf = 0.f;
        }
      }
    }
    sm.ts[v][r] = s;
  }
}

// Reduce-scatter over the warp's 8 rows (lane bits 2..4) of 8 values per lane:
// afterwards lane l holds, for its quad g = l & 3, the sum over the rows of
// value (l >> 2).
__device__ __forceinline__ float rows_reduce_scatter8(float (&v)[8]) {
  const unsigned lane = threadIdx.x & 31u;
#pragma unroll
  for (int step = 0; step < 3; ++step) {
    const int half = 4 >> step;             // values kept after this step: 4, 2, 1
    const unsigned bit = 16u >> step;       // lane bit exchanged: 16, 8, 4
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
  }
  return v[0];
}

template <typename T>
__global__ void __launch_bounds__(kBwdThreads, 3) scan_bwd_kernel(const BwdArgs p) {
  using AT = Act<T>;
  constexpr bool FAST = AT::kFast;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int N = (int)p.N;
  const int64_t L = p.L;
  const int64_t b = blockIdx.x / p.ctiles;
  const int64_t c0 = (int64_t)(blockIdx.x % p.ctiles) * kBwdRows;
  const int nrows = (int)((p.d_inner - c0) < kBwdRows ? (p.d_inner - c0) : kBwdRows);
  const int r = threadIdx.x / kBwdTpr, g = threadIdx.x % kBwdTpr;
  const bool row_ok = r < nrows;
  const int64_t c = c0 + (row_ok ? r : 0);
  const int64_t row = b * p.d_inner + c;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // this thread's states n = 4g + k: A and 1/A (0 for |A| < 2^-60 and padded states)
  float a[kBwdG], ia[kBwdG];
#pragma unroll
  for (int k = 0; k < kBwdG; ++k) {
    const int n = kBwdG * g + k;
    const float av = (row_ok && n < N) ? p.A[c * N + n] : 0.f;
    const bool zero = fabsf(av) < 8.673617e-19f;
    a[k] = zero ? 0.f : av;
    ia[k] = zero ? 0.f : 1.f / av;
  }
  const float Dc = (row_ok && p.D) ? p.D[c] : 0.f;
  const float biasc = (row_ok && p.bias) ? p.bias[c] : 0.f;
  const int64_t nblk = p.nblk;
  // this thread's checkpoints: [nblk] float4 (its quad of the row's state)
  float4* ck = reinterpret_cast<float4*>(p.ckpt) + ((int64_t)blockIdx.x * kBwdThreads + threadIdx.x) * nblk;

  // packed path: bf16 arithmetic and no A = 0 state among this thread's four
  const bool packed = FAST && a[0] != 0.f && a[1] != 0.f && a[2] != 0.f && a[3] != 0.f;
  const float2 aP[2] = {make_float2(a[0], a[1]), make_float2(a[2], a[3])};
  const float2 iaP[2] = {make_float2(ia[0], ia[1]), make_float2(ia[2], ia[3])};
  // Ā - 1 and Ā of states (2j, 2j+1) at step size dt (packed path)
  auto disc2 = [&](float dt, int j, float2& abar, float2& phi) {
    const float dl = dt * kLog2e;
    const float2 e = __fmul2_rn(make_float2(dl, dl), aP[j]);
    abar = make_float2(ex2_approx(e.x), ex2_approx(e.y));
    phi = __fmul2_rn(__fadd2_rn(abar, make_float2(-1.f, -1.f)), iaP[j]);
  };
  auto discretise = [&](float dt, int k, float& abar, float& phi) {
    if (a[k] != 0.f) {
      abar = FAST ? ex2_approx(dt * a[k] * kLog2e) : expf(dt * a[k]);
      phi = (FAST ? abar - 1.f : expm1f(dt * a[k])) * ia[k];
    } else {
      abar = 1.f;
      phi = dt;
    }
  };

  // ---------------- pass one: forward, checkpoint every kBwdTok tokens ----------------
  float h[kBwdG] = {0.f, 0.f, 0.f, 0.f};
  for (int64_t blk = 0; blk < nblk; ++blk) {
    const int64_t t0 = blk * kBwdTok;
    const int nv = (int)(L - t0 < kBwdTok ? L - t0 : kBwdTok);
    ck[blk] = make_float4(h[0], h[1], h[2], h[3]);
    __syncthreads();  // the previous block's bc and ts are no longer read
    stage_bc<T>(sm, p, b, t0, nv);
    row_scalars<T>(sm, p, r, g, row_ok, row, t0, nv, biasc, false);
    __syncthreads();
    for (int v = 0; v < nv; ++v) {
      const TokScalars s = sm.ts[v][r];
      if (packed) {
        const float2 xx = make_float2(s.x, s.x);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float2 abar, phi;
          disc2(s.dt, j, abar, phi);
          const float2 bb = *reinterpret_cast<const float2*>(&sm.bc[v][0][kBwdG * g + 2 * j]);
          const float2 hh = __ffma2_rn(abar, make_float2(h[2 * j], h[2 * j + 1]), __fmul2_rn(__fmul2_rn(phi, bb), xx));
          h[2 * j] = hh.x;
          h[2 * j + 1] = hh.y;
        }
      } else {
#pragma unroll
        for (int k = 0; k < kBwdG; ++k) {
          float abar, phi;
          discretise(s.dt, k, abar, phi);
          h[k] = fmaf(abar, h[k], phi * sm.bc[v][0][kBwdG * g + k] * s.x);
        }
      }
    }
  }

  // ---------------- pass two: blocks in reverse, adjoint recurrence ----------------
  float dh[kBwdG] = {0.f, 0.f, 0.f, 0.f}, dA_acc[kBwdG] = {0.f, 0.f, 0.f, 0.f};
  float dD_acc = 0.f, db_acc = 0.f;
  for (int64_t blk = nblk - 1; blk >= 0; --blk) {
    const int64_t t0 = blk * kBwdTok;
    const int nv = (int)(L - t0 < kBwdTok ? L - t0 : kBwdTok);
    __syncthreads();  // bc, ts, hs and red of the previous block are no longer read
    stage_bc<T>(sm, p, b, t0, nv);
    row_scalars<T>(sm, p, r, g, row_ok, row, t0, nv, biasc, true);
    const float4 h0v = ck[blk];
    h[0] = h0v.x; h[1] = h0v.y; h[2] = h0v.z; h[3] = h0v.w;
    sm.hs[0][r][g] = h0v;
    __syncthreads();  // bc and ts staged
    // recompute the block's states
    for (int v = 0; v < nv; ++v) {
      const TokScalars s = sm.ts[v][r];
      if (packed) {
        const float2 xx = make_float2(s.x, s.x);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float2 abar, phi;
          disc2(s.dt, j, abar, phi);
          const float2 bb = *reinterpret_cast<const float2*>(&sm.bc[v][0][kBwdG * g + 2 * j]);
          const float2 hh = __ffma2_rn(abar, make_float2(h[2 * j], h[2 * j + 1]), __fmul2_rn(__fmul2_rn(phi, bb), xx));
          h[2 * j] = hh.x;
          h[2 * j + 1] = hh.y;
        }
      } else {
#pragma unroll
        for (int k = 0; k < kBwdG; ++k) {
          float abar, phi;
          discretise(s.dt, k, abar, phi);
          h[k] = fmaf(abar, h[k], phi * sm.bc[v][0][kBwdG * g + k] * s.x);
        }
      }
      sm.hs[v + 1][r][g] = make_float4(h[0], h[1], h[2], h[3]);
    }
    // adjoint over the block, last token first
    for (int v = nv - 1; v >= 0; --v) {
      const int64_t i = row * L + t0 + v;
      const TokScalars s = sm.ts[v][r];
      const float4 hv4 = sm.hs[v + 1][r][g], hp4 = sm.hs[v][r][g];
      const float hv[kBwdG] = {hv4.x, hv4.y, hv4.z, hv4.w};
      const float hp[kBwdG] = {hp4.x, hp4.y, hp4.z, hp4.w};
      // y = Σ_n C h + D x over the row's four threads
      float y = 0.f;
#pragma unroll
      for (int k = 0; k < kBwdG; ++k) y = fmaf(sm.bc[v][1][kBwdG * g + k], hv[k], y);
      y += __shfl_xor_sync(0xffffffffu, y, 1);
      y += __shfl_xor_sync(0xffffffffu, y, 2);
      y = fmaf(Dc, s.x, y);
      const float dy = s.dy;
      float dx = 0.f, ddt = 0.f;
      float slots[8];  // [0..3] dB, [4..7] dC of this thread's states
      if (packed) {
        const float2 dy2 = make_float2(dy, dy), xx = make_float2(s.x, s.x), dt2 = make_float2(s.dt, s.dt);
        float2 dx2 = make_float2(0.f, 0.f), ddt2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int n = kBwdG * g + 2 * j;
          const float2 Bn = *reinterpret_cast<const float2*>(&sm.bc[v][0][n]);
          const float2 Cn = *reinterpret_cast<const float2*>(&sm.bc[v][1][n]);
          const float2 hv2 = make_float2(hv[2 * j], hv[2 * j + 1]), hp2 = make_float2(hp[2 * j], hp[2 * j + 1]);
          const float2 gk = __ffma2_rn(dy2, Cn, make_float2(dh[2 * j], dh[2 * j + 1]));
          const float2 sc = __fmul2_rn(dy2, hv2);
          float2 abar, phi;
          disc2(s.dt, j, abar, phi);
          const float2 bx = __fmul2_rn(Bn, xx);
          const float2 gphi = __fmul2_rn(gk, phi);
          const float2 sb = __fmul2_rn(gphi, xx);
          dx2 = __ffma2_rn(gphi, Bn, dx2);
          ddt2 = __ffma2_rn(__fmul2_rn(gk, abar), __ffma2_rn(aP[j], hp2, bx), ddt2);
          const float2 dta = __fmul2_rn(dt2, abar);
          const float2 tb = __fmul2_rn(__fmul2_rn(bx, __fadd2_rn(dta, make_float2(-phi.x, -phi.y))), iaP[j]);
          const float2 da = __fmul2_rn(gk, __ffma2_rn(dta, hp2, tb));
          dA_acc[2 * j] += da.x;
          dA_acc[2 * j + 1] += da.y;
          const float2 dhn = __fmul2_rn(gk, abar);
          dh[2 * j] = dhn.x;
          dh[2 * j + 1] = dhn.y;
          slots[2 * j] = sb.x;
          slots[2 * j + 1] = sb.y;
          slots[4 + 2 * j] = sc.x;
          slots[4 + 2 * j + 1] = sc.y;
        }
        dx = dx2.x + dx2.y;
        ddt = ddt2.x + ddt2.y;
      } else
#pragma unroll
      for (int k = 0; k < kBwdG; ++k) {
        const int n = kBwdG * g + k;
        const float Bn = sm.bc[v][0][n], Cn = sm.bc[v][1][n];
        const float gk = fmaf(dy, Cn, dh[k]);  // dℓ/dh_t
        slots[4 + k] = dy * hv[k];
        float abar, phi;
        discretise(s.dt, k, abar, phi);
        const float bx = Bn * s.x;
        slots[k] = gk * phi * s.x;
        dx = fmaf(gk * phi, Bn, dx);
        if (a[k] != 0.f) {
          ddt = fmaf(gk * abar, fmaf(a[k], hp[k], bx), ddt);
          dA_acc[k] = fmaf(gk, fmaf(s.dt * abar, hp[k], bx * (s.dt * abar - phi) * ia[k]), dA_acc[k]);
        } else {
          ddt = fmaf(gk, bx, ddt);
          dA_acc[k] = fmaf(gk, fmaf(s.dt, hp[k], 0.5f * bx * s.dt * s.dt), dA_acc[k]);
        }
        dh[k] = gk * abar;
      }
      dx += __shfl_xor_sync(0xffffffffu, dx, 1);
      dx += __shfl_xor_sync(0xffffffffu, dx, 2);
      ddt += __shfl_xor_sync(0xffffffffu, ddt, 1);
      ddt += __shfl_xor_sync(0xffffffffu, ddt, 2);
      dx = fmaf(dy, Dc, dx);
      const float dr = ddt * s.sig;
      if (g == 0) {
        dD_acc = fmaf(dy, s.x, dD_acc);
        db_acc += dr;
        if (row_ok) {
          stf<T>(p.du, i, dx);
          stf<T>(p.ddelta, i, dr);
          if (p.z) stf<T>(p.dz, i, s.dzf * y);
        }
      }
      // Σ over the CTA's rows of the 32 (B|C, n) slots: warp reduce-scatter, then shared memory
      sm.red[warp][v][lane] = rows_reduce_scatter8(slots);
    }
    __syncthreads();  // red complete
    for (int sidx = threadIdx.x; sidx < nv * 32; sidx += kBwdThreads) {
      const int v = sidx >> 5, l = sidx & 31;
      const int qg = l & 3, slot = l >> 2;               // lane l held quad qg, value slot
      const int n = kBwdG * qg + (slot & 3);
      if (n >= N) continue;
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) sum += sm.red[w][v][l];
      atomicAdd((slot < 4 ? p.dB : p.dC) + (b * L + t0 + v) * N + n, sum);
    }
  }
  if (row_ok) {
#pragma unroll
    for (int k = 0; k < kBwdG; ++k) {
      const int n = kBwdG * g + k;
      if (n < N) atomicAdd(p.dA + c * N + n, dA_acc[k]);
    }
    if (g == 0) {
      if (p.dD) atomicAdd(p.dD + c, dD_acc);
      if (p.dbias) atomicAdd(p.dbias + c, db_acc);
    }
  }
}

template <typename T>
cudaError_t bwd_launch_t(const BwdArgs& p, cudaStream_t s) {
  const cudaError_t e =
      cudaFuncSetAttribute(scan_bwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(BwdSmem));
  if (e != cudaSuccess) return e;
  scan_bwd_kernel<T><<<(unsigned)(p.batch * p.ctiles), kBwdThreads, sizeof(BwdSmem), s>>>(p);
  return cudaGetLastError();
}

}  // namespace

int scan_bwd_rows_per_cta() { return kBwdRows; }

size_t scan_bwd_workspace_bytes(int64_t batch, int64_t d_inner, int64_t L) {
  const int64_t ctiles = (d_inner + kBwdRows - 1) / kBwdRows;
  const int64_t nblk = (L + kBwdTok - 1) / kBwdTok;
  return (size_t)(batch * ctiles * kBwdThreads) * (size_t)nblk * sizeof(float4);
}

cudaError_t scan_bwd_launch(BwdArgs p, cudaStream_t stream) {
  p.ctiles = (int)((p.d_inner + kBwdRows - 1) / kBwdRows);
  p.nblk = (p.L + kBwdTok - 1) / kBwdTok;
  return p.act == 1 ? bwd_launch_t<__nv_bfloat16>(p, stream) : bwd_launch_t<float>(p, stream);
}

}  // namespace ssm

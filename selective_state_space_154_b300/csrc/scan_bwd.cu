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
// Organisation: a CTA holds kBwdRows rows of one batch and one chunk of the sequence,
// so that the grid is (row tiles) × (chunks) and short batches still fill the GPU;
// four threads per (batch, channel) row, four states each, in general, and one
// thread per row for bf16 rows of 16 states (the kernels further below, which keep
// the same workspace layout).  Two launches, neither waiting on another CTA:
//   1. scan_bwd_chunk_kernel runs each chunk forward from h = 0 and saves, every
//      kBwdTok tokens, that local state and the Δ summed since the chunk's start;
//      at the chunk's end it saves the local end state, the chunk's ΣΔ and the
//      adjoint the chunk sends to its left neighbour when nothing comes in from
//      its right, Σ_t (Π_{s≤t} Ā_s) dy_t C_t (the adjoint is linear in what
//      comes in and needs no state, so it can be summed in forward order).
//   2. scan_bwd_kernel first combines the chunks' summaries: the true state
//      entering its chunk, h_in = Σ_{j<k} (Π_{j<i<k} e^{a S_i}) H_j, and the true
//      adjoint entering from the right.  It then walks its chunk's kBwdTok-token
//      blocks backwards: it rebuilds the block's starting state as
//      local + e^{a ΣΔ} h_in, recomputes the block's states into shared memory,
//      and runs the adjoint recurrence over the block in reverse.
// Per (row, token) scalars (Δ, x, the gate terms) are evaluated once per row
// into shared memory; sums over a row's states take two shuffles; the sums of
// dB and dC over channels are reduced across the warp's rows (reduce-scatter by
// shuffles), across the CTA's warps in shared memory, and added to global memory
// once per CTA; dA, dD and dbias are accumulated in registers over the chunk and
// added once per row and chunk.
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
constexpr int kBwdMaxChunks = 32;               // chunk summaries kept per row tile
constexpr int64_t kBwdMinChunkBlocks = 2;       // a chunk spans at least 16 tokens

// chunks the workspace provides for nblk blocks of kBwdTok tokens
__host__ __device__ constexpr int64_t bwd_max_chunks(int64_t nblk) {
  return nblk / kBwdMinChunkBlocks < 1 ? 1 : (nblk / kBwdMinChunkBlocks > kBwdMaxChunks ? kBwdMaxChunks
                                                                                           : nblk / kBwdMinChunkBlocks);
}

// The workspace, per row tile rt (batch-major, then channel tile):
//   ck   [rt][nblk][kBwdThreads] float4  chunk-local state at each block's start
//   scum [rt][nblk][kBwdRows]    float   ΣΔ from the chunk's start to the block's
//   hend [rt][kmax][kBwdThreads] float4  chunk-local state after the chunk
//   gcar [rt][kmax][kBwdThreads] float4  adjoint sent left with none coming in
//   stot [rt][kmax][kBwdRows]    float   the chunk's ΣΔ
struct BwdWs {
  float4* ck;
  float* scum;
  float4* hend;
  float4* gcar;
  float* stot;
};

// per (row, token) scalars of a block
struct TokScalars {
  float x;      // u
  float dt;     // Δ = softplus(Δraw + bias)
  float sig;    // sigmoid(Δraw + bias) = dΔ/dΔraw
  float dy;     // dout·silu(z) (dout without a gate)
  float dzf;    // dout·silu'(z): dz = dzf·y
};

// The per-block staging both kernels share, followed (second kernel) by the
// recomputed states and the partial sums of dB and dC.
struct StageSmem {
  TokScalars ts[kBwdTok][kBwdRows];
  float bc[kBwdTok][2][kBwdN];                // B | C of the block's tokens, fp32
};
struct BwdSmem {
  StageSmem st;
  float4 hs[kBwdTok + 1][kBwdRows][kBwdTpr];  // h_{t0-1} .. h_{t0+7}, [step][row][quad]
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
__device__ __forceinline__ void stage_bc(StageSmem& sm, const BwdArgs& p, int64_t b, int64_t t0, int nv) {
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
__device__ __forceinline__ void row_scalars(StageSmem& sm, const BwdArgs& p, int r, int g, bool row_ok, int64_t row,
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

// The next block's raw inputs, copied by cp.async while the current block computes
// (bf16, d_state 16, rows of 16-byte aligned 8-token pieces: L % 8 == 0); the block's
// scalars are then formed from shared memory instead of waiting on global loads.
struct RawBlock {
  uint4 act[4][kBwdRows];   // u, Δraw, dout, z: a row's 8 tokens (bf16)
  uint4 bc[2][16];          // B, C: 8 tokens × 16 states (bf16)
  float4 ck[kBwdThreads];   // the block's chunk-local starting state (gradient kernel)
  float scum[kBwdRows];     // ΣΔ from the chunk's start to the block (gradient kernel)
};

__device__ __forceinline__ void raw_issue(RawBlock& rb, const BwdArgs& p, const BwdWs& w, int64_t b, int64_t c0,
                                          int64_t rt, int64_t blk, bool with_grad, bool with_ck) {
  const int64_t t0 = blk * kBwdTok;
  const int tid = threadIdx.x;
  {  // 4 tensors × 64 rows: one 16-byte piece per thread
    const int wt = tid / kBwdRows, rr = tid % kBwdRows;
    const void* base = wt == 0 ? p.u : (wt == 1 ? p.delta : (wt == 2 ? p.dout : p.z));
    const int64_t c = c0 + rr;
    const bool ok = c < p.d_inner && base != nullptr && (wt < 2 || with_grad);
    const __nv_bfloat16* src =
        static_cast<const __nv_bfloat16*>(ok ? base : p.u) + (ok ? (b * p.d_inner + c) * p.L + t0 : 0);
    cp_async16(&rb.act[wt][rr], src, ok ? 16 : 0);
  }
  if (tid < 32) {  // B and C: 256 bytes each
    const int wt = tid / 16, qq = tid % 16;
    cp_async16(&rb.bc[wt][qq], static_cast<const __nv_bfloat16*>(wt ? p.C : p.B) + (b * p.L + t0) * kBwdN + qq * 8,
               16);
  }
  if (with_ck) {
    const int64_t slot = rt * p.nblk + blk;
    cp_async16(&rb.ck[tid], w.ck + slot * kBwdThreads + tid, 16);
    if (tid < kBwdRows / 4) cp_async16(&rb.scum[tid * 4], w.scum + slot * kBwdRows + tid * 4, 16);
  }
}

// stage_bc and row_scalars from a raw copy (bf16, full blocks)
__device__ __forceinline__ void stage_bc_raw(StageSmem& sm, const RawBlock& rb) {
  for (int i = threadIdx.x; i < kBwdTok * 2 * kBwdN; i += kBwdThreads) {
    const int v = i / (2 * kBwdN), wt = (i / kBwdN) & 1, n = i % kBwdN;
    sm.bc[v][wt][n] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(rb.bc[wt])[v * kBwdN + n]);
  }
}
__device__ __forceinline__ void row_scalars_raw(StageSmem& sm, const RawBlock& rb, const BwdArgs& p, int r, int g,
                                                bool row_ok, float biasc, bool with_grad) {
  const __nv_bfloat16* U = reinterpret_cast<const __nv_bfloat16*>(&rb.act[0][r]);
  const __nv_bfloat16* Dr = reinterpret_cast<const __nv_bfloat16*>(&rb.act[1][r]);
  const __nv_bfloat16* Go = reinterpret_cast<const __nv_bfloat16*>(&rb.act[2][r]);
  const __nv_bfloat16* Z = reinterpret_cast<const __nv_bfloat16*>(&rb.act[3][r]);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int v = g + 4 * k;
    TokScalars s{};
    if (row_ok) {
      s.x = __bfloat162float(U[v]);
      const float rr = __bfloat162float(Dr[v]) + biasc;
      s.dt = softplus_fast(rr);
      if (with_grad) {
        s.sig = rcp_approx(1.f + ex2_approx(-rr * kLog2e));
        const float go = __bfloat162float(Go[v]);
        if (p.z) {
          const float zv = __bfloat162float(Z[v]);
          const float sz = rcp_approx(1.f + ex2_approx(-zv * kLog2e));
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

// A thread's four states n = 4g + k of its row: A and 1/A (both 0 for |A| < 2^-60
// and for padded states), their pairs for packed f32x2 arithmetic, and whether
// the packed path applies (bf16 arithmetic and no A = 0 state among the four).
struct Quad {
  float a[kBwdG], ia[kBwdG];
  float2 aP[2], iaP[2];
  bool packed;
};

template <bool FAST>
__device__ __forceinline__ Quad load_quad(const float* A, int64_t c, int g, int N, bool row_ok) {
  Quad q;
#pragma unroll
  for (int k = 0; k < kBwdG; ++k) {
    const int n = kBwdG * g + k;
    const float av = (row_ok && n < N) ? A[c * N + n] : 0.f;
    const bool zero = fabsf(av) < 8.673617e-19f;
    q.a[k] = zero ? 0.f : av;
    q.ia[k] = zero ? 0.f : 1.f / av;
  }
  q.packed = FAST && q.a[0] != 0.f && q.a[1] != 0.f && q.a[2] != 0.f && q.a[3] != 0.f;
  q.aP[0] = make_float2(q.a[0], q.a[1]);
  q.aP[1] = make_float2(q.a[2], q.a[3]);
  q.iaP[0] = make_float2(q.ia[0], q.ia[1]);
  q.iaP[1] = make_float2(q.ia[2], q.ia[3]);
  return q;
}

// Ā = e^{Δa} and φ = (Ā − 1)/a (Δ for a = 0) of state k
template <bool FAST>
__device__ __forceinline__ void discretise(const Quad& q, float dt, int k, float& abar, float& phi) {
  if (q.a[k] != 0.f) {
    abar = FAST ? ex2_approx(dt * q.a[k] * kLog2e) : expf(dt * q.a[k]);
    phi = (FAST ? abar - 1.f : expm1f(dt * q.a[k])) * q.ia[k];
  } else {
    abar = 1.f;
    phi = dt;
  }
}
// the same for states (2j, 2j+1) on the packed path
__device__ __forceinline__ void disc2(const Quad& q, float dt, int j, float2& abar, float2& phi) {
  const float dl = dt * kLog2e;
  const float2 e = __fmul2_rn(make_float2(dl, dl), q.aP[j]);
  abar = make_float2(ex2_approx(e.x), ex2_approx(e.y));
  phi = __fmul2_rn(__fadd2_rn(abar, make_float2(-1.f, -1.f)), q.iaP[j]);
}

// e^{a S} for the four states (the decay over a stretch whose Δ sum to S)
template <bool FAST>
__device__ __forceinline__ void decay4(const Quad& q, float S, float (&e)[kBwdG]) {
#pragma unroll
  for (int k = 0; k < kBwdG; ++k) e[k] = FAST ? ex2_approx(q.a[k] * S * kLog2e) : expf(q.a[k] * S);
}

// One token of the recurrence h ← Ā h + φ B x for the thread's four states
// (bq: their four B values); abar receives Ā.
template <bool FAST>
__device__ __forceinline__ void fwd_token(const Quad& q, float (&h)[kBwdG], float (&abar)[kBwdG], float dt, float x,
                                          const float* bq) {
  if (q.packed) {
    const float2 xx = make_float2(x, x);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float2 ab, phi;
      disc2(q, dt, j, ab, phi);
      const float2 bb = *reinterpret_cast<const float2*>(bq + 2 * j);
      const float2 hh = __ffma2_rn(ab, make_float2(h[2 * j], h[2 * j + 1]), __fmul2_rn(__fmul2_rn(phi, bb), xx));
      h[2 * j] = hh.x;
      h[2 * j + 1] = hh.y;
      abar[2 * j] = ab.x;
      abar[2 * j + 1] = ab.y;
    }
  } else {
#pragma unroll
    for (int k = 0; k < kBwdG; ++k) {
      float phi;
      discretise<FAST>(q, dt, k, abar[k], phi);
      h[k] = fmaf(abar[k], h[k], phi * bq[k] * x);
    }
  }
}

// Where this CTA sits: row tile blockIdx.x (batch-major), chunk blockIdx.y.
struct CtaPos {
  int64_t rt, b, c, row, blk0, blk1;
  int chunk, r, g;
  bool row_ok;
};
__device__ __forceinline__ CtaPos cta_pos(const BwdArgs& p) {
  CtaPos o;
  o.rt = blockIdx.x;
  o.chunk = (int)blockIdx.y;
  o.b = o.rt / p.ctiles;
  const int64_t c0 = (o.rt % p.ctiles) * kBwdRows;
  const int nrows = (int)((p.d_inner - c0) < kBwdRows ? (p.d_inner - c0) : kBwdRows);
  o.r = threadIdx.x / kBwdTpr;
  o.g = threadIdx.x % kBwdTpr;
  o.row_ok = o.r < nrows;
  o.c = c0 + (o.row_ok ? o.r : 0);
  o.row = o.b * p.d_inner + o.c;
  o.blk0 = o.chunk * p.cblk;
  o.blk1 = o.blk0 + p.cblk < p.nblk ? o.blk0 + p.cblk : p.nblk;
  return o;
}

// Launch 1: each chunk forward from h = 0, saving the local states, the prefix
// sums of Δ and the chunk's summary (end state, ΣΔ, adjoint sent left).
template <typename T, bool PF>
__global__ void __launch_bounds__(kBwdThreads, 4) scan_bwd_chunk_kernel(const BwdArgs p, const BwdWs w) {
  constexpr bool FAST = Act<T>::kFast;
  __shared__ StageSmem sm;
  __shared__ RawBlock raw[PF ? 2 : 1];
  const CtaPos o = cta_pos(p);
  const int r = o.r, g = o.g;
  const Quad q = load_quad<FAST>(p.A, o.c, g, (int)p.N, o.row_ok);
  const float biasc = (o.row_ok && p.bias) ? p.bias[o.c] : 0.f;
  const bool want_g = o.chunk > 0;  // chunk 0 sends no adjoint further left
  float h[kBwdG] = {0.f, 0.f, 0.f, 0.f}, P[kBwdG] = {1.f, 1.f, 1.f, 1.f}, G[kBwdG] = {0.f, 0.f, 0.f, 0.f};
  float S = 0.f;
  const int64_t c0 = (o.rt % p.ctiles) * kBwdRows;
  if (PF && o.blk0 < o.blk1) {
    raw_issue(raw[0], p, w, o.b, c0, o.rt, o.blk0, want_g, false);
    cp_async_commit();
  }
  for (int64_t blk = o.blk0; blk < o.blk1; ++blk) {
    const int64_t t0 = blk * kBwdTok;
    const int nv = (int)(p.L - t0 < kBwdTok ? p.L - t0 : kBwdTok);
    const int64_t slot = o.rt * p.nblk + blk;
    w.ck[slot * kBwdThreads + threadIdx.x] = make_float4(h[0], h[1], h[2], h[3]);
    if (g == 0) w.scum[slot * kBwdRows + r] = S;
    __syncthreads();  // the previous block's staging is no longer read
    if (PF) {
      const int i = (int)(blk - o.blk0);
      if (blk + 1 < o.blk1) raw_issue(raw[(i + 1) & 1], p, w, o.b, c0, o.rt, blk + 1, want_g, false);
      cp_async_commit();
      cp_async_wait<1>();  // this block's copies (the next block's may still be in flight)
      __syncthreads();
      stage_bc_raw(sm, raw[i & 1]);
      row_scalars_raw(sm, raw[i & 1], p, r, g, o.row_ok, biasc, want_g);
    } else {
      stage_bc<T>(sm, p, o.b, t0, nv);
      row_scalars<T>(sm, p, r, g, o.row_ok, o.row, t0, nv, biasc, want_g);
    }
    __syncthreads();
    auto token = [&](int v) {
      const TokScalars s = sm.ts[v][r];
      float ab[kBwdG];
      fwd_token<FAST>(q, h, ab, s.dt, s.x, &sm.bc[v][0][kBwdG * g]);
      if (want_g) {
        // P = Π Ā over the chunk so far; G += P dy C
        const float* cq = &sm.bc[v][1][kBwdG * g];
        if (q.packed) {
          const float2 dy2 = make_float2(s.dy, s.dy);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float2 pp = __fmul2_rn(make_float2(P[2 * j], P[2 * j + 1]), make_float2(ab[2 * j], ab[2 * j + 1]));
            const float2 cc = *reinterpret_cast<const float2*>(cq + 2 * j);
            const float2 gg = __ffma2_rn(pp, __fmul2_rn(dy2, cc), make_float2(G[2 * j], G[2 * j + 1]));
            P[2 * j] = pp.x;
            P[2 * j + 1] = pp.y;
            G[2 * j] = gg.x;
            G[2 * j + 1] = gg.y;
          }
        } else {
#pragma unroll
          for (int k = 0; k < kBwdG; ++k) {
            P[k] *= ab[k];
            G[k] = fmaf(P[k], s.dy * cq[k], G[k]);
          }
        }
      }
      S += s.dt;
    };
    if (nv == kBwdTok) {  // full blocks: unrolled, shared-memory offsets fixed at compile time
#pragma unroll
      for (int v = 0; v < kBwdTok; ++v) token(v);
    } else {
      for (int v = 0; v < nv; ++v) token(v);
    }
  }
  const int64_t cs = o.rt * p.kmax + o.chunk;
  w.hend[cs * kBwdThreads + threadIdx.x] = make_float4(h[0], h[1], h[2], h[3]);
  w.gcar[cs * kBwdThreads + threadIdx.x] = make_float4(G[0], G[1], G[2], G[3]);
  if (g == 0) w.stot[cs * kBwdRows + r] = S;
}

// Launch 2: the gradients over one chunk, from the combined chunk summaries.
template <typename T, bool PF>
__global__ void __launch_bounds__(kBwdThreads, 3) scan_bwd_kernel(const BwdArgs p, const BwdWs w) {
  constexpr bool FAST = Act<T>::kFast;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  RawBlock* raw = reinterpret_cast<RawBlock*>(smem_raw + sizeof(BwdSmem));  // [2] when PF
  const int N = (int)p.N;
  const int64_t L = p.L;
  const CtaPos o = cta_pos(p);
  const int r = o.r, g = o.g;
  const bool row_ok = o.row_ok;
  const int64_t b = o.b, c = o.c, row = o.row;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Quad q = load_quad<FAST>(p.A, c, g, N, row_ok);
  const float Dc = (row_ok && p.D) ? p.D[c] : 0.f;
  const float biasc = (row_ok && p.bias) ? p.bias[c] : 0.f;

  // the state entering the chunk and the adjoint entering it from the right
  float hin[kBwdG] = {0.f, 0.f, 0.f, 0.f}, dh[kBwdG] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < o.chunk; ++j) {
    const int64_t cs = o.rt * p.kmax + j;
    const float4 H = w.hend[cs * kBwdThreads + threadIdx.x];
    float e[kBwdG];
    decay4<FAST>(q, w.stot[cs * kBwdRows + r], e);
    hin[0] = fmaf(e[0], hin[0], H.x);
    hin[1] = fmaf(e[1], hin[1], H.y);
    hin[2] = fmaf(e[2], hin[2], H.z);
    hin[3] = fmaf(e[3], hin[3], H.w);
  }
  for (int j = p.nchunks - 1; j > o.chunk; --j) {
    const int64_t cs = o.rt * p.kmax + j;
    const float4 Gj = w.gcar[cs * kBwdThreads + threadIdx.x];
    float e[kBwdG];
    decay4<FAST>(q, w.stot[cs * kBwdRows + r], e);
    dh[0] = fmaf(e[0], dh[0], Gj.x);
    dh[1] = fmaf(e[1], dh[1], Gj.y);
    dh[2] = fmaf(e[2], dh[2], Gj.z);
    dh[3] = fmaf(e[3], dh[3], Gj.w);
  }

  // blocks in reverse, adjoint recurrence
  float h[kBwdG], dA_acc[kBwdG] = {0.f, 0.f, 0.f, 0.f};
  float dD_acc = 0.f, db_acc = 0.f;
  const int64_t c0 = (o.rt % p.ctiles) * kBwdRows;
  if (PF && o.blk0 < o.blk1) {
    raw_issue(raw[0], p, w, b, c0, o.rt, o.blk1 - 1, true, true);
    cp_async_commit();
  }
  for (int64_t blk = o.blk1 - 1; blk >= o.blk0; --blk) {
    const int64_t t0 = blk * kBwdTok;
    const int nv = (int)(L - t0 < kBwdTok ? L - t0 : kBwdTok);
    const int64_t slot = o.rt * p.nblk + blk;
    __syncthreads();  // bc, ts, hs and red of the previous block are no longer read
    float4 h0v;
    float scum;
    if (PF) {
      const int i = (int)(o.blk1 - 1 - blk);
      if (blk - 1 >= o.blk0) raw_issue(raw[(i + 1) & 1], p, w, b, c0, o.rt, blk - 1, true, true);
      cp_async_commit();
      cp_async_wait<1>();  // this block's copies (the next block's may still be in flight)
      __syncthreads();
      stage_bc_raw(sm.st, raw[i & 1]);
      row_scalars_raw(sm.st, raw[i & 1], p, r, g, row_ok, biasc, true);
      h0v = raw[i & 1].ck[threadIdx.x];
      scum = raw[i & 1].scum[r];
    } else {
      stage_bc<T>(sm.st, p, b, t0, nv);
      row_scalars<T>(sm.st, p, r, g, row_ok, row, t0, nv, biasc, true);
      h0v = w.ck[slot * kBwdThreads + threadIdx.x];
      scum = w.scum[slot * kBwdRows + r];
    }
    // the block's starting state: chunk-local + decay since the chunk's start × h_in
    if (o.chunk > 0) {
      float e[kBwdG];
      decay4<FAST>(q, scum, e);
      h0v.x = fmaf(e[0], hin[0], h0v.x);
      h0v.y = fmaf(e[1], hin[1], h0v.y);
      h0v.z = fmaf(e[2], hin[2], h0v.z);
      h0v.w = fmaf(e[3], hin[3], h0v.w);
    }
    h[0] = h0v.x; h[1] = h0v.y; h[2] = h0v.z; h[3] = h0v.w;
    sm.hs[0][r][g] = h0v;
    __syncthreads();  // bc and ts staged
    // recompute the block's states
    auto recompute = [&](int v) {
      const TokScalars s = sm.st.ts[v][r];
      float ab[kBwdG];
      fwd_token<FAST>(q, h, ab, s.dt, s.x, &sm.st.bc[v][0][kBwdG * g]);
      sm.hs[v + 1][r][g] = make_float4(h[0], h[1], h[2], h[3]);
    };
    if (nv == kBwdTok) {  // full blocks: unrolled, shared-memory offsets fixed at compile time
#pragma unroll
      for (int v = 0; v < kBwdTok; ++v) recompute(v);
    } else {
      for (int v = 0; v < nv; ++v) recompute(v);
    }
    // adjoint over the block, last token first
    auto adjoint = [&](int v) {
      const TokScalars s = sm.st.ts[v][r];
      const float4 hv4 = sm.hs[v + 1][r][g], hp4 = sm.hs[v][r][g];
      const float hv[kBwdG] = {hv4.x, hv4.y, hv4.z, hv4.w};
      const float hp[kBwdG] = {hp4.x, hp4.y, hp4.z, hp4.w};
      const float(&bcv)[2][kBwdN] = sm.st.bc[v];
      // y = Σ_n C h + D x over the row's four threads
      float y = 0.f;
#pragma unroll
      for (int k = 0; k < kBwdG; ++k) y = fmaf(bcv[1][kBwdG * g + k], hv[k], y);
      y += __shfl_xor_sync(0xffffffffu, y, 1);
      y += __shfl_xor_sync(0xffffffffu, y, 2);
      y = fmaf(Dc, s.x, y);
      const float dy = s.dy;
      float dx = 0.f, ddt = 0.f;
      float slots[8];  // [0..3] dB, [4..7] dC of this thread's states
      if (q.packed) {
        const float2 dy2 = make_float2(dy, dy), xx = make_float2(s.x, s.x), dt2 = make_float2(s.dt, s.dt);
        float2 dx2 = make_float2(0.f, 0.f), ddt2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int n = kBwdG * g + 2 * j;
          const float2 Bn = *reinterpret_cast<const float2*>(&bcv[0][n]);
          const float2 Cn = *reinterpret_cast<const float2*>(&bcv[1][n]);
          const float2 hv2 = make_float2(hv[2 * j], hv[2 * j + 1]), hp2 = make_float2(hp[2 * j], hp[2 * j + 1]);
          const float2 gk = __ffma2_rn(dy2, Cn, make_float2(dh[2 * j], dh[2 * j + 1]));
          const float2 sc = __fmul2_rn(dy2, hv2);
          float2 abar, phi;
          disc2(q, s.dt, j, abar, phi);
          const float2 bx = __fmul2_rn(Bn, xx);
          const float2 gphi = __fmul2_rn(gk, phi);
          const float2 sb = __fmul2_rn(gphi, xx);
          dx2 = __ffma2_rn(gphi, Bn, dx2);
          ddt2 = __ffma2_rn(__fmul2_rn(gk, abar), __ffma2_rn(q.aP[j], hp2, bx), ddt2);
          const float2 dta = __fmul2_rn(dt2, abar);
          const float2 tb = __fmul2_rn(__fmul2_rn(bx, __fadd2_rn(dta, make_float2(-phi.x, -phi.y))), q.iaP[j]);
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
        const float Bn = bcv[0][n], Cn = bcv[1][n];
        const float gk = fmaf(dy, Cn, dh[k]);  // dℓ/dh_t
        slots[4 + k] = dy * hv[k];
        float abar, phi;
        discretise<FAST>(q, s.dt, k, abar, phi);
        const float bx = Bn * s.x;
        slots[k] = gk * phi * s.x;
        dx = fmaf(gk * phi, Bn, dx);
        if (q.a[k] != 0.f) {
          ddt = fmaf(gk * abar, fmaf(q.a[k], hp[k], bx), ddt);
          dA_acc[k] = fmaf(gk, fmaf(s.dt * abar, hp[k], bx * (s.dt * abar - phi) * q.ia[k]), dA_acc[k]);
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
        // the token's du, Δraw gradient and dz wait in this thread's slot of h_t, which no
        // later (earlier-in-time) token reads, until the block's end
        sm.hs[v + 1][r][0] = make_float4(dx, dr, s.dzf * y, 0.f);
      }
      // Σ over the CTA's rows of the 32 (B|C, n) slots: warp reduce-scatter, then shared memory
      sm.red[warp][v][lane] = rows_reduce_scatter8(slots);
    };
    if (nv == kBwdTok) {
#pragma unroll
      for (int v = kBwdTok - 1; v >= 0; --v) adjoint(v);
    } else {
      for (int v = nv - 1; v >= 0; --v) adjoint(v);
    }
    __syncwarp();  // the row's staged outputs are visible to its four threads
    if (row_ok && g < (p.z ? 3 : 2)) {  // thread g stores the block's tokens of du, dΔraw, dz
      T* d = static_cast<T*>(g == 0 ? p.du : (g == 1 ? p.ddelta : p.dz)) + row * L + t0;
      auto staged = [&](int v) {
        const float4 t4 = sm.hs[v + 1][r][0];
        return g == 0 ? t4.x : (g == 1 ? t4.y : t4.z);
      };
      if (nv == kBwdTok && (reinterpret_cast<uintptr_t>(d) & 15u) == 0) {
        float ov[kBwdTok];
#pragma unroll
        for (int v = 0; v < kBwdTok; ++v) ov[v] = staged(v);
        if (sizeof(T) == 2) {
          uint4 pk;
          unsigned* pw = &pk.x;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 t = __floats2bfloat162_rn(ov[2 * j], ov[2 * j + 1]);
            pw[j] = *reinterpret_cast<unsigned*>(&t);
          }
          *reinterpret_cast<uint4*>(d) = pk;
        } else {
          float4* d4 = reinterpret_cast<float4*>(d);
          d4[0] = make_float4(ov[0], ov[1], ov[2], ov[3]);
          d4[1] = make_float4(ov[4], ov[5], ov[6], ov[7]);
        }
      } else {
        for (int v = 0; v < nv; ++v) stf<T>(d, v, staged(v));
      }
    }
    __syncthreads();  // red complete
    for (int sidx = threadIdx.x; sidx < nv * 32; sidx += kBwdThreads) {
      const int v = sidx >> 5, l = sidx & 31;
      const int qg = l & 3, slot_id = l >> 2;            // lane l held quad qg, value slot_id
      const int n = kBwdG * qg + (slot_id & 3);
      if (n >= N) continue;
      float sum = 0.f;
#pragma unroll
      for (int wi = 0; wi < kWarps; ++wi) sum += sm.red[wi][v][l];
      const int w = slot_id < 4 ? 0 : 1;
      if (p.det)  // this CTA's channel tile's share, summed over the tiles by the reduce launch
        p.part_bc[(((o.rt % p.ctiles) * p.batch + b) * L + t0 + v) * 2 * N + w * N + n] = sum;
      else
        atomicAdd((w ? p.dC : p.dB) + (b * L + t0 + v) * N + n, sum);
    }
  }
  if (row_ok && p.det) {
    float* pr = p.part_row + ((b * p.nchunks + o.chunk) * p.d_inner + c) * (N + 2);
#pragma unroll
    for (int k = 0; k < kBwdG; ++k) {
      const int n = kBwdG * g + k;
      if (n < N) pr[n] = dA_acc[k];
    }
    if (g == 0) {
      pr[N] = dD_acc;
      pr[N + 1] = db_acc;
    }
  } else if (row_ok) {
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

// ---------------------------------------------------------------------------
// The gradient pass with one thread per row (bf16, d_state 16, L % 8 == 0, 16-byte
// aligned rows): a thread holds all 16 states of its row, so the readout and the sums
// over states stay in registers, and the state arithmetic runs on packed f32x2 pairs.
// A CTA is the same 64-row tile as above (two warps), over one chunk, reading the same
// checkpoints and chunk summaries.
//  * Per 8-token block: the block's raw inputs arrive by cp.async into one buffer,
//    which is refilled with the next block's as soon as they are converted (the
//    per-token scalars of each row to shared memory); the forward is recomputed from
//    the block's starting state, each h_{t-1} kept in shared memory ([token][quad][row],
//    conflict-free); the adjoint then runs over the block in reverse.
//  * dA uses a·∂h/∂a = Δ·∂h/∂Δ − φ B x (a ≠ 0): per state one sum over the chunk,
//    Σ [Δ dh Ā (a h_{t-1} + B x) − dh φ x · B x], which times 1/a is the same
//    Σ dh (Δ Ā h_{t-1} + B x (Δ Ā − φ)/a) as the general form, with 1/a factored out of
//    the time sum.  The fast path carries −1/a, so that the terms with −φ come out of
//    fused multiply-adds.  A CTA with an A = 0 state takes the general form per state
//    (PRECISE).
//  * dB and dC, sums over the rows: each thread writes its 32 (B | C, n) terms of a
//    token to a [32 rows][32] tile (16-byte groups XOR-swizzled by row, so that the 8
//    lanes of each 128-bit access hit distinct banks); lane j sums 8 rows × 4 terms
//    from it, and two exchanges over lane bits 4 and 3 finish the warp's sum of one
//    term per lane; the two warps' sums meet in shared memory and leave once per
//    (token, term) per CTA.
constexpr int kLaneThreads = kBwdRows;  // one thread per row

struct LaneRaw {
  uint4 act[4][kBwdRows];     // u, Δraw, dout, z: a row's 8 tokens (bf16)
  uint4 bc[2][16];            // B, C: 8 tokens × 16 states (bf16)
  float4 ck[kBwdRows][4];     // the block's chunk-local starting state, 16 floats per row
  float scum[kBwdRows];       // ΣΔ from the chunk's start to the block
};
struct LaneTok {              // a row's per-token scalars, [token][row]
  float x[kBwdTok][kBwdRows];    // u
  float dt[kBwdTok][kBwdRows];   // Δ
  float sig[kBwdTok][kBwdRows];  // sigmoid(Δraw + bias)
  float dy[kBwdTok][kBwdRows];   // dout·silu(z)
  float dzf[kBwdTok][kBwdRows];  // dout·silu'(z)
};
// 56 KB: four CTAs fill an SM's 228 KB with their reserved kilobyte each.
struct LaneSmem {
  // h_{t-1} of tokens 1..7, [token - 1][quad][row] (token 0's stays in registers); once a
  // token's adjoint has read its slot, the slot's first quad holds each warp's sums of the
  // token's 32 terms
  float4 hp[kBwdTok - 1][4][kBwdRows];
  float bc[kBwdTok][2][kBwdN];       // B | C of the block's tokens, fp32
  float xs[2][32][32];               // per warp: a token's dB | dC terms, [row][term], the
                                     // 16-byte groups of row j at group g ^ (j & 7)
  float red0[2][32];                 // per warp: token 0's sums
  LaneTok ts;
  LaneRaw raw;
};
static_assert(sizeof(LaneSmem) <= 56 * 1024, "four CTAs per SM");

// where warp w's sums of token v's 32 terms go
__device__ __forceinline__ float* lane_red(LaneSmem& sm, int v, int w) {
  return v > 0 ? reinterpret_cast<float*>(&sm.hp[v - 1][0][32 * w]) : &sm.red0[w][0];
}

__device__ __forceinline__ void lane_issue(LaneRaw& rb, const BwdArgs& p, const BwdWs& w, int64_t b, int64_t c0,
                                           int64_t rt, int64_t blk) {
  const int64_t t0 = blk * kBwdTok;
  const int r = threadIdx.x;
  const int64_t c = c0 + r;
  const bool row_ok = c < p.d_inner;
#pragma unroll
  for (int wt = 0; wt < 4; ++wt) {
    const void* base = wt == 0 ? p.u : (wt == 1 ? p.delta : (wt == 2 ? p.dout : p.z));
    const bool ok = row_ok && base != nullptr;
    const __nv_bfloat16* src =
        static_cast<const __nv_bfloat16*>(ok ? base : p.u) + (ok ? (b * p.d_inner + c) * p.L + t0 : 0);
    cp_async16(&rb.act[wt][r], src, ok ? 16 : 0);
  }
  if (r < 32) {  // B and C: 256 bytes each
    const int wt = r / 16, qq = r % 16;
    cp_async16(&rb.bc[wt][qq], static_cast<const __nv_bfloat16*>(wt ? p.C : p.B) + (b * p.L + t0) * kBwdN + qq * 8,
               16);
  }
  const int64_t slot = rt * p.nblk + blk;
#pragma unroll
  for (int q = 0; q < 4; ++q) cp_async16(&rb.ck[r][q], w.ck + slot * kBwdThreads + 4 * r + q, 16);
  if (r < kBwdRows / 4) cp_async16(&rb.scum[r * 4], w.scum + slot * kBwdRows + r * 4, 16);
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// na: −1/a (fast path) or 1/a (PRECISE); both 0 where a = 0
template <bool PRECISE>
__device__ __forceinline__ void lane_body(LaneSmem& sm, const BwdArgs& p, const BwdWs& w, const CtaPos& o,
                                          const float (&a)[kBwdN], const float (&na)[kBwdN], float Dc, float biasc) {
  const int r = threadIdx.x, warp = r >> 5, lane = r & 31;
  const bool row_ok = o.row_ok;
  const int64_t b = o.b, L = p.L;
  const int64_t c0 = (o.rt % p.ctiles) * kBwdRows;

  // The chunk pass's chunks ("fine") f_lo..f_hi make up this chunk.  The adjoint entering
  // it from the right comes from the fine chunks after f_hi; the state entering each fine
  // chunk, h_in, is formed when the walk reaches it.
  const int f_hi = min((o.chunk + 1) * p.sub, p.nfine) - 1;
  float hin[kBwdN], dh[kBwdN];
#pragma unroll
  for (int n = 0; n < kBwdN; ++n) hin[n] = dh[n] = 0.f;
  int f_cur = -1;
  for (int j = p.nfine - 1; j > f_hi; --j) {
    const int64_t cs = o.rt * p.kmax + j;
    const float st = w.stot[cs * kBwdRows + r] * kLog2e;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 G = w.gcar[cs * kBwdThreads + 4 * r + q];
      const float gv[4] = {G.x, G.y, G.z, G.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) dh[4 * q + k] = fmaf(ex2_approx(a[4 * q + k] * st), dh[4 * q + k], gv[k]);
    }
  }

  // dA before the factor 1/a (fast path), or dA itself (PRECISE)
  float dAs[kBwdN];
#pragma unroll
  for (int n = 0; n < kBwdN; ++n) dAs[n] = 0.f;
  float dD_acc = 0.f, db_acc = 0.f;

  if (o.blk0 < o.blk1) {
    lane_issue(sm.raw, p, w, b, c0, o.rt, o.blk1 - 1);
    cp_async_commit();
  }
  for (int64_t blk = o.blk1 - 1; blk >= o.blk0; --blk) {
    const int64_t t0 = blk * kBwdTok;
    const int f = (int)(blk / p.cblk_f);
    if (f != f_cur) {  // h_in = Σ_{j<f} (Π_{j<i<f} e^{a S_i}) H_j over the fine chunks
      f_cur = f;
#pragma unroll
      for (int n = 0; n < kBwdN; ++n) hin[n] = 0.f;
      for (int j = 0; j < f; ++j) {
        const int64_t cs = o.rt * p.kmax + j;
        const float st = w.stot[cs * kBwdRows + r] * kLog2e;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 H = w.hend[cs * kBwdThreads + 4 * r + q];
          const float hv[4] = {H.x, H.y, H.z, H.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) hin[4 * q + k] = fmaf(ex2_approx(a[4 * q + k] * st), hin[4 * q + k], hv[k]);
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // the raw copy is in; red of the previous block has been read
    // B and C to fp32 (4 values per thread)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = r * 4 + k;  // [token][B|C][n]
      const int v = i / (2 * kBwdN), wt = (i / kBwdN) & 1, n = i % kBwdN;
      sm.bc[v][wt][n] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(&sm.raw.bc[wt][0])[v * kBwdN + n]);
    }
    // this row's per-token scalars
    {
      const uint4 U = sm.raw.act[0][r], Dr = sm.raw.act[1][r], Go = sm.raw.act[2][r], Z = sm.raw.act[3][r];
      const __nv_bfloat16* u8 = reinterpret_cast<const __nv_bfloat16*>(&U);
      const __nv_bfloat16* d8 = reinterpret_cast<const __nv_bfloat16*>(&Dr);
      const __nv_bfloat16* g8 = reinterpret_cast<const __nv_bfloat16*>(&Go);
      const __nv_bfloat16* z8 = reinterpret_cast<const __nv_bfloat16*>(&Z);
#pragma unroll
      for (int v = 0; v < kBwdTok; ++v) {
        sm.ts.x[v][r] = __bfloat162float(u8[v]);
        const float rr = __bfloat162float(d8[v]) + biasc;
        sm.ts.dt[v][r] = softplus_fast(rr);
        sm.ts.sig[v][r] = rcp_approx(1.f + ex2_approx(-rr * kLog2e));
        const float go = __bfloat162float(g8[v]);
        if (p.z) {
          const float zv = __bfloat162float(z8[v]);
          const float sz = rcp_approx(1.f + ex2_approx(-zv * kLog2e));
          sm.ts.dy[v][r] = go * zv * sz;
          sm.ts.dzf[v][r] = go * sz * (1.f + zv * (1.f - sz));
        } else {
          sm.ts.dy[v][r] = go;
          sm.ts.dzf[v][r] = 0.f;
        }
      }
    }
    // the block's starting state: chunk-local + decay since the chunk's start × h_in
    float h[kBwdN], h0[kBwdN];
    {
      const float sc = sm.raw.scum[r] * kLog2e;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 c4 = sm.raw.ck[r][q];
        const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) h0[4 * q + k] = h[4 * q + k] = fmaf(ex2_approx(a[4 * q + k] * sc), hin[4 * q + k], cv[k]);
      }
    }
    __syncthreads();  // bc converted, the raw buffer read: the next block's copy may land
    if (blk - 1 >= o.blk0) {
      lane_issue(sm.raw, p, w, b, c0, o.rt, blk - 1);
      cp_async_commit();
    }

    // recompute the block's states, keeping each token's h_{t-1}
#pragma unroll
    for (int v = 0; v < kBwdTok; ++v) {
      if (v > 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          sm.hp[v - 1][q][r] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
      }
      const float dtv = sm.ts.dt[v][r], x = sm.ts.x[v][r];
      const float dl = dtv * kLog2e;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 B4 = *reinterpret_cast<const float4*>(&sm.bc[v][0][4 * q]);
        const float bq[4] = {B4.x, B4.y, B4.z, B4.w};
        if (PRECISE) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int n = 4 * q + k;
            const float ab = a[n] != 0.f ? ex2_approx(dl * a[n]) : 1.f;
            const float phi = a[n] != 0.f ? (ab - 1.f) * na[n] : dtv;
            h[n] = fmaf(ab, h[n], phi * bq[k] * x);
          }
        } else {
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int n = 4 * q + 2 * k2;
            // h ← (Ā − 1)(h + x B/a) + h
            const float2 e = __fmul2_rn(f2(dl, dl), f2(a[n], a[n + 1]));
            const float2 em = __fadd2_rn(f2(ex2_approx(e.x), ex2_approx(e.y)), f2(-1.f, -1.f));
            const float2 xp = __fmul2_rn(f2(-x, -x), f2(na[n], na[n + 1]));
            const float2 hb = f2(h[n], h[n + 1]);
            const float2 hn = __ffma2_rn(em, __ffma2_rn(xp, f2(bq[2 * k2], bq[2 * k2 + 1]), hb), hb);
            h[n] = hn.x;
            h[n + 1] = hn.y;
          }
        }
      }
    }

    // the adjoint over the block, last token first; h = h_t, hp = h_{t-1}
    float* xsw = &sm.xs[warp][0][0];
    float* xrow = xsw + lane * 32;  // this row's 32 terms: dB, then dC (groups swizzled)
    const int sw = lane & 7;
    const int64_t i0 = o.row * L + t0;
    float4 o0 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int v = kBwdTok - 1; v >= 0; --v) {
      float hp[kBwdN];
      if (v > 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 t4 = sm.hp[v - 1][q][r];
          hp[4 * q] = t4.x; hp[4 * q + 1] = t4.y; hp[4 * q + 2] = t4.z; hp[4 * q + 3] = t4.w;
        }
      } else {
#pragma unroll
        for (int n = 0; n < kBwdN; ++n) hp[n] = h0[n];
      }
      const float x = sm.ts.x[v][r], dtv = sm.ts.dt[v][r], dyv = sm.ts.dy[v][r];
      const float dl = dtv * kLog2e;
      float y = 0.f, dx = 0.f, ddt = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 B4 = *reinterpret_cast<const float4*>(&sm.bc[v][0][4 * q]);
        const float4 C4 = *reinterpret_cast<const float4*>(&sm.bc[v][1][4 * q]);
        const float bq[4] = {B4.x, B4.y, B4.z, B4.w}, cq[4] = {C4.x, C4.y, C4.z, C4.w};
        float slot[8];  // the quad's dB terms, then its dC terms
        if (PRECISE) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int n = 4 * q + k;
            const float ab = a[n] != 0.f ? ex2_approx(dl * a[n]) : 1.f;
            const float phi = a[n] != 0.f ? (ab - 1.f) * na[n] : dtv;
            y = fmaf(cq[k], h[n], y);
            const float g = fmaf(dyv, cq[k], dh[n]);
            slot[4 + k] = dyv * h[n];
            slot[k] = g * phi * x;
            dx = fmaf(g * phi, bq[k], dx);
            const float bx = bq[k] * x;
            if (a[n] != 0.f) {
              ddt = fmaf(g * ab, fmaf(a[n], hp[n], bx), ddt);
              dAs[n] = fmaf(g, fmaf(dtv * ab, hp[n], bx * (dtv * ab - phi) * na[n]), dAs[n]);
            } else {
              ddt = fmaf(g, bx, ddt);
              dAs[n] = fmaf(g, fmaf(dtv, hp[n], 0.5f * bx * dtv * dtv), dAs[n]);
            }
            dh[n] = g * ab;
          }
        } else {
          // with nphi = −φ: dB term = (g nphi)(−x); dx = −Σ (g nphi) B;
          // dAs += Δ gd + (g nphi) B x
          float2 y2 = f2(0.f, 0.f), ndx2 = f2(0.f, 0.f), ddt2 = f2(0.f, 0.f);
          const float2 xx = f2(x, x), nxx = f2(-x, -x), dt2 = f2(dtv, dtv), dy2 = f2(dyv, dyv);
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int n = 4 * q + 2 * k2;
            const float2 bb = f2(bq[2 * k2], bq[2 * k2 + 1]), cc = f2(cq[2 * k2], cq[2 * k2 + 1]);
            const float2 hv2 = f2(h[n], h[n + 1]), hp2 = f2(hp[n], hp[n + 1]);
            const float2 an = f2(a[n], a[n + 1]);
            y2 = __ffma2_rn(cc, hv2, y2);
            const float2 g = __ffma2_rn(dy2, cc, f2(dh[n], dh[n + 1]));
            const float2 e = __fmul2_rn(f2(dl, dl), an);
            const float2 ab = f2(ex2_approx(e.x), ex2_approx(e.y));
            const float2 nphi = __fmul2_rn(__fadd2_rn(ab, f2(-1.f, -1.f)), f2(na[n], na[n + 1]));
            const float2 gnp = __fmul2_rn(g, nphi);
            const float2 sb = __fmul2_rn(gnp, nxx);
            const float2 sc = __fmul2_rn(dy2, hv2);
            ndx2 = __ffma2_rn(gnp, bb, ndx2);
            const float2 ga = __fmul2_rn(g, ab);
            const float2 bx = __fmul2_rn(bb, xx);
            const float2 gd = __fmul2_rn(ga, __ffma2_rn(an, hp2, bx));
            ddt2 = __fadd2_rn(ddt2, gd);
            const float2 da = __ffma2_rn(gnp, bx, __ffma2_rn(dt2, gd, f2(dAs[n], dAs[n + 1])));
            dAs[n] = da.x; dAs[n + 1] = da.y;
            dh[n] = ga.x; dh[n + 1] = ga.y;
            slot[2 * k2] = sb.x; slot[2 * k2 + 1] = sb.y;
            slot[4 + 2 * k2] = sc.x; slot[4 + 2 * k2 + 1] = sc.y;
          }
          y += y2.x + y2.y;
          dx -= ndx2.x + ndx2.y;
          ddt += ddt2.x + ddt2.y;
        }
        *reinterpret_cast<float4*>(xrow + 4 * (q ^ sw)) = make_float4(slot[0], slot[1], slot[2], slot[3]);
        *reinterpret_cast<float4*>(xrow + 4 * ((4 + q) ^ sw)) = make_float4(slot[4], slot[5], slot[6], slot[7]);
      }
      y = fmaf(Dc, x, y);
      dx = fmaf(dyv, Dc, dx);
      const float dr = ddt * sm.ts.sig[v][r];
      // the token's du, Δraw gradient and dz wait in the row's spent state slot (token 0's in
      // registers) and leave with the block's other tokens
      const float dzv = sm.ts.dzf[v][r] * y;
      if (v > 0)
        sm.hp[v - 1][1][r] = make_float4(dx, dr, dzv, 0.f);
      else
        o0 = make_float4(dx, dr, dzv, 0.f);
      dD_acc = fmaf(dyv, x, dD_acc);
      db_acc += dr;
      // Σ over the warp's rows of the 32 terms
      __syncwarp();
      const int sg = lane & 7, rg = lane >> 3;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 t4 = *reinterpret_cast<const float4*>(xsw + (8 * rg + i) * 32 + 4 * (sg ^ i));
        acc.x += t4.x; acc.y += t4.y; acc.z += t4.z; acc.w += t4.w;
      }
      __syncwarp();  // the tile is read before the next token's terms overwrite it
      // over lane bit 4, then bit 3: lane keeps term 4 sg + 2 b4 + b3
      const bool up4 = (lane & 16) != 0, up3 = (lane & 8) != 0;
      const float s0 = up4 ? acc.x : acc.z, s1 = up4 ? acc.y : acc.w;
      const float k0 = up4 ? acc.z : acc.x, k1 = up4 ? acc.w : acc.y;
      const float m0 = k0 + __shfl_xor_sync(0xffffffffu, s0, 16);
      const float m1 = k1 + __shfl_xor_sync(0xffffffffu, s1, 16);
      const float sfin = (up3 ? m1 : m0) + __shfl_xor_sync(0xffffffffu, up3 ? m0 : m1, 8);
      lane_red(sm, v, warp)[4 * sg + 2 * (up4 ? 1 : 0) + (up3 ? 1 : 0)] = sfin;
#pragma unroll
      for (int n = 0; n < kBwdN; ++n) h[n] = hp[n];
    }
    if (row_ok) {  // the block's 8 tokens of du, the Δraw gradient and dz of this row
      float ov[3][kBwdTok];
      ov[0][0] = o0.x; ov[1][0] = o0.y; ov[2][0] = o0.z;
#pragma unroll
      for (int v = 1; v < kBwdTok; ++v) {
        const float4 t4 = sm.hp[v - 1][1][r];
        ov[0][v] = t4.x; ov[1][v] = t4.y; ov[2][v] = t4.z;
      }
      void* dst[3] = {p.du, p.ddelta, p.dz};
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        if (k == 2 && !p.z) break;
        __nv_bfloat16* d = static_cast<__nv_bfloat16*>(dst[k]) + i0;
        if ((reinterpret_cast<uintptr_t>(d) & 15u) == 0) {
          uint4 pk;
          unsigned* pw = &pk.x;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 t = __floats2bfloat162_rn(ov[k][2 * j], ov[k][2 * j + 1]);
            pw[j] = *reinterpret_cast<unsigned*>(&t);
          }
          *reinterpret_cast<uint4*>(d) = pk;
        } else {
#pragma unroll
          for (int v = 0; v < kBwdTok; ++v) d[v] = __float2bfloat16_rn(ov[k][v]);
        }
      }
    }
    __syncthreads();  // both warps' sums are in red
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = r + kLaneThreads * k;  // [token][term]
      const int v = idx >> 5, term = idx & 31;
      const float sum = lane_red(sm, v, 0)[term] + lane_red(sm, v, 1)[term];
      const int wt = term >> 4, n = term & 15;
      if (p.det)
        p.part_bc[(((o.rt % p.ctiles) * p.batch + b) * L + t0 + v) * 2 * kBwdN + wt * kBwdN + n] = sum;
      else
        atomicAdd((wt ? p.dC : p.dB) + (b * L + t0 + v) * kBwdN + n, sum);
    }
  }
  if (!row_ok) return;
  float dA[kBwdN];
#pragma unroll
  for (int n = 0; n < kBwdN; ++n) dA[n] = PRECISE ? dAs[n] : -na[n] * dAs[n];
  if (p.det) {
    float* pr = p.part_row + ((b * p.nchunks + o.chunk) * p.d_inner + o.c) * (kBwdN + 2);
#pragma unroll
    for (int n = 0; n < kBwdN; ++n) pr[n] = dA[n];
    pr[kBwdN] = dD_acc;
    pr[kBwdN + 1] = db_acc;
  } else {
#pragma unroll
    for (int n = 0; n < kBwdN; ++n) atomicAdd(p.dA + o.c * kBwdN + n, dA[n]);
    if (p.dD) atomicAdd(p.dD + o.c, dD_acc);
    if (p.dbias) atomicAdd(p.dbias + o.c, db_acc);
  }
}

// split: CTAs per 64-row tile (thread t of CTA x serves row (x % split) · 64/split + t)
__device__ __forceinline__ CtaPos lane_pos(const BwdArgs& p, int split, int64_t cblk) {
  CtaPos o;
  o.rt = blockIdx.x / split;
  o.chunk = (int)blockIdx.y;
  o.b = o.rt / p.ctiles;
  const int64_t c0 = (o.rt % p.ctiles) * kBwdRows;
  o.r = threadIdx.x + (int)(blockIdx.x % split) * (kBwdRows / split);
  o.g = 0;
  o.row_ok = c0 + o.r < p.d_inner;
  o.c = c0 + (o.row_ok ? o.r : 0);
  o.row = o.b * p.d_inner + o.c;
  o.blk0 = o.chunk * cblk;
  o.blk1 = o.blk0 + cblk < p.nblk ? o.blk0 + cblk : p.nblk;
  return o;
}
// A of the row (0 for |A| < 2^-60; rows past d_inner take A = -1); true if a state has A = 0
__device__ __forceinline__ bool lane_a(const BwdArgs& p, const CtaPos& o, float (&a)[kBwdN]) {
  bool zero = false;
#pragma unroll
  for (int n = 0; n < kBwdN; ++n) {
    const float av = o.row_ok ? p.A[o.c * kBwdN + n] : -1.f;
    const bool tiny = fabsf(av) < 8.673617e-19f;
    zero = zero || tiny;
    a[n] = tiny ? 0.f : av;
  }
  return zero;
}

__global__ void __launch_bounds__(kLaneThreads, 4) scan_bwd_lane_kernel(const BwdArgs p, const BwdWs w) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  LaneSmem& sm = *reinterpret_cast<LaneSmem*>(smem_raw);
  const CtaPos o = lane_pos(p, 1, p.cblk);
  float a[kBwdN];
  const bool zero = lane_a(p, o, a);
  const float Dc = (o.row_ok && p.D) ? p.D[o.c] : 0.f;
  const float biasc = (o.row_ok && p.bias) ? p.bias[o.c] : 0.f;
  float na[kBwdN];
  if (__syncthreads_or(zero)) {
#pragma unroll
    for (int n = 0; n < kBwdN; ++n) na[n] = a[n] != 0.f ? 1.f / a[n] : 0.f;
    lane_body<true>(sm, p, w, o, a, na, Dc, biasc);
  } else {
#pragma unroll
    for (int n = 0; n < kBwdN; ++n) na[n] = -1.f / a[n];
    lane_body<false>(sm, p, w, o, a, na, Dc, biasc);
  }
}

// Launch 1 in one thread per row: each chunk forward from h = 0, saving the local states
// every block, the prefix sums of Δ and the chunk's summary (end state, ΣΔ and the adjoint
// sent left, G = Σ_t (Π_{s≤t} Ā_s) dy_t C_t), in the layout the gradient passes read.  A CTA
// is one warp over half a tile (the grid has twice the CTAs of the gradient pass, so that
// short grids still fill the SMs); only the block's raw inputs, its B, C and the rows'
// per-token scalars live in shared memory (6.5 KB).
constexpr int kLaneChunkRows = 32;
struct LaneChunkSmem {
  float bc[kBwdTok][2][kBwdN];
  float x[kBwdTok][kLaneChunkRows], dt[kBwdTok][kLaneChunkRows], dy[kBwdTok][kLaneChunkRows];
  uint4 act[4][kLaneChunkRows];  // u, Δraw, dout, z: a row's 8 tokens (bf16)
  uint4 bcr[2][16];              // B, C: 8 tokens × 16 states (bf16)
};

// the raw inputs of block blk for the CTA's rows (thread l: row o.r = first + l)
__device__ __forceinline__ void lane_chunk_issue(LaneChunkSmem& sm, const BwdArgs& p, const CtaPos& o, int64_t blk) {
  const int64_t t0 = blk * kBwdTok;
  const int l = threadIdx.x;
  const bool row_ok = o.row_ok;
#pragma unroll
  for (int wt = 0; wt < 4; ++wt) {
    const void* base = wt == 0 ? p.u : (wt == 1 ? p.delta : (wt == 2 ? p.dout : p.z));
    const bool ok = row_ok && base != nullptr;
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(ok ? base : p.u) + (ok ? o.row * p.L + t0 : 0);
    cp_async16(&sm.act[wt][l], src, ok ? 16 : 0);
  }
  {  // B and C: 256 bytes each
    const int wt = l / 16, qq = l % 16;
    cp_async16(&sm.bcr[wt][qq], static_cast<const __nv_bfloat16*>(wt ? p.C : p.B) + (o.b * p.L + t0) * kBwdN + qq * 8,
               16);
  }
}

template <bool PRECISE>
__device__ __forceinline__ void lane_chunk_body(LaneChunkSmem& sm, const BwdArgs& p, const BwdWs& w,
                                                const CtaPos& o, const float (&a)[kBwdN], const float (&na)[kBwdN],
                                                float biasc) {
  const int l = threadIdx.x, r = o.r;  // r: the row within the 64-row tile
  const bool want_g = o.chunk > 0;  // chunk 0 sends no adjoint further left
  float h[kBwdN], P[kBwdN], G[kBwdN];
#pragma unroll
  for (int n = 0; n < kBwdN; ++n) {
    h[n] = 0.f;
    P[n] = 1.f;
    G[n] = 0.f;
  }
  float S = 0.f;
  if (o.blk0 < o.blk1) {
    lane_chunk_issue(sm, p, o, o.blk0);
    cp_async_commit();
  }
  for (int64_t blk = o.blk0; blk < o.blk1; ++blk) {
    const int64_t slot = o.rt * p.nblk + blk;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w.ck[slot * kBwdThreads + 4 * r + q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    w.scum[slot * kBwdRows + r] = S;
    cp_async_wait<0>();
    __syncthreads();  // the raw copy is in; the previous block's B, C are no longer read
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = l * 8 + k;  // [token][B|C][n]
      const int v = i / (2 * kBwdN), wt = (i / kBwdN) & 1, n = i % kBwdN;
      sm.bc[v][wt][n] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(&sm.bcr[wt][0])[v * kBwdN + n]);
    }
    {
      const uint4 U = sm.act[0][l], Dr = sm.act[1][l], Go = sm.act[2][l], Z = sm.act[3][l];
      const __nv_bfloat16* u8 = reinterpret_cast<const __nv_bfloat16*>(&U);
      const __nv_bfloat16* d8 = reinterpret_cast<const __nv_bfloat16*>(&Dr);
      const __nv_bfloat16* g8 = reinterpret_cast<const __nv_bfloat16*>(&Go);
      const __nv_bfloat16* z8 = reinterpret_cast<const __nv_bfloat16*>(&Z);
#pragma unroll
      for (int v = 0; v < kBwdTok; ++v) {
        sm.x[v][l] = __bfloat162float(u8[v]);
        sm.dt[v][l] = softplus_fast(__bfloat162float(d8[v]) + biasc);
        const float go = __bfloat162float(g8[v]);
        if (p.z) {
          const float zv = __bfloat162float(z8[v]);
          sm.dy[v][l] = go * zv * rcp_approx(1.f + ex2_approx(-zv * kLog2e));
        } else {
          sm.dy[v][l] = go;
        }
      }
    }
    __syncthreads();  // B, C converted and the raw buffer read: the next block's copy may land
    if (blk + 1 < o.blk1) {
      lane_chunk_issue(sm, p, o, blk + 1);
      cp_async_commit();
    }
#pragma unroll 1
    for (int v = 0; v < kBwdTok; ++v) {
      const float xv = sm.x[v][l], dtv = sm.dt[v][l], dyv = sm.dy[v][l], dl = dtv * kLog2e;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 B4 = *reinterpret_cast<const float4*>(&sm.bc[v][0][4 * q]);
        const float4 C4 = *reinterpret_cast<const float4*>(&sm.bc[v][1][4 * q]);
        const float bq[4] = {B4.x, B4.y, B4.z, B4.w}, cq[4] = {C4.x, C4.y, C4.z, C4.w};
        if (PRECISE) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int n = 4 * q + k;
            const float ab = a[n] != 0.f ? ex2_approx(dl * a[n]) : 1.f;
            const float phi = a[n] != 0.f ? (ab - 1.f) * na[n] : dtv;
            h[n] = fmaf(ab, h[n], phi * bq[k] * xv);
            if (want_g) {
              P[n] *= ab;
              G[n] = fmaf(P[n], dyv * cq[k], G[n]);
            }
          }
        } else {
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int n = 4 * q + 2 * k2;
            const float2 e = __fmul2_rn(f2(dl, dl), f2(a[n], a[n + 1]));
            const float2 em = __fadd2_rn(f2(ex2_approx(e.x), ex2_approx(e.y)), f2(-1.f, -1.f));
            const float2 xp = __fmul2_rn(f2(-xv, -xv), f2(na[n], na[n + 1]));
            const float2 hb = f2(h[n], h[n + 1]);
            const float2 hn = __ffma2_rn(em, __ffma2_rn(xp, f2(bq[2 * k2], bq[2 * k2 + 1]), hb), hb);
            h[n] = hn.x;
            h[n + 1] = hn.y;
            if (want_g) {  // P ← P Ā = P + P (Ā − 1); G += P dy C
              const float2 pb = f2(P[n], P[n + 1]);
              const float2 pp = __ffma2_rn(pb, em, pb);
              const float2 gg = __ffma2_rn(pp, __fmul2_rn(f2(dyv, dyv), f2(cq[2 * k2], cq[2 * k2 + 1])),
                                           f2(G[n], G[n + 1]));
              P[n] = pp.x; P[n + 1] = pp.y;
              G[n] = gg.x; G[n + 1] = gg.y;
            }
          }
        }
      }
      S += dtv;
    }
  }
  const int64_t cs = o.rt * p.kmax + o.chunk;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    w.hend[cs * kBwdThreads + 4 * r + q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    w.gcar[cs * kBwdThreads + 4 * r + q] = make_float4(G[4 * q], G[4 * q + 1], G[4 * q + 2], G[4 * q + 3]);
  }
  w.stot[cs * kBwdRows + r] = S;
}

__global__ void __launch_bounds__(kLaneChunkRows, 16) scan_bwd_lane_chunk_kernel(const BwdArgs p, const BwdWs w) {
  __shared__ __align__(16) LaneChunkSmem sm;
  const CtaPos o = lane_pos(p, kBwdRows / kLaneChunkRows, p.cblk_f);
  float a[kBwdN];
  const bool zero = lane_a(p, o, a);
  const float biasc = (o.row_ok && p.bias) ? p.bias[o.c] : 0.f;
  float na[kBwdN];
  if (__syncthreads_or(zero)) {
#pragma unroll
    for (int n = 0; n < kBwdN; ++n) na[n] = a[n] != 0.f ? 1.f / a[n] : 0.f;
    lane_chunk_body<true>(sm, p, w, o, a, na, biasc);
  } else {
#pragma unroll
    for (int n = 0; n < kBwdN; ++n) na[n] = -1.f / a[n];
    lane_chunk_body<false>(sm, p, w, o, a, na, biasc);
  }
}

// Launch 3 (deterministic mode): the sums over channel tiles (dB, dC) and over batch and
// chunks (dA, dD, dbias) of the partials, each in ascending index order, so that the result
// does not depend on which CTA ran first.
__global__ void __launch_bounds__(256) scan_bwd_reduce_kernel(const BwdArgs p) {
  const int64_t N = p.N;
  const int64_t nbc = p.batch * p.L * 2 * N;  // one channel tile's partials
  const int64_t nrow = p.d_inner * (N + 2);
  const int64_t nparts = p.batch * p.nchunks;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nbc + nrow;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < nbc) {
      float s = 0.f;
      for (int ct = 0; ct < p.ctiles; ++ct) s += __ldcs(p.part_bc + ct * nbc + i);
      const int64_t n = i % N, w = (i / N) & 1, bt = i / (2 * N);
      (w ? p.dC : p.dB)[bt * N + n] = s;
    } else {
      const int64_t j = i - nbc;
      float s = 0.f;
      for (int64_t q = 0; q < nparts; ++q) s += __ldcs(p.part_row + q * nrow + j);
      const int64_t c = j / (N + 2), k = j % (N + 2);
      if (k < N)
        p.dA[c * N + k] = s;
      else if (k == N) {
        if (p.dD) p.dD[c] = s;
      } else if (p.dbias) {
        p.dbias[c] = s;
      }
    }
  }
}

BwdWs ws_layout(float* base, int64_t R, int64_t nblk, int64_t kmax) {
  unsigned char* p = reinterpret_cast<unsigned char*>(base);
  BwdWs w;
  w.ck = reinterpret_cast<float4*>(p);
  p += (size_t)(R * nblk * kBwdThreads) * sizeof(float4);
  w.scum = reinterpret_cast<float*>(p);
  p += (size_t)(R * nblk * kBwdRows) * sizeof(float);
  w.hend = reinterpret_cast<float4*>(p);
  p += (size_t)(R * kmax * kBwdThreads) * sizeof(float4);
  w.gcar = reinterpret_cast<float4*>(p);
  p += (size_t)(R * kmax * kBwdThreads) * sizeof(float4);
  w.stot = reinterpret_cast<float*>(p);
  return w;
}

// Chunks for R row tiles of nblk blocks on `slots` resident CTAs: fewest
// block-steps per slot, counting whole waves and about two blocks' worth of
// fixed cost per CTA (the summaries, the atomics at the end).
int pick_bwd_chunks(int64_t R, int64_t nblk, int64_t slots, int64_t kmax) {
  int best = 1;
  int64_t best_cost = INT64_MAX;
  for (int64_t k = 1; k <= kmax; ++k) {
    const int64_t cb = (nblk + k - 1) / k;
    const int64_t ke = (nblk + cb - 1) / cb;
    const int64_t waves = (R * ke + slots - 1) / slots;
    const int64_t cost = waves * (cb + 2);
    if (cost < best_cost) {
      best_cost = cost;
      best = (int)ke;
    }
  }
  return best;
}

// lane: the gradient pass with one thread per row (bf16 with the raw-copy prefetch only)
template <typename T, bool PF>
cudaError_t bwd_launch_t(BwdArgs p, cudaStream_t s, bool lane) {
  const void* grad = lane ? reinterpret_cast<const void*>(scan_bwd_lane_kernel)
                          : reinterpret_cast<const void*>(scan_bwd_kernel<T, PF>);
  const size_t smem = lane ? sizeof(LaneSmem) : sizeof(BwdSmem) + (PF ? 2 * sizeof(RawBlock) : 0);
  const int threads = lane ? kLaneThreads : kBwdThreads;
  cudaError_t e = cudaFuncSetAttribute(grad, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t R = p.batch * p.ctiles;
  if (R == 0) return cudaSuccess;
  int64_t k = p.force_chunks;
  if (k <= 0) {
    int dev = 0, sms = 0, occ = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, grad, threads, smem)) != cudaSuccess) return e;
    k = pick_bwd_chunks(R, p.nblk, (int64_t)(sms > 0 ? sms : 1) * (occ > 0 ? occ : 1), p.kmax);
  }
  if (k > p.kmax) k = p.kmax;
  if (k > p.nblk) k = p.nblk;
  if (k < 1) k = 1;
  p.cblk = (p.nblk + k - 1) / k;
  p.nchunks = p.cblk > 0 ? (int)((p.nblk + p.cblk - 1) / p.cblk) : 1;
  // The one-thread-per-row chunk pass runs two one-warp CTAs per tile and chunk, sixteen
  // per SM; when the gradient pass's chunks leave it under half of those slots, it takes
  // each of them as two chunks of its own.
  p.sub = 1;
  if (lane && p.cblk >= 2 && 2 * p.nchunks <= p.kmax) {
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (R * p.nchunks * (kBwdRows / kLaneChunkRows) * 2 <= (int64_t)sms * 16) p.sub = 2;
  }
  p.cblk_f = (p.cblk + p.sub - 1) / p.sub;
  p.cblk = p.cblk_f * p.sub;
  p.nchunks = (int)((p.nblk + p.cblk - 1) / p.cblk);
  p.nfine = (int)((p.nblk + p.cblk_f - 1) / p.cblk_f);
  const BwdWs w = ws_layout(p.ckpt, R, p.nblk, p.kmax);
  const dim3 grid((unsigned)R, (unsigned)p.nchunks);
  if (lane)
    scan_bwd_lane_chunk_kernel<<<dim3(grid.x * (kBwdRows / kLaneChunkRows), (unsigned)p.nfine), kLaneChunkRows, 0,
                                 s>>>(p, w);
  else
    scan_bwd_chunk_kernel<T, PF><<<grid, kBwdThreads, 0, s>>>(p, w);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (lane)
    scan_bwd_lane_kernel<<<grid, kLaneThreads, smem, s>>>(p, w);
  else
    scan_bwd_kernel<T, PF><<<grid, kBwdThreads, smem, s>>>(p, w);
  if ((e = cudaGetLastError()) != cudaSuccess || !p.det) return e;
  const int64_t items = p.batch * p.L * 2 * p.N + p.d_inner * (p.N + 2);
  const int64_t blocks = (items + 255) / 256;
  scan_bwd_reduce_kernel<<<(unsigned)(blocks < 148 * 16 ? blocks : 148 * 16), 256, 0, s>>>(p);
  return cudaGetLastError();
}

// The raw-copy prefetch needs bf16 rows of whole 16-byte pieces: d_state 16, L % 8 == 0
// and every activation array 16-byte aligned.
bool bwd_prefetch_ok(const BwdArgs& p) {
  auto a16 = [](const void* q) { return q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  return p.act == 1 && p.N == kBwdN && p.L % kBwdTok == 0 && a16(p.u) && a16(p.delta) && a16(p.dout) &&
         a16(p.z) && a16(p.B) && a16(p.C);
}


}  // namespace

int scan_bwd_rows_per_cta() { return kBwdRows; }

namespace {
// Workspace: [checkpoints and chunk summaries][partials of dB, dC][partials of dA, dD, dbias]
struct BwdWsSizes {
  size_t base, part_bc, part_row;
};
size_t round256(size_t v) { return (v + 255) & ~size_t(255); }
BwdWsSizes bwd_ws_sizes(int64_t batch, int64_t d_inner, int64_t N, int64_t L) {
  const int64_t ctiles = (d_inner + kBwdRows - 1) / kBwdRows;
  const int64_t R = batch * ctiles;
  const int64_t nblk = (L + kBwdTok - 1) / kBwdTok;
  const int64_t kmax = bwd_max_chunks(nblk);
  BwdWsSizes z;
  z.base = round256((size_t)(R * nblk) * (kBwdThreads * sizeof(float4) + kBwdRows * sizeof(float)) +
                    (size_t)(R * kmax) * (2 * kBwdThreads * sizeof(float4) + kBwdRows * sizeof(float)));
  z.part_bc = round256((size_t)(ctiles * batch * L * 2 * N) * sizeof(float));
  z.part_row = round256((size_t)(batch * kmax * d_inner * (N + 2)) * sizeof(float));
  return z;
}
}  // namespace

size_t scan_bwd_workspace_bytes(int64_t batch, int64_t d_inner, int64_t N, int64_t L, bool deterministic) {
  const BwdWsSizes z = bwd_ws_sizes(batch, d_inner, N, L);
  return deterministic ? z.base + z.part_bc + z.part_row : z.base;
}

cudaError_t scan_bwd_launch(BwdArgs p, cudaStream_t stream) {
  p.ctiles = (int)((p.d_inner + kBwdRows - 1) / kBwdRows);
  p.nblk = (p.L + kBwdTok - 1) / kBwdTok;
  p.kmax = (int)bwd_max_chunks(p.nblk);
  if (p.det) {
    const BwdWsSizes z = bwd_ws_sizes(p.batch, p.d_inner, p.N, p.L);
    unsigned char* base = reinterpret_cast<unsigned char*>(p.ckpt);
    p.part_bc = reinterpret_cast<float*>(base + z.base);
    p.part_row = reinterpret_cast<float*>(base + z.base + z.part_bc);
  }
  if (p.act != 1) return bwd_launch_t<float, false>(p, stream, false);
  if (!bwd_prefetch_ok(p)) return bwd_launch_t<__nv_bfloat16, false>(p, stream, false);
  return bwd_launch_t<__nv_bfloat16, true>(p, stream, p.form != 1);
}

}  // namespace ssm

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
// holds kBwdRows rows of one batch and one chunk of the sequence, so that the
// grid is (row tiles) × (chunks) and short batches still fill the GPU.  Two
// launches, neither waiting on another CTA:
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
      const int64_t i = row * L + t0 + v;
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
        if (row_ok) {
          stf<T>(p.du, i, dx);
          stf<T>(p.ddelta, i, dr);
          if (p.z) stf<T>(p.dz, i, s.dzf * y);
        }
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

template <typename T, bool PF>
cudaError_t bwd_launch_t(BwdArgs p, cudaStream_t s) {
  const size_t smem = sizeof(BwdSmem) + (PF ? 2 * sizeof(RawBlock) : 0);
  cudaError_t e = cudaFuncSetAttribute(scan_bwd_kernel<T, PF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t R = p.batch * p.ctiles;
  if (R == 0) return cudaSuccess;
  int64_t k = p.force_chunks;
  if (k <= 0) {
    int dev = 0, sms = 0, occ = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, scan_bwd_kernel<T, PF>, kBwdThreads, smem)) !=
        cudaSuccess)
      return e;
    k = pick_bwd_chunks(R, p.nblk, (int64_t)(sms > 0 ? sms : 1) * (occ > 0 ? occ : 1), p.kmax);
  }
  if (k > p.kmax) k = p.kmax;
  if (k > p.nblk) k = p.nblk;
  if (k < 1) k = 1;
  p.cblk = (p.nblk + k - 1) / k;
  p.nchunks = p.cblk > 0 ? (int)((p.nblk + p.cblk - 1) / p.cblk) : 1;
  const BwdWs w = ws_layout(p.ckpt, R, p.nblk, p.kmax);
  const dim3 grid((unsigned)R, (unsigned)p.nchunks);
  scan_bwd_chunk_kernel<T, PF><<<grid, kBwdThreads, 0, s>>>(p, w);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
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
  if (p.act != 1) return bwd_launch_t<float, false>(p, stream);
  return bwd_prefetch_ok(p) ? bwd_launch_t<__nv_bfloat16, true>(p, stream)
                            : bwd_launch_t<__nv_bfloat16, false>(p, stream);
}

}  // namespace ssm

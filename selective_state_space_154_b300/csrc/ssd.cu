// The Mamba-2 layer scan (state space duality, SSD) for sm_103a, on the
// fifth-generation tensor cores.  Each head has one scalar A, so its state
// update is h_t = Ā_t h_{t-1} + φ_t x_t B_tᵀ (h: headdim × d_state) and the layer
// is causal linear attention with queries C, keys B, values φ x and the decay
// mask e^{Σ Δa} between tokens ("Mambaとは？Transformer以外の系列モデル", section
// Mamba-2とTransformerとの関係性; "State Space Models（SSM）とMamba" §4.6 Mamba-2).
// Discretisation is the zero-order hold of the Mamba-1 scan (Ā = e^{Δa},
// φ = (e^{Δa} − 1)/a) with Δ = softplus(Δraw + dt_bias).
//
// The sequence is cut into chunks of kQ = 128 tokens; per (batch, head, chunk):
//   1. ssd_chunk_state_kernel: the chunk's own end state
//        H_c = Bᵀ diag(w) X,   w_s = e^{Σ_{s<k≤end} Δa} φ_s        (tensor cores)
//      and its total log decay Σ Δa;
//   2. ssd_state_pass_kernel: h_in[c+1] = e^{Σ_c Δa} h_in[c] + H_c along the chunks
//      (one thread per state element, h_in[0] = the initial state, carried in
//      fp32), h_in stored as two bf16 terms for the next launch's tensor cores,
//      the last state in fp32;
//   3. ssd_chunk_out_kernel: S = C Bᵀ and Y_in = C h_inᵀ (tensor cores), the
//      masked G_ts = S_ts e^{Σ_{s<k≤t} Δa} φ_s (s ≤ t) in registers, then
//      Y = G X (tensor cores), y_t = Y_t + e^{Σ_{k≤t} Δa} Y_in,t + D x_t, gated
//      by silu(z).
// Operands are staged in shared memory in the no-swizzle K-major layout
// (tc_sm100.cuh), by cp.async where global memory already has K contiguous and
// through an 8 × 8 register transpose where it does not; accumulators live in
// tensor memory.  The operands computed by the kernels (G, w·x of the chunk
// state, and the state h_in entering a chunk) are passed to the tensor cores
// as two bf16 terms, hi = bf16(v) and lo = bf16(v − hi), each multiplied in
// turn: about 16 significant bits instead of 8, which keeps their rounding
// below that of the bf16 output.
// No CTA waits on another; each tensor-core wait is bounded and reports
// through the workspace's error word.
#include <cstdint>

#include <cuda_bf16.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "tc_sm100.cuh"

namespace ssm {
namespace {

constexpr int kQ = kSsdChunk;
constexpr int kP = kSsdHeadDim;
constexpr int kN = kSsdState;
constexpr int kThreads = 256;
constexpr int kDefaultTimeoutMs = 2000;

static_assert(kQ == 128 && kThreads == 2 * kQ && kN == 128 && kP == 64,
              "tile shapes assume 128 tokens, 128 states, headdim 64, 256 threads");

// Workspace: error words | H_c fp32 [b][H][nch][P][N] | Σ Δa [b][H][nch] |
// h_in as bf16 hi and lo terms [b][H][nch][2][P][N]
struct SsdWs {
  unsigned* err;
  float* hc;
  float* ctot;
  __nv_bfloat16* hin;
};
constexpr size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
struct WsSizes {
  size_t hc, ctot, hin;
};
WsSizes ws_sizes(int64_t b, int64_t H, int64_t nch) {
  const size_t cells = (size_t)(b * H * nch);
  return {align256(cells * kP * kN * sizeof(float)), align256(cells * sizeof(float)),
          align256(cells * 2 * kP * kN * sizeof(__nv_bfloat16))};
}
SsdWs ws_layout(void* base, int64_t b, int64_t H, int64_t nch) {
  const WsSizes z = ws_sizes(b, H, nch);
  unsigned char* p = static_cast<unsigned char*>(base);
  SsdWs w;
  w.err = reinterpret_cast<unsigned*>(p) + 1;
  p += 256;
  w.hc = reinterpret_cast<float*>(p);
  p += z.hc;
  w.ctot = reinterpret_cast<float*>(p);
  p += z.ctot;
  w.hin = reinterpret_cast<__nv_bfloat16*>(p);
  return w;
}

__device__ __forceinline__ const __nv_bfloat16* bf(const void* p) { return static_cast<const __nv_bfloat16*>(p); }

constexpr int kMaxHeadsPerCta = 8;

// Per-token scalars of one chunk for the CTA's heads j < hb (head h0 + j).
struct TokenSmem {
  float cs2[kMaxHeadsPerCta][kQ];   // inclusive prefix sums of Δa since the chunk's start, log2 units
  float phi[kMaxHeadsPerCta][kQ];   // φ of the token (0 past the sequence's end)
  float wsum[2][4];
  float total[kMaxHeadsPerCta];     // Σ Δa over the chunk (natural units)
};

// Threads 0..127 take heads 0, 2, 4, ... and threads 128..255 heads 1, 3, 5, ...,
// token i = thread % 128; a block scan over the 128 tokens per head.
__device__ void chunk_tokens(const SsdArgs& p, int64_t b, int h0, int hb, int64_t t0, int q, TokenSmem& ts) {
  const int i = threadIdx.x & (kQ - 1), half = threadIdx.x >> 7, lane = threadIdx.x & 31,
            wq = (threadIdx.x >> 5) & 3;
  for (int r = 0; r < (hb + 1) / 2; ++r) {
    const int j = 2 * r + half;
    const bool on = j < hb;
    float la = 0.f, ph = 0.f;
    if (on && i < q) {
      const int h = h0 + j;
      const float a = p.A[h];
      const float rr =
          __bfloat162float(bf(p.dt)[(b * p.L + t0 + i) * p.H + h]) + (p.dt_bias ? p.dt_bias[h] : 0.f);
      const float d = softplus_precise(rr);
      la = d * a;
      ph = a != 0.f ? expm1f(la) / a : d;
    }
    float v = la;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) ts.wsum[half][wq] = v;
    __syncthreads();
    for (int w = 0; w < wq; ++w) v += ts.wsum[half][w];
    if (on) {
      ts.cs2[j][i] = v * kLog2e;
      ts.phi[j][i] = ph;
      if (i == kQ - 1) ts.total[j] = v;
    }
    __syncthreads();
  }
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int m) {
  return m == 0 ? v.x : (m == 1 ? v.y : (m == 2 ? v.z : v.w));
}
// 8 × 8 transpose of 16-bit values: in[i] is row i, out[j] receives column j.
__device__ __forceinline__ void transpose8x8(const uint4 (&in)[8], uint4 (&out)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k] = __byte_perm(word_of(in[2 * k], j >> 1), word_of(in[2 * k + 1], j >> 1), (j & 1) ? 0x7632 : 0x5410);
    out[j] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}
// hi = bf16(v·s) and lo = bf16(v·s − hi) of a bf16 pair v
__device__ __forceinline__ void scale_split_bf16x2(uint32_t v, float s, uint32_t& hi, uint32_t& lo) {
  const float a = __uint_as_float(v << 16) * s, b = __uint_as_float(v & 0xffff0000u) * s;
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Rows [0, R) × 128 columns of a K-major operand whose rows are contiguous in
// global memory (row r at g + r·stride); rows ≥ valid are zero.  cp.async.
template <int R>
__device__ __forceinline__ void stage_rows_async(unsigned char* s, const __nv_bfloat16* g, int64_t stride,
                                                 int valid) {
#pragma unroll 4
  for (int i = threadIdx.x; i < R * 16; i += kThreads) {
    const int r = i >> 4, kg = i & 15;
    const bool ok = r < valid;
    cp_async16(s + tc::kmajor_offset(R, r, kg * 8), ok ? static_cast<const void*>(g + r * stride + kg * 8) : g,
               ok ? 16 : 0);
  }
}

// Bᵀ (N rows × 128 tokens, K-major over the tokens) from B [token][n]; one core
// matrix (n group = thread % 16, token group = thread / 16) per thread.
__device__ __forceinline__ void stage_bt(unsigned char* s, const __nv_bfloat16* g, int64_t stride, int valid) {
  const int jg = threadIdx.x % (kN / 8), ig = threadIdx.x / (kN / 8);
  uint4 in[8], out[8];
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) {
    const int i = ig * 8 + ii;
    in[ii] = i < valid ? *reinterpret_cast<const uint4*>(g + i * stride + jg * 8) : make_uint4(0, 0, 0, 0);
  }
  transpose8x8(in, out);
  unsigned char* dst = s + (size_t)((ig * (kN / 8)) + jg) * 128;
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) *reinterpret_cast<uint4*>(dst + jj * 16) = out[jj];
}

// One head's X over the chunk, [token][p]: threads 0..127 each hold the 8 × 8 block
// (p group = thread % 8, token group = thread / 8), read into registers ahead of use.
__device__ __forceinline__ void load_x_block(const __nv_bfloat16* xg, int64_t stride, int valid, uint4 (&in)[8]) {
  const int jg = threadIdx.x % (kP / 8), ig = threadIdx.x / (kP / 8);
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) {
    const int i = ig * 8 + ii;
    in[ii] = i < valid ? *reinterpret_cast<const uint4*>(xg + i * stride + jg * 8) : make_uint4(0, 0, 0, 0);
  }
}
// Xᵀ (P rows × 128 tokens, K-major over the tokens) from the block of load_x_block
__device__ __forceinline__ void store_xt(unsigned char* s, const uint4 (&in)[8]) {
  const int jg = threadIdx.x % (kP / 8), ig = threadIdx.x / (kP / 8);
  uint4 out[8];
  transpose8x8(in, out);
  unsigned char* dst = s + (size_t)((ig * (kP / 8)) + jg) * 128;
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) *reinterpret_cast<uint4*>(dst + jj * 16) = out[jj];
}
// (diag(w) X)ᵀ as hi and lo terms, w = token weights of the head
__device__ __forceinline__ void store_xw(unsigned char* s_hi, unsigned char* s_lo, const uint4 (&in)[8],
                                         const float* w) {
  const int jg = threadIdx.x % (kP / 8), ig = threadIdx.x / (kP / 8);
  uint4 hi[8], lo[8], out[8];
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) {
    const float wi = w[ig * 8 + ii];
    uint32_t h[4], l[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) scale_split_bf16x2(word_of(in[ii], m), wi, h[m], l[m]);
    hi[ii] = make_uint4(h[0], h[1], h[2], h[3]);
    lo[ii] = make_uint4(l[0], l[1], l[2], l[3]);
  }
  const size_t off = (size_t)((ig * (kP / 8)) + jg) * 128;
  transpose8x8(hi, out);
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) *reinterpret_cast<uint4*>(s_hi + off + jj * 16) = out[jj];
  transpose8x8(lo, out);
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) *reinterpret_cast<uint4*>(s_lo + off + jj * 16) = out[jj];
}

// Bounded wait for an mbarrier phase; on timeout the error word is set.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const SsdArgs& p, unsigned* err) {
  const unsigned long long start = globaltimer_ns();
  for (int it = 0; it < (1 << 28); ++it) {
    if (tc::mbar_test(bar, parity)) return true;
    if ((it & 63) == 63 && (long long)(globaltimer_ns() - start) > p.timeout_ns) break;
  }
  atomicOr(err, kErrTimeout);
  return false;
}
// every thread's tcgen05 work and shared-memory writes before, the elected
// thread's tensor-core work after
__device__ __forceinline__ void sync_for_mma() {
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

// After giving up on a wait: one more commit, which completes once every MMA
// this CTA's issuing thread has started is done, and a bounded wait for it, so
// that tensor memory is not released under a running product.
__device__ __forceinline__ void drain_mmas(uint32_t bar, const SsdArgs& p, unsigned* err) {
  if (threadIdx.x == 0) tc::mma_commit(bar);
  wait_phase(bar, 0, p, err);
}

// Where the CTA sits: chunk blockIdx.x, heads h0 .. h0 + hb − 1 (one group), batch blockIdx.z.
struct CtaPos {
  int64_t b, t0;
  int c, h0, hb, g, q;
};
__device__ __forceinline__ CtaPos cta_pos(const SsdArgs& p) {
  CtaPos o;
  o.c = blockIdx.x;
  o.hb = p.heads_per_cta;
  o.h0 = blockIdx.y * o.hb;
  o.b = blockIdx.z;
  o.g = (int)(o.h0 / (p.H / p.G));
  o.t0 = (int64_t)o.c * kQ;
  o.q = (int)(p.L - o.t0 < kQ ? p.L - o.t0 : kQ);
  return o;
}

// ---------------------------------------------------------------------------
// Launch 1: each head's chunk end state H_c = Bᵀ diag(w) X and the chunk's Σ Δa.
// Bᵀ is staged once for the CTA's heads; per head the (w X)ᵀ tile and the
// tensor-memory accumulator are double-buffered, so a head's product runs while
// the previous head's state is written out and the next head's X is read.
struct StateSmem {
  unsigned char bt[kN * kQ * 2];          // Bᵀ: N rows × Q tokens, K-major
  unsigned char xw[2][2][kP * kQ * 2];    // [buffer][hi, lo] (diag(w) X)ᵀ: P rows × Q tokens
  TokenSmem ts;
  uint64_t bar, bar_drain;
  uint32_t tslot;
};
constexpr int kStateCols = 128;  // two 64-column accumulators

__global__ void __launch_bounds__(kThreads, 2) ssd_chunk_state_kernel(const SsdArgs p, const SsdWs ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  StateSmem& sm = *reinterpret_cast<StateSmem*>(smem_raw);
  const CtaPos o = cta_pos(p);
  const int warp = threadIdx.x >> 5, wq = warp & 3, hf = warp >> 2;
  const uint32_t bar = tc::smem_addr(&sm.bar), bar_drain = tc::smem_addr(&sm.bar_drain);
  if (threadIdx.x == 0) {
    tc::mbar_init1(bar);
    tc::mbar_init1(bar_drain);
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_addr(&sm.tslot), kStateCols);
  const __nv_bfloat16* xbase = bf(p.x) + (o.b * p.L + o.t0) * p.H * kP;
  const int64_t xstride = p.H * kP;
  uint4 xin[8];
  if (threadIdx.x < kQ) load_x_block(xbase + (int64_t)o.h0 * kP, xstride, o.q, xin);
  stage_bt(sm.bt, bf(p.B) + ((o.b * p.L + o.t0) * p.G + o.g) * kN, p.G * kN, o.q);
  chunk_tokens(p, o.b, o.h0, o.hb, o.t0, o.q, sm.ts);  // (its barriers publish the mbarrier's initialisation)
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tslot;
  const uint32_t idesc = tc::idesc_bf16_f32(kN, kP);
  bool ok = true;
  auto write_state = [&](int j) {  // accumulator of head j → H_c [p][n] (fp32)
    const int n = wq * 32 + (threadIdx.x & 31);
    float v[32];
    tc::tmem_ld32(tc::tmem_lane_addr(tmem + (uint32_t)((j & 1) * 64), wq * 32, hf * 32), v);
    float* dst = ws.hc + (((o.b * p.H + o.h0 + j) * p.nchunks + o.c) * kP + hf * 32) * kN + n;
#pragma unroll
    for (int k = 0; k < 32; ++k) dst[k * kN] = v[k];
    if (threadIdx.x == 0) ws.ctot[(o.b * p.H + o.h0 + j) * p.nchunks + o.c] = sm.ts.total[j];
  };
  for (int j = 0; j < o.hb; ++j) {
    const int k = j & 1;
    bool done = true;
    if (j > 0) done = wait_phase(bar, (uint32_t)((j - 1) & 1), p, ws.err);  // head j−1's product
    if (threadIdx.x < kQ) {
      // token weights w_s = 2^(cs2_end − cs2_s) φ_s of head j, over φ (each thread its own token)
      const int i = threadIdx.x;
      sm.ts.phi[j][i] *= ex2_approx(sm.ts.cs2[j][kQ - 1] - sm.ts.cs2[j][i]);
    }
    ok = __syncthreads_and(ok && done) != 0;  // the same decision in every thread
    if (!ok) break;
    tc::fence_after_sync();
    if (threadIdx.x < kQ) store_xw(sm.xw[k][0], sm.xw[k][1], xin, sm.ts.phi[j]);
    sync_for_mma();
    if (threadIdx.x == 0) {
      const uint32_t abase = tc::smem_addr(sm.bt), bhi = tc::smem_addr(sm.xw[k][0]),
                     blo = tc::smem_addr(sm.xw[k][1]), d = tmem + (uint32_t)(k * 64);
#pragma unroll
      for (int kk = 0; kk < kQ / 16; ++kk)
        tc::mma_bf16(d, tc::kslice_desc(abase, kN, kk), tc::kslice_desc(bhi, kP, kk), idesc, kk > 0);
#pragma unroll
      for (int kk = 0; kk < kQ / 16; ++kk)
        tc::mma_bf16(d, tc::kslice_desc(abase, kN, kk), tc::kslice_desc(blo, kP, kk), idesc, true);
      tc::mma_commit(bar);
    }
    if (threadIdx.x < kQ && j + 1 < o.hb) load_x_block(xbase + (int64_t)(o.h0 + j + 1) * kP, xstride, o.q, xin);
    if (j > 0) write_state(j - 1);
  }
  if (ok && o.hb > 0) ok = __syncthreads_and(wait_phase(bar, (uint32_t)((o.hb - 1) & 1), p, ws.err)) != 0;
  if (ok && o.hb > 0) {
    tc::fence_after_sync();
    write_state(o.hb - 1);
  }
  if (!ok) drain_mmas(bar_drain, p, ws.err);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kStateCols);
}

// ---------------------------------------------------------------------------
// Launch 2: states entering each chunk, one thread per (batch, head, p, n).
__global__ void __launch_bounds__(256) ssd_state_pass_kernel(const SsdArgs p, const SsdWs ws) {
  const int64_t bh = blockIdx.x;                 // b * H + h
  const int e = blockIdx.y * 256 + threadIdx.x;  // p * N + n
  float hv = p.h0 ? p.h0[bh * kP * kN + e] : 0.f;
  const int64_t nch = p.nchunks;
  const float* hc = ws.hc + bh * nch * kP * kN + e;
  const float* ct = ws.ctot + bh * nch;
  __nv_bfloat16* hin = ws.hin + bh * nch * 2 * kP * kN + e;
  auto put = [&](int64_t cc, float v) {  // hi and lo terms of the state entering chunk cc
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    hin[cc * 2 * kP * kN] = hi;
    hin[cc * 2 * kP * kN + kP * kN] = __float2bfloat16_rn(v - __bfloat162float(hi));
  };
  int64_t c = 0;
  for (; c + 4 <= nch; c += 4) {
    float hcv[4], dec[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hcv[j] = hc[(c + j) * kP * kN];
      dec[j] = expf(ct[c + j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      put(c + j, hv);
      hv = fmaf(dec[j], hv, hcv[j]);
    }
  }
  for (; c < nch; ++c) {
    put(c, hv);
    hv = fmaf(expf(ct[c]), hv, hc[c * kP * kN]);
  }
  if (p.final_state) p.final_state[bh * kP * kN + e] = hv;
}

// ---------------------------------------------------------------------------
// Launch 3: the outputs of the CTA's heads over one chunk.  S = C Bᵀ is computed
// once for all of them; per head j (buffers k = j & 1):
//   Y_in = C h_inᵀ and, once head j−1's product is done, G_j → shared memory and
//   Y = G_j X_j; head j−1's epilogue runs while head j's products do.
struct OutSmem {
  unsigned char c[kQ * kN * 2];          // C: Q rows × N, K-major (A of S and of every Y_in)
  unsigned char bg[kQ * kN * 2];         // B: Q rows × N (B of S); then G's hi term (A of Y)
  unsigned char glo[kQ * kQ * 2];        // G's lo term
  unsigned char hin[2][2][kP * kN * 2];  // [buffer][hi, lo] h_in: P rows × N (B of Y_in)
  unsigned char xt[2][kP * kQ * 2];      // [buffer] Xᵀ: P rows × Q tokens (B of Y)
  TokenSmem ts;
  uint64_t bar_s, bar_y, bar_drain, bar_never;  // bar_never: the test hook's wait (nothing arrives)
  uint32_t tslot;
};
constexpr int kColS = 0, kOutCols = 512;
__device__ __forceinline__ int col_y(int k) { return 128 + 128 * k; }
__device__ __forceinline__ int col_yin(int k) { return 192 + 128 * k; }

__global__ void __launch_bounds__(kThreads, 1) ssd_chunk_out_kernel(const SsdArgs p, const SsdWs ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  OutSmem& sm = *reinterpret_cast<OutSmem*>(smem_raw);
  const CtaPos o = cta_pos(p);
  const int warp = threadIdx.x >> 5, wq = warp & 3, hf = warp >> 2;
  const int t = wq * 32 + (threadIdx.x & 31);  // this thread's token row (tensor-memory lane)
  const uint32_t bar_s = tc::smem_addr(&sm.bar_s), bar_y = tc::smem_addr(&sm.bar_y),
                 bar_drain = tc::smem_addr(&sm.bar_drain), bar_never = tc::smem_addr(&sm.bar_never);
  if (threadIdx.x == 0) {
    tc::mbar_init1(bar_s);
    tc::mbar_init1(bar_y);
    tc::mbar_init1(bar_drain);
    tc::mbar_init1(bar_never);
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_addr(&sm.tslot), kOutCols);
  const __nv_bfloat16* hin_base = ws.hin + ((o.b * p.H + o.h0) * p.nchunks + o.c) * 2 * kP * kN;
  const int64_t hin_head = p.nchunks * 2 * kP * kN;  // from one head to the next
  auto stage_hin = [&](int j) {
    const __nv_bfloat16* g = hin_base + (int64_t)j * hin_head;
    stage_rows_async<kP>(sm.hin[j & 1][0], g, kN, kP);
    stage_rows_async<kP>(sm.hin[j & 1][1], g + kP * kN, kN, kP);
    cp_async_commit();
  };
  stage_rows_async<kQ>(sm.c, bf(p.C) + ((o.b * p.L + o.t0) * p.G + o.g) * kN, p.G * kN, o.q);
  stage_rows_async<kQ>(sm.bg, bf(p.B) + ((o.b * p.L + o.t0) * p.G + o.g) * kN, p.G * kN, o.q);
  cp_async_commit();
  stage_hin(0);
  const __nv_bfloat16* xbase = bf(p.x) + (o.b * p.L + o.t0) * p.H * kP;
  const int64_t xstride = p.H * kP;
  uint4 xin[8];
  if (threadIdx.x < kQ) load_x_block(xbase + (int64_t)o.h0 * kP, xstride, o.q, xin);
  chunk_tokens(p, o.b, o.h0, o.hb, o.t0, o.q, sm.ts);
  cp_async_wait<1>();  // C and B
  sync_for_mma();
  const uint32_t tmem = sm.tslot;
  const uint32_t a_c = tc::smem_addr(sm.c), a_bg = tc::smem_addr(sm.bg), a_glo = tc::smem_addr(sm.glo);
  const uint32_t id_s = tc::idesc_bf16_f32(kQ, kQ), id_y = tc::idesc_bf16_f32(kQ, kP);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int kk = 0; kk < kN / 16; ++kk)
      tc::mma_bf16(tmem + kColS, tc::kslice_desc(a_c, kQ, kk), tc::kslice_desc(a_bg, kQ, kk), id_s, kk > 0);
    tc::mma_commit(bar_s);
  }
  // head j's x and z at row t, columns hf·32 .. hf·32 + 31, read ahead of its epilogue
  uint4 xv[4], zv[4];
  auto prefetch_xz = [&](int j) {
    const int64_t row = ((o.b * p.L + o.t0 + t) * p.H + o.h0 + j) * kP + hf * 32;
    const uint4* xr = reinterpret_cast<const uint4*>(bf(p.x) + row);
    const uint4* zr = p.z ? reinterpret_cast<const uint4*>(bf(p.z) + row) : nullptr;
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4) {
      xv[v4] = t < o.q ? xr[v4] : make_uint4(0, 0, 0, 0);
      zv[v4] = (zr && t < o.q) ? zr[v4] : make_uint4(0, 0, 0, 0);
    }
  };
  auto epilogue = [&](int j) {  // head j's outputs, row t, columns hf·32 .. hf·32 + 31
    const int k = j & 1, h = o.h0 + j;
    float y[32], yin[32];
    tc::tmem_ld32(tc::tmem_lane_addr(tmem + (uint32_t)col_y(k), wq * 32, hf * 32), y);
    tc::tmem_ld32(tc::tmem_lane_addr(tmem + (uint32_t)col_yin(k), wq * 32, hf * 32), yin);
    if (t >= o.q) return;
    const float et = ex2_approx(sm.ts.cs2[j][t]);
    const float Dh = p.D ? p.D[h] : 0.f;
    const bool gated = p.z != nullptr;
    const int64_t row = ((o.b * p.L + o.t0 + t) * p.H + h) * kP + hf * 32;
    uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + row);
#pragma unroll
    for (int v4 = 0; v4 < 4; ++v4) {
      uint32_t ow[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t xw = word_of(xv[v4], m), zw = word_of(zv[v4], m);
        float r2[2];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int jj = v4 * 8 + m * 2 + kk;
          const float xf = __uint_as_float(kk ? (xw & 0xffff0000u) : (xw << 16));
          float yv = fmaf(et, yin[jj], y[jj]);
          yv = fmaf(Dh, xf, yv);
          if (gated) yv *= silu_fast(__uint_as_float(kk ? (zw & 0xffff0000u) : (zw << 16)));
          r2[kk] = yv;
        }
        ow[m] = pack_bf16x2(r2[0], r2[1]);
      }
      orow[v4] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
  };
  bool ok = true;
  for (int j = 0; j < o.hb; ++j) {
    const int k = j & 1;
    if (j > 0) prefetch_xz(j - 1);
    cp_async_wait<0>();  // head j's h_in
    sync_for_mma();
    if (threadIdx.x == 0) {
      const uint32_t hhi = tc::smem_addr(sm.hin[k][0]), hlo = tc::smem_addr(sm.hin[k][1]),
                     d = tmem + (uint32_t)col_yin(k);
#pragma unroll
      for (int kk = 0; kk < kN / 16; ++kk)
        tc::mma_bf16(d, tc::kslice_desc(a_c, kQ, kk), tc::kslice_desc(hhi, kP, kk), id_y, kk > 0);
#pragma unroll
      for (int kk = 0; kk < kN / 16; ++kk)
        tc::mma_bf16(d, tc::kslice_desc(a_c, kQ, kk), tc::kslice_desc(hlo, kP, kk), id_y, true);
    }
    // S (first head) or head j−1's products: G and the other buffers are free after it
    const bool done = j == 0 ? wait_phase(p.fault ? bar_never : bar_s, 0, p, ws.err)
                             : wait_phase(bar_y, (uint32_t)((j - 1) & 1), p, ws.err);
    ok = __syncthreads_and(ok && done) != 0;  // the same decision in every thread
    if (!ok) break;
    tc::fence_after_sync();
    if (j + 1 < o.hb) stage_hin(j + 1);
    if (threadIdx.x < kQ) {
      store_xt(sm.xt[k], xin);
      if (j + 1 < o.hb) load_x_block(xbase + (int64_t)(o.h0 + j + 1) * kP, xstride, o.q, xin);
    }
    // G_ts = S_ts · 2^(cs2_t − cs2_s) · φ_s for s ≤ t as hi (over B's tile) and lo terms;
    // this thread: row t, column blocks 2·hf and 2·hf + 1
    const float cst = sm.ts.cs2[j][t];
    const float* cs2 = sm.ts.cs2[j];
    const float* phi = sm.ts.phi[j];
#pragma unroll 1
    for (int bi = 0; bi < 2; ++bi) {
      const int blk = 2 * hf + bi;
      uint32_t hi[16], lo[16];
      if (blk <= wq) {  // warp-uniform: some s of the block is ≤ some t of the warp
        float v[32];
        tc::tmem_ld32(tc::tmem_lane_addr(tmem + kColS, wq * 32, blk * 32), v);
#pragma unroll
        for (int jj = 0; jj < 32; jj += 2) {
          const int s0 = blk * 32 + jj;
          const float g0 = s0 <= t ? v[jj] * ex2_approx(cst - cs2[s0]) * phi[s0] : 0.f;
          const float g1 = s0 + 1 <= t ? v[jj + 1] * ex2_approx(cst - cs2[s0 + 1]) * phi[s0 + 1] : 0.f;
          const __nv_bfloat162 gh = __floats2bfloat162_rn(g0, g1);
          const float2 ghf = __bfloat1622float2(gh);
          hi[jj / 2] = *reinterpret_cast<const uint32_t*>(&gh);
          lo[jj / 2] = pack_bf16x2(g0 - ghf.x, g1 - ghf.y);
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) hi[jj] = lo[jj] = 0u;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t off = tc::kmajor_offset(kQ, t, blk * 32 + m * 8);
        *reinterpret_cast<uint4*>(sm.bg + off) = make_uint4(hi[4 * m], hi[4 * m + 1], hi[4 * m + 2], hi[4 * m + 3]);
        *reinterpret_cast<uint4*>(sm.glo + off) = make_uint4(lo[4 * m], lo[4 * m + 1], lo[4 * m + 2], lo[4 * m + 3]);
      }
    }
    sync_for_mma();
    if (threadIdx.x == 0) {
      const uint32_t a_x = tc::smem_addr(sm.xt[k]), d = tmem + (uint32_t)col_y(k);
#pragma unroll
      for (int kk = 0; kk < kQ / 16; ++kk)
        tc::mma_bf16(d, tc::kslice_desc(a_bg, kQ, kk), tc::kslice_desc(a_x, kP, kk), id_y, kk > 0);
#pragma unroll
      for (int kk = 0; kk < kQ / 16; ++kk)
        tc::mma_bf16(d, tc::kslice_desc(a_glo, kQ, kk), tc::kslice_desc(a_x, kP, kk), id_y, true);
      tc::mma_commit(bar_y);  // covers Y_in and Y of head j
    }
    if (j > 0) epilogue(j - 1);
  }
  if (ok && o.hb > 0) prefetch_xz(o.hb - 1);
  if (ok && o.hb > 0) ok = __syncthreads_and(wait_phase(bar_y, (uint32_t)((o.hb - 1) & 1), p, ws.err)) != 0;
  if (ok && o.hb > 0) {
    tc::fence_after_sync();
    epilogue(o.hb - 1);
  }
  if (!ok) drain_mmas(bar_drain, p, ws.err);
  cp_async_wait<0>();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kOutCols);
}

}  // namespace

// The walking form (ssd_walk.cu) needs batch · heads CTAs to fill the GPU; below
// that the chunk-parallel form runs.
bool ssd_use_walk(int64_t batch, int64_t L, int64_t H) {
  const int f = runtime_knobs().force_ssd;
  if (f == 1) return true;
  if (f == 2) return false;
  (void)L;
  return batch * H >= kSsdWalkMinPairs;
}

size_t ssd_workspace_bytes(int64_t batch, int64_t L, int64_t H) {
  if (ssd_use_walk(batch, L, H)) return ssd_walk_workspace_bytes(ssd_walk_split(batch, H, L));
  const int64_t nch = (L + kQ - 1) / kQ;
  const WsSizes z = ws_sizes(batch, H, nch < 1 ? 1 : nch);
  return 256 + z.hc + z.ctot + z.hin;
}

cudaError_t ssd_launch(SsdArgs p, cudaStream_t stream) {
  if (ssd_use_walk(p.batch, p.L, p.H))
    return ssd_walk_launch(p, p.ws, stream);
  p.nchunks = (p.L + kQ - 1) / kQ;
  if (p.timeout_ns <= 0) p.timeout_ns = (long long)kDefaultTimeoutMs * 1000000ll;
  // heads per CTA: the largest divisor of the heads of a group up to kMaxHeadsPerCta
  const int64_t hpg = p.H / p.G;
  p.heads_per_cta = 1;
  for (int d = kMaxHeadsPerCta; d >= 1; --d)
    if (hpg % d == 0) {
      p.heads_per_cta = d;
      break;
    }
  const SsdWs ws = ws_layout(p.ws, p.batch, p.H, p.nchunks < 1 ? 1 : p.nchunks);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(ssd_chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(StateSmem))) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(ssd_chunk_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(OutSmem))) != cudaSuccess)
    return e;
  const dim3 grid((unsigned)p.nchunks, (unsigned)(p.H / p.heads_per_cta), (unsigned)p.batch);
  if (p.nchunks > 0) {
    ssd_chunk_state_kernel<<<grid, kThreads, sizeof(StateSmem), stream>>>(p, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  ssd_state_pass_kernel<<<dim3((unsigned)(p.batch * p.H), kP * kN / 256), 256, 0, stream>>>(p, ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.nchunks > 0) {
    ssd_chunk_out_kernel<<<grid, kThreads, sizeof(OutSmem), stream>>>(p, ws);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace ssm

// ---------------------------------------------------------------------------
// Recurrent (decode) mode of the Mamba-2 layer: one token for every (batch, head),
// the state (headdim × d_state, fp32) updated in place:
//   H ← Ā H + φ x Bᵀ,   out = (H C + D x) · silu(z)
// ("State Space Models（SSM）とMamba" §2.4 二つのモード; the per-head structure of
// §4.6 Mamba-2).  One CTA of 8 warps per (batch, head); warp w takes rows
// p = w, w + 8, ...; lane l holds states 4l .. 4l + 3 of a row (d_state 128), so a
// row's 512 bytes are one coalesced warp access, and the readout is a warp sum.
// Memory-bound: the state is read and written once.
namespace ssm {
namespace {

constexpr int kStepRowsPerIter = 8;  // rows per warp whose loads are issued together

__global__ void __launch_bounds__(256, 3) ssd_step_kernel(const SsdStepArgs p) {
  const int64_t bh = blockIdx.x;  // b * H + h
  const int64_t b = bh / p.H, h = bh % p.H, g = h / (p.H / p.G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float4* st = reinterpret_cast<float4*>(p.state + bh * p.P * kSsdState) + lane;
  const __nv_bfloat16* xr = static_cast<const __nv_bfloat16*>(p.x) + bh * p.P;
  // the first rows' states are requested before the per-head scalars are computed
  float4 s[kStepRowsPerIter];
  float xv[kStepRowsPerIter];
#pragma unroll
  for (int k = 0; k < kStepRowsPerIter; ++k) {
    const int64_t row = warp + 8 * k;
    if (row < p.P) {
      s[k] = st[row * (kSsdState / 4)];
      xv[k] = __bfloat162float(xr[row]);
    }
  }
  const __nv_bfloat16* bf_dt = static_cast<const __nv_bfloat16*>(p.dt);
  const float a = p.A[h];
  const float d = softplus_precise(__bfloat162float(bf_dt[bh]) + (p.dt_bias ? p.dt_bias[h] : 0.f));
  const float abar = expf(d * a);
  const float phi = a != 0.f ? expm1f(d * a) / a : d;
  const float Dh = p.D ? p.D[h] : 0.f;
  // this lane's four states of B and C (bf16 → fp32)
  const uint2 bw = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.B) + (b * p.G + g) * kSsdState + 4 * lane);
  const uint2 cw = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.C) + (b * p.G + g) * kSsdState + 4 * lane);
  const float Bv[4] = {__uint_as_float(bw.x << 16), __uint_as_float(bw.x & 0xffff0000u), __uint_as_float(bw.y << 16),
                       __uint_as_float(bw.y & 0xffff0000u)};
  const float Cv[4] = {__uint_as_float(cw.x << 16), __uint_as_float(cw.x & 0xffff0000u), __uint_as_float(cw.y << 16),
                       __uint_as_float(cw.y & 0xffff0000u)};
  const __nv_bfloat16* zr = p.z ? static_cast<const __nv_bfloat16*>(p.z) + bh * p.P : nullptr;
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + bh * p.P;
  for (int64_t base = warp; base < p.P; base += 8 * kStepRowsPerIter) {
    if (base != warp) {
#pragma unroll
      for (int k = 0; k < kStepRowsPerIter; ++k) {
        const int64_t row = base + 8 * k;
        if (row < p.P) {
          s[k] = st[row * (kSsdState / 4)];
          xv[k] = __bfloat162float(xr[row]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kStepRowsPerIter; ++k) {
      const int64_t row = base + 8 * k;
      if (row >= p.P) break;
      const float px = phi * xv[k];
      float4 v = s[k];
      v.x = fmaf(abar, v.x, px * Bv[0]);
      v.y = fmaf(abar, v.y, px * Bv[1]);
      v.z = fmaf(abar, v.z, px * Bv[2]);
      v.w = fmaf(abar, v.w, px * Bv[3]);
      st[row * (kSsdState / 4)] = v;
      float y = v.x * Cv[0];
      y = fmaf(v.y, Cv[1], y);
      y = fmaf(v.z, Cv[2], y);
      y = fmaf(v.w, Cv[3], y);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
      if (lane == 0) {
        y = fmaf(Dh, xv[k], y);
        if (zr) y *= silu_precise(__bfloat162float(zr[row]));
        orow[row] = __float2bfloat16_rn(y);
      }
    }
  }
}

}  // namespace

cudaError_t ssd_step_launch(const SsdStepArgs& p, cudaStream_t stream) {
  if (p.batch * p.H == 0) return cudaSuccess;
  ssd_step_kernel<<<(unsigned)(p.batch * p.H), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ssm

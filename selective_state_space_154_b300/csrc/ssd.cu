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
constexpr int kThreads = 128;
constexpr int kDefaultTimeoutMs = 2000;

static_assert(kQ == kThreads && kN == 128 && kP == 64, "tile shapes assume 128 tokens, 128 states, headdim 64");

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

// Per-token scalars of one chunk, thread i = token t0 + i.
struct TokenSmem {
  float cs2[kQ];   // inclusive prefix sums of Δa since the chunk's start, in log2 units
  float phi[kQ];   // φ of the token (0 past the sequence's end)
  float wsum[kThreads / 32];
  float total;     // Σ Δa over the chunk (natural units)
};

__device__ void chunk_tokens(const SsdArgs& p, int64_t b, int h, int64_t t0, int q, TokenSmem& ts) {
  const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
  const float a = p.A[h];
  float la = 0.f, ph = 0.f;
  if (i < q) {
    const float r = __bfloat162float(bf(p.dt)[(b * p.L + t0 + i) * p.H + h]) + (p.dt_bias ? p.dt_bias[h] : 0.f);
    const float d = softplus_precise(r);
    la = d * a;
    ph = a != 0.f ? expm1f(la) / a : d;
  }
  float v = la;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) ts.wsum[warp] = v;
  __syncthreads();
  for (int w = 0; w < warp; ++w) v += ts.wsum[w];
  ts.cs2[i] = v * kLog2e;
  ts.phi[i] = ph;
  if (i == kThreads - 1) ts.total = v;
  __syncthreads();
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

// The transpose of a [128 tokens][R] block (token i at g + i·stride, R contiguous
// values) as an R-row K-major operand over the tokens; tokens ≥ valid are zero.
// With wt given, token i's row is scaled by wt[i] and written as the two terms
// hi (to s) and lo (to s_lo).  Thread k builds core matrices k, k + 128, ...
// (column group fastest, so a warp's loads of one token are contiguous).
template <int R>
__device__ __forceinline__ void stage_transposed(unsigned char* s, unsigned char* s_lo, const __nv_bfloat16* g,
                                                 int64_t stride, int valid, const float* wt) {
  constexpr int kCores = (R / 8) * (kQ / 8);
#pragma unroll
  for (int core = threadIdx.x; core < kCores; core += kThreads) {
    const int jg = core % (R / 8), ig = core / (R / 8);
    uint4 in[8], out[8];
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) {
      const int i = ig * 8 + ii;
      in[ii] = i < valid ? *reinterpret_cast<const uint4*>(g + i * stride + jg * 8) : make_uint4(0, 0, 0, 0);
    }
    const size_t off = (size_t)((ig * (R / 8)) + jg) * 128;
    if (wt) {
      uint4 lo[8];
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        const float w = wt[ig * 8 + ii];
        uint32_t h[4], l[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) scale_split_bf16x2(word_of(in[ii], m), w, h[m], l[m]);
        in[ii] = make_uint4(h[0], h[1], h[2], h[3]);
        lo[ii] = make_uint4(l[0], l[1], l[2], l[3]);
      }
      transpose8x8(lo, out);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) *reinterpret_cast<uint4*>(s_lo + off + jj * 16) = out[jj];
    }
    transpose8x8(in, out);
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) *reinterpret_cast<uint4*>(s + off + jj * 16) = out[jj];
  }
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

// ---------------------------------------------------------------------------
// Launch 1: the chunk's own end state H_c = Bᵀ diag(w) X and its Σ Δa.
struct StateSmem {
  unsigned char bt[kN * kQ * 2];     // Bᵀ: N rows × Q tokens, K-major
  unsigned char xw[kP * kQ * 2];     // (diag(w) X)ᵀ, hi term: P rows × Q tokens, K-major
  unsigned char xw_lo[kP * kQ * 2];  // its lo term
  TokenSmem ts;
  float w[kQ];
  uint64_t bar;
  uint32_t tslot;
};

__global__ void __launch_bounds__(kThreads) ssd_chunk_state_kernel(const SsdArgs p, const SsdWs ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  StateSmem& sm = *reinterpret_cast<StateSmem*>(smem_raw);
  const int c = blockIdx.x, h = blockIdx.y;
  const int64_t b = blockIdx.z;
  const int g = (int)(h / (p.H / p.G));
  const int64_t t0 = (int64_t)c * kQ;
  const int q = (int)(p.L - t0 < kQ ? p.L - t0 : kQ);
  const int warp = threadIdx.x >> 5;
  const uint32_t bar = tc::smem_addr(&sm.bar);
  if (threadIdx.x == 0) tc::mbar_init1(bar);
  if (warp == 0) tc::tmem_alloc(tc::smem_addr(&sm.tslot), 64);
  chunk_tokens(p, b, h, t0, q, sm.ts);  // (its barriers also publish the mbarrier's initialisation)
  sm.w[threadIdx.x] = ex2_approx(sm.ts.cs2[kQ - 1] - sm.ts.cs2[threadIdx.x]) * sm.ts.phi[threadIdx.x];
  __syncthreads();
  stage_transposed<kN>(sm.bt, nullptr, bf(p.B) + ((b * p.L + t0) * p.G + g) * kN, p.G * kN, q, nullptr);
  stage_transposed<kP>(sm.xw, sm.xw_lo, bf(p.x) + ((b * p.L + t0) * p.H + h) * kP, p.H * kP, q, sm.w);
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tslot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = tc::idesc_bf16_f32(kN, kP);
    const uint32_t abase = tc::smem_addr(sm.bt), bhi = tc::smem_addr(sm.xw), blo = tc::smem_addr(sm.xw_lo);
#pragma unroll
    for (int kk = 0; kk < kQ / 16; ++kk)
      tc::mma_bf16(tmem, tc::kslice_desc(abase, kN, kk), tc::kslice_desc(bhi, kP, kk), idesc, kk > 0);
#pragma unroll
    for (int kk = 0; kk < kQ / 16; ++kk)
      tc::mma_bf16(tmem, tc::kslice_desc(abase, kN, kk), tc::kslice_desc(blo, kP, kk), idesc, true);
    tc::mma_commit(bar);
  }
  if (wait_phase(bar, 0, p, ws.err)) {
    tc::fence_after_sync();
    // thread = state row n; columns = headdim p
    const int n = threadIdx.x;
    float* dst = ws.hc + (((b * p.H + h) * p.nchunks + c) * kP) * kN + n;
#pragma unroll
    for (int half = 0; half < kP / 32; ++half) {
      float v[32];
      tc::tmem_ld32(tc::tmem_lane_addr(tmem, warp * 32, half * 32), v);
#pragma unroll
      for (int j = 0; j < 32; ++j) dst[(half * 32 + j) * kN] = v[j];
    }
    if (threadIdx.x == 0) ws.ctot[(b * p.H + h) * p.nchunks + c] = sm.ts.total;
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 64);
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
// Launch 3: the chunk's outputs.
struct OutSmem {
  unsigned char c[kQ * kN * 2];    // C: Q rows × N, K-major (A of S and of Y_in); then G's lo term
  unsigned char bg[kQ * kN * 2];   // B: Q rows × N (B of S); then G's hi term: Q rows × Q (A of Y)
  unsigned char hin[kP * kN * 2];  // h_in, hi term: P rows × N (B of Y_in); then Xᵀ: P rows × Q (B of Y)
  unsigned char hlo[kP * kN * 2];  // h_in, lo term
  TokenSmem ts;
  uint64_t bar;
  uint32_t tslot;
};
constexpr int kColS = 0, kColY = 128, kColYin = 192, kOutCols = 256;

__global__ void __launch_bounds__(kThreads) ssd_chunk_out_kernel(const SsdArgs p, const SsdWs ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  OutSmem& sm = *reinterpret_cast<OutSmem*>(smem_raw);
  const int c = blockIdx.x, h = blockIdx.y;
  const int64_t b = blockIdx.z;
  const int g = (int)(h / (p.H / p.G));
  const int64_t t0 = (int64_t)c * kQ;
  const int q = (int)(p.L - t0 < kQ ? p.L - t0 : kQ);
  const int warp = threadIdx.x >> 5;
  const uint32_t bar = tc::smem_addr(&sm.bar);
  if (threadIdx.x == 0) tc::mbar_init1(bar);
  if (warp == 0) tc::tmem_alloc(tc::smem_addr(&sm.tslot), kOutCols);
  // operands with K contiguous in global memory go by cp.async while the token scalars are computed
  stage_rows_async<kQ>(sm.c, bf(p.C) + ((b * p.L + t0) * p.G + g) * kN, p.G * kN, q);
  stage_rows_async<kQ>(sm.bg, bf(p.B) + ((b * p.L + t0) * p.G + g) * kN, p.G * kN, q);
  const __nv_bfloat16* hin_g = ws.hin + ((b * p.H + h) * p.nchunks + c) * 2 * kP * kN;
  stage_rows_async<kP>(sm.hin, hin_g, kN, kP);
  stage_rows_async<kP>(sm.hlo, hin_g + kP * kN, kN, kP);
  cp_async_commit();
  // X (B of the last product, transposed) is read now and written over h_in's
  // hi tile once the first products are done: core matrix (p group, token
  // group) = (threadIdx % 8, threadIdx / 8)
  uint4 xin[8];
  const int xjg = threadIdx.x % (kP / 8), xig = threadIdx.x / (kP / 8);
  {
    const __nv_bfloat16* xg = bf(p.x) + ((b * p.L + t0) * p.H + h) * kP;
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) {
      const int i = xig * 8 + ii;
      xin[ii] = i < q ? *reinterpret_cast<const uint4*>(xg + (int64_t)i * p.H * kP + xjg * 8) : make_uint4(0, 0, 0, 0);
    }
  }
  chunk_tokens(p, b, h, t0, q, sm.ts);
  cp_async_wait<0>();
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tslot;
  const uint32_t a_c = tc::smem_addr(sm.c), a_bg = tc::smem_addr(sm.bg), a_h = tc::smem_addr(sm.hin),
                 a_hlo = tc::smem_addr(sm.hlo), a_x = a_h;
  if (threadIdx.x == 0) {
    const uint32_t id_s = tc::idesc_bf16_f32(kQ, kQ), id_y = tc::idesc_bf16_f32(kQ, kP);
#pragma unroll
    for (int kk = 0; kk < kN / 16; ++kk)
      tc::mma_bf16(tmem + kColS, tc::kslice_desc(a_c, kQ, kk), tc::kslice_desc(a_bg, kQ, kk), id_s, kk > 0);
#pragma unroll
    for (int kk = 0; kk < kN / 16; ++kk)
      tc::mma_bf16(tmem + kColYin, tc::kslice_desc(a_c, kQ, kk), tc::kslice_desc(a_h, kP, kk), id_y, kk > 0);
#pragma unroll
    for (int kk = 0; kk < kN / 16; ++kk)
      tc::mma_bf16(tmem + kColYin, tc::kslice_desc(a_c, kQ, kk), tc::kslice_desc(a_hlo, kP, kk), id_y, true);
    tc::mma_commit(bar);
  }
  bool ok = wait_phase(bar, 0, p, ws.err);
  if (ok) {
    tc::fence_after_sync();
    {  // Xᵀ over h_in's hi tile (its product is complete)
      uint4 xo[8];
      transpose8x8(xin, xo);
      unsigned char* dst = sm.hin + (size_t)((xig * (kP / 8)) + xjg) * 128;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) *reinterpret_cast<uint4*>(dst + jj * 16) = xo[jj];
    }
    // G_ts = S_ts · 2^(cs2_t − cs2_s) · φ_s for s ≤ t, written as the K-major A
    // operand over s in two terms: hi over B's tile, lo over C's (both MMAs that
    // read them have completed)
    const int t = threadIdx.x;
    const float cst = sm.ts.cs2[t];
#pragma unroll 1
    for (int blk = 0; blk < kQ / 32; ++blk) {
      uint32_t hi[16], lo[16];
      if (blk * 32 <= warp * 32 + 31) {  // warp-uniform: some s of the block is ≤ some t of the warp
        float v[32];
        tc::tmem_ld32(tc::tmem_lane_addr(tmem + kColS, warp * 32, blk * 32), v);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int s0 = blk * 32 + j;
          const float g0 = s0 <= t ? v[j] * ex2_approx(cst - sm.ts.cs2[s0]) * sm.ts.phi[s0] : 0.f;
          const float g1 = s0 + 1 <= t ? v[j + 1] * ex2_approx(cst - sm.ts.cs2[s0 + 1]) * sm.ts.phi[s0 + 1] : 0.f;
          const __nv_bfloat162 gh = __floats2bfloat162_rn(g0, g1);
          const float2 ghf = __bfloat1622float2(gh);
          hi[j / 2] = *reinterpret_cast<const uint32_t*>(&gh);
          lo[j / 2] = pack_bf16x2(g0 - ghf.x, g1 - ghf.y);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) hi[j] = lo[j] = 0u;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t off = tc::kmajor_offset(kQ, t, blk * 32 + m * 8);
        *reinterpret_cast<uint4*>(sm.bg + off) = make_uint4(hi[4 * m], hi[4 * m + 1], hi[4 * m + 2], hi[4 * m + 3]);
        *reinterpret_cast<uint4*>(sm.c + off) = make_uint4(lo[4 * m], lo[4 * m + 1], lo[4 * m + 2], lo[4 * m + 3]);
      }
    }
  }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (ok && threadIdx.x == 0) {
    const uint32_t id_y = tc::idesc_bf16_f32(kQ, kP);
#pragma unroll
    for (int kk = 0; kk < kQ / 16; ++kk)
      tc::mma_bf16(tmem + kColY, tc::kslice_desc(a_bg, kQ, kk), tc::kslice_desc(a_x, kP, kk), id_y, kk > 0);
#pragma unroll
    for (int kk = 0; kk < kQ / 16; ++kk)
      tc::mma_bf16(tmem + kColY, tc::kslice_desc(a_c, kQ, kk), tc::kslice_desc(a_x, kP, kk), id_y, true);
    tc::mma_commit(bar);
  }
  if (ok) ok = wait_phase(bar, 1, p, ws.err);
  if (ok) {
    tc::fence_after_sync();
    const int t = threadIdx.x;
    const float et = ex2_approx(sm.ts.cs2[t]);
    const float Dh = p.D ? p.D[h] : 0.f;
    const int64_t row = ((b * p.L + t0 + t) * p.H + h) * kP;
#pragma unroll 1
    for (int half = 0; half < kP / 32; ++half) {
      float y[32], yin[32];
      tc::tmem_ld32(tc::tmem_lane_addr(tmem + kColY, warp * 32, half * 32), y);
      tc::tmem_ld32(tc::tmem_lane_addr(tmem + kColYin, warp * 32, half * 32), yin);
      if (t < q) {
        const uint4* xr = reinterpret_cast<const uint4*>(bf(p.x) + row + half * 32);
        const uint4* zr = p.z ? reinterpret_cast<const uint4*>(bf(p.z) + row + half * 32) : nullptr;
        uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + row + half * 32);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          const uint4 xv = xr[v4];
          const uint4 zv = zr ? zr[v4] : make_uint4(0, 0, 0, 0);
          uint32_t o[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t xw = word_of(xv, m), zw = word_of(zv, m);
            float r2[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int j = v4 * 8 + m * 2 + k;
              const float xf = __uint_as_float(k ? (xw & 0xffff0000u) : (xw << 16));
              float yv = fmaf(et, yin[j], y[j]);
              yv = fmaf(Dh, xf, yv);
              if (zr) yv *= silu_fast(__uint_as_float(k ? (zw & 0xffff0000u) : (zw << 16)));
              r2[k] = yv;
            }
            o[m] = pack_bf16x2(r2[0], r2[1]);
          }
          orow[v4] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kOutCols);
}

}  // namespace

size_t ssd_workspace_bytes(int64_t batch, int64_t L, int64_t H) {
  const int64_t nch = (L + kQ - 1) / kQ;
  const WsSizes z = ws_sizes(batch, H, nch < 1 ? 1 : nch);
  return 256 + z.hc + z.ctot + z.hin;
}

cudaError_t ssd_launch(SsdArgs p, cudaStream_t stream) {
  p.nchunks = (p.L + kQ - 1) / kQ;
  if (p.timeout_ns <= 0) p.timeout_ns = (long long)kDefaultTimeoutMs * 1000000ll;
  const SsdWs ws = ws_layout(p.ws, p.batch, p.H, p.nchunks < 1 ? 1 : p.nchunks);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(ssd_chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(StateSmem))) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(ssd_chunk_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(OutSmem))) != cudaSuccess)
    return e;
  if (p.nchunks > 0) {
    const dim3 grid((unsigned)p.nchunks, (unsigned)p.H, (unsigned)p.batch);
    ssd_chunk_state_kernel<<<grid, kThreads, sizeof(StateSmem), stream>>>(p, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  ssd_state_pass_kernel<<<dim3((unsigned)(p.batch * p.H), kP * kN / 256), 256, 0, stream>>>(p, ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.nchunks > 0) {
    const dim3 grid((unsigned)p.nchunks, (unsigned)p.H, (unsigned)p.batch);
    ssd_chunk_out_kernel<<<grid, kThreads, sizeof(OutSmem), stream>>>(p, ws);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace ssm

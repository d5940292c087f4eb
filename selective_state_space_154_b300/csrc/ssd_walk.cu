// The Mamba-2 layer scan (SSD) with one CTA walking the whole sequence of one
// (batch, head), for sm_103a.  The operation is the one of ssd.cu
// ("Mambaとは？Transformer以外の系列モデル", section Mamba-2とTransformerとの関係性;
// "State Space Models（SSM）とMamba" §4.6 Mamba-2): per 128-token chunk,
//   S = C Bᵀ,  G_ts = S_ts e^{Σ_{s<k≤t} Δa} φ_s (s ≤ t),
//   y_t = (G X)_t + e^{Σ_{k≤t} Δa} (C h_inᵀ)_t + D x_t, gated by silu(z_t),
//   h_out = e^{Σ Δa} h_in + Bᵀ diag(w) X,   w_s = e^{Σ_{s<k≤end} Δa} φ_s,
// with the four products on the tensor cores and the state h (headdim × d_state)
// carried from chunk to chunk in fp32 registers.  Nothing goes through global
// memory but the layer's own inputs and outputs: no chunk-state workspace and one
// launch.  The chunk-parallel form of ssd.cu is kept for problems with too few
// (batch, head) pairs to fill the GPU this way.
//
// Warp roles (18 warps):
//  * the MMA warp (one lane) issues the tensor-core products, and the load warp (one
//    lane) the tensor copies of each chunk's C, B and X tiles, each as soon as the
//    previous chunk's last reader of the tile is done; both wait on mbarriers only;
//  * 16 compute warps (tensor-memory lane quarter = warp % 4, column quarter =
//    warp / 4) build the operands the kernel computes, read the accumulators and
//    write the outputs.  Per chunk c, in order: diag(w) X (the six warps whose block
//    of G lies above the diagonal, all zeros), G (the other ten), then, while G X
//    runs, chunk c − 1's outputs and chunk c + 1's token scalars (with the decay
//    weights that spare G below the diagonal and diag(w) X an exponential per
//    element), then the state update.  Each warp
//    writes its outputs to a staging tile of its own and stores it with one tensor
//    store, so no global store of a compute thread is in flight at its next fence.
// The tensor cores run, per chunk: S, then C h_inᵀ and the chunk state Bᵀ diag(w) X
// while G is built, then G X; the next chunk's C and B are copied while G X runs,
// so its S follows right behind, and its X once G X is done.
// Handoffs are mbarriers: tensor copies complete on bar_ldcb (C, B) and bar_ldx (X),
// products on bar_a (S), bar_cb (the last reader of C and B) and bar_c (G X and all
// before it) through tcgen05.commit; the compute warps arrive (one lane per warp, 16
// arrivals) on bar_wx, bar_g and bar_h once their shared-memory writes are fenced
// for the tensor cores.
//
// Operand tiles in shared memory (tc_sm100.cuh).  The copied ones arrive by tensor
// copies of [128 tokens × 64 elements] boxes in the 128-byte swizzle, five per chunk:
//   C [t][n]   K-major A of S and of C h_inᵀ;
//   B [s][n]   K-major B of S and, read MN-major, A (= Bᵀ) of the chunk state;
//   X [s][p]   MN-major B of G X.
// The ones the compute warps write use the layout without swizzle:
//   diag(w) X [s][p] MN-major B of the chunk state;  G [t][s] K-major A of G X;
//   h [n][p]   MN-major B of C h_inᵀ.
// The operands the kernel computes (G, diag(w) X, h_in) go to the tensor cores as
// two bf16 terms, hi = bf16(v) and lo = bf16(v − hi).
// Every wait is bounded.  A timeout sets the error word (workspace byte 4) and a
// shared abort flag; from then on no wait blocks, every warp runs its loop to the
// end, the issued copies and products are drained and the CTA leaves.
#include <algorithm>
#include <cstdint>

#include <cuda_bf16.h>

#include "async_copy.cuh"
#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "tc_sm100.cuh"

namespace ssm {
namespace {

constexpr int kQ = kSsdChunk;
constexpr int kP = kSsdHeadDim;
constexpr int kN = kSsdState;
constexpr int kComputeWarps = 16;
constexpr int kCtrlWarp = kComputeWarps;      // issues the tensor-core products
constexpr int kLoadWarp = kComputeWarps + 1;  // issues the tensor copies
constexpr int kThreads = (kComputeWarps + 2) * 32;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kDefaultTimeoutMs = 2000;
constexpr uint32_t kBoxBytes = kQ * 128;                  // one [128 tokens × 64 elements] copy

static_assert(kQ == 128 && kN == 128 && kP == 64, "tile shapes assume 128 tokens, 128 states, headdim 64");

// tensor-memory columns: S (128), the chunk state (128: the products with the hi and
// the lo terms of diag(w) X side by side), Y = G X and Y_in = C h_inᵀ (64 each) in
// two buffers by chunk parity
constexpr int kColS = 0, kColHc = 128, kCols = 512;
__device__ __forceinline__ uint32_t col_y(int k) { return 256u + 128u * (uint32_t)k; }
__device__ __forceinline__ uint32_t col_yin(int k) { return 320u + 128u * (uint32_t)k; }

// named barriers (0 is __syncthreads): all compute warps; the token-scalar warps 0..3
constexpr int kBarCompute = 1, kBarTokens = 2;

// Work: CTA i < full_units walks (batch, head) unit i over the whole sequence.  The
// units left over after the launch's full rounds of CTAs are cut into seg_k segments
// of chunks each, so that the last round's few units use every SM.  The CTA of
// segment s walks its chunks twice: first for the state alone (the chunk-state
// products, no S, G or outputs; from the initial state for s = 0, from zero else),
// and publishes that end state and its total log decay in the workspace behind a
// release flag (s < seg_k − 1); then it combines the published states of segments
// 0 .. s − 1 in order (decoupled look-back: each is 2^{decay}·(state so far) + its
// own) into the state entering its chunks, and walks them in full.  The last segment
// needs no first walk.  CTAs then take their work by ticket, in the order they start.
struct WalkParams {
  CUtensorMap tm_c, tm_b, tm_x, tm_out;
  SsdArgs a;
  unsigned* err;
  int64_t full_units;
  int seg_k;
  int64_t slots;
  unsigned* seg_flag;  // [slot] 1 once the segment's state is published; then the ticket counter
  float* seg_decay;    // [slot] Σ Δa over the segment, log2 units
  float* seg_state;    // [slot][P][N] the segment's end state (fp32)
};

struct WalkSmem {
  unsigned char c[kQ * kN * 2];
  unsigned char b[kQ * kN * 2];
  unsigned char x[kQ * kP * 2];
  unsigned char g[2][kQ * kQ * 2];   // hi, lo
  unsigned char wx[2][kQ * kP * 2];  // hi, lo
  unsigned char h[2][kN * kP * 2];   // hi, lo
  unsigned char stage[kComputeWarps][16 * 32];  // each warp's outputs: 16 tokens × 16 p (bf16)
  float cs2[3][kQ];                  // by chunk mod 3: inclusive prefix sums of Δa, log2 units
  float phi[2][kQ];                  // by chunk parity: φ of the token (0 past the sequence's end)
  float ep[2][kQ];                   // by chunk parity: 2^(cs2 at the end of the token's 32-block − cs2) φ
  float wgt[2][kQ];                  // by chunk parity: w = 2^(cs2 at the chunk's end − cs2) φ
  float wsum[2][4];
  uint64_t bar_ldcb, bar_ldx, bar_a, bar_cb, bar_c, bar_wx, bar_g, bar_h, bar_drain, bar_never;
  uint32_t tslot;
  int abort;
  long long ticket;
};

__device__ __forceinline__ const __nv_bfloat16* bf(const void* p) { return static_cast<const __nv_bfloat16*>(p); }
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&r);
}
// eight fp32 values as hi and lo bf16 terms (16 bytes each)
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const __nv_bfloat162 hh = __floats2bfloat162_rn(v[2 * m], v[2 * m + 1]);
    const float2 hf = __bfloat1622float2(hh);
    h[m] = *reinterpret_cast<const uint32_t*>(&hh);
    l[m] = pack2(v[2 * m] - hf.x, v[2 * m + 1] - hf.y);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t word_of(const uint4& v, int m) {
  return m == 0 ? v.x : (m == 1 ? v.y : (m == 2 ? v.z : v.w));
}
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ bool aborted(const WalkSmem& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.abort) != 0;
}
// Bounded wait for the phase of `parity`; gives up at once if another thread has
// given up (abort flag), or sets the error word and the flag after `timeout_ns`.
// Waiting threads sleep in the barrier (up to kSleepNs per try) rather than spin.
constexpr uint32_t kSleepNs = 20000;
__device__ __forceinline__ bool wait_bar(WalkSmem& sm, uint32_t bar, uint32_t parity, long long timeout_ns,
                                         unsigned* err) {
  if (tc::mbar_test(bar, parity)) return true;
  const unsigned long long start = globaltimer_ns();
  for (int it = 0; it < (1 << 28); ++it) {
    if (tc::mbar_test_sleep(bar, parity, kSleepNs)) return true;
    if (aborted(sm)) return false;
    if ((long long)(globaltimer_ns() - start) > timeout_ns) break;
  }
  atomicOr(err, kErrTimeout);
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
  return false;
}
// the same without the abort flag: the drain after a timeout
__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity, long long timeout_ns) {
  const unsigned long long start = globaltimer_ns();
  for (int it = 0; it < (1 << 28); ++it) {
    if (tc::mbar_test(bar, parity)) return;
    if ((it & 63) == 63 && (long long)(globaltimer_ns() - start) > timeout_ns) return;
  }
}
// a compute warp's arrival: its shared-memory writes are made visible to the tensor
// cores and its tensor-memory reads are ordered before what the waiter issues
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ac::mbar_arrive(bar);
}
// the same for a warp that wrote nothing the tensor cores read since its last arrival
// (the proxy fence would wait for its global loads and stores in flight)
__device__ __forceinline__ void warp_arrive_plain(uint32_t bar) {
  tc::fence_before_sync();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ac::mbar_arrive(bar);
}

// Chunk c's C and B, two boxes each (n 0..63 and 64..127), 65,536 bytes on bar_ldcb
// (B alone for a chunk walked for its state only).
__device__ __forceinline__ void issue_cb(WalkSmem& sm, const WalkParams& w, int64_t c, int b, int g, bool with_c) {
  const uint32_t bar = ac::smem_u32(&sm.bar_ldcb);
  const int t0 = (int)(c * kQ);
  ac::mbar_arrive_expect_tx(bar, (with_c ? 4 : 2) * kBoxBytes);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (with_c) ac::tma_load_4d(ac::smem_u32(sm.c + j * kBoxBytes), &w.tm_c, j * 64, g, t0, b, bar);
    ac::tma_load_4d(ac::smem_u32(sm.b + j * kBoxBytes), &w.tm_b, j * 64, g, t0, b, bar);
  }
}
// The head's X over chunk c, one box, 16,384 bytes on bar_ldx.
__device__ __forceinline__ void issue_x(WalkSmem& sm, const WalkParams& w, int64_t c, int b, int h) {
  const uint32_t bar = ac::smem_u32(&sm.bar_ldx);
  ac::mbar_arrive_expect_tx(bar, kBoxBytes);
  ac::tma_load_4d(ac::smem_u32(sm.x), &w.tm_x, 0, h, (int)(c * kQ), b, bar);
}

__global__ void __launch_bounds__(kThreads, 1) ssd_walk_kernel(const __grid_constant__ WalkParams w) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  WalkSmem& sm = *reinterpret_cast<WalkSmem*>(smem_raw);
  const SsdArgs& p = w.a;
  const int64_t nch = p.nchunks;
  // With split units, CTAs take their work in the order they start (a ticket), so the
  // segments a segment waits for have started before it; else by index.
  if (threadIdx.x == 0)
    sm.ticket = w.seg_k > 1 ? (long long)atomicAdd(w.seg_flag + w.slots, 1u) : (long long)blockIdx.x;
  __syncthreads();
  // this CTA's (batch, head) and its chunks [c0, c0 + m); a split unit's segment seg
  int64_t bh = sm.ticket, c0 = 0, c1 = nch, slot0 = 0;
  int seg = 0, nseg = 1;
  if (bh >= w.full_units) {
    const int64_t j = bh - w.full_units;
    seg = (int)(j % w.seg_k);
    nseg = w.seg_k;
    slot0 = j - seg;  // slot of the unit's segment 0
    bh = w.full_units + j / w.seg_k;
    c0 = (int64_t)seg * nch / nseg;
    c1 = (int64_t)(seg + 1) * nch / nseg;
  }
  const int64_t m = c1 - c0;
  const bool pre = seg < nseg - 1;   // a first walk for the state alone, then publish
  const bool need_in = seg > 0;      // the state entering the chunks comes from the others
  // steps: the first walk (m chunks, state alone) if pre, then the full walk
  const int64_t nv = pre ? 2 * m : m;
  auto chunk_of = [&](int64_t v) { return c0 + (pre && v >= m ? v - m : v); };
  auto full_of = [&](int64_t v) { return !pre || v >= m; };
  const int64_t b = bh / p.H, h = bh % p.H, g = h / (p.H / p.G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wq = warp & 3, cq = warp >> 2;
  const int row = wq * 32 + lane;  // a compute thread's tensor-memory lane: token t or state n
  const uint32_t bar_ldcb = ac::smem_u32(&sm.bar_ldcb), bar_ldx = ac::smem_u32(&sm.bar_ldx),
                 bar_a = ac::smem_u32(&sm.bar_a), bar_cb = ac::smem_u32(&sm.bar_cb), bar_c = ac::smem_u32(&sm.bar_c),
                 bar_wx = ac::smem_u32(&sm.bar_wx), bar_g = ac::smem_u32(&sm.bar_g), bar_h = ac::smem_u32(&sm.bar_h),
                 bar_drain = ac::smem_u32(&sm.bar_drain), bar_never = ac::smem_u32(&sm.bar_never);
  const long long tmo = p.timeout_ns;
  const bool compute = warp < kComputeWarps;
  if (threadIdx.x == 0) {
    ac::mbar_init(bar_ldcb, 1);
    ac::mbar_init(bar_ldx, 1);
    ac::mbar_init(bar_a, 1);
    ac::mbar_init(bar_cb, 1);
    ac::mbar_init(bar_c, 1);
    ac::mbar_init(bar_wx, kComputeWarps);
    ac::mbar_init(bar_g, kComputeWarps);
    ac::mbar_init(bar_h, kComputeWarps);
    ac::mbar_init(bar_drain, 1);
    ac::mbar_init(bar_never, 1);
    ac::fence_mbar_init();
    sm.abort = 0;
  }
  if (warp == kCtrlWarp) tc::tmem_alloc(tc::smem_addr(&sm.tslot), kCols);

  // compute threads: the state h[p][n] for n = row, p = 16·cq .. 16·cq + 15
  float hs[16];
  const int64_t sbase = bh * kP * kN + (int64_t)(16 * cq) * kN + row;
  auto put_state = [&]() {  // hi and lo terms of hs into the h tile ([n][p], MN-major over p)
#pragma unroll
    for (int g2 = 0; g2 < 2; ++g2) {
      uint4 hi, lo;
      split8(hs + 8 * g2, hi, lo);
      const uint32_t off = tc::kmajor_offset(kQ, row, 16 * cq + 8 * g2);
      *reinterpret_cast<uint4*>(sm.h[0] + off) = hi;
      *reinterpret_cast<uint4*>(sm.h[1] + off) = lo;
    }
  };
  // The state entering this segment: the published end states of segments 0 .. seg − 1
  // folded in order (segment 0's is its true end state, each later one its own end state
  // from zero, added to the state so far decayed over it).  Bounded waits on the flags.
  auto combine_in = [&](float (&out)[16]) {
    for (int j = 0; j < seg; ++j) {
      const int64_t slot = slot0 + j;
      const unsigned long long start = globaltimer_ns();
      for (int it = 0; it < (1 << 28); ++it) {
        if (ld_acquire_gpu(w.seg_flag + slot) != 0u) break;
        if ((it & 15) == 15) {
          if (aborted(sm)) break;
          if ((long long)(globaltimer_ns() - start) > p.timeout_ns) {
            atomicOr(w.err, kErrTimeout);
            *reinterpret_cast<volatile int*>(&sm.abort) = 1;
            break;
          }
        }
        __nanosleep(200);
      }
      const float dec = ex2_approx(w.seg_decay[slot]);
      const float* st = w.seg_state + slot * kP * kN + (int64_t)(16 * cq) * kN + row;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) out[jj] = j == 0 ? st[jj * kN] : fmaf(dec, out[jj], st[jj * kN]);
    }
  };
  const float a = p.A[h];
  const float inv_a = a != 0.f ? 1.f / a : 0.f;
  const float bias = p.dt_bias ? p.dt_bias[h] : 0.f;
  const float Dh = p.D ? p.D[h] : 0.f;
  auto chunk_len = [&](int64_t c) { return (int)(p.L - c * kQ < kQ ? p.L - c * kQ : kQ); };
  auto load_dt = [&](int64_t v) {  // token threadIdx.x of step v's chunk (warps 0..3), 0 past the end
    const int64_t t = chunk_of(v) * kQ + threadIdx.x;
    return (v < nv && t < p.L) ? __bfloat162float(bf(p.dt)[(b * p.L + t) * p.H + h]) : 0.f;
  };
  // token scalars of step v's chunk into buffers v % 3 (cs2) and v & 1 (the others)
  // (warps 0..3, token = threadIdx.x)
  auto token_scalars = [&](int64_t step, float dtv) {
    const int i = threadIdx.x, par = (int)(step & 1);
    float la = 0.f, ph = 0.f;
    if (step < nv && i < chunk_len(chunk_of(step))) {
      // Δ = softplus(Δraw + bias) and φ = (e^{Δa} − 1)/a with the MUFU ex2 / lg2: e^x − 1
      // as 2^{x log2 e} − 1 for |x| ≥ 1/16 (relative error below 2^-18), by its series
      // to x^6 below (truncation below 2^-36)
      const float r = dtv + bias;
      const float d = r > 15.f ? r : kLn2 * lg2_approx(1.f + ex2_approx(r * kLog2e));
      la = d * a;
      if (fabsf(la) < 0.0625f) {
        const float ser = 1.f + la * (0.5f + la * (1.f / 6 + la * (1.f / 24 + la * (1.f / 120 + la * (1.f / 720)))));
        ph = d * ser;
      } else {
        ph = (ex2_approx(la * kLog2e) - 1.f) * inv_a;
      }
    }
    float v = la;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) sm.wsum[par][warp] = v;
    named_sync(kBarTokens, 128);
    float before = 0.f, total = 0.f;
    for (int k = 0; k < 4; ++k) {
      before += k < warp ? sm.wsum[par][k] : 0.f;
      total += sm.wsum[par][k];
    }
    v += before;
    const float c2 = v * kLog2e;
    // the token's 32-block is this warp's: its last prefix sum is lane 31's
    const float block_end = __shfl_sync(0xffffffffu, c2, 31);
    sm.cs2[step % 3][i] = c2;
    sm.phi[par][i] = ph;
    sm.ep[par][i] = ex2_approx(block_end - c2) * ph;
    sm.wgt[par][i] = ex2_approx(total * kLog2e - c2) * ph;
  };

  float dt_next = 0.f;
  if (compute) {
    if (!pre && need_in) {
      combine_in(hs);  // the last segment of a split unit walks once, from the others' states
    } else {
      // the initial state, or zero for the first walk of a later segment
#pragma unroll
      for (int j = 0; j < 16; ++j) hs[j] = (p.h0 && !need_in) ? p.h0[sbase + j * kN] : 0.f;
    }
    put_state();
    // G blocks above the diagonal (tokens s of column block cq all after the warp's t) stay zero
    if (cq > wq) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t off = tc::kmajor_offset(kQ, row, cq * 32 + m * 8);
        *reinterpret_cast<uint4*>(sm.g[0] + off) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sm.g[1] + off) = make_uint4(0, 0, 0, 0);
      }
    }
    if (warp < 4) {
      token_scalars(0, load_dt(0));
      dt_next = load_dt(1);
    }
    tc::fence_smem_to_async();
  }
  tc::fence_before_sync();
  __syncthreads();  // barriers initialised, tensor memory allocated, h_in and chunk 0's scalars written
  tc::fence_after_sync();
  const uint32_t tmem = sm.tslot;

  if (warp == kCtrlWarp) {
    // ------------------------------------------------------------ MMA warp, one lane
    if (lane == 0) {
      const uint32_t a_c = tc::smem_addr(sm.c), a_b = tc::smem_addr(sm.b), a_x = tc::smem_addr(sm.x);
      const uint32_t a_g0 = tc::smem_addr(sm.g[0]), a_g1 = tc::smem_addr(sm.g[1]);
      const uint32_t a_w0 = tc::smem_addr(sm.wx[0]);  // hi, then lo: one N = 128 operand
      const uint32_t a_h0 = tc::smem_addr(sm.h[0]), a_h1 = tc::smem_addr(sm.h[1]);
      const uint32_t id_s = tc::idesc_bf16_f32(kQ, kQ);                       // C · Bᵀ
      const uint32_t id_yin = tc::idesc_bf16_f32_major(kQ, kP, false, true);  // C · h_inᵀ
      const uint32_t id_hc = tc::idesc_bf16_f32_major(kN, 2 * kP, true, true);  // Bᵀ · (diag(w) X), hi | lo
      const uint32_t id_y = tc::idesc_bf16_f32_major(kQ, kP, false, true);    // G · X
      // The tiles never move, so every descriptor is its tile's K-slice-0 descriptor
      // plus a constant byte offset (the start address is the descriptor's low field).
      const uint64_t dc = tc::sw128_kslice_desc(a_c, kQ, 0), db = tc::sw128_kslice_desc(a_b, kQ, 0);
      const uint64_t dbt = tc::sw128_mn_kslice_desc(a_b, kBoxBytes, 0), dx = tc::sw128_mn_kslice_desc(a_x, kBoxBytes, 0);
      const uint64_t dh0 = tc::mn_kslice_desc(a_h0, 0), dh1 = tc::mn_kslice_desc(a_h1, 0);
      const uint64_t dw = tc::mn_kslice_desc(a_w0, 0);
      const uint64_t dg0 = tc::kslice_desc(a_g0, kQ, 0), dg1 = tc::kslice_desc(a_g1, kQ, 0);
      auto at = [](uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); };
      constexpr uint32_t kSw = (uint32_t)kQ * 128;  // 128-byte swizzle: K 64..127 column block
      for (int64_t v = 0; v < nv; ++v) {
        const uint32_t par = (uint32_t)(v & 1), prev = (uint32_t)((v - 1) & 1);
        const int k = (int)(v & 1);
        const bool full = full_of(v);  // else the chunk state alone
        // S: C and B of the chunk landed (the previous step's G has read S: bar_g awaited before its Y)
        if (!wait_bar(sm, p.fault && v == 0 ? bar_never : bar_ldcb, par, tmo, w.err)) break;
        tc::fence_after_sync();
        if (full) {
#pragma unroll
          for (int kk = 0; kk < kN / 16; ++kk) {
            const uint32_t o = (kk >> 2) * kSw + (kk & 3) * 32;
            tc::mma_bf16(tmem + kColS, at(dc, o), at(db, o), id_s, kk > 0);
          }
        }
        tc::mma_commit(bar_a);
        if (v > 0) {
          // h_in of the chunk written (and step v − 2's outputs have read Y[k], Y_in[k])
          if (!wait_bar(sm, bar_h, prev, tmo, w.err)) break;
          tc::fence_after_sync();
        }
        if (full) {
#pragma unroll
          for (int kk = 0; kk < kN / 16; ++kk)
            tc::mma_bf16(tmem + col_yin(k), at(dc, (kk >> 2) * kSw + (kk & 3) * 32), at(dh0, kk * 256), id_yin,
                         kk > 0);
#pragma unroll
          for (int kk = 0; kk < kN / 16; ++kk)
            tc::mma_bf16(tmem + col_yin(k), at(dc, (kk >> 2) * kSw + (kk & 3) * 32), at(dh1, kk * 256), id_yin,
                         true);
        }
        // the chunk state, hi and lo terms of diag(w) X side by side (N = 128)
        if (!wait_bar(sm, bar_wx, par, tmo, w.err)) break;
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kQ / 16; ++kk)
          tc::mma_bf16(tmem + kColHc, at(dbt, kk * 2048), at(dw, kk * 256), id_hc, kk > 0);
        tc::mma_commit(bar_cb);  // C and B are free once S, Y_in and the chunk state are done
        if (!wait_bar(sm, bar_g, par, tmo, w.err)) break;
        tc::fence_after_sync();
        if (full) {
#pragma unroll
          for (int kk = 0; kk < kQ / 16; ++kk)
            tc::mma_bf16(tmem + col_y(k), at(dg0, kk * 4096), at(dx, kk * 2048), id_y, kk > 0);
#pragma unroll
          for (int kk = 0; kk < kQ / 16; ++kk)
            tc::mma_bf16(tmem + col_y(k), at(dg1, kk * 4096), at(dx, kk * 2048), id_y, true);
        }
        tc::mma_commit(bar_c);  // covers Y_in, the chunk state and Y
      }
    }
    __syncwarp();
  } else if (warp == kLoadWarp) {
    // ------------------------------------------------------------ load warp, one lane
    if (lane == 0 && nch > 0) {
      ac::prefetch_tensormap(&w.tm_c);
      ac::prefetch_tensormap(&w.tm_b);
      ac::prefetch_tensormap(&w.tm_x);
      issue_cb(sm, w, chunk_of(0), (int)b, (int)g, full_of(0));
      issue_x(sm, w, chunk_of(0), (int)b, (int)h);
      int64_t cb_issued = 1, x_issued = 1;
      for (int64_t v = 1; v < nv; ++v) {
        const uint32_t prev = (uint32_t)((v - 1) & 1);
        // C and B take step v's chunk once step v − 1's S, C h_inᵀ and chunk state are done
        if (!wait_bar(sm, bar_cb, prev, tmo, w.err)) break;
        issue_cb(sm, w, chunk_of(v), (int)b, (int)g, full_of(v));
        cb_issued = v + 1;
        // X takes it once step v − 1's G X (and diag(w) X, before it) are done
        if (!wait_bar(sm, bar_c, prev, tmo, w.err)) break;
        issue_x(sm, w, chunk_of(v), (int)b, (int)h);
        x_issued = v + 1;
      }
      // the last copies have landed before the CTA leaves (at once unless a wait timed out)
      wait_bar_drain(bar_ldcb, (uint32_t)((cb_issued - 1) & 1), tmo);
      wait_bar_drain(bar_ldx, (uint32_t)((x_issued - 1) & 1), tmo);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps
    const int widx = cq > wq ? cq * (cq - 1) / 2 + wq : -1;  // the six warps that build diag(w) X
    unsigned char* stage = sm.stage[warp];
    // Outputs of chunk oc: token rows 32·wq .., p = 16·cq .. 16·cq + 15 of this warp,
    // through its staging tile and one tensor store (rows past L are clipped).
    // x and z of this thread's outputs of chunk oc (token row, p = 16·cq ..), zero past the end
    auto load_xz = [&](int64_t ov, uint4 (&xv)[2], uint4 (&zv)[2]) {
      const int64_t oc = chunk_of(ov);
      const int64_t off = ((b * p.L + oc * kQ + row) * p.H + h) * kP + 16 * cq;
      const bool in = row < chunk_len(oc);
      const uint4* xr = reinterpret_cast<const uint4*>(bf(p.x) + off);
      const uint4* zr = p.z ? reinterpret_cast<const uint4*>(bf(p.z) + off) : nullptr;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        xv[m] = in ? xr[m] : make_uint4(0, 0, 0, 0);
        zv[m] = (in && zr) ? zr[m] : make_uint4(0, 0, 0, 0);
      }
    };
    auto outputs = [&](int64_t ov, bool ok, const uint4 (&xv)[2], const uint4 (&zv)[2]) {
      const int ok_k = (int)(ov & 1), t0 = (int)(chunk_of(ov) * kQ);
      float y[16], yi[16];
      tc::tmem_ld16(tc::tmem_lane_addr(tmem + col_y(ok_k), wq * 32, cq * 16), y);
      tc::tmem_ld16(tc::tmem_lane_addr(tmem + col_yin(ok_k), wq * 32, cq * 16), yi);
      const float et = ex2_approx(sm.cs2[ov % 3][row]);
      uint32_t ow[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint32_t xw = word_of(xv[m >> 2], m & 3), zw = word_of(zv[m >> 2], m & 3);
        float r2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = 2 * m + e;
          float yv = fmaf(et, yi[j], y[j]);
          yv = fmaf(Dh, e ? bf_hi(xw) : bf_lo(xw), yv);
          if (p.z) {
            const float hz = 0.5f * (e ? bf_hi(zw) : bf_lo(zw));
            yv *= fmaf(hz, tanh_approx(hz), hz);  // silu(z) = z/2 + (z/2)·tanh(z/2)
          }
          r2[e] = yv;
        }
        ow[m] = pack2(r2[0], r2[1]);
      }
      // two stores of 16 token rows each through the warp's staging tile, which is free
      // once the previous store has read it
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if (lane == 0) ac::bulk_wait_read0();
        __syncwarp();
        if ((lane >> 4) == half) {
          *reinterpret_cast<uint4*>(stage + (lane & 15) * 32) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
          *reinterpret_cast<uint4*>(stage + (lane & 15) * 32 + 16) = make_uint4(ow[4], ow[5], ow[6], ow[7]);
        }
        ac::fence_proxy_async_smem();
        __syncwarp();
        const int r0 = t0 + 32 * wq + 16 * half;
        if (lane == 0 && ok && r0 < p.L && !aborted(sm)) {
          ac::tma_store_4d(&w.tm_out, ac::smem_u32(stage), 16 * cq, (int)h, r0, (int)b);
          ac::bulk_commit();
        }
      }
    };
    float logdec = 0.f;  // Σ Δa over the first walk so far, log2 units
    for (int64_t v = 0; v < nv; ++v) {
      const uint32_t par = (uint32_t)(v & 1);
      const bool full = full_of(v), prev_out = v > 0 && full_of(v - 1);
      named_sync(kBarCompute, kComputeThreads);  // step v's scalars visible
      const float* cs2 = sm.cs2[v % 3];
      const float* phi = sm.phi[v & 1];
      const float cs_end = cs2[kQ - 1];
      uint4 xv[2], zv[2];
      if (widx >= 0) {
        // diag(w) X as hi and lo terms, w_s = 2^(cs2_end − cs2_s) φ_s; 16-byte granules
        // (8 p of token s), consecutive threads on consecutive tokens
        if (__all_sync(0xffffffffu, wait_bar(sm, bar_ldx, par, tmo, w.err))) {
#pragma unroll 1
          for (int i = widx * 32 + lane; i < kQ * kP / 8; i += 6 * 32) {
            const int s = i & (kQ - 1), pg = i >> 7;
            const uint32_t off = tc::kmajor_offset(kQ, s, pg * 8);
            // X granule pg of token s in the 128-byte swizzle of its tensor copy
            const uint4 xw = *reinterpret_cast<const uint4*>(sm.x + s * 128 + ((pg ^ (s & 7)) << 4));
            const float wgt = sm.wgt[v & 1][s];
            float f[8];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              f[2 * m] = bf_lo(word_of(xw, m)) * wgt;
              f[2 * m + 1] = bf_hi(word_of(xw, m)) * wgt;
            }
            uint4 hi, lo;
            split8(f, hi, lo);
            *reinterpret_cast<uint4*>(sm.wx[0] + off) = hi;
            *reinterpret_cast<uint4*>(sm.wx[1] + off) = lo;
          }
        }
        warp_arrive(bar_wx);
        warp_arrive_plain(bar_g);
        if (prev_out) load_xz(v - 1, xv, zv);
      } else if (!full) {  // a chunk walked for its state: no G (bar_a still awaited, phase by phase)
        warp_arrive_plain(bar_wx);
        (void)__all_sync(0xffffffffu, wait_bar(sm, bar_a, par, tmo, w.err));
        warp_arrive_plain(bar_g);
      } else {
        warp_arrive_plain(bar_wx);
        if (prev_out) load_xz(v - 1, xv, zv);  // read ahead of the wait for S
        // G_ts for this thread's token row t and tokens s = 32·cq .. 32·cq + 31 (s ≤ t)
        const bool ok = __all_sync(0xffffffffu, wait_bar(sm, bar_a, par, tmo, w.err));
        tc::fence_after_sync();
        float sv[32];
        tc::tmem_ld32(tc::tmem_lane_addr(tmem + kColS, wq * 32, cq * 32), sv);
        if (ok) {
          const int t = row;
          const float cst = cs2[t];
          const bool diag = cq == wq;
          // below the diagonal every s of the block is before t:
          // 2^(cs2_t − cs2_s) φ_s = 2^(cs2_t − cs2_end(block)) · ep_s, both factors ≤ 1
          const float ft = ex2_approx(cst - cs2[cq * 32 + 31]);
          const float* ep = sm.ep[v & 1];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int s0 = cq * 32 + m * 8;
            float f[8];
            if (diag) {
              const float4 ca = *reinterpret_cast<const float4*>(cs2 + s0);
              const float4 cb = *reinterpret_cast<const float4*>(cs2 + s0 + 4);
              const float4 pa = *reinterpret_cast<const float4*>(phi + s0);
              const float4 pb = *reinterpret_cast<const float4*>(phi + s0 + 4);
              const float cv[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
              const float pv[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = s0 + e <= t ? sv[m * 8 + e] * ex2_approx(cst - cv[e]) * pv[e] : 0.f;
            } else {
              const float4 ea = *reinterpret_cast<const float4*>(ep + s0);
              const float4 eb = *reinterpret_cast<const float4*>(ep + s0 + 4);
              const float ev[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = sv[m * 8 + e] * ft * ev[e];
            }
            uint4 hi, lo;
            split8(f, hi, lo);
            const uint32_t off = tc::kmajor_offset(kQ, t, s0);
            *reinterpret_cast<uint4*>(sm.g[0] + off) = hi;
            *reinterpret_cast<uint4*>(sm.g[1] + off) = lo;
          }
        }
        warp_arrive(bar_g);
      }
      // while G X runs: the previous chunk's outputs, the next chunk's token scalars
      if (prev_out) outputs(v - 1, true, xv, zv);
      if (warp < 4) {
        token_scalars(v + 1, dt_next);
        dt_next = load_dt(v + 2);
      }
      // chunk c's products done: the state entering chunk c + 1
      const bool okc = __all_sync(0xffffffffu, wait_bar(sm, bar_c, par, tmo, w.err));
      tc::fence_after_sync();
      {
        float hc[16], hl[16];
        tc::tmem_ld16(tc::tmem_lane_addr(tmem + kColHc, wq * 32, cq * 16), hc);
        tc::tmem_ld16(tc::tmem_lane_addr(tmem + kColHc + kP, wq * 32, cq * 16), hl);
        const float dec = ex2_approx(cs_end);
#pragma unroll
        for (int j = 0; j < 16; ++j) hs[j] = fmaf(dec, hs[j], hc[j] + hl[j]);
        if (!full) logdec += cs_end;
        if (pre && v == m - 1) {
          // the first walk is done: publish its end state, then start the full walk from the
          // initial state (segment 0) or from the combined states of the segments before
          const int64_t slot = slot0 + seg;
#pragma unroll
          for (int j = 0; j < 16; ++j) w.seg_state[slot * kP * kN + (16 * cq + j) * kN + row] = hs[j];
          if (threadIdx.x == 0) w.seg_decay[slot] = logdec;
          __threadfence();
          named_sync(kBarCompute, kComputeThreads);
          if (threadIdx.x == 0) st_release_gpu(w.seg_flag + slot, 1u);
          if (need_in) {
            combine_in(hs);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) hs[j] = p.h0 ? p.h0[sbase + j * kN] : 0.f;
          }
        }
        put_state();
      }
      warp_arrive(bar_h);  // h_in of the next step written; step v − 1's outputs read Y, Y_in
      if (v + 1 == nv) {
        load_xz(v, xv, zv);
        outputs(v, okc, xv, zv);
      }
    }
    // every tensor store of this warp has completed before the CTA leaves
    if (lane == 0) ac::bulk_wait0();
    __syncwarp();
    if (!aborted(sm) && p.final_state && seg == nseg - 1) {
#pragma unroll
      for (int j = 0; j < 16; ++j) p.final_state[sbase + j * kN] = hs[j];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  // every product this CTA issued is complete before tensor memory is released
  if (warp == kCtrlWarp) {
    if (lane == 0 && nch > 0) {
      tc::mma_commit(bar_drain);
      wait_bar_drain(bar_drain, 0, tmo);
    }
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kCols);
  }
}

}  // namespace

WalkSplit ssd_walk_split(int64_t batch, int64_t H, int64_t L) {
  WalkSplit sp{};
  const int64_t units = batch * H, nch = (L + kQ - 1) / kQ;
  sp.full_units = units;
  sp.seg_k = 1;
  const int force = runtime_knobs().ssd_split;
  if (force > 0) {
    sp.full_units = 0;
    sp.seg_k = (int)(force < nch ? force : (nch > 0 ? nch : 1));
  } else if (nch >= 2) {
    // one CTA per SM: the units beyond the last full round of SMs are cut into segments
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0) {
      (void)cudaGetLastError();
      sms = 148;  // no device to ask (sizing only): a B300
    }
    const int64_t rem = units % sms;
    const int64_t k = rem > 0 ? std::min<int64_t>(nch, sms / rem) : 1;
    if (k > 1) {
      sp.full_units = units - rem;
      sp.seg_k = (int)k;
    }
  }
  sp.slots = sp.seg_k > 1 ? (units - sp.full_units) * sp.seg_k : 0;
  return sp;
}

// Workspace: 256 bytes of error words | flags [slots] and the ticket counter | decays
// [slots] | states [slots][P][N]; only the error words when no unit is split
size_t ssd_walk_workspace_bytes(const WalkSplit& sp) {
  if (sp.slots == 0) return 256;
  auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
  return 256 + al((size_t)(sp.slots + 1) * 4) + al((size_t)sp.slots * 4) + (size_t)sp.slots * kP * kN * 4;
}

cudaError_t ssd_walk_launch(SsdArgs p, void* ws, cudaStream_t stream) {
  p.nchunks = (p.L + kQ - 1) / kQ;
  if (p.timeout_ns <= 0) p.timeout_ns = (long long)kDefaultTimeoutMs * 1000000ll;
  WalkParams w{};
  w.a = p;
  unsigned char* base = static_cast<unsigned char*>(ws);
  w.err = reinterpret_cast<unsigned*>(base) + 1;
  const WalkSplit sp = ssd_walk_split(p.batch, p.H, p.L);
  w.full_units = sp.full_units;
  w.seg_k = sp.seg_k;
  w.slots = sp.slots;
  auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
  w.seg_flag = reinterpret_cast<unsigned*>(base + 256);
  w.seg_decay = reinterpret_cast<float*>(base + 256 + al((size_t)(sp.slots + 1) * 4));
  w.seg_state = reinterpret_cast<float*>(base + 256 + al((size_t)(sp.slots + 1) * 4) + al((size_t)sp.slots * 4));
  cudaError_t e;
  if (sp.slots > 0 && (e = cudaMemsetAsync(w.seg_flag, 0, (size_t)(sp.slots + 1) * 4, stream)) != cudaSuccess)
    return e;
  if (p.L > 0) {
    const CUtensorMapDataType bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    const CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
    // C, B [batch][L][G][N] and X [batch][L][H][P]: boxes of 64 elements × 1 × 128 tokens × 1
    // in the 128-byte swizzle; tokens past L read as zeros
    const uint64_t dims_bc[4] = {(uint64_t)kN, (uint64_t)p.G, (uint64_t)p.L, (uint64_t)p.batch};
    const uint64_t str_bc[3] = {(uint64_t)kN * 2, (uint64_t)(p.G * kN * 2), (uint64_t)(p.L * p.G * kN * 2)};
    const uint64_t dims_x[4] = {(uint64_t)kP, (uint64_t)p.H, (uint64_t)p.L, (uint64_t)p.batch};
    const uint64_t str_x[3] = {(uint64_t)kP * 2, (uint64_t)(p.H * kP * 2), (uint64_t)(p.L * p.H * kP * 2)};
    const uint32_t box[4] = {64, 1, (uint32_t)kQ, 1};
    const uint32_t box_out[4] = {16, 1, 16, 1};  // 16 tokens × 16 p of a compute warp
    if (!encode_tensor_map(&w.tm_c, bf16, 4, p.C, dims_bc, str_bc, box, sw, promo) ||
        !encode_tensor_map(&w.tm_b, bf16, 4, p.B, dims_bc, str_bc, box, sw, promo) ||
        !encode_tensor_map(&w.tm_x, bf16, 4, p.x, dims_x, str_x, box, sw, promo) ||
        !encode_tensor_map(&w.tm_out, bf16, 4, p.out, dims_x, str_x, box_out, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE))
      return cudaErrorInvalidValue;
  }
  if ((e = cudaFuncSetAttribute(ssd_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(WalkSmem))) != cudaSuccess)
    return e;
  const int64_t grid = sp.full_units + (p.batch * p.H - sp.full_units) * sp.seg_k;
  ssd_walk_kernel<<<(unsigned)grid, kThreads, sizeof(WalkSmem), stream>>>(w);
  return cudaGetLastError();
}

}  // namespace ssm

// Selective-scan forward, bf16 activations, d_state 16: the streamed row kernel (sm_103a).
//
// The operation is the one of scan_fwd.cu ("State Space Models（SSM）とMamba" §2.2 離散化;
// "Mambaとは？Transformer以外の系列モデル", sections 状態空間モデルを一つの式から理解する
// and Mamba blockのarchitecture).  Organisation:
//  * one thread per (batch, channel) row holds the row's 16 states, A and 1/A in
//    registers; the readout Σ_n C_n h_n needs no other thread;
//  * a CTA owns RB rows of one batch over one chunk of the sequence, walked in stages
//    of 32 tokens, and no warp ever waits for another warp's rows:
//      - each warp copies its own 32 rows' u, Δraw and z tiles ([32 rows × 32 tokens]
//        tensor copies issued by its lane 0, counted on an mbarrier of its own) into a
//        double buffer of its own, one stage ahead, and writes its outputs back the same
//        way: in place of u in shared memory, then one tensor store;
//      - B and C of a stage, shared by all rows, come by tensor (TMA) copy into a ring of
//        four stages; the warp that releases a stage last refills it, and every warp
//        converts a share of each stage to fp32 two stages before its use (an mbarrier
//        counts the shares);
//  * the step size enters the exponent in base 2: Δ' = log2(1 + 2^{(Δraw+bias)·log2 e})
//    = Δ / ln 2, so Ā_n = 2^{Δ'·A_n} with no further scaling, and Σ Δ' is the chunk's
//    decay exponent;
//  * chunks compose as affine maps, (A₂,b₂)∘(A₁,b₁) = (A₂A₁, A₂b₁+b₂) ("Mambaとは？…",
//    Selective Scanは選択機構そのものではない).  Every chunk first scans from h = 0
//    keeping S = ΣΔ', then each warp publishes (S, h_local) for its 32 rows and
//    combines those of all preceding chunks, in a fixed order, into its carried-in
//    state h_in; its end state is 2^{A S}·h_in + h_local.  The chunk's first blocks,
//    those whose outputs h_in still changes (2^{A_n S} ≥ 2^-12 for the slowest-decaying
//    state, bf16 outputs), are not written by the first pass: a second pass scans them
//    again from h_in and writes them, so every output is rounded once.  How many
//    stages the second pass needs is known during the first, so its copies start
//    before the carry is combined.
#include "async_copy.cuh"
#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <mutex>

namespace ssm {

namespace {
thread_local int g_driver_error = 0;  // CUresult of this thread's last failed driver call
}  // namespace

int take_driver_error() {
  const int e = g_driver_error;
  g_driver_error = 0;
  return e;
}

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
  using Fn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                          const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                          CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(f);
  });
  if (!fn) {
    g_driver_error = (int)CUDA_ERROR_NOT_FOUND;
    return false;
  }
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  const CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, e,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) g_driver_error = (int)r;
  return r == CUDA_SUCCESS;
}

namespace {

constexpr int NS = 16;        // states per row

// Stage geometry: TS = 32 tokens per stage.  Each warp double-buffers its own 32 rows'
// tiles (64 bytes of a row per tensor and stage, copied by the warp itself); B and C
// of a stage, shared by all rows, sit in a ring of NB = 4 stages filled by tensor
// copies and converted to fp32 kAhead = 2 stages before their use.
constexpr int TS = kStreamTokensPerStage;
constexpr int NB = 4;
constexpr int kAhead = 2;
constexpr int kRowBytes = TS * 2;
// 16-byte granule g of row r of a tile: XOR-swizzled by (r / 2) mod 4, so that eight
// lanes reading the same granule of eight consecutive rows hit different banks
__device__ __forceinline__ int swz(int r, int g) { return g ^ ((r >> 1) & 3); }

// Work items: the (row tile, stage) pairs of all tiles, tile after tile, cut into `items`
// ranges of nearly equal length; item j holds flattened stages [j·ptot/items,
// (j+1)·ptot/items).  A range lies in one tile or straddles two; the part of a range in
// one tile is a segment of that tile's sequence (a chunk), and the segments of a tile,
// in order, belong to consecutive items.
struct StreamParams {
  CUtensorMap tm_b, tm_c, tm_out;
  CUtensorMap tm_u, tm_d, tm_z;  // the row tensors, [32 rows × 32 tokens] boxes in the tiles' swizzle
  ScanArgs a;
  int rtiles;   // row tiles per batch
  int sl;       // stages per tile (ceil(L / 32))
  int items;    // work items (CTAs)
  int multi;    // some tile has more than one segment (the carry and the workspace are used)
  int64_t ptot; // flattened stages: batch · rtiles · sl
  StreamWs ws;
  long long timeout_ns;
  int fault_lookback;
};

// A segment of one tile's sequence as one work item sees it.
struct Segment {
  int tile;      // row tile, batch-major
  int s0, s1;    // its stages [s0, s1) of the tile's sequence
  int q;         // its index among the tile's segments (0: starts from the initial state)
  int64_t slot;  // where its aggregate is published
  int64_t item;  // the work item holding it
};

// Shared memory of one CTA (the dynamic allocation is aligned up to 1024 bytes).
template <int RB>
struct StreamSmem {
  uint8_t tile[2][3][RB * kRowBytes];  // [buffer][u|Δraw|z][row][TS tokens], swizzled; warp w owns rows 32w..32w+31
  uint16_t bc_raw[NB][2][TS * NS];     // [stage][B|C][token][state] bf16
  float bcf[NB][TS][2 * NS];           // [stage][token][B 0..15 | C 0..15] fp32
  uint64_t full[NB];  // the stage's B and C copies landed (bytes counted)
  uint64_t conv[NB];  // every warp converted its share of the stage's B and C
  uint64_t settled;   // every warp knows how far pass two must go
  uint64_t rowbar[RB / 32][2];  // [warp][buffer]: the warp's row tiles of a stage landed (bytes counted)
  int rissued[RB / 32];         // ring stages whose row tiles the warp has requested (the last + 1)
  int done[NB];       // warps that released the stage's B and C
  int n2;             // stages of the second pass (max over warps)
  int issued;         // B/C stages issued so far (the last one + 1)
  int nseg;           // this CTA's segments: 1, or 2 (the next tile's first one runs first)
  Segment seg[2];
};
template <int RB>
constexpr size_t stream_smem_bytes() {
  return sizeof(StreamSmem<RB>) + 1024;
}

__device__ __forceinline__ float bf_lo(unsigned w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(unsigned w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ bool wait_flag(const unsigned* flag, unsigned want, long long timeout_ns,
                                          unsigned* value) {
  const unsigned long long start = ac::globaltimer();
  unsigned ns = 32;
  for (long long it = 0; it < (1ll << 28); ++it) {
    const unsigned v = ld_acquire_gpu(flag);
    if (v >= want) {
      *value = v;
      return true;
    }
    if ((long long)(ac::globaltimer() - start) > timeout_ns) break;
    __nanosleep(ns);
    ns = ns < 256 ? ns * 2 : ns;
  }
  return false;
}

enum StreamPass {
  kAll = 0,        // the first chunk: every block written, S not needed
  kSettled = 1,    // other chunks, pass one from h = 0: the settled blocks
  kUnsettled = 2,  // other chunks, pass two from h_in: the rest
};

// Per-thread (row) constants.
struct RowConst {
  float a2[NS], ia[NS];  // A (the exponent base is 2: Ā = 2^{Δ' A}) and 1/A; 0 for A = 0
  float a2max, Dc, bl2;  // slowest decay, D, bias · log2 e
  bool precise;          // a row of this warp has an A = 0 state: the exact branch
  bool row_ok;
};

// What every warp knows about its CTA's stages: the chunk's tokens and stage counts.
// Stage k < n1 is pass one's stage k, stage n1 + i pass two's stage i (tokens from the
// chunk start again).  Copies for the first stages of pass two are issued before pass
// two's length is known (every chunk after the first re-scans at least one stage);
// later ones once it is.
struct Ring {
  const StreamParams* p;
  unsigned long long deadline;
  int c0, b, tc0, tc1, n1;
  int kb;         // ring stages the CTA used before this segment (the ring's slots and phases run on)
  int spec_rows;  // row-tile stages a warp may copy without knowing pass two's length
  int spec_bc;    // B/C stages that may be issued without knowing it
};

__device__ __forceinline__ int stage_t0(const Ring& g, int k) { return g.tc0 + (k < g.n1 ? k : k - g.n1) * TS; }
// position of the segment's stage k in the CTA's ring (buffer k & 1, B/C slot k % NB)
__device__ __forceinline__ int ring(const Ring& g, int k) { return g.kb + k; }

// This warp's 32 rows of stage k's u, Δraw, z tiles into row buffer k % 2: three tensor
// copies of [32 rows × 32 tokens] issued by lane 0, completion counted in bytes on the
// warp's mbarrier of that buffer (rows past d_inner and tokens past the sequence are
// zero-filled).  The boxes land in the tiles' 64-byte swizzle, the layout swz() reads.
template <int RB, bool HAS_Z>
__device__ __forceinline__ void rows_issue(StreamSmem<RB>& sm, const Ring& g, int k, int warp, int lane) {
  if (lane != 0) return;
  const StreamParams& p = *g.p;
  const int rk = ring(g, k), buf = rk & 1;
  const uint32_t bar = ac::smem_u32(&sm.rowbar[warp][buf]);
  constexpr int ntens = HAS_Z ? 3 : 2;
  ac::mbar_arrive_expect_tx(bar, (uint32_t)(ntens * 32 * kRowBytes));
  const int t0 = stage_t0(g, k), y = g.c0 + 32 * warp;
  ac::tma_load_3d(ac::smem_u32(sm.tile[buf][0] + 32 * warp * kRowBytes), &p.tm_u, t0, y, g.b, bar);
  ac::tma_load_3d(ac::smem_u32(sm.tile[buf][1] + 32 * warp * kRowBytes), &p.tm_d, t0, y, g.b, bar);
  if (HAS_Z) ac::tma_load_3d(ac::smem_u32(sm.tile[buf][2] + 32 * warp * kRowBytes), &p.tm_z, t0, y, g.b, bar);
  sm.rissued[warp] = rk + 1;
}

// Lane 0: wait until every row-tile copy this warp requested has landed (the ones a
// second pass shorter than its speculation never consumed included).
template <int RB>
__device__ __forceinline__ bool rows_drain(StreamSmem<RB>& sm, int warp, unsigned long long deadline) {
  bool ok = true;
  const int n = sm.rissued[warp];
  for (int j = n - 2 < 0 ? 0 : n - 2; j < n; ++j)
    ok = ac::mbar_wait(ac::smem_u32(&sm.rowbar[warp][j & 1]), (uint32_t)(j >> 1) & 1u, deadline) && ok;
  return ok;
}

// Issue the tensor copies of stage j's B and C (one thread).
template <int RB>
__device__ __forceinline__ void bc_issue(StreamSmem<RB>& sm, const Ring& g, int j) {
  const int s = ring(g, j) % NB;
  const int t0 = stage_t0(g, j);
  const StreamParams& p = *g.p;
  const uint32_t fb = ac::smem_u32(&sm.full[s]);
  ac::mbar_arrive_expect_tx(fb, (uint32_t)(2 * TS * NS * 2));
  ac::tma_load_3d(ac::smem_u32(sm.bc_raw[s][0]), &p.tm_b, 0, t0, g.b, fb);
  ac::tma_load_3d(ac::smem_u32(sm.bc_raw[s][1]), &p.tm_c, 0, t0, g.b, fb);
  atomicMax(&sm.issued, ring(g, j) + 1);
}

// This warp's share of stage j's B and C to fp32: [B|C][token][state] -> [token][B | C].
template <int RB>
__device__ __forceinline__ void bc_convert(StreamSmem<RB>& sm, const Ring& g, int j, int warp, int lane, int& err) {
  constexpr int NW = RB / 32;
  constexpr int kWords = TS * NS;      // 32-bit words of B and C together
  constexpr int kShare = kWords / NW;  // words per warp
  const int s = ring(g, j) % NB;
  if (!ac::mbar_wait(ac::smem_u32(&sm.full[s]), (uint32_t)(ring(g, j) / NB) & 1u, g.deadline)) err = 1;
  const unsigned* raw = reinterpret_cast<const unsigned*>(sm.bc_raw[s][0]);
#pragma unroll
  for (int q = 0; q < (kShare + 31) / 32; ++q) {
    const int k = lane + 32 * q;
    if (kShare % 32 == 0 || k < kShare) {
      const int i = warp * kShare + k;  // word i: tensor i / (kWords / 2), token (i mod kWords/2) / 8, pair i mod 8
      const unsigned wv = raw[i];
      const int w = i / (kWords / 2), tok = (i % (kWords / 2)) / (NS / 2), np = i % (NS / 2);
      *reinterpret_cast<float2*>(&sm.bcf[s][tok][w * NS + 2 * np]) = make_float2(bf_lo(wv), bf_hi(wv));
    }
  }
  __syncwarp();
  if (lane == 0) ac::mbar_arrive(ac::smem_u32(&sm.conv[s]));
}

// Whether stage j is ever used: pass one, the first stages of pass two, or pass two's
// remaining stages once its length n2 (< 0: unknown) is known.
__device__ __forceinline__ bool stage_has(int j, int spec_end, int n1, int n2) {
  return j < spec_end || (n2 >= 0 && j < n1 + n2);
}

// After this warp finished stage k: copy its rows of stage k + 2 into the row buffer
// just freed; release stage k's B and C (the warp releasing them last issues the copies
// of stage k + NB into that slot) and convert its share of stage k + kAhead.
template <int RB, bool HAS_Z>
__device__ __forceinline__ void stage_advance(StreamSmem<RB>& sm, const Ring& g, int k, int n2, int warp, int lane,
                                              int& err) {
  constexpr int NW = RB / 32;
  if (lane == 0) ac::bulk_wait_read0();  // the tensor store has read stage k's outputs out of the buffer
  __syncwarp();
  if (stage_has(k + 2, g.spec_rows, g.n1, n2)) rows_issue<RB, HAS_Z>(sm, g, k + 2, warp, lane);
  const int s = ring(g, k) % NB;
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();  // this warp's reads of the slot precede its release
    if (atomicAdd(&sm.done[s], 1) == NW - 1) {
      sm.done[s] = 0;
      // stage k + NB > k ≥ n1 only once pass two runs, when n2 is known to every warp
      if (stage_has(k + NB, g.spec_bc, g.n1, n2)) bc_issue<RB>(sm, g, k + NB);
    }
  }
  if (stage_has(k + kAhead, g.spec_bc, g.n1, n2)) bc_convert<RB>(sm, g, k + kAhead, warp, lane, err);
}

// The warp's outputs of a stage, written in place of u in shared memory, to HBM by one
// tensor store (lane 0), after the lanes' shared-memory writes are made visible to it.
__device__ __forceinline__ void fence_store_and_issue(const Ring& g, const uint8_t* slice, int ts, int warp,
                                                      int lane) {
  ac::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ac::tma_store_3d(&g.p->tm_out, ac::smem_u32(slice), ts, g.c0 + 32 * warp, g.b);
    ac::bulk_commit();
  }
}

// The 32 tokens of one stage for one row, in groups of four: steps, updates, readout,
// gate; outputs (bf16) replace u in the tile; returns the stage's ΣΔ' (P != kAll).
// MASKED: tokens past t_valid (the sequence's or chunk's end, or a row past d_inner)
// take Δ' = 0; a stage the whole warp has inside needs no mask.  OUT = false: the
// state updates alone (no readout, gate or outputs), for a stage pass two writes.
template <int RB, bool HAS_Z, int P, bool PRECISE, bool MASKED, bool OUT>
__device__ __forceinline__ float stage_tokens(const StreamSmem<RB>& sm, int s, const RowConst& c, int r, uint2* tu,
                                              const uint2* td, const uint2* tz, int ts, int t_valid,
                                              float (&h)[NS]) {
  float Sst = 0.f;
#pragma unroll 1
  for (int q4 = 0; q4 < TS / 4; ++q4) {
    // four tokens per iteration: 8 bytes of each of u, Δraw, z (half a swizzled granule)
    const int t = ts + q4 * 4;
    const int gi = swz(r, q4 >> 1) * 2 + (q4 & 1);  // 8-byte unit of the row
    const uint2 wu = tu[gi], wd = td[gi];
    uint2 wz = make_uint2(0u, 0u);
    if (HAS_Z && OUT) wz = tz[gi];
    const float* bcs = sm.bcf[s][q4 * 4];
    unsigned packed0 = 0u, packed1 = 0u;
    float Sb = 0.f;
#pragma unroll
    for (int v = 0; v < 4; v += 2) {
      const unsigned uw = v ? wu.y : wu.x, dw = v ? wd.y : wd.x;
      // Δ' = log2(1 + 2^{r log2 e}) for two tokens (r = Δraw + bias); r log2 e above 15 log2 e
      const float2 rl = __ffma2_rn(make_float2(bf_lo(dw), bf_hi(dw)), make_float2(kLog2e, kLog2e),
                                   make_float2(c.bl2, c.bl2));
      const float2 q = __fadd2_rn(make_float2(ex2_approx(rl.x), ex2_approx(rl.y)), make_float2(1.f, 1.f));
      float d0 = rl.x > 15.f * kLog2e ? rl.x : lg2_approx(q.x);
      float d1 = rl.y > 15.f * kLog2e ? rl.y : lg2_approx(q.y);
      if (MASKED) {
        d0 = t + v < t_valid ? d0 : 0.f;
        d1 = t + v + 1 < t_valid ? d1 : 0.f;
      }
      float2 gz = make_float2(1.f, 1.f);
      if (HAS_Z && OUT) {
        const unsigned zw = v ? wz.y : wz.x;
        const float2 zz = make_float2(bf_lo(zw), bf_hi(zw));
        // silu(z) = z/2 + (z/2)·tanh(z/2): one MUFU operation per token
        const float2 hz = __fmul2_rn(zz, make_float2(0.5f, 0.5f));
        gz = __ffma2_rn(hz, make_float2(tanh_approx(hz.x), tanh_approx(hz.y)), hz);
      }
      const float xs[2] = {bf_lo(uw), bf_hi(uw)};
      const float ds[2] = {d0, d1};
      float ys[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float dlt = ds[j], x = xs[j];
        const float4* bc4 = reinterpret_cast<const float4*>(bcs + (v + j) * 2 * NS);
        const float2 dd = make_float2(dlt, dlt), xx = make_float2(x, x);
        // rows with an A = 0 state (PRECISE): Ā = 1, B̄ = Δ B exactly there (Δ = Δ' ln 2)
        const float2 dx = PRECISE ? make_float2(dlt * kLn2 * x, dlt * kLn2 * x) : make_float2(0.f, 0.f);
        float2 ya = make_float2(0.f, 0.f);
#pragma unroll
        for (int qd = 0; qd < NS / 4; ++qd) {
          const float4 bq = bc4[qd];
          const float4 cq = OUT ? bc4[NS / 4 + qd] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int n = 4 * qd + 2 * k2;
            const float2 e = __fmul2_rn(dd, make_float2(c.a2[n], c.a2[n + 1]));
            const float2 em = __fadd2_rn(make_float2(ex2_approx(e.x), ex2_approx(e.y)), make_float2(-1.f, -1.f));
            const float2 xp = __fmul2_rn(xx, make_float2(c.ia[n], c.ia[n + 1]));
            const float2 hb = make_float2(h[n], h[n + 1]);
            const float2 bb = k2 ? make_float2(bq.z, bq.w) : make_float2(bq.x, bq.y);
            const float2 cc = k2 ? make_float2(cq.z, cq.w) : make_float2(cq.x, cq.y);
            float2 hn = __ffma2_rn(em, __ffma2_rn(xp, bb, hb), hb);
            if (PRECISE) {
              const float2 h0 = __ffma2_rn(dx, bb, hb);
              hn.x = c.ia[n] != 0.f ? hn.x : h0.x;
              hn.y = c.ia[n + 1] != 0.f ? hn.y : h0.y;
            }
            h[n] = hn.x;
            h[n + 1] = hn.y;
            if (OUT) ya = __ffma2_rn(cc, hn, ya);
          }
        }
        ys[j] = fmaf(c.Dc, x, ya.x + ya.y);
      }
      const float2 yo = __fmul2_rn(make_float2(ys[0], ys[1]), gz);
      __nv_bfloat162 p2 = __floats2bfloat162_rn(yo.x, yo.y);
      const unsigned pw = *reinterpret_cast<unsigned*>(&p2);
      packed0 = v ? packed0 : pw;
      packed1 = v ? pw : packed1;
      if (P != kAll) Sb += d0 + d1;
    }
    if (P != kAll) Sst += Sb;
    if (OUT) tu[gi] = make_uint2(packed0, packed1);
  }
  return Sst;
}

// One pass of a thread over stages [k0, k0 + nst), tokens from t_lo, writing the
// 4-token groups that P selects.  h: the row's states; S: ΣΔ' since the chunk start
// (P != kAll), with Kahan compensation `comp`.  In pass one (kSettled), lane 0
// publishes the warp's stage count for pass two as soon as it is known.
template <int RB, bool HAS_Z, int P, bool PRECISE>
__device__ __forceinline__ void consume(StreamSmem<RB>& sm, const Ring& g, const RowConst& c,
                                        int r, int warp, int lane, int k0, int nst, int n2, float (&h)[NS],
                                        float& S, float& comp, int& err) {
  constexpr float kStop = corr_stop_log2<__nv_bfloat16>();
  const int t_lo = g.tc0, t_hi = g.tc1;
  const int t_valid = c.row_ok ? t_hi : t_lo;  // rows past d_inner compute nothing useful
  bool published = P != kSettled;
#pragma unroll 1
  for (int kk = 0; kk < nst; ++kk) {
    const int k = k0 + kk;
    const int s = ring(g, k) % NB;
    const uint32_t ph = (uint32_t)(ring(g, k) / NB) & 1u;
    // this warp's rows of stage k (stage k + 1's may still be in flight), then its B and C
    if (!ac::mbar_wait(ac::smem_u32(&sm.rowbar[warp][ring(g, k) & 1]), (uint32_t)(ring(g, k) >> 1) & 1u,
                       g.deadline))
      err = 1;
    if (!ac::mbar_wait(ac::smem_u32(&sm.conv[s]), ph, g.deadline)) err = 1;
    const int ts = t_lo + kk * TS;
    const int buf = ring(g, k) & 1;
    uint2* tu = reinterpret_cast<uint2*>(sm.tile[buf][0] + r * kRowBytes);  // outputs replace u in place
    const uint2* td = reinterpret_cast<const uint2*>(sm.tile[buf][1] + r * kRowBytes);
    const uint2* tz = reinterpret_cast<const uint2*>(sm.tile[buf][2] + r * kRowBytes);
    float Sst;
    // in pass one, a stage that starts with the warp's rows unsettled is one pass two
    // writes again (its stage count only grows): the state updates alone
    const bool out = published;
    const bool whole = __all_sync(0xffffffffu, ts + TS <= t_valid);
    if (P == kSettled && !out)
      Sst = whole ? stage_tokens<RB, HAS_Z, P, PRECISE, false, false>(sm, s, c, r, tu, td, tz, ts, t_valid, h)
                  : stage_tokens<RB, HAS_Z, P, PRECISE, true, false>(sm, s, c, r, tu, td, tz, ts, t_valid, h);
    else
      Sst = whole ? stage_tokens<RB, HAS_Z, P, PRECISE, false, true>(sm, s, c, r, tu, td, tz, ts, t_valid, h)
                  : stage_tokens<RB, HAS_Z, P, PRECISE, true, true>(sm, s, c, r, tu, td, tz, ts, t_valid, h);
    if (P != kAll) {  // S += the stage's sum with Kahan compensation (S feeds 2^{A S} over long chunks)
      const float yk = Sst - comp;
      const float tk = S + yk;
      comp = (tk - S) - yk;
      S = tk;
    }
    // the stage's outputs, in place of u, leave by one tensor store of the warp's
    // [32 rows × 32 tokens] (rows past d_inner and tokens past L are clipped).  Pass one
    // of a chunk after the first stores the stages after its rows settled; pass two
    // stores the others, computed from the carried-in state.
    if (out) fence_store_and_issue(g, sm.tile[buf][0] + 32 * warp * kRowBytes, ts, warp, lane);
    if (!published) {
      // pass two must cover this stage unless every row of the warp is settled after it
      const bool settled = !c.row_ok || !(c.a2max * S > kStop - 1.f);
      if (__all_sync(0xffffffffu, settled)) {
        published = true;
        if (lane == 0) {
          atomicMax(&sm.n2, kk + 1);
          ac::mbar_arrive(ac::smem_u32(&sm.settled));
        }
      }
    }
    stage_advance<RB, HAS_Z>(sm, g, k, n2, warp, lane, err);
  }
  if (!published && lane == 0) {  // never settled: pass two covers the whole chunk
    atomicMax(&sm.n2, nst);
    ac::mbar_arrive(ac::smem_u32(&sm.settled));
  }
}

// Threads of a CTA: one per row (an SM's 16 warps of 128 registers fill its register
// file).  RB 512: one CTA per SM; RB 128: three.
template <int RB>
struct StreamCta {
  static_assert(RB == 512 || RB == 128, "rows per CTA");
  static constexpr int kThreads = RB;
  static constexpr int kMaxRegs = 128;
};

// Work-item geometry (see StreamParams): the first flattened stage of item j, and the
// item whose range holds flattened stage P.
__device__ __forceinline__ int64_t item_start(const StreamParams& p, int64_t j) { return j * p.ptot / p.items; }
__device__ __forceinline__ int64_t item_owner(const StreamParams& p, int64_t P) {
  return ((P + 1) * p.items - 1) / p.ptot;
}
// Workspace slot of an item's segment: 2j for the segment its range starts in, 2j + 1 for
// the first segment of the next tile where its range ends.
__device__ __forceinline__ int64_t seg_slot(const StreamParams& p, int64_t owner, int tile, int m) {
  return (m == 0 && item_start(p, owner) < (int64_t)tile * p.sl) ? 2 * owner + 1 : 2 * owner;
}


template <int RB, bool HAS_Z, bool PRECISE>
__device__ __forceinline__ void row_program(StreamSmem<RB>& sm, const StreamParams& p, const Ring& g,
                                            const RowConst& cs, float (&h)[NS], const Segment& sg, int64_t row,
                                            int r, int warp, int lane, int& err) {
  constexpr int NW = RB / 32;
  const int n1 = g.n1;
  const bool last = sg.s1 == p.sl;  // no later segment in this tile
  float S = 0.f, comp = 0.f;
  if (sg.q == 0)
    consume<RB, HAS_Z, kAll, PRECISE>(sm, g, cs, r, warp, lane, 0, n1, 0, h, S, comp, err);
  else
    consume<RB, HAS_Z, kSettled, PRECISE>(sm, g, cs, r, warp, lane, 0, n1, -1, h, S, comp, err);
  // pass one's stores complete before pass two stores its stages again
  if (lane == 0) ac::bulk_wait0();

  // ---------------- carry between the segments of a tile ----------------
  // Each warp publishes its rows' aggregate (S, h from h = 0; the first segment's h is
  // its end state from the initial state) and combines those of all preceding
  // segments in a fixed order, h_in = Σ_m 2^{A (S_{m+1} + … + S_{q-1})} h_m, so the
  // result does not depend on which segment finished first.  The aggregates are
  // published right after pass one, so no segment waits for another's carry.
  float hin[NS];
#pragma unroll
  for (int n = 0; n < NS; ++n) hin[n] = 0.f;
  if (p.multi) {
    if (!last) {
      float4* ah = reinterpret_cast<float4*>(p.ws.agg_h + (sg.slot * RB + r) * NS);
#pragma unroll
      for (int q = 0; q < NS / 4; ++q) ah[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
      p.ws.agg_s[sg.slot * RB + r] = S;
      __threadfence();
      __syncwarp();
      if (lane == 0) st_release_gpu(p.ws.flags + sg.slot * NW + warp, 1u);
    }
    if (sg.q > 0) {
      // every preceding segment's aggregate (segment m belongs to item sg.item - q + m):
      // lanes wait on different segments' flags
      const unsigned want = p.fault_lookback ? 3u : 1u;  // 3 is never written
      bool all_ok = true;
      for (int base = 0; base < sg.q; base += 32) {
        const int m = base + lane;
        unsigned v = 0;
        bool ok = true;
        if (m < sg.q) {
          const int64_t sl_m = seg_slot(p, sg.item - sg.q + m, sg.tile, m);
          ok = wait_flag(p.ws.flags + sl_m * NW + warp, want, p.timeout_ns, &v);
        }
        all_ok = __all_sync(0xffffffffu, ok) && all_ok;
      }
      __syncwarp();
      if (!all_ok) {
        err = 1;  // the carry is left out; the error word reports it
      } else {
        float acc = 0.f;
        for (int m = sg.q - 1; m >= 0; --m) {
          const int64_t sl_m = seg_slot(p, sg.item - sg.q + m, sg.tile, m);
          const float4* src = reinterpret_cast<const float4*>(p.ws.agg_h + (sl_m * RB + r) * NS);
#pragma unroll
          for (int q = 0; q < NS / 4; ++q) {
            const float4 x = __ldcg(src + q);
            const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int n = 4 * q + i;
              hin[n] = fmaf(PRECISE ? exp2f(cs.a2[n] * acc) : ex2_approx(cs.a2[n] * acc), xv[i], hin[n]);
            }
          }
          acc += __ldcg(p.ws.agg_s + sl_m * RB + r);
        }
      }
#pragma unroll
      for (int n = 0; n < NS; ++n)
        h[n] = fmaf(PRECISE ? exp2f(cs.a2[n] * S) : ex2_approx(cs.a2[n] * S), hin[n], h[n]);
    }
  }
  if (p.a.final_state && last && cs.row_ok) {
    float4* fs = reinterpret_cast<float4*>(p.a.final_state + row * NS);
#pragma unroll
    for (int q = 0; q < NS / 4; ++q) fs[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
  }

  // ---------------- pass two: the segment's first stages again, from h_in ----------------
  if (sg.q > 0) {
    if (!ac::mbar_wait(ac::smem_u32(&sm.settled), 0u, g.deadline)) err = 1;
    const int n2 = *reinterpret_cast<volatile int*>(&sm.n2);
    float S2 = 0.f, comp2 = 0.f;
    consume<RB, HAS_Z, kUnsettled, PRECISE>(sm, g, cs, r, warp, lane, n1, n2, n2, hin, S2, comp2, err);
  }
}

// The row's constants (channel ch); `precise` is made warp-uniform: the exact branch
// serves every row of a warp that has an A = 0 state.
__device__ __forceinline__ RowConst row_const(const StreamParams& p, int64_t ch, bool row_ok) {
  RowConst c;
  c.row_ok = row_ok;
  c.precise = false;
  c.a2max = -INFINITY;
  const float* arow = p.a.A + ch * NS;
#pragma unroll
  for (int n = 0; n < NS; ++n) {
    const float a = row_ok ? arow[n] : 0.f;
    const bool tiny = fabsf(a) < 8.673617e-19f;  // |A| < 2^-60 counts as A = 0
    if (row_ok && tiny) c.precise = true;
    c.a2[n] = tiny ? 0.f : a;
    c.ia[n] = tiny ? 0.f : 1.f / a;
    if (row_ok) c.a2max = fmaxf(c.a2max, c.a2[n]);
  }
  c.precise = __any_sync(0xffffffffu, c.precise);
  c.Dc = (row_ok && p.a.D) ? p.a.D[ch] : 0.f;
  c.bl2 = (row_ok && p.a.bias) ? p.a.bias[ch] * kLog2e : 0.f;
  return c;
}

// One segment, from the ring's prologue to its last store: thread r owns row c0 + r.
template <int RB, bool HAS_Z>
__device__ __forceinline__ void run_segment(StreamSmem<RB>& sm, const StreamParams& p, const Segment& sg, int kb,
                                            unsigned long long deadline, int warp, int lane, int& err) {
  Ring g;
  g.p = &p;
  g.deadline = deadline;
  g.kb = kb;
  g.b = sg.tile / p.rtiles;
  g.c0 = (sg.tile % p.rtiles) * RB;
  g.tc0 = sg.s0 * TS;
  g.tc1 = (int)min((int64_t)p.a.L, (int64_t)sg.s1 * TS);
  g.n1 = sg.s1 - sg.s0;
  g.spec_rows = g.n1 + (sg.q > 0 ? min(2, g.n1) : 0);
  g.spec_bc = g.n1 + (sg.q > 0 ? min(NB, g.n1) : 0);

  // the first two stages of this warp's rows; the B/C ring filled; every warp converts
  // its share of the first kAhead stages
  for (int k = 0; k < 2; ++k)
    if (k < g.spec_rows) rows_issue<RB, HAS_Z>(sm, g, k, warp, lane);
  if (threadIdx.x == 0)
    for (int j = 0; j < NB && j < g.spec_bc; ++j) bc_issue<RB>(sm, g, j);
  for (int j = 0; j < kAhead && j < g.spec_bc; ++j) bc_convert<RB>(sm, g, j, warp, lane, err);

  const int r = threadIdx.x;
  const int nrows = min(RB, (int)p.a.d_inner - g.c0);
  const bool row_ok = r < nrows;
  const int64_t ch = g.c0 + (row_ok ? r : 0);
  const int64_t row = (int64_t)g.b * p.a.d_inner + ch;
  const RowConst cs = row_const(p, ch, row_ok);
  float h[NS];
#pragma unroll
  for (int n = 0; n < NS; ++n) h[n] = (sg.q == 0 && p.a.h0 && row_ok) ? p.a.h0[row * NS + n] : 0.f;
  if (cs.precise)
    row_program<RB, HAS_Z, true>(sm, p, g, cs, h, sg, row, r, warp, lane, err);
  else
    row_program<RB, HAS_Z, false>(sm, p, g, cs, h, sg, row, r, warp, lane, err);
}

template <int RB, bool HAS_Z>
__global__ void __launch_bounds__(StreamCta<RB>::kThreads) __maxnreg__(StreamCta<RB>::kMaxRegs)
    scan_stream_kernel(const __grid_constant__ StreamParams p) {
  constexpr int NW = RB / 32;
  extern __shared__ unsigned char smem_raw[];
  // aligned by offsetting the shared array itself, so that the compiler keeps
  // shared-memory (32-bit) addressing
  StreamSmem<RB>& sm = *reinterpret_cast<StreamSmem<RB>*>(
      smem_raw + ((1024u - (ac::smem_u32(smem_raw) & 1023u)) & 1023u));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NB; ++s) {
      ac::mbar_init(ac::smem_u32(&sm.full[s]), 1);  // the issuing thread's arrival + the copies' bytes
      ac::mbar_init(ac::smem_u32(&sm.conv[s]), NW);
      sm.done[s] = 0;
    }
    ac::mbar_init(ac::smem_u32(&sm.settled), NW);
    for (int w = 0; w < NW; ++w) {
      ac::mbar_init(ac::smem_u32(&sm.rowbar[w][0]), 1);  // the issuing lane's arrival + the copies' bytes
      ac::mbar_init(ac::smem_u32(&sm.rowbar[w][1]), 1);
      sm.rissued[w] = 0;
    }
    ac::fence_mbar_init();
    sm.n2 = 0;
    sm.issued = 0;
    // tickets in start order: the items a segment's carry waits on started earlier
    const int64_t item = p.multi ? (int64_t)atomicAdd(p.ws.hdr, 1u) : (int64_t)blockIdx.x;
    // the item's range of flattened stages, in one tile or across the end of one tile
    // and the start of the next; with two segments, the next tile's first segment runs
    // first: it waits for nothing, and later items wait on it
    const int64_t P0 = item_start(p, item), P1 = item_start(p, item + 1);
    const int ta = (int)(P0 / p.sl), tb = (int)((P1 - 1) / p.sl);
    sm.nseg = tb > ta ? 2 : 1;
    Segment& sa = sm.seg[sm.nseg - 1];
    sa.item = item;
    sa.tile = ta;
    sa.s0 = (int)(P0 - (int64_t)ta * p.sl);
    sa.s1 = tb > ta ? p.sl : (int)(P1 - (int64_t)ta * p.sl);
    sa.q = (int)(item - item_owner(p, (int64_t)ta * p.sl));
    sa.slot = 2 * item;
    if (tb > ta) {
      Segment& sb = sm.seg[0];
      sb.item = item;
      sb.tile = tb;
      sb.s0 = 0;
      sb.s1 = (int)(P1 - (int64_t)tb * p.sl);
      sb.q = 0;
      sb.slot = 2 * item + 1;
    }
    ac::prefetch_tensormap(&p.tm_b);
    ac::prefetch_tensormap(&p.tm_c);
    ac::prefetch_tensormap(&p.tm_u);
    ac::prefetch_tensormap(&p.tm_d);
    if (HAS_Z) ac::prefetch_tensormap(&p.tm_z);
  }
  __syncthreads();
  const unsigned long long deadline = ac::globaltimer() + (unsigned long long)p.timeout_ns;
  int err = 0;
  const int nseg = sm.nseg;
  int kb = 0;
#pragma unroll 1
  for (int sgi = 0; sgi < nseg; ++sgi) {
    run_segment<RB, HAS_Z>(sm, p, sm.seg[sgi], kb, deadline, warp, lane, err);
    if (sgi + 1 < nseg) {
      kb = sm.seg[sgi].s1;  // every ring stage of a first segment was issued and consumed
      if (lane == 0) {
        if (!rows_drain(sm, warp, deadline + 1000000000ull)) err = 1;
        ac::bulk_wait0();
      }
      __syncthreads();  // the ring and the row buffers are free for the next segment
    }
  }

  // copies issued ahead of a pass two shorter than the ring, never consumed, must land,
  // and the tensor stores complete, before the CTA exits
  if (lane == 0) {
    if (!rows_drain(sm, warp, deadline + 1000000000ull)) err = 1;
    ac::bulk_wait0();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int issued = sm.issued;
    for (int j = issued - NB < 0 ? 0 : issued - NB; j < issued; ++j)
      if (!ac::mbar_wait(ac::smem_u32(&sm.full[j % NB]), (uint32_t)(j / NB) & 1u, deadline + 1000000000ull))
        err = 1;
  }
  if (err && p.ws.hdr) atomicOr(p.ws.hdr + 1, kErrTimeout);
}

template <int RB, bool HAS_Z>
cudaError_t stream_launch_t(const StreamParams& p, int grid, cudaStream_t s) {
  auto kern = scan_stream_kernel<RB, HAS_Z>;
  const cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stream_smem_bytes<RB>());
  if (e != cudaSuccess) return e;
  kern<<<grid, StreamCta<RB>::kThreads, stream_smem_bytes<RB>(), s>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t stream_smem_bytes_for(int rb) { return rb == 512 ? stream_smem_bytes<512>() : stream_smem_bytes<128>(); }

StreamWs stream_ws_layout(unsigned char* ws, int64_t items, int rb, size_t* total) {
  // [header][flags: 2 items × warps][aggregate h: 2 items × rows × 16][aggregate S: 2 items × rows]
  // (an item publishes at most two segments: the one its range starts in and the next tile's first)
  StreamWs w{};
  const int64_t slots = 2 * items;
  size_t off = kWsHeaderBytes;
  const size_t flags_off = off;
  off += ((size_t)slots * (rb / 32) * 4 + 255) & ~size_t(255);
  w.flags_bytes = off;
  const size_t aggh_off = off;
  off += (size_t)slots * rb * NS * 4;
  const size_t aggs_off = off;
  off += ((size_t)slots * rb * 4 + 255) & ~size_t(255);
  *total = off;
  if (ws) {
    w.hdr = reinterpret_cast<unsigned*>(ws);
    w.flags = reinterpret_cast<unsigned*>(ws + flags_off);
    w.agg_h = reinterpret_cast<float*>(ws + aggh_off);
    w.agg_s = reinterpret_cast<float*>(ws + aggs_off);
  }
  return w;
}

bool stream_supported(const ScanArgs& a) {
  if (a.act != 1 || a.N != NS || a.L < 1) return false;
  if (a.L % 8 != 0 || a.L > (int64_t)INT32_MAX - 64 || a.d_inner > (int64_t)INT32_MAX - 512 || a.batch > 65535)
    return false;
  auto a16 = [](const void* q) { return q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  return a16(a.u) && a16(a.delta) && a16(a.z) && a16(a.B) && a16(a.C) && a16(a.out);
}

cudaError_t scan_stream_launch(const ScanArgs& a, const ScanPlan& plan, cudaStream_t stream) {
  StreamParams p{};
  p.a = a;
  p.rtiles = plan.ctiles;
  p.sl = (int)((a.L + TS - 1) / TS);
  p.items = plan.nchunks;
  const int64_t tiles = a.batch * plan.ctiles;
  p.ptot = tiles * p.sl;
  p.multi = p.items > tiles ? 1 : 0;
  const RuntimeKnobs knobs = runtime_knobs();
  p.timeout_ns = knobs.lookback_timeout_ns > 0 ? knobs.lookback_timeout_ns
                                               : 1000ll * 1000 * 1000 + plan.chunk_len * 100ll;
  p.fault_lookback = knobs.fault_lookback ? 1 : 0;
  const int rb = plan.rows_per_cta;
  size_t total = 0;
  // one segment per tile: no workspace is required; if one is given its header takes the error word
  p.ws = stream_ws_layout(p.multi ? a.ws : nullptr, p.items, rb, &total);
  if (!p.multi) p.ws.hdr = reinterpret_cast<unsigned*>(a.ws);
  // tensor maps of B and C as [batch][L][16] bf16 (tokens past L read as zero)
  const uint64_t L = (uint64_t)a.L, Bt = (uint64_t)a.batch;
  const uint64_t dims_bc[3] = {(uint64_t)NS, L, Bt}, str_bc[2] = {NS * 2, L * NS * 2};
  const uint32_t box_bc[3] = {(uint32_t)NS, (uint32_t)TS, 1};
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto none = CU_TENSOR_MAP_SWIZZLE_NONE;
  const auto promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  // out as [batch][d_inner][L] bf16, stored in [32 rows × 32 tokens] boxes with the
  // 64-byte swizzle of the row tiles (rows past d_inner, tokens past L clipped)
  const uint64_t D = (uint64_t)a.d_inner;
  const uint64_t dims_row[3] = {L, D, Bt}, str_row[2] = {L * 2, L * D * 2};
  const uint32_t box_row[3] = {(uint32_t)TS, 32u, 1u};
  const auto sw64 = CU_TENSOR_MAP_SWIZZLE_64B;
  if (!encode_tensor_map(&p.tm_b, bf, 3, a.B, dims_bc, str_bc, box_bc, none, promo) ||
      !encode_tensor_map(&p.tm_c, bf, 3, a.C, dims_bc, str_bc, box_bc, none, promo) ||
      !encode_tensor_map(&p.tm_out, bf, 3, a.out, dims_row, str_row, box_row, sw64, CU_TENSOR_MAP_L2_PROMOTION_NONE) ||
      !encode_tensor_map(&p.tm_u, bf, 3, a.u, dims_row, str_row, box_row, sw64, promo) ||
      !encode_tensor_map(&p.tm_d, bf, 3, a.delta, dims_row, str_row, box_row, sw64, promo) ||
      (a.z && !encode_tensor_map(&p.tm_z, bf, 3, a.z, dims_row, str_row, box_row, sw64, promo)))
    return cudaErrorInvalidValue;
  if (p.multi) {
    const cudaError_t e = cudaMemsetAsync(a.ws, 0, p.ws.flags_bytes, stream);
    if (e != cudaSuccess) return e;
  }
  const int grid = p.items;
  const bool hz = a.z != nullptr;
  if (rb == 512) return hz ? stream_launch_t<512, true>(p, grid, stream) : stream_launch_t<512, false>(p, grid, stream);
  return hz ? stream_launch_t<128, true>(p, grid, stream) : stream_launch_t<128, false>(p, grid, stream);
}

}  // namespace ssm

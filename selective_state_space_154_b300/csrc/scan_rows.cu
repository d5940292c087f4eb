// Selective-scan forward for long sequences (d_state ≤ 16), sm_103a.
//
// Same operation as scan_fwd.cu ("State Space Models（SSM）とMamba" §2.2 離散化;
// "Mambaとは？Transformer以外の系列モデル", sections 状態空間モデルを一つの式から
// 理解する and Mamba blockのarchitecture).  Organisation:
//  * a thread owns one (batch, channel) row and all its states: h, A·log2e and
//    1/A live in registers, the readout Σ_n C_n h_n needs no other thread, and
//    softplus / silu are evaluated once per (row, token);
//  * a CTA owns 128 rows of one batch over one chunk of the sequence and walks it
//    in stages of 32 tokens.  Per stage the CTA copies [128 rows × 64 bytes] tiles
//    of u, Δraw and z with cp.async, four lanes per 64-byte row segment, so every
//    DRAM access covers 64 contiguous bytes of one row (rows are L·2 bytes apart;
//    one lane streaming 16 bytes of its own row per request reaches only a small
//    fraction of the HBM bandwidth), plus B and C of the 32 tokens, which all 128
//    rows share and which are converted to fp32 once.  Stages are double-buffered;
//    tiles are XOR-swizzled so that a lane reading its own row is conflict-free;
//  * chunks compose as affine maps, (A₂,b₂)∘(A₁,b₁) = (A₂A₁, A₂b₁+b₂)
//    ("Mambaとは？…", Selective Scanは選択機構そのものではない): every chunk scans
//    from h = 0 at once keeping S = ΣΔ, then takes the end state h_in of the
//    previous chunk (in chunk order, bounded wait) and publishes its own end state
//    exp(A S)·h_in + h_local.  Its first blocks, those whose outputs the carried-in
//    state still changes (exp(A_n S) ≥ 2^-24 for fp32 outputs, 2^-12 for bf16, for
//    the row's slowest-decaying state), are not written by that pass: a second pass
//    scans them again from h_in and writes them, rounding each output once.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int TS = kRowTokensPerStage;  // tokens per stage
constexpr int NS = 16;                  // states per row held by one thread

struct RowParams {
  ScanArgs a;
  int rtiles, nchunks;
  int64_t chunk_len;
  int vec_rows, vec_bc;
  unsigned* hdr;
  unsigned* flags;  // [nchunks][batch*rtiles]
  float* incl;      // [nchunks][batch*rtiles*RB][NS] end state of each chunk
  long long timeout_ns;
  int fault_lookback;
};

__device__ __forceinline__ int64_t min64r(int64_t a, int64_t b) { return a < b ? a : b; }

// Shared memory of one CTA.  A row tile holds TS tokens of RB rows; granule g
// (16 bytes) of row r sits at granule index g ^ swz(r) of that row.
template <typename T, int RB>
struct Smem {
  static constexpr int kRowBytes = TS * (int)sizeof(T);  // 64 (bf16) or 128 (fp32)
  static constexpr int kGran = kRowBytes / 16;           // 16-byte granules per row and stage
  uint4 tile[2][3][RB][kGran];                           // [stage][u|delta|z][row][granule]
  uint4 raw_bc[2][2 * TS * NS * sizeof(T) / 16];         // [stage][B|C][TS][N] raw
  float bcf[TS * 2 * NS];                                // converted stage, [TS][B|C][16]
  // two ints used outside the passes (ticket, wait result) share bcf's storage,
  // which keeps the CTA at 56 KB of shared memory (four CTAs per SM)
  __device__ int* misc() { return reinterpret_cast<int*>(bcf); }
};

// XOR swizzle of the granule index: lanes r..r+7 reading the same granule of
// their rows then hit eight different 16-byte bank groups.
template <typename T>
__device__ __forceinline__ int swz(int r) {
  constexpr int kRowBytes = TS * (int)sizeof(T), kGran = kRowBytes / 16;
  return (r / (128 / kRowBytes)) & (kGran - 1);
}

// Issue the copies of stage [t0, t0 + TS) ∩ [t0, t_end): three row tiles and B, C.
template <typename T, int RB, int NT, bool VEC>
__device__ __forceinline__ void issue_stage(Smem<T, RB>& sm, int buf, const RowParams& p, int64_t b, int64_t row0, int nrows,
                                            int64_t t0, int64_t t_end) {
  constexpr int G = Smem<T, RB>::kGran;
  constexpr int RSTEP = NT / G;        // rows apart of one thread's copies
  constexpr int NPER = RB / RSTEP;     // copies per thread and tensor
  static_assert(NT % G == 0 && RB % RSTEP == 0, "a stage splits evenly over the CTA's threads");
  constexpr int E = sizeof(T);
  const int64_t L = p.a.L;
  const T* srcs[3] = {static_cast<const T*>(p.a.u), static_cast<const T*>(p.a.delta),
                      static_cast<const T*>(p.a.z)};
  const int ntens = p.a.z ? 3 : 2;
  const int g = threadIdx.x % G;
  const int r_first = threadIdx.x / G;
  const int64_t t = t0 + (int64_t)g * (16 / E);
  for (int w = 0; w < ntens; ++w) {
    const T* base = srcs[w] + (row0 + r_first) * L + t;
    for (int k = 0; k < NPER; ++k) {
      const int r = r_first + k * RSTEP;
      uint4* dst = &sm.tile[buf][w][r][g ^ swz<T>(r)];
      const bool ok = r < nrows && t < t_end;
      if (VEC) {
        cp_async16(dst, ok ? static_cast<const void*>(base + (int64_t)k * RSTEP * L) : static_cast<const void*>(srcs[w]),
                   ok ? 16 : 0);
      } else {
        // element copies for rows that are not 16-byte aligned
        unsigned wv[4] = {0u, 0u, 0u, 0u};
        if (ok) {
          const T* s = srcs[w] + (row0 + r) * L;
          for (int e = 0; e < 16 / E; ++e) {
            if (t + e < t_end) {
              unsigned bits;
              if (E == 2) bits = reinterpret_cast<const unsigned short*>(s)[t + e];
              else bits = __float_as_uint(reinterpret_cast<const float*>(s)[t + e]);
              wv[(e * E) / 4] |= bits << ((e * E) % 4 * 8);
            }
          }
        }
        *dst = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
    }
  }
  // B and C of the stage, [B|C][TS][N] raw
  const int N = (int)p.a.N;
  const int64_t ntok = min64r(TS, t_end - t0);
  const int64_t nvalid = ntok > 0 ? ntok * N : 0;
  const T* bcsrc[2] = {static_cast<const T*>(p.a.B), static_cast<const T*>(p.a.C)};
  T* raw = reinterpret_cast<T*>(sm.raw_bc[buf]);
  for (int w = 0; w < 2; ++w) {
    T* dst = raw + w * TS * N;
    const T* s0 = bcsrc[w] + (b * L + t0) * N;
    if (p.vec_bc) {
      constexpr int VPT = 16 / E;
      const int nvec = TS * N / VPT;
      for (int i = threadIdx.x; i < nvec; i += NT) {
        const bool ok = (int64_t)(i + 1) * VPT <= nvalid;
        cp_async16(dst + i * VPT, ok ? s0 + (int64_t)i * VPT : bcsrc[w], ok ? 16 : 0);
      }
    } else {
      for (int i = threadIdx.x; i < TS * N; i += NT) dst[i] = (i < nvalid) ? s0[i] : T(0.f);
    }
  }
}

template <typename T, int NT>
__device__ __forceinline__ void convert_bc(float* bc, const T* raw, int N) {
  for (int i = threadIdx.x; i < TS * 2 * NS; i += NT) {
    const int t = i / (2 * NS), w = (i / NS) & 1, n = i % NS;
    bc[i] = n < N ? Act<T>::to_f(raw[(w * TS + t) * N + n]) : 0.f;
  }
}

// element i of the 8-token group held in raw 16-byte words (bf16: 1 word, fp32: 2 words)
template <typename T>
__device__ __forceinline__ float get8(const uint4* w, int i) {
  if constexpr (sizeof(T) == 2) {
    const unsigned x = (&w[0].x)[i >> 1];
    return __uint_as_float((i & 1) ? (x & 0xffff0000u) : (x << 16));
  } else {
    return __uint_as_float((&w[i >> 2].x)[i & 3]);
  }
}

template <typename T, bool VEC>
__device__ __forceinline__ void store8(T* row, int64_t t, int64_t t_end, const float (&y)[8]) {
  if constexpr (sizeof(T) == 2) {
    if (VEC && t + 8 <= t_end) {
      uint4 w;
      unsigned* wp = &w.x;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 p2 = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
        wp[i] = *reinterpret_cast<unsigned*>(&p2);
      }
      *reinterpret_cast<uint4*>(row + t) = w;
    } else {
      for (int i = 0; i < 8; ++i)
        if (t + i < t_end) row[t + i] = __float2bfloat16_rn(y[i]);
    }
  } else {
    if (VEC && t + 8 <= t_end) {
      *reinterpret_cast<float4*>(row + t) = make_float4(y[0], y[1], y[2], y[3]);
      *reinterpret_cast<float4*>(row + t + 4) = make_float4(y[4], y[5], y[6], y[7]);
    } else {
      for (int i = 0; i < 8; ++i)
        if (t + i < t_end) row[t + i] = y[i];
    }
  }
}

// silu for bf16 outputs: z / (1 + 2^(-z log2 e)) with the MUFU ex2 and rcp
// approximations (no cancellation for z < 0, unlike (z/2)(1 + tanh(z/2)),
// whose 1 + tanh loses all accuracy there); precise form otherwise.
template <bool FAST>
__device__ __forceinline__ float silu_t(float z) {
  return FAST ? silu_fast(z) : silu_precise(z);
}

__device__ bool wait_flag_rows(const RowParams& p, const unsigned* flag, unsigned want) {
  const unsigned long long start = globaltimer_ns();
  unsigned ns = 32;
  for (long long it = 0; it < (1ll << 28); ++it) {
    if (ld_acquire_gpu(flag) >= want) return true;
    if ((long long)(globaltimer_ns() - start) > p.timeout_ns) break;
    __nanosleep(ns);
    ns = ns < 256 ? ns * 2 : ns;
  }
  atomicOr(p.hdr + 1, kErrTimeout);
  return false;
}

// Which 8-token blocks a pass writes.  A block of a chunk after the first is
// "settled" when exp(A_n S) < 2^stop for every state at the block's start
// (S = ΣΔ from the chunk start, the same sequence in both passes), i.e. when
// the chunk's carried-in state can no longer change its outputs.
enum WritePolicy {
  kWriteAll = 0,        // the first chunk (or the only one): every block
  kWriteSettled = 1,    // other chunks, first pass from h = 0: the settled blocks
  kWriteUnsettled = 2,  // other chunks, second pass from the carried-in state: the rest,
                        // stopping once every row of the CTA is settled
};

// One pass of the CTA over tokens [t_lo, t_hi): the scan from the registers' h,
// writing the blocks that WP selects.  a2max = max_n A_n log2e over the row's
// states (-inf for rows past d_inner): the slowest decay decides when a row is
// settled.  TPR threads share a row: thread j of the row holds states
// [j·SPT, (j+1)·SPT) and the readout is summed over the row's threads with shuffles.
template <typename T, int RB, int TPR, bool HAS_Z, bool VEC, int WP>
__device__ __forceinline__ void row_pass(Smem<T, RB>& sm, const RowParams& p, int64_t b, int64_t row0, int nrows,
                                         int64_t t_lo, int64_t t_hi, float (&h)[NS / TPR], const float (&a2)[NS / TPR],
                                         const float (&ia)[NS / TPR], const float* arow, bool precise, float Dc,
                                         float biasc, float a2max, float& S) {
  using AT = Act<T>;
  constexpr bool FAST = AT::kFast;
  constexpr int NT = RB * TPR;
  constexpr int SPT = NS / TPR;
  constexpr int GPB = (8 * (int)sizeof(T)) / 16;  // granules per 8-token block
  const int N = (int)p.a.N;
  const int r = threadIdx.x / TPR;
  const int jpart = threadIdx.x % TPR;
  const int n0 = jpart * SPT;
  const bool row_ok = r < nrows;
  T* orow = static_cast<T*>(p.a.out) + (row0 + (row_ok ? r : 0)) * p.a.L;
  const int nst = (int)((t_hi - t_lo + TS - 1) / TS);
  if (nst <= 0) return;
  issue_stage<T, RB, NT, VEC>(sm, 0, p, b, row0, nrows, t_lo, t_hi);
  cp_async_commit();
  float comp = 0.f;  // Kahan compensation of S
  for (int st = 0; st < nst; ++st) {
    const int64_t ts = t_lo + (int64_t)st * TS;
    const int buf = st & 1;
    if (st + 1 < nst) issue_stage<T, RB, NT, VEC>(sm, buf ^ 1, p, b, row0, nrows, ts + TS, t_hi);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();  // stage st landed for every thread
    convert_bc<T, NT>(sm.bcf, reinterpret_cast<const T*>(sm.raw_bc[buf]), N);
    __syncthreads();
    const int64_t t_valid = row_ok ? t_hi : ts;  // rows past d_inner compute nothing useful
#pragma unroll 1
    for (int blk = 0; blk < TS / 8; ++blk) {
      const int64_t t = ts + blk * 8;
      // S: ΣΔ before this block.  Pass two takes the threshold one power of two
      // looser, so a block near the boundary may be written twice (pass two last)
      // but never by neither pass.
      const bool write_blk = WP == kWriteAll || (WP == kWriteSettled ? !(a2max * S > corr_stop_log2<T>())
                                                                     : a2max * S > corr_stop_log2<T>() - 1.f);
      uint4 wu[GPB], wd[GPB], wz[GPB];
#pragma unroll
      for (int j = 0; j < GPB; ++j) {
        const int g = (blk * GPB + j) ^ swz<T>(r);
        wu[j] = sm.tile[buf][0][r][g];
        wd[j] = sm.tile[buf][1][r][g];
        if (HAS_Z) wz[j] = sm.tile[buf][2][r][g];
      }
      const float* bcs = sm.bcf + blk * 8 * 2 * NS;
      float yv[8];
      float Sb = 0.f;
      float dlt8[8], gz8[8];
      if (FAST) {  // per-token scalars first, two tokens per packed instruction
#pragma unroll
        for (int v = 0; v < 8; v += 2) {
          const float2 rr = __fadd2_rn(make_float2(get8<T>(wd, v), get8<T>(wd, v + 1)), make_float2(biasc, biasc));
          const float2 e = __fmul2_rn(rr, make_float2(kLog2e, kLog2e));
          const float2 q = __fadd2_rn(make_float2(ex2_approx(e.x), ex2_approx(e.y)), make_float2(1.f, 1.f));
          const float2 sp = __fmul2_rn(make_float2(lg2_approx(q.x), lg2_approx(q.y)), make_float2(kLn2, kLn2));
          dlt8[v] = t + v < t_valid ? (rr.x > 15.f ? rr.x : sp.x) : 0.f;
          dlt8[v + 1] = t + v + 1 < t_valid ? (rr.y > 15.f ? rr.y : sp.y) : 0.f;
          if (HAS_Z) {
            const float2 zz = make_float2(get8<T>(wz, v), get8<T>(wz, v + 1));
            const float2 ez = __fmul2_rn(zz, make_float2(-kLog2e, -kLog2e));
            const float2 dz = __fadd2_rn(make_float2(ex2_approx(ez.x), ex2_approx(ez.y)), make_float2(1.f, 1.f));
            const float2 gz = __fmul2_rn(zz, make_float2(rcp_approx(dz.x), rcp_approx(dz.y)));
            gz8[v] = gz.x;
            gz8[v + 1] = gz.y;
          } else {
            gz8[v] = gz8[v + 1] = 1.f;
          }
        }
      } else {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const bool tok_ok = t + v < t_valid;
          const float rr = get8<T>(wd, v) + biasc;
          dlt8[v] = tok_ok ? softplus_precise(rr) : 0.f;
          gz8[v] = HAS_Z ? silu_precise(get8<T>(wz, v)) : 1.f;
        }
      }
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float dlt = dlt8[v];
        const float x = get8<T>(wu, v);
        const float4* bc4 = reinterpret_cast<const float4*>(bcs + v * 2 * NS);
        float y;
        {
          if (!precise) {
            const float2 dd = make_float2(dlt, dlt), xx = make_float2(x, x);
            float2 ya = make_float2(0.f, 0.f), yb = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < SPT / 4; ++q) {
              const float4 bq = bc4[n0 / 4 + q];
              const float4 cq = bc4[NS / 4 + n0 / 4 + q];
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2) {
                const int n = 4 * q + 2 * k2;
                const float2 e = __fmul2_rn(dd, make_float2(a2[n], a2[n + 1]));
                const float2 ab = make_float2(ex2_approx(e.x), ex2_approx(e.y));
                const float2 em = __fadd2_rn(ab, make_float2(-1.f, -1.f));
                const float2 xp = __fmul2_rn(xx, make_float2(ia[n], ia[n + 1]));
                const float2 hb = make_float2(h[n], h[n + 1]);
                const float2 bb = k2 ? make_float2(bq.z, bq.w) : make_float2(bq.x, bq.y);
                const float2 cc = k2 ? make_float2(cq.z, cq.w) : make_float2(cq.x, cq.y);
                const float2 hn = __ffma2_rn(em, __ffma2_rn(xp, bb, hb), hb);
                h[n] = hn.x;
                h[n + 1] = hn.y;
                if (k2) yb = __ffma2_rn(cc, hn, yb); else ya = __ffma2_rn(cc, hn, ya);
              }
            }
            y = (ya.x + yb.x) + (ya.y + yb.y);
          } else {
            y = 0.f;
#pragma unroll
            for (int q = 0; q < SPT / 4; ++q) {
              const float4 bq = bc4[n0 / 4 + q];
              const float4 cq = bc4[NS / 4 + n0 / 4 + q];
              const float bb[4] = {bq.x, bq.y, bq.z, bq.w};
              const float cc[4] = {cq.x, cq.y, cq.z, cq.w};
#pragma unroll
              for (int k2 = 0; k2 < 4; ++k2) {
                const int n = 4 * q + k2;
                const float an0 = (row_ok && n0 + n < N) ? __ldg(arow + n) : 0.f;  // arow starts at state n0
                const float an = fabsf(an0) < 8.673617e-19f ? 0.f : an0;
                if (an != 0.f) {
                  const float em1 = FAST ? ex2_approx(dlt * a2[n]) - 1.f : expm1f(dlt * an);
                  h[n] = fmaf(em1, fmaf(x * ia[n], bb[k2], h[n]), h[n]);
                } else {
                  h[n] = fmaf(dlt * x, bb[k2], h[n]);  // A = 0: Ā = 1, B̄ = Δ B
                }
                y = fmaf(cc[k2], h[n], y);
              }
            }
          }
#pragma unroll
          for (int off = TPR / 2; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
          y = fmaf(Dc, x, y);
          if (HAS_Z) y *= gz8[v];
          Sb += dlt;
        }
        yv[v] = y;
      }
      {  // S += Sb with Kahan compensation (S feeds exp(A S) over long chunks)
        const float yk = Sb - comp;
        const float tk = S + yk;
        comp = (tk - S) - yk;
        S = tk;
      }
      if (row_ok && jpart == 0 && t < t_hi && write_blk) store8<T, VEC>(orow, t, t_hi, yv);
    }
    if (WP == kWriteUnsettled) {
      // stop once every row of the CTA is settled: pass one wrote the rest
      const bool unsettled = a2max * S > corr_stop_log2<T>() - 1.f;
      if (!__syncthreads_or(unsettled)) break;  // also orders the reuse of this stage's buffers
    } else {
      __syncthreads();  // this stage's buffers are refilled two stages later
    }
  }
  cp_async_wait<0>();
  __syncthreads();
}

// RB rows (threads) per CTA: 128 (four CTAs per SM) or 512 / 256 (one CTA per SM
// for bf16 / fp32).  With one CTA per SM all of an SM's rows advance in lock-step
// through the per-stage barriers, so chunks finish together; co-resident CTAs
// with equal work were seen to finish up to 1.6x apart.
// TPR = 2 (two threads per row, 8 states each) doubles the threads for layers
// with too few rows to fill the GPU at one thread per row.
template <int RB, int TPR>
struct RowCta {
  static constexpr int kThreads = RB * TPR;
  static constexpr int kMinBlocks = TPR == 1 ? 512 / RB : 3;
};

template <typename T, int RB, int TPR, bool HAS_Z, bool VEC>
__global__ void __launch_bounds__(RowCta<RB, TPR>::kThreads, RowCta<RB, TPR>::kMinBlocks)
    scan_rows_kernel(const RowParams p) {
  constexpr int SPT = NS / TPR;
  using AT = Act<T>;
  constexpr bool FAST = AT::kFast;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem<T, RB>& sm = *reinterpret_cast<Smem<T, RB>*>(smem_raw);

  const int N = (int)p.a.N;
  const int per_chunk = (int)p.a.batch * p.rtiles;
  int item;
  if (p.nchunks > 1) {
    if (threadIdx.x == 0) sm.misc()[0] = (int)atomicAdd(p.hdr, 1u);
    __syncthreads();
    item = sm.misc()[0];
  } else {
    item = blockIdx.x;
  }
  const int chunk = item / per_chunk;  // chunk-major tickets: a chunk's predecessor started earlier
  const int rem = item % per_chunk;
  const int64_t b = rem / p.rtiles;
  const int64_t c0 = (int64_t)(rem % p.rtiles) * RB;
  const int nrows = (int)min64r(RB, p.a.d_inner - c0);
  const int64_t row0 = b * p.a.d_inner + c0;
  const int64_t tc0 = min64r(p.a.L, (int64_t)chunk * p.chunk_len);
  const int64_t tc1 = min64r(p.a.L, tc0 + p.chunk_len);
  const int r = (int)threadIdx.x / TPR;
  const int n0 = ((int)threadIdx.x % TPR) * SPT;
  const bool row_ok = r < nrows;
  const int64_t c = c0 + (row_ok ? r : 0);
  const int64_t row = row0 + (row_ok ? r : 0);

  // per-row constants of this thread's states; padded states (n >= N) are inert: A = 0, B = C = 0
  float a2[SPT], ia[SPT], h[SPT];
  bool precise = !FAST;
  const float* arow = p.a.A + c * N + n0;
#pragma unroll
  for (int n = 0; n < SPT; ++n) {
    const float a = (row_ok && n0 + n < N) ? arow[n] : 0.f;
    const bool tiny = fabsf(a) < 8.673617e-19f;  // |A| < 2^-60 counts as A = 0
    if (row_ok && n0 + n < N && tiny) precise = true;
    a2[n] = tiny ? 0.f : a * kLog2e;
    ia[n] = tiny ? 0.f : 1.f / a;
    // the first chunk starts from the initial state; later chunks start from 0 and take their carry
    h[n] = (chunk == 0 && p.a.h0 && row_ok && n0 + n < N) ? p.a.h0[row * N + n0 + n] : 0.f;
  }
  // slowest decay of the row (its real states only): decides which blocks the carry still changes
  float a2max = -INFINITY;
#pragma unroll
  for (int n = 0; n < SPT; ++n)
    if (row_ok && n0 + n < N) a2max = fmaxf(a2max, a2[n]);
  // a row's threads take the same path (the precise one if any of its states has A = 0)
  if (TPR > 1) {
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) {
      precise |= __shfl_xor_sync(0xffffffffu, (int)precise, off) != 0;
      a2max = fmaxf(a2max, __shfl_xor_sync(0xffffffffu, a2max, off));
    }
  }
  const float Dc = (row_ok && p.a.D) ? p.a.D[c] : 0.f;
  const float biasc = (row_ok && p.a.bias) ? p.a.bias[c] : 0.f;

  // pass one: the chunk from h = 0 (the initial state for the first chunk); later
  // chunks write only the blocks their carried-in state can no longer change
  float S = 0.f;
  if (chunk > 0)
    row_pass<T, RB, TPR, HAS_Z, VEC, kWriteSettled>(sm, p, b, row0, nrows, tc0, tc1, h, a2, ia, arow, precise, Dc,
                                                    biasc, a2max, S);
  else
    row_pass<T, RB, TPR, HAS_Z, VEC, kWriteAll>(sm, p, b, row0, nrows, tc0, tc1, h, a2, ia, arow, precise, Dc,
                                                biasc, a2max, S);

  // ---------------- carry between chunks ----------------
  float hin[SPT];
#pragma unroll
  for (int n = 0; n < SPT; ++n) hin[n] = 0.f;
  if (p.nchunks > 1) {
    const size_t slot = (size_t)per_chunk * RB * NS;  // RB: this instantiation's rows per CTA
    const size_t my = ((size_t)rem * RB + r) * NS + n0;
    if (chunk > 0) {
      if (threadIdx.x == 0) {
        const unsigned* f = p.flags + (size_t)(chunk - 1) * per_chunk + rem;
        sm.misc()[1] = wait_flag_rows(p, f, p.fault_lookback ? 3u : 1u) ? 1 : 0;  // 3 is never written
      }
      __syncthreads();
      __threadfence();
      const bool ok = sm.misc()[1] != 0;
      const float4* prev = reinterpret_cast<const float4*>(p.incl + (size_t)(chunk - 1) * slot + my);
#pragma unroll
      for (int q = 0; q < SPT / 4; ++q) {
        const float4 v = ok ? __ldcg(prev + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        hin[4 * q] = v.x; hin[4 * q + 1] = v.y; hin[4 * q + 2] = v.z; hin[4 * q + 3] = v.w;
      }
#pragma unroll
      for (int n = 0; n < SPT; ++n) {
        const float P = precise ? exp2f(a2[n] * S) : ex2_approx(a2[n] * S);
        h[n] = fmaf(P, hin[n], h[n]);
      }
    }
    if (chunk + 1 < p.nchunks) {
      float4* mine = reinterpret_cast<float4*>(p.incl + (size_t)chunk * slot + my);
#pragma unroll
      for (int q = 0; q < SPT / 4; ++q) mine[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) st_release_gpu(p.flags + (size_t)chunk * per_chunk + rem, 1u);
    }
  }
  if (p.a.final_state && chunk == p.nchunks - 1 && row_ok) {
#pragma unroll
    for (int n = 0; n < SPT; ++n)
      if (n0 + n < N) p.a.final_state[row * N + n0 + n] = h[n];
  }
  if (chunk == 0 || p.nchunks == 1) return;

  // ---------------- pass two: the chunk's first blocks again, from the carried-in state ----------------
  // The same arithmetic as an unchunked scan, so these outputs are rounded once;
  // it runs until every row of the CTA is settled.
  float S2 = 0.f;
  row_pass<T, RB, TPR, HAS_Z, VEC, kWriteUnsettled>(sm, p, b, row0, nrows, tc0, tc1, hin, a2, ia, arow, precise, Dc,
                                                    biasc, a2max, S2);
}

template <typename T, int RB, int TPR, bool HAS_Z, bool VEC>
cudaError_t rows_launch_v(const RowParams& p, int grid, cudaStream_t s) {
  auto kern = scan_rows_kernel<T, RB, TPR, HAS_Z, VEC>;
  const cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem<T, RB>));
  if (e != cudaSuccess) return e;
  kern<<<grid, RowCta<RB, TPR>::kThreads, sizeof(Smem<T, RB>), s>>>(p);
  return cudaGetLastError();
}

template <typename T, int RB, int TPR, bool HAS_Z>
cudaError_t rows_launch_t(const RowParams& p, int grid, cudaStream_t s) {
  return p.vec_rows ? rows_launch_v<T, RB, TPR, HAS_Z, true>(p, grid, s)
                    : rows_launch_v<T, RB, TPR, HAS_Z, false>(p, grid, s);
}

template <typename T, bool HAS_Z>
cudaError_t rows_launch_dt(const RowParams& p, int rb, int tpr, int grid, cudaStream_t s) {
  if (tpr == 2) return rows_launch_t<T, 128, 2, HAS_Z>(p, grid, s);
  if (rb == 128) return rows_launch_t<T, 128, 1, HAS_Z>(p, grid, s);
  return rows_launch_t<T, (sizeof(T) == 2 ? 512 : 256), 1, HAS_Z>(p, grid, s);
}

}  // namespace

int rows_big_cta_rows(int act) { return act == 1 ? 512 : 256; }

cudaError_t scan_rows_launch(const ScanArgs& a, const ScanPlan& plan, cudaStream_t stream) {
  RowParams p{};
  p.a = a;
  p.rtiles = plan.ctiles;
  p.nchunks = plan.nchunks;
  p.chunk_len = plan.chunk_len;
  const int esize = a.act == 1 ? 2 : 4;
  auto a16 = [](const void* q) { return q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  p.vec_rows = ((a.L * esize) % 16 == 0 && a16(a.u) && a16(a.delta) && a16(a.z) && a16(a.out)) ? 1 : 0;
  p.vec_bc = ((a.N * esize) % 16 == 0 && a16(a.B) && a16(a.C)) ? 1 : 0;
  const RuntimeKnobs knobs = runtime_knobs();
  p.timeout_ns = knobs.lookback_timeout_ns > 0 ? knobs.lookback_timeout_ns
                                               : 1000ll * 1000 * 1000 + plan.chunk_len * 100ll;
  p.fault_lookback = knobs.fault_lookback ? 1 : 0;
  if (plan.nchunks > 1) {
    p.hdr = reinterpret_cast<unsigned*>(a.ws);
    p.flags = reinterpret_cast<unsigned*>(a.ws + plan.ws_flags_off);
    p.incl = reinterpret_cast<float*>(a.ws + plan.ws_agg_off);
    cudaError_t e = cudaMemsetAsync(a.ws, 0, plan.ws_agg_off, stream);
    if (e != cudaSuccess) return e;
  }
  const int grid = (int)((int64_t)plan.nchunks * a.batch * plan.ctiles);
  const int rb = plan.rows_per_cta, tpr = plan.threads / plan.rows_per_cta;
  if (a.act == 1)
    return a.z ? rows_launch_dt<__nv_bfloat16, true>(p, rb, tpr, grid, stream)
               : rows_launch_dt<__nv_bfloat16, false>(p, rb, tpr, grid, stream);
  return a.z ? rows_launch_dt<float, true>(p, rb, tpr, grid, stream)
             : rows_launch_dt<float, false>(p, rb, tpr, grid, stream);
}

}  // namespace ssm

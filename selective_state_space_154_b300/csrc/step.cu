// Recurrent (decode) mode for sm_103a: one token per (batch, channel) row,
// fixed-size state updated in place ("Mambaとは？Transformer以外の系列モデル",
// section training、prefill、decodeでは計算の姿が違う; "State Space Models（SSM）
// とMamba" §2.4 二つのモード).
//
// The step is bound by memory: per row it moves the fp32 state (4·N bytes read
// and written) plus x, Δ, z, out.  Two kernels:
//
//  * step_pipe_kernel (d_state ∈ {4, 8, 16, 32, 64}, d_inner a multiple of the
//    tile's rows, state / x / Δ / z 16-byte aligned): a tile is 512 (row, quad
//    of 4 states) items = 8 KB of state, 512 / (d_state / 4) consecutive
//    channels of one batch row.  Each CTA keeps one block of channels (so A,
//    bias and D are read once per CTA) and walks the batch.  One thread per CTA
//    streams each tile's state, x, Δ and z into shared memory with
//    cp.async.bulk (completion counted in bytes on an mbarrier) several tiles
//    ahead; all threads update the tile in place in shared memory, and the same
//    thread writes it back with a bulk store.  Loads of later tiles, the
//    arithmetic of the current one and the stores of earlier ones overlap, so
//    HBM stays busy without a large register footprint.
//  * step_kernel (any shape): work items (row, quad) spread over the grid; each
//    thread issues the loads of kItems items before any arithmetic.
//
// In both, a warp's lanes take consecutive items, so the state moves as
// contiguous 16-byte vectors, and the readout Σ_n C_n h_n is reduced across the
// lanes of a row with shuffles.  The per-state arithmetic is that of the scan.
#include <algorithm>
#include <cstdint>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kItems = 4;
constexpr int kBlock = 256;

template <typename T, int QR, bool VEC>
__global__ void __launch_bounds__(kBlock) step_kernel(const StepArgs p, int64_t nthreads) {
  using AT = Act<T>;
  const int N = (int)p.N;
  const int64_t rows = p.batch * p.d_inner;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const T* xp = static_cast<const T*>(p.x);
  const T* dp = static_cast<const T*>(p.delta);
  const T* zp = static_cast<const T*>(p.z);

  bool ok[kItems];
  int64_t rowv[kItems], cv[kItems];
  int n0v[kItems];
  float hs[kItems][4], av[kItems][4], bv[kItems][4], cc[kItems][4];
  float xv[kItems], rr[kItems], zv[kItems];
  // ---- loads for all items first ----
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const int64_t item = tid + j * nthreads;
    const int64_t row = item / QR;
    const int q = (int)(item % QR);
    const int n0 = q * 4;
    ok[j] = row < rows && n0 < N;  // lanes past the last state of a row hold nothing
    const int64_t rw = ok[j] ? row : 0;
    const int64_t b = rw / p.d_inner, c = rw % p.d_inner;
    rowv[j] = rw;
    cv[j] = c;
    n0v[j] = ok[j] ? n0 : 0;
    float* st = p.state + rw * N + n0v[j];
    const float* ap = p.A + c * N + n0v[j];
    const T* bp = static_cast<const T*>(p.B) + b * N + n0v[j];
    const T* cp = static_cast<const T*>(p.C) + b * N + n0v[j];
    if (VEC) {
      const float4 h4 = ok[j] ? __ldcs(reinterpret_cast<const float4*>(st)) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 a4 = ok[j] ? __ldg(reinterpret_cast<const float4*>(ap)) : make_float4(0.f, 0.f, 0.f, 0.f);
      hs[j][0] = h4.x; hs[j][1] = h4.y; hs[j][2] = h4.z; hs[j][3] = h4.w;
      av[j][0] = a4.x; av[j][1] = a4.y; av[j][2] = a4.z; av[j][3] = a4.w;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bv[j][k] = ok[j] ? AT::load(bp + k) : 0.f;
        cc[j][k] = ok[j] ? AT::load(cp + k) : 0.f;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const bool e = ok[j] && n0v[j] + k < N;
        hs[j][k] = e ? st[k] : 0.f;
        av[j][k] = e ? ap[k] : 0.f;
        bv[j][k] = e ? AT::load(bp + k) : 0.f;
        cc[j][k] = e ? AT::load(cp + k) : 0.f;
      }
    }
    xv[j] = ok[j] ? AT::load(xp + rw) : 0.f;
    rr[j] = ok[j] ? AT::load(dp + rw) + (p.bias ? p.bias[c] : 0.f) : 0.f;
    zv[j] = (ok[j] && zp) ? AT::load(zp + rw) : 0.f;
  }
  // ---- update, readout, store ----
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const float dlt = AT::kFast ? softplus_fast(rr[j]) : softplus_precise(rr[j]);
    float y = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = av[j][k];
      if (fabsf(a) < 8.673617e-19f) {
        hs[j][k] = fmaf(dlt * xv[j], bv[j][k], hs[j][k]);  // A = 0: Ā = 1, B̄ = Δ B
      } else if (AT::kFast) {
        const float em1 = ex2_approx(dlt * (a * kLog2e)) - 1.f;
        hs[j][k] = fmaf(em1, fmaf(xv[j] * (1.f / a), bv[j][k], hs[j][k]), hs[j][k]);
      } else {
        const float em1 = expm1f(dlt * a);
        hs[j][k] = fmaf(em1, fmaf(xv[j] * (1.f / a), bv[j][k], hs[j][k]), hs[j][k]);
      }
      y = fmaf(cc[j][k], hs[j][k], y);
    }
    float* st = p.state + rowv[j] * N + n0v[j];
    if (ok[j]) {
      if (VEC) {
        __stcs(reinterpret_cast<float4*>(st), make_float4(hs[j][0], hs[j][1], hs[j][2], hs[j][3]));
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (n0v[j] + k < N) st[k] = hs[j][k];
      }
    }
    // lanes of one row are adjacent and aligned to QR (nthreads is a multiple of 32)
#pragma unroll
    for (int off = QR / 2; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
    if (ok[j] && n0v[j] == 0) {
      if (p.D) y = fmaf(p.D[cv[j]], xv[j], y);
      if (zp) y *= AT::kFast ? silu_fast(zv[j]) : silu_precise(zv[j]);
      static_cast<T*>(p.out)[rowv[j]] = AT::from_f(y);
    }
  }
}


// ------------------------------------------------------------ pipelined kernel
constexpr int kTileFloats = 2048;   // fp32 state per tile: 8 KB
constexpr int kPipeStages = 5;      // tiles in shared memory per CTA
constexpr int kRefillLag = 1;       // a tile's buffer is refilled this many tiles after its store was issued
constexpr int kPipeBarBytes = 128;  // mbarriers (one per stage + one never-completed) at the front

__device__ unsigned g_step_error;  // sticky: a pipelined step gave up waiting (read by ssm_step_check)

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded wait for the phase of `parity` to complete: false once the deadline
// (globaltimer, ns) has passed or after 2^26 polls, whichever comes first.
__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity, unsigned long long deadline) {
  for (int it = 0; it < (1 << 26); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15) == 15 && globaltimer_ns() > deadline) return false;
  }
  return false;
}
// global -> shared bulk copy, completion signalled on `bar` (bytes: multiple of 16)
__device__ __forceinline__ void bulk_load(unsigned dst, const void* src, unsigned bytes, unsigned bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// shared -> global bulk copy in the current bulk group
__device__ __forceinline__ void bulk_store(void* dst, unsigned src, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Tile geometry for d_state = N: a thread holds SPT = min(N, 16) states of one
// row, TPR = N / SPT threads share a row, a tile is kRows = 2048 / N rows
// (8 KB of state) of one batch row.  Per stage, shared memory holds the state
// tile, x / Δ / z of its rows and B / C of its batch, all bulk-copied.
template <typename T, int N>
struct RowTile {
  static constexpr int SPT = N < 16 ? N : 16;
  static constexpr int TPR = N / SPT;
  static constexpr int Q = SPT / 4;  // float4 groups per thread
  static constexpr int kRows = kTileFloats / N;
  static constexpr int kThreads = kRows * TPR;
  static constexpr int kMinBlocks = 512 / kThreads > 0 ? 512 / kThreads : 1;
  static constexpr int kStateBytes = kTileFloats * 4;
  static constexpr int kInBytes = kRows * (int)sizeof(T);  // x, Δ or z of the tile's rows
  static constexpr int kBCBytes = N * (int)sizeof(T);      // B or C of the tile's batch
  static constexpr int kOffX = kStateBytes, kOffD = kOffX + kInBytes, kOffZ = kOffD + kInBytes;
  static constexpr int kOffB = kOffZ + kInBytes, kOffC = kOffB + kBCBytes;
  static constexpr int kStageBytes = kOffC + kBCBytes;
  static constexpr int kSmemBytes = kPipeBarBytes + kPipeStages * kStageBytes;
  static_assert(kInBytes % 16 == 0 && kBCBytes % 16 == 0, "bulk copies move multiples of 16 bytes");
};

// Four consecutive activation values read from shared memory as one vector.
template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&v)[4]) {
  if constexpr (sizeof(T) == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(w.x << 16);
    v[1] = __uint_as_float(w.x & 0xffff0000u);
    v[2] = __uint_as_float(w.y << 16);
    v[3] = __uint_as_float(w.y & 0xffff0000u);
  } else {
    const float4 w = *reinterpret_cast<const float4*>(p);
    v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
  }
}

struct PipeArgs {
  StepArgs a;
  int64_t ncb;  // channel blocks of kRows channels: d_inner / kRows (the grid is a multiple of it)
  unsigned long long timeout_ns;
  int fault;  // test hook: the first wait is on a barrier that never completes
};

// CTA j owns channel block cb = j mod ncb for its whole life and walks the batch
// rows b = j / ncb, + gridDim / ncb, ...: a tile is (b, cb).  A, bias and D of its
// channels are loaded once.  Thread t reads its SPT states as float4 groups in
// the rotated order (k + rot) mod Q, so that the eight lanes of each shared-memory
// phase hit eight different bank groups; A, B and C are taken in the same order.
template <typename T, int N, bool HAS_Z>
__global__ void __launch_bounds__(RowTile<T, N>::kThreads, RowTile<T, N>::kMinBlocks)
    step_pipe_kernel(const PipeArgs pa) {
  using AT = Act<T>;
  using RT = RowTile<T, N>;
  constexpr int SPT = RT::SPT, TPR = RT::TPR, Q = RT::Q;
  extern __shared__ __align__(128) unsigned char smem[];
  const StepArgs& p = pa.a;
  const int t = threadIdx.x;
  const int r = t / TPR;                   // row within the tile
  const int n0 = (t % TPR) * SPT;          // first state of this thread
  const int rot = (t * SPT / 32) & (Q - 1);
  const unsigned bar0 = smem_u32(smem);
  const unsigned stage0 = bar0 + kPipeBarBytes;
  const unsigned long long deadline = globaltimer_ns() + pa.timeout_ns;

  const int64_t cb = blockIdx.x % pa.ncb;
  const int64_t b0 = blockIdx.x / pa.ncb, bstride = gridDim.x / pa.ncb;
  const int my_tiles = b0 < p.batch ? (int)((p.batch - 1 - b0) / bstride + 1) : 0;
  const int64_t c = cb * RT::kRows + r;
  auto batch_of = [&](int i) { return b0 + (int64_t)i * bstride; };
  const uint8_t* xg = static_cast<const uint8_t*>(p.x);
  const uint8_t* dg = static_cast<const uint8_t*>(p.delta);
  const uint8_t* zg = static_cast<const uint8_t*>(p.z);
  const uint8_t* bg = static_cast<const uint8_t*>(p.B);
  const uint8_t* cg = static_cast<const uint8_t*>(p.C);
  auto issue = [&](int s, int i) {  // one thread: all copies of tile i into stage s
    const unsigned st = stage0 + s * RT::kStageBytes;
    const unsigned bar = bar0 + 8 * s;
    const int64_t b = batch_of(i);
    const int64_t row0 = b * p.d_inner + cb * RT::kRows;
    constexpr int64_t E = sizeof(T);
    mbar_expect_tx(bar, RT::kStateBytes + (HAS_Z ? 3 : 2) * RT::kInBytes + 2 * RT::kBCBytes);
    bulk_load(st, p.state + row0 * N, RT::kStateBytes, bar);
    bulk_load(st + RT::kOffX, xg + row0 * E, RT::kInBytes, bar);
    bulk_load(st + RT::kOffD, dg + row0 * E, RT::kInBytes, bar);
    if (HAS_Z) bulk_load(st + RT::kOffZ, zg + row0 * E, RT::kInBytes, bar);
    bulk_load(st + RT::kOffB, bg + b * N * E, RT::kBCBytes, bar);
    bulk_load(st + RT::kOffC, cg + b * N * E, RT::kBCBytes, bar);
  };

  if (t == 0) {
    for (int s = 0; s <= kPipeStages; ++s) mbar_init(bar0 + 8 * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (t == 0)
    for (int i = 0; i < my_tiles && i < kPipeStages; ++i) issue(i, i);

  // per-channel constants, once per CTA, in this thread's rotated state order
  float a2[SPT], ia[SPT], av[AT::kFast ? 1 : SPT];  // A·log2e, 1/A (0 where |A| < 2^-60: Ā = 1, B̄ = Δ B)
  bool zero_a = false;
#pragma unroll
  for (int k = 0; k < Q; ++k) {
    const int qq = (k + rot) & (Q - 1);
    const float4 a4 = my_tiles > 0 ? __ldg(reinterpret_cast<const float4*>(p.A + c * N + n0) + qq)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    const float a[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool z0 = fabsf(a[j]) < 8.673617e-19f;
      zero_a |= z0;
      a2[4 * k + j] = z0 ? 0.f : a[j] * kLog2e;
      ia[4 * k + j] = z0 ? 0.f : 1.f / a[j];
      if constexpr (!AT::kFast) av[4 * k + j] = a[j];
    }
  }
  const float biasc = (p.bias && my_tiles > 0) ? __ldg(p.bias + c) : 0.f;
  const float Dc = (p.D && my_tiles > 0) ? __ldg(p.D + c) : 0.f;

  int i = 0;
  bool failed = false;
  for (; i < my_tiles; ++i) {
    const int s = i % kPipeStages;
    const int64_t row0 = batch_of(i) * p.d_inner + cb * RT::kRows;
    const unsigned wait_bar = (pa.fault && i == 0) ? bar0 + 8 * kPipeStages : bar0 + 8 * s;
    const bool ok = mbar_wait(wait_bar, (unsigned)(i / kPipeStages) & 1u, deadline);
    unsigned char* st = smem + kPipeBarBytes + s * RT::kStageBytes;
    float4* hq = reinterpret_cast<float4*>(st) + t * Q;
    const T* bs = reinterpret_cast<const T*>(st + RT::kOffB) + n0;
    const T* cs = reinterpret_cast<const T*>(st + RT::kOffC) + n0;
    const float x = AT::to_f(reinterpret_cast<const T*>(st + RT::kOffX)[r]);
    const float rr = AT::to_f(reinterpret_cast<const T*>(st + RT::kOffD)[r]) + biasc;
    const float dlt = AT::kFast ? softplus_fast(rr) : softplus_precise(rr);
    float y = 0.f;
#pragma unroll
    for (int k = 0; k < Q; ++k) {
      const int qq = (k + rot) & (Q - 1);
      const float4 h4 = hq[qq];
      float h[4] = {h4.x, h4.y, h4.z, h4.w}, bb[4], cc[4];
      load4<T>(bs + 4 * qq, bb);
      load4<T>(cs + 4 * qq, cc);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = 4 * k + j;
        if (AT::kFast && !zero_a) {
          const float em1 = ex2_approx(dlt * a2[n]) - 1.f;
          h[j] = fmaf(em1, fmaf(x * ia[n], bb[j], h[j]), h[j]);
        } else if (a2[n] == 0.f) {
          h[j] = fmaf(dlt * x, bb[j], h[j]);  // A = 0: Ā = 1, B̄ = Δ B
        } else {
          float em1;
          if constexpr (AT::kFast) em1 = ex2_approx(dlt * a2[n]) - 1.f;
          else em1 = expm1f(dlt * av[n]);
          h[j] = fmaf(em1, fmaf(x * ia[n], bb[j], h[j]), h[j]);
        }
        y = fmaf(cc[j], h[j], y);
      }
      hq[qq] = make_float4(h[0], h[1], h[2], h[3]);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
    if (n0 == 0 && ok) {
      y = fmaf(Dc, x, y);
      if (HAS_Z) {
        const float zv = AT::to_f(reinterpret_cast<const T*>(st + RT::kOffZ)[r]);
        y *= AT::kFast ? silu_fast(zv) : silu_precise(zv);
      }
      static_cast<T*>(p.out)[row0 + r] = AT::from_f(y);
    }
    fence_async_smem();  // the bulk store below reads what the threads wrote
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    if (t == 0) {
      // refill the buffer of tile j = i - kRefillLag once its store has read it,
      // ahead of this tile's store in the copy queue
      const int j = i - kRefillLag;
      if (j >= 0 && j + kPipeStages < my_tiles) {
        bulk_wait_read<kRefillLag - 1>();
        issue(j % kPipeStages, j + kPipeStages);
      }
      bulk_store(p.state + row0 * N, stage0 + s * RT::kStageBytes, RT::kStateBytes);
      bulk_commit();
    }
  }
  if (t == 0) {
    if (failed) {
      atomicOr(&g_step_error, 1u);
      // let every load still in flight land before the CTA's shared memory is released
      const int last = min(my_tiles, max(kPipeStages, i - kRefillLag + kPipeStages));  // tiles issued so far
      for (int j = i; j < last; ++j)
        mbar_wait(bar0 + 8 * (j % kPipeStages), (unsigned)(j / kPipeStages) & 1u,
                  globaltimer_ns() + pa.timeout_ns);
    }
    bulk_wait_all();
  }
}

template <typename T, int N>
cudaError_t launch_pipe_n(const PipeArgs& pa, cudaStream_t stream) {
  using RT = RowTile<T, N>;
  // per device and instantiation: shared-memory opt-in and resident CTAs per SM, set up once
  constexpr int kMaxDev = 64;
  static int grid_cap[2][kMaxDev] = {};
  const bool has_z = pa.a.z != nullptr;
  auto kern = has_z ? step_pipe_kernel<T, N, true> : step_pipe_kernel<T, N, false>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  int& cap = grid_cap[has_z][dev];
  if (!cap) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RT::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, RT::kThreads, RT::kSmemBytes);
    if (e != cudaSuccess) return e;
    cap = sms * std::max(per_sm, 1);
  }
  // a multiple of the channel blocks, at most one CTA per (batch, channel block)
  const int64_t per_cb = std::max<int64_t>(1, std::min<int64_t>(pa.a.batch, cap / pa.ncb));
  const int64_t grid = pa.ncb * per_cb;
  if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)grid, RT::kThreads, RT::kSmemBytes, stream>>>(pa);
  return cudaGetLastError();
}

// The pipelined kernel takes the step when its tiles fit the shape exactly and
// every bulk-copied array is 16-byte aligned with 16-byte rows of B and C;
// otherwise step_kernel does.
template <typename T>
bool pipe_launch_dt(const StepArgs& a, const StepKnobs& k, cudaStream_t stream, cudaError_t* err) {
  const int N = (int)a.N;
  if (k.force_plain) return false;
  if (N != 4 && N != 8 && N != 16 && N != 32 && N != 64) return false;
  if ((N * (int)sizeof(T)) % 16 != 0) return false;  // B, C rows of one batch
  const int rows_per_tile = kTileFloats / N;
  if (a.d_inner % rows_per_tile != 0) return false;
  auto al = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
  if (!al(a.state) || !al(a.x) || !al(a.delta) || (a.z && !al(a.z)) || !al(a.B) || !al(a.C)) return false;
  PipeArgs pa{};
  pa.a = a;
  pa.ncb = a.d_inner / rows_per_tile;
  pa.timeout_ns = k.timeout_ns > 0 ? (unsigned long long)k.timeout_ns : 1000000000ull;
  pa.fault = k.fault ? 1 : 0;
  switch (N) {
    case 4: *err = launch_pipe_n<T, (sizeof(T) == 4 ? 4 : 8)>(pa, stream); break;  // bf16 N = 4 excluded above
    case 8: *err = launch_pipe_n<T, 8>(pa, stream); break;
    case 16: *err = launch_pipe_n<T, 16>(pa, stream); break;
    case 32: *err = launch_pipe_n<T, 32>(pa, stream); break;
    default: *err = launch_pipe_n<T, 64>(pa, stream); break;
  }
  return true;
}

template <typename T, int QR>
cudaError_t launch_q(const StepArgs& a, bool vec, cudaStream_t stream) {
  const int64_t items = a.batch * a.d_inner * QR;
  int64_t nthreads = (items + kItems - 1) / kItems;
  nthreads = (nthreads + 31) / 32 * 32;
  const int64_t grid = (nthreads + kBlock - 1) / kBlock;
  if (vec)
    step_kernel<T, QR, true><<<(unsigned)grid, kBlock, 0, stream>>>(a, nthreads);
  else
    step_kernel<T, QR, false><<<(unsigned)grid, kBlock, 0, stream>>>(a, nthreads);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dt(const StepArgs& a, cudaStream_t stream) {
  const int quads = (int)((a.N + 3) / 4);
  // float4 state / A loads need rows of a multiple of 4 states (state and A are 16-byte aligned)
  const bool vec = (a.N % 4) == 0;
  if (quads <= 1) return launch_q<T, 1>(a, vec, stream);
  if (quads <= 2) return launch_q<T, 2>(a, vec, stream);
  if (quads <= 4) return launch_q<T, 4>(a, vec, stream);
  if (quads <= 8) return launch_q<T, 8>(a, vec, stream);
  return launch_q<T, 16>(a, vec, stream);
}

}  // namespace

cudaError_t step_launch(const StepArgs& a, const StepKnobs& k, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (a.act == 1) {
    if (pipe_launch_dt<__nv_bfloat16>(a, k, stream, &e)) return e;
    return launch_dt<__nv_bfloat16>(a, stream);
  }
  if (pipe_launch_dt<float>(a, k, stream, &e)) return e;
  return launch_dt<float>(a, stream);
}

cudaError_t step_error_fetch_clear(unsigned* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_step_error, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_step_error, &zero, sizeof(unsigned));
}

}  // namespace ssm

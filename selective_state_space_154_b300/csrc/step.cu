// Recurrent (decode) mode for sm_103a: one token per (batch, channel) row,
// fixed-size state updated in place ("Mambaとは？Transformer以外の系列モデル",
// section training、prefill、decodeでは計算の姿が違う; "State Space Models（SSM）
// とMamba" §2.4 二つのモード).
//
// The step is bound by memory: per row it moves the fp32 state (4·N bytes read
// and written) plus x, Δ, z, out.  Work items are (row, quad of 4 states); a
// warp's lanes take consecutive items, so the state moves as contiguous 16-byte
// vectors, and the readout Σ_n C_n h_n is reduced across the lanes of a row with
// shuffles.  Each thread handles kItems items spread over the grid and issues
// all their loads before any arithmetic, so enough bytes are in flight per SM to
// cover the memory latency.  The per-state arithmetic is that of the scan.
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

cudaError_t step_launch(const StepArgs& a, cudaStream_t stream) {
  return a.act == 1 ? launch_dt<__nv_bfloat16>(a, stream) : launch_dt<float>(a, stream);
}

}  // namespace ssm

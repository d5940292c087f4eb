// Recurrent (decode) mode for sm_103a: one token per (batch, channel) row,
// fixed-size state updated in place ("Mambaとは？Transformer以外の系列モデル",
// section training、prefill、decodeでは計算の姿が違う; "State Space Models（SSM）
// とMamba" §2.4 二つのモード).
//
// The step is bound by HBM (or L2 when the fp32 state stays resident): per row it
// moves the state (4·N bytes read + written) plus x, Δ, z, out.  Each thread
// owns four consecutive states of one row, so a warp reads and writes the state
// as contiguous 16-byte vectors; the readout Σ_n C_n h_n is reduced across the
// row's lanes with shuffles and the lane holding state 0 writes the output.
// The arithmetic per state is the same as in the scan kernel.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

template <typename T, int QR, bool VEC>
__global__ void __launch_bounds__(256) step_kernel(const StepArgs p) {
  using AT = Act<T>;
  const int N = (int)p.N;
  const int64_t rows = p.batch * p.d_inner;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = tid / QR;
  const int q = (int)(tid % QR);
  const bool row_ok = row < rows;
  const int64_t b = row_ok ? row / p.d_inner : 0;
  const int64_t c = row_ok ? row % p.d_inner : 0;

  float y = 0.f;
  float dlt = 0.f, xv = 0.f;
  const bool q_ok = q * 4 < N;  // lanes past the last state of a row hold nothing
  if (row_ok && q_ok) {
    const T* xp = static_cast<const T*>(p.x);
    const T* dp = static_cast<const T*>(p.delta);
    xv = AT::load(xp + row);
    const float rr = AT::load(dp + row) + (p.bias ? p.bias[c] : 0.f);
    dlt = AT::kFast ? softplus_fast(rr) : softplus_precise(rr);
    const int n0 = q * 4;
    float hs[4], av[4], bv[4], cv[4];
    float* st = p.state + row * N + n0;
    const float* ap = p.A + c * N + n0;
    const T* bp = static_cast<const T*>(p.B) + b * N + n0;
    const T* cp = static_cast<const T*>(p.C) + b * N + n0;
    if (VEC) {
      const float4 h4 = *reinterpret_cast<const float4*>(st);
      const float4 a4 = *reinterpret_cast<const float4*>(ap);
      hs[0] = h4.x; hs[1] = h4.y; hs[2] = h4.z; hs[3] = h4.w;
      av[0] = a4.x; av[1] = a4.y; av[2] = a4.z; av[3] = a4.w;
#pragma unroll
      for (int k = 0; k < 4; ++k) { bv[k] = AT::load(bp + k); cv[k] = AT::load(cp + k); }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const bool ok = n0 + k < N;
        hs[k] = ok ? st[k] : 0.f;
        av[k] = ok ? ap[k] : 0.f;
        bv[k] = ok ? AT::load(bp + k) : 0.f;
        cv[k] = ok ? AT::load(cp + k) : 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = av[k];
      if (fabsf(a) < 8.673617e-19f) {
        hs[k] = fmaf(dlt * xv, bv[k], hs[k]);  // A = 0: Ā = 1, B̄ = Δ B
      } else if (AT::kFast) {
        const float em1 = ex2_approx(dlt * (a * kLog2e)) - 1.f;
        hs[k] = fmaf(em1, fmaf(xv * (1.f / a), bv[k], hs[k]), hs[k]);
      } else {
        const float em1 = expm1f(dlt * a);
        hs[k] = fmaf(em1, fmaf(xv * (1.f / a), bv[k], hs[k]), hs[k]);
      }
      y = fmaf(cv[k], hs[k], y);
    }
    if (VEC) {
      *reinterpret_cast<float4*>(st) = make_float4(hs[0], hs[1], hs[2], hs[3]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (n0 + k < N) st[k] = hs[k];
    }
  }
  // reduce the readout over the QR lanes of the row (lanes of a row are adjacent)
#pragma unroll
  for (int off = QR / 2; off > 0; off >>= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
  if (row_ok && q == 0) {
    xv = AT::load(static_cast<const T*>(p.x) + row);
    if (p.D) y = fmaf(p.D[c], xv, y);
    if (p.z) {
      const float zv = AT::load(static_cast<const T*>(p.z) + row);
      y *= AT::kFast ? silu_fast(zv) : silu_precise(zv);
    }
    static_cast<T*>(p.out)[row] = AT::from_f(y);
  }
}

template <typename T, int QR>
cudaError_t launch_q(const StepArgs& a, bool vec, cudaStream_t stream) {
  const int64_t threads_total = a.batch * a.d_inner * QR;
  const int block = 256;
  const int64_t grid = (threads_total + block - 1) / block;
  if (vec)
    step_kernel<T, QR, true><<<(unsigned)grid, block, 0, stream>>>(a);
  else
    step_kernel<T, QR, false><<<(unsigned)grid, block, 0, stream>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dt(const StepArgs& a, cudaStream_t stream) {
  const int quads = (int)((a.N + 3) / 4);
  // float4 state / A loads need rows of a multiple of 4 states (pointers are 16-byte aligned)
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

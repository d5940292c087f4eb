// Selective-scan forward for small problems (few rows × states, short sequences), for
// sm_103a: the sequence is parallelised inside a warp instead of walked by one thread.
//
// The operation is the one of scan_fwd.cu ("State Space Models（SSM）とMamba" §2.2 離散化;
// "Mambaとは？Transformer以外の系列モデル", sections 状態空間モデルを一つの式から理解する and
// Mamba blockのarchitecture).  Each token applies to a state the affine map
// h ↦ Ā_t h + B̄_t x_t, and maps compose associatively, (A₂,b₂)∘(A₁,b₁) = (A₂A₁, A₂b₁+b₂)
// ("Mambaとは？…", Selective Scanは選択機構そのものではない).  So:
//  * a CTA holds one (batch, channel) row, a warp per state n (32·N threads);
//  * lane l takes a segment of ⌈L/32⌉ consecutive tokens (at most kSeg), forms each
//    token's map in registers and composes them;
//  * a five-step shuffle scan of the segments' maps gives every lane the composition of
//    the segments before its own, hence the state entering its segment (from the
//    initial state, or 0);
//  * each lane replays its segment from that state, token by token with the same update
//    as the row kernels, and leaves C_n h_n per token in shared memory;
//  * the row's outputs Σ_n C_n h_n + D x, gated by silu(z), are summed over the states in
//    a fixed order and written once; the lane holding the last token writes the final
//    state.
// For a handful of rows this replaces a sequential walk of L dependent updates by about
// ⌈L/32⌉ + 5 + ⌈L/32⌉ steps.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kSeg = kTinyMaxSeq / 32;  // tokens per lane at most

template <typename T>
__global__ void __launch_bounds__(1024) scan_tiny_kernel(const ScanArgs a, int seg) {
  constexpr bool FAST = Act<T>::kFast;
  extern __shared__ float ys[];  // [N][L]: C_n h_n of every token
  const int n = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = (int)a.N;
  const int64_t L = a.L;
  const int64_t row = blockIdx.x;  // b · d_inner + c
  const int64_t b = row / a.d_inner, c = row % a.d_inner;
  const T* u = static_cast<const T*>(a.u) + row * L;
  const T* dr = static_cast<const T*>(a.delta) + row * L;
  const T* Bp = static_cast<const T*>(a.B) + b * L * N + n;
  const T* Cp = static_cast<const T*>(a.C) + b * L * N + n;
  const float av = a.A[c * N + n];
  const bool zero = fabsf(av) < 8.673617e-19f;  // |A| < 2^-60 counts as A = 0
  const float ia = zero ? 0.f : 1.f / av;
  const float biasc = a.bias ? a.bias[c] : 0.f;
  const int64_t t0 = (int64_t)lane * seg;

  // the segment's tokens: Ā − 1 and w (the update is h ← h + (Ā − 1)(h + w), i.e.
  // Ā h + B̄ x with B̄ x = (Ā − 1) x B / A; for A = 0 it is h ← h + w with w = Δ x B)
  float em[kSeg], w[kSeg];
  float Ac = 1.f, bc = 0.f;  // the segment's composed map
#pragma unroll
  for (int k = 0; k < kSeg; ++k) {
    em[k] = 0.f;
    w[k] = 0.f;
    const int64_t t = t0 + k;
    if (k < seg && t < L) {
      const float x = Act<T>::to_f(u[t]);
      const float r = Act<T>::to_f(dr[t]) + biasc;
      const float dt = FAST ? softplus_fast(r) : softplus_precise(r);
      const float Bv = Act<T>::to_f(Bp[t * N]);
      float abar, bb;
      if (zero) {
        w[k] = dt * x * Bv;
        abar = 1.f;
        bb = w[k];
      } else {
        em[k] = FAST ? ex2_approx(dt * av * kLog2e) - 1.f : expm1f(dt * av);
        w[k] = x * Bv * ia;
        abar = 1.f + em[k];
        bb = em[k] * w[k];
      }
      bc = fmaf(abar, bc, bb);
      Ac *= abar;
    }
  }
  // inclusive scan of the segments' maps over the lanes: lane l ends with segments 0..l
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float Au = __shfl_up_sync(0xffffffffu, Ac, off), bu = __shfl_up_sync(0xffffffffu, bc, off);
    if (lane >= off) {
      bc = fmaf(Ac, bu, bc);
      Ac *= Au;
    }
  }
  float Ax = __shfl_up_sync(0xffffffffu, Ac, 1), bx = __shfl_up_sync(0xffffffffu, bc, 1);
  if (lane == 0) {
    Ax = 1.f;
    bx = 0.f;
  }
  const float h0 = a.h0 ? a.h0[row * N + n] : 0.f;
  float h = fmaf(Ax, h0, bx);  // the state entering this lane's segment
#pragma unroll
  for (int k = 0; k < kSeg; ++k) {
    const int64_t t = t0 + k;
    if (k < seg && t < L) {
      h = zero ? h + w[k] : fmaf(em[k], h + w[k], h);
      ys[n * L + t] = Act<T>::to_f(Cp[t * N]) * h;
      if (t == L - 1 && a.final_state) a.final_state[row * N + n] = h;
    }
  }
  __syncthreads();
  const float Dc = a.D ? a.D[c] : 0.f;
  T* out = static_cast<T*>(a.out) + row * L;
  const T* z = a.z ? static_cast<const T*>(a.z) + row * L : nullptr;
  for (int64_t t = threadIdx.x; t < L; t += blockDim.x) {
    float y = 0.f;
    for (int k = 0; k < N; ++k) y += ys[k * L + t];
    y = fmaf(Dc, Act<T>::to_f(u[t]), y);
    if (z) {
      const float zv = Act<T>::to_f(z[t]);
      y *= FAST ? silu_fast(zv) : silu_precise(zv);
    }
    out[t] = Act<T>::from_f(y);
  }
}

}  // namespace

bool tiny_supported(const ScanArgs& a) {
  return a.N <= 32 && a.L >= 1 && a.L <= kTinyMaxSeq && a.batch * a.d_inner <= (int64_t)INT32_MAX;
}

cudaError_t scan_tiny_launch(const ScanArgs& a, cudaStream_t stream) {
  const int seg = (int)((a.L + 31) / 32);
  const unsigned threads = 32u * (unsigned)a.N;
  const size_t smem = (size_t)a.N * (size_t)a.L * sizeof(float);
  const unsigned grid = (unsigned)(a.batch * a.d_inner);
  if (a.act == 1)
    scan_tiny_kernel<__nv_bfloat16><<<grid, threads, smem, stream>>>(a, seg);
  else
    scan_tiny_kernel<float><<<grid, threads, smem, stream>>>(a, seg);
  return cudaGetLastError();
}

}  // namespace ssm

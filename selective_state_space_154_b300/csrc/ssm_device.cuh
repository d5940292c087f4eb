// Device-side helpers for the selective-scan kernels (sm_103a).
//
// Two arithmetic variants are used:
//  * fast    (bf16 activations): MUFU ex2/lg2/rcp approximations.  The
//    discretisation takes one ex2 per state and forms expm1 as Ā - 1, which is
//    exact in fp32 for Ā in [0.5, 2]; Ā and B̄ then form the exact
//    zero-order-hold pair of a step size that differs from Δ by the ex2
//    rounding (about 2^-22 / |Δ·A| relative).
//  * precise (fp32 activations, or a state with A = 0): expf / expm1f /
//    log1pf from the CUDA math library, IEEE division.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// hardware tanh (one MUFU operation; absolute error about 2^-11)
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus(r) = log(1 + e^r).  Fast form, without branches:
// ln2 · log2(1 + 2^{r log2 e}) for r ≤ 15 and r itself above (relative error < e^-15).
// Where e^r is small the rounding of 1 + e^r leaves an absolute error of about
// 2^-24 in Δ, which moves the output by far less than the bf16 rounding of it.
__device__ __forceinline__ float softplus_fast(float r) {
  const float sp = kLn2 * lg2_approx(1.f + ex2_approx(r * kLog2e));
  return r > 15.f ? r : sp;
}
__device__ __forceinline__ float softplus_precise(float r) {
  return r > 20.f ? r : log1pf(expf(r));
}

// silu(z) = z · sigmoid(z)
__device__ __forceinline__ float silu_fast(float z) {
  return z * rcp_approx(1.f + ex2_approx(-z * kLog2e));
}
__device__ __forceinline__ float silu_precise(float z) { return z / (1.f + expf(-z)); }

// Activation element type traits.
template <typename T> struct Act;
template <> struct Act<float> {
  static constexpr int kBytes = 4;
  static constexpr bool kFast = false;
  __device__ __forceinline__ static float load(const float* p) { return *p; }
  __device__ __forceinline__ static float to_f(float v) { return v; }
  __device__ __forceinline__ static float from_f(float v) { return v; }
};
template <> struct Act<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr bool kFast = true;
  __device__ __forceinline__ static float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// 16-byte asynchronous global->shared copy; src_bytes = 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, int src_bytes) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem_src), "r"(src_bytes)
               : "memory");
}
// The same with an L2 prefetch hint: the L2 fetches the aligned 256 bytes around the
// copied 16 (a row's next stages, for row-streaming kernels).
__device__ __forceinline__ void cp_async16_l2_256(void* smem_dst, const void* gmem_src, int src_bytes) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem_src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

}  // namespace ssm

// Throughput probe of the SM arithmetic pipes that bound the selective scan (sm_103a).
//
// Not part of the scan library: the benchmark loads it to measure, on the GPU it runs
// on, how many FP32 lane operations, MUFU ex2 and state updates of the scan's inner
// loop one SM completes per clock.  Each kernel runs register-resident independent
// chains (no memory traffic inside the timed loop), every CTA times itself with the
// SM clock counter, and the host divides the work by the cycles.
//
// Variants (argument `which`):
//   0  FFMA, 16 independent scalar chains per thread
//   1  FFMA2 (packed f32x2), 8 independent chains per thread
//   2  MUFU ex2, 16 independent chains per thread
//   3  one state update of the scan per state, packed form: Δ·a, ex2 ×2, Ā-1,
//      x·(1/A), (x/A)·B + h, (Ā-1)·s + h, C·h (16 states per thread)
//   4  the same update with scalar instructions only
//   5  integer ALU: LOP3 / PRMT chains (bf16 -> fp32 unpacking), 16 chains per thread
//   6  FFMA2 and MUFU ex2 mixed, 12 packed and 4 ex2 chains per thread (no dependency
//      between them): do the two pipes overlap?
//   7  the same with 6 packed and 4 ex2 chains
//   8  the packed state update with the ex2 replaced by an FMUL: the FP32 work alone
//   9  the scan's per-token work as the row kernels do it, B and C read from shared
//      memory: softplus and silu (ex2, lg2, rcp), 16 state updates, readout, D skip,
//      gate; one thread per row, 8 tokens unrolled
//  10  the same, 4 tokens unrolled
//  11  the same with two threads per row (8 states each, readout summed by a shuffle)
//  12  variant 9 software-pipelined by one token: the ex2 of token t+1's states and
//      its softplus are issued in the loop body that updates token t
//  13  the same with the token loop unrolled twice
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ float ex2a(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void stamp(long long t0, long long* cyc) {
  __syncthreads();
  if (threadIdx.x == 0) cyc[blockIdx.x] = clock64() - t0;
}

__global__ void k_ffma(int iters, float s, float* out, long long* cyc) {
  float a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = threadIdx.x * 1e-3f + i;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int i = 0; i < 16; ++i) a[i] = fmaf(a[i], s, 0.5f);
  }
  stamp(t0, cyc);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc += a[i];
  if (acc == 12345.f) out[threadIdx.x] = acc;
}

__global__ void k_ffma2(int iters, float s, float* out, long long* cyc) {
  float2 a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = make_float2(threadIdx.x * 1e-3f + i, i * 0.5f);
  const float2 ss = make_float2(s, s), hh = make_float2(0.5f, 0.5f);
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = __ffma2_rn(a[i], ss, hh);
  }
  stamp(t0, cyc);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc += a[i].x + a[i].y;
  if (acc == 12345.f) out[threadIdx.x] = acc;
}

__global__ void k_ex2(int iters, float s, float* out, long long* cyc) {
  float a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = (threadIdx.x & 7) * 0.1f + i * 0.01f;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int i = 0; i < 16; ++i) a[i] = ex2a(-a[i]);
  }
  stamp(t0, cyc);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc += a[i];
  if (acc == 12345.f) out[threadIdx.x] = acc * s;
}

// The scan's state update, 16 states, token scalars varied per iteration so that
// nothing is loop-invariant.
template <bool PACKED, bool NO_MUFU = false>
__global__ void k_update(int iters, float s, const float* __restrict__ params, float* out, long long* cyc) {
  // per-thread constants read from memory, so that the compiler cannot rematerialise them
  float h[16], a2[16], ia[16], bb[16], cc[16];
  const float* q = params + (threadIdx.x & 31) * 64;
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    h[n] = 0.f;
    a2[n] = q[n];
    ia[n] = q[16 + n];
    bb[n] = q[32 + n];
    cc[n] = q[48 + n];
  }
  float dlt = 0.01f + (threadIdx.x & 15) * 1e-3f, x = 0.5f, yacc = 0.f;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int tok = 0; tok < 8; ++tok) {
      float y;
      if (PACKED) {
        const float2 dd = make_float2(dlt, dlt), xx = make_float2(x, x);
        float2 ya = make_float2(0.f, 0.f);
#pragma unroll
        for (int n = 0; n < 16; n += 2) {
          const float2 e = __fmul2_rn(dd, make_float2(a2[n], a2[n + 1]));
          const float2 ab = NO_MUFU ? __fmul2_rn(e, make_float2(0.5f, 0.5f)) : make_float2(ex2a(e.x), ex2a(e.y));
          const float2 em = __fadd2_rn(ab, make_float2(-1.f, -1.f));
          const float2 xp = __fmul2_rn(xx, make_float2(ia[n], ia[n + 1]));
          const float2 hb = make_float2(h[n], h[n + 1]);
          const float2 hn = __ffma2_rn(em, __ffma2_rn(xp, make_float2(bb[n], bb[n + 1]), hb), hb);
          h[n] = hn.x;
          h[n + 1] = hn.y;
          ya = __ffma2_rn(make_float2(cc[n], cc[n + 1]), hn, ya);
        }
        y = ya.x + ya.y;
      } else {
        y = 0.f;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          const float em = ex2a(dlt * a2[n]) - 1.f;
          h[n] = fmaf(em, fmaf(x * ia[n], bb[n], h[n]), h[n]);
          y = fmaf(cc[n], h[n], y);
        }
      }
      yacc += y;
      dlt = dlt * s + 1e-4f;
      x = x * s + 0.25f;
    }
  }
  stamp(t0, cyc);
  float acc = yacc;
#pragma unroll
  for (int n = 0; n < 16; ++n) acc += h[n];
  if (acc == 12345.f) out[threadIdx.x] = acc;
}

__device__ __forceinline__ float lg2a(float x) {
  float y;
  asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcpa(float x) {
  float y;
  asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// SPT states per thread (16 / SPT threads per row), TOK tokens per unrolled loop body.
template <int SPT, int TOK>
__global__ void k_row(int iters, float s, const float* __restrict__ params, float* out, long long* cyc) {
  constexpr int TPR = 16 / SPT;
  __shared__ float4 bcs[TOK][8];  // per token: B 0..15, C 0..15
  const int part = threadIdx.x % TPR;
  const float* q = params + (threadIdx.x & 31) * 64;
  float h[SPT], a2[SPT], ia[SPT];
#pragma unroll
  for (int n = 0; n < SPT; ++n) {
    h[n] = 0.f;
    a2[n] = q[part * SPT + n];
    ia[n] = q[16 + part * SPT + n];
  }
  for (int i = threadIdx.x; i < TOK * 8; i += blockDim.x)
    bcs[i / 8][i % 8] = make_float4(q[32 + (i % 4) * 4], q[33 + (i % 4) * 4], q[34 + (i % 4) * 4], q[35 + (i % 4) * 4]);
  float r = -3.f + (threadIdx.x & 7) * 0.1f, z = 0.3f, x = 0.5f, yacc = 0.f, S = 0.f;
  const float D = q[63], bl2 = q[62];
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters * (8 / TOK); ++it) {
#pragma unroll
    for (int tok = 0; tok < TOK; ++tok) {
      const float rl = fmaf(r, 1.4426950408889634f, bl2);
      const float dl = rl > 21.6f ? rl : lg2a(1.f + ex2a(rl));
      const float g = z * rcpa(1.f + ex2a(z * -1.4426950408889634f));
      const float2 dd = make_float2(dl, dl), xx = make_float2(x, x);
      float2 ya = make_float2(0.f, 0.f);
#pragma unroll
      for (int qd = 0; qd < SPT / 4; ++qd) {
        const float4 bq = bcs[tok][part * (SPT / 4) + qd];
        const float4 cq = bcs[tok][4 + part * (SPT / 4) + qd];
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          const int n = 4 * qd + 2 * k2;
          const float2 e = __fmul2_rn(dd, make_float2(a2[n], a2[n + 1]));
          const float2 em = __fadd2_rn(make_float2(ex2a(e.x), ex2a(e.y)), make_float2(-1.f, -1.f));
          const float2 xp = __fmul2_rn(xx, make_float2(ia[n], ia[n + 1]));
          const float2 hb = make_float2(h[n], h[n + 1]);
          const float2 bb = k2 ? make_float2(bq.z, bq.w) : make_float2(bq.x, bq.y);
          const float2 cc = k2 ? make_float2(cq.z, cq.w) : make_float2(cq.x, cq.y);
          const float2 hn = __ffma2_rn(em, __ffma2_rn(xp, bb, hb), hb);
          h[n] = hn.x;
          h[n + 1] = hn.y;
          ya = __ffma2_rn(cc, hn, ya);
        }
      }
      float y = ya.x + ya.y;
      if (TPR == 2) y += __shfl_xor_sync(0xffffffffu, y, 1);
      yacc = fmaf(fmaf(D, x, y), g, yacc);
      S += dl;
      r = r * s + 1e-3f;
      z = z * s + 0.01f;
      x = x * s + 0.25f;
    }
  }
  stamp(t0, cyc);
  float acc = yacc + S;
#pragma unroll
  for (int n = 0; n < SPT; ++n) acc += h[n];
  if (acc == 12345.f) out[threadIdx.x] = acc;
}

// One thread per row, 16 states, the MUFU work of token t+1 issued in the body of token t.
template <int UNR>
__global__ void k_rowsp(int iters, float s, const float* __restrict__ params, float* out, long long* cyc) {
  __shared__ float4 bcs[8][8];
  const float* q = params + (threadIdx.x & 31) * 64;
  float h[16], a2[16], ia[16], ab[16];
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    h[n] = 0.f;
    a2[n] = q[n];
    ia[n] = q[16 + n];
  }
  for (int i = threadIdx.x; i < 64; i += blockDim.x)
    bcs[i / 8][i % 8] = make_float4(q[32 + (i % 4) * 4], q[33 + (i % 4) * 4], q[34 + (i % 4) * 4], q[35 + (i % 4) * 4]);
  float r = -3.f + (threadIdx.x & 7) * 0.1f, z = 0.3f, x = 0.5f, yacc = 0.f, S = 0.f;
  const float D = q[63], bl2 = q[62];
  // token 0's step and its states' ex2
  float dl = lg2a(1.f + ex2a(fmaf(r, 1.4426950408889634f, bl2)));
#pragma unroll
  for (int n = 0; n < 16; ++n) ab[n] = ex2a(dl * a2[n]);
  __syncthreads();
  const long long t0 = clock64();
  const int ntok = iters * 8;
#pragma unroll UNR
  for (int tok = 0; tok < ntok; ++tok) {
    // next token's step size (its MUFU chain runs under this token's FMA work)
    const float r1 = r * s + 1e-3f;
    const float rl1 = fmaf(r1, 1.4426950408889634f, bl2);
    const float dl1 = rl1 > 21.6f ? rl1 : lg2a(1.f + ex2a(rl1));
    const float g = z * rcpa(1.f + ex2a(z * -1.4426950408889634f));
    const float2 xx = make_float2(x, x), dd1 = make_float2(dl1, dl1);
    float2 ya = make_float2(0.f, 0.f);
    const int slot = tok & 7;
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      const float4 bq = bcs[slot][qd];
      const float4 cq = bcs[slot][4 + qd];
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const int n = 4 * qd + 2 * k2;
        const float2 em = __fadd2_rn(make_float2(ab[n], ab[n + 1]), make_float2(-1.f, -1.f));
        const float2 xp = __fmul2_rn(xx, make_float2(ia[n], ia[n + 1]));
        const float2 hb = make_float2(h[n], h[n + 1]);
        const float2 bb = k2 ? make_float2(bq.z, bq.w) : make_float2(bq.x, bq.y);
        const float2 cc = k2 ? make_float2(cq.z, cq.w) : make_float2(cq.x, cq.y);
        const float2 hn = __ffma2_rn(em, __ffma2_rn(xp, bb, hb), hb);
        h[n] = hn.x;
        h[n + 1] = hn.y;
        ya = __ffma2_rn(cc, hn, ya);
        const float2 e1 = __fmul2_rn(dd1, make_float2(a2[n], a2[n + 1]));
        ab[n] = ex2a(e1.x);
        ab[n + 1] = ex2a(e1.y);
      }
    }
    const float y = ya.x + ya.y;
    yacc = fmaf(fmaf(D, x, y), g, yacc);
    S += dl;
    dl = dl1;
    r = r1;
    z = z * s + 0.01f;
    x = x * s + 0.25f;
  }
  stamp(t0, cyc);
  float acc = yacc + S;
#pragma unroll
  for (int n = 0; n < 16; ++n) acc += h[n];
  if (acc == 12345.f) out[threadIdx.x] = acc;
}

// F packed FMA chains and M ex2 chains per thread, independent of each other
template <int F, int M>
__global__ void k_mix(int iters, float s, float* out, long long* cyc) {
  float2 a[F];
  float m[M];
#pragma unroll
  for (int i = 0; i < F; ++i) a[i] = make_float2(threadIdx.x * 1e-3f + i, i * 0.5f);
#pragma unroll
  for (int i = 0; i < M; ++i) m[i] = (threadIdx.x & 7) * 0.1f + i * 0.01f;
  const float2 ss = make_float2(s, s), hh = make_float2(0.5f, 0.5f);
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
#pragma unroll
      for (int i = 0; i < F; ++i) a[i] = __ffma2_rn(a[i], ss, hh);
#pragma unroll
      for (int i = 0; i < M; ++i) m[i] = ex2a(-m[i]);
    }
  }
  stamp(t0, cyc);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < F; ++i) acc += a[i].x + a[i].y;
#pragma unroll
  for (int i = 0; i < M; ++i) acc += m[i];
  if (acc == 12345.f) out[threadIdx.x] = acc;
}

__global__ void k_alu(int iters, float s, float* out, long long* cyc) {
  unsigned a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = threadIdx.x * 2654435761u + i;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        a[i] = __byte_perm(a[i], 0u, 0x1044) ^ (a[i] & 0xffff0000u);  // PRMT + LOP3
      }
  }
  stamp(t0, cyc);
  unsigned acc = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc += a[i];
  if (acc == 12345u) out[threadIdx.x] = s;
}

}  // namespace

extern "C" {

// Runs variant `which` with `ctas` CTAs of `threads` threads for `iters` loop
// iterations; returns 0 and writes the per-CTA SM cycles (host array of `ctas`
// entries) and the work per thread (lane operations; state updates for 3, 4 and 8;
// rounds of the mix for 6 and 7), or a CUDA error code.  All memory is allocated
// and freed here.
__attribute__((visibility("default"))) int ssm_probe_pipe_rates(int which, int ctas, int threads, int iters, long long* cycles_host,
                         double* work_per_thread) {
  float* out = nullptr;
  long long* cyc = nullptr;
  float* params = nullptr;
  cudaError_t e = cudaMalloc(&out, sizeof(float) * 1024);
  if (e != cudaSuccess) return (int)e;
  e = cudaMalloc(&params, sizeof(float) * 32 * 64);
  if (e != cudaSuccess) {
    cudaFree(out);
    return (int)e;
  }
  {
    float hp[32 * 64];
    for (int l = 0; l < 32; ++l)
      for (int n = 0; n < 16; ++n) {
        hp[l * 64 + n] = -(n + 1) * 1.4426950408889634f;
        hp[l * 64 + 16 + n] = -1.f / (n + 1);
        hp[l * 64 + 32 + n] = 0.01f * (n + (l & 3));
        hp[l * 64 + 48 + n] = 0.02f * (16 - n);
      }
    e = cudaMemcpy(params, hp, sizeof(hp), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaMalloc(&cyc, sizeof(long long) * ctas);
  if (e != cudaSuccess) {
    cudaFree(out);
    cudaFree(params);
    return (int)e;
  }
  const float s = 0.999f;
  double w = 0;
  switch (which) {
    case 0: k_ffma<<<ctas, threads>>>(iters, s, out, cyc); w = 8.0 * 16 * iters; break;
    case 1: k_ffma2<<<ctas, threads>>>(iters, s, out, cyc); w = 8.0 * 16 * iters; break;
    case 2: k_ex2<<<ctas, threads>>>(iters, s, out, cyc); w = 8.0 * 16 * iters; break;
    case 3: k_update<true><<<ctas, threads>>>(iters, s, params, out, cyc); w = 8.0 * 16 * iters; break;
    case 4: k_update<false><<<ctas, threads>>>(iters, s, params, out, cyc); w = 8.0 * 16 * iters; break;
    case 5: k_alu<<<ctas, threads>>>(iters, s, out, cyc); w = 4.0 * 16 * 2 * iters; break;
    case 6: k_mix<12, 4><<<ctas, threads>>>(iters, s, out, cyc); w = 8.0 * iters; break;
    case 7: k_mix<6, 4><<<ctas, threads>>>(iters, s, out, cyc); w = 8.0 * iters; break;
    case 8: k_update<true, true><<<ctas, threads>>>(iters, s, params, out, cyc); w = 8.0 * 16 * iters; break;
    case 9: k_row<16, 8><<<ctas, threads>>>(iters, s, params, out, cyc); w = 8.0 * 16 * iters; break;
    case 10: k_row<16, 4><<<ctas, threads>>>(iters, s, params, out, cyc); w = 8.0 * 16 * iters; break;
    case 11: k_row<8, 8><<<ctas, threads>>>(iters, s, params, out, cyc); w = 8.0 * 8 * iters; break;
    case 12: k_rowsp<1><<<ctas, threads>>>(iters, s, params, out, cyc); w = 8.0 * 16 * iters; break;
    case 13: k_rowsp<2><<<ctas, threads>>>(iters, s, params, out, cyc); w = 8.0 * 16 * iters; break;
    default: cudaFree(out); cudaFree(cyc); cudaFree(params); return (int)cudaErrorInvalidValue;
  }
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(cycles_host, cyc, sizeof(long long) * ctas, cudaMemcpyDeviceToHost);
  cudaFree(out);
  cudaFree(cyc);
  cudaFree(params);
  *work_per_thread = w;
  return (int)e;
}

}  // extern "C"

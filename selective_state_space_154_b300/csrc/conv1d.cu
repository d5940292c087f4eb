// Causal depthwise Conv1D + SiLU for sm_103a: the short convolution of the
// Mamba block's main branch, in front of the selective SSM
// ("Mambaとは？Transformer以外の系列モデル", section Mamba blockのarchitecture,
// steps 2 and 3), and its one-token decode form with the carried state
// (same page, section training、prefill、decodeでは計算の姿が違う).
//
//   pre[t] = bias + Σ_{k<W} w[k] · x̃[t - (W-1) + k],   out[t] = silu(pre[t])
//
// x̃ is the row prefixed by the W-1 inputs before it (the carried state, or
// zeros).  Both kernels are bound by memory: per (row, token) one input read
// and one output written.
//
// conv1d_fwd_kernel: a thread owns 32 consecutive tokens of one row (four
// 16-byte vectors in bf16, eight in fp32, all loaded before any arithmetic).
// The 8 tokens before a thread's own come from the lane to its left by
// shuffles; lane 0 loads them (or takes the carried state at the start of the
// row).  The thread
// holding the row's last token writes the final state.
// conv1d_step_kernel: one thread per row shifts the W-1 carried inputs, appends
// x and writes out; conv1d_step4_kernel does the same for four consecutive channels
// with vector accesses (bf16, width 4).
#include <algorithm>
#include <cstdint>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kTok = 8;            // tokens per 16-byte vector (bf16)
constexpr int kVec = 4;            // vectors per thread in the sequence kernel
constexpr int kSpan = kTok * kVec; // tokens per thread in the sequence kernel
constexpr int kConvBlock = 256;    // threads per CTA (at most)

template <typename T>
__device__ __forceinline__ float ld_act(const T* p) {
  return Act<T>::to_f(*p);
}

// 8 consecutive values at p (16-byte aligned)
template <typename T>
__device__ __forceinline__ void load8_vec(const T* p, float* v) {
  if constexpr (sizeof(T) == 2) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const unsigned u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(u[i] << 16);
      v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
  } else {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

template <typename T>
__device__ __forceinline__ void store8_vec(T* p, const float* v) {
  if constexpr (sizeof(T) == 2) {
    unsigned u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      u[i] = *reinterpret_cast<unsigned*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(u[0], u[1], u[2], u[3]);
  } else {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

// silu(v) = v·sigmoid(v): v / (1 + 2^(-v log2 e)) with the MUFU ex2 and rcp
// approximations for bf16 outputs (accurate for v < 0 too), the precise form otherwise.
template <bool FAST>
__device__ __forceinline__ float silu_c(float v) {
  return FAST ? silu_fast(v) : silu_precise(v);
}

struct ConvArgs {
  const void* x;
  const float* w;      // [d_inner][W]
  const float* bias;   // [d_inner] or nullptr
  const void* state0;  // [rows][W-1] or nullptr
  void* out;
  void* stateT;        // [rows][W-1] or nullptr
  int64_t rows, d_inner, L;
  int W;               // taps (runtime copy; the forward kernel is instantiated per width)
};

// Grid: x = segments of blockDim.x * kSpan tokens of a row, y = channel, z = batch
// (no division per thread).  A thread owns kSpan consecutive tokens, loaded as
// kVec vectors before any arithmetic.
template <typename T, int W, bool VEC>
__global__ void __launch_bounds__(kConvBlock) conv1d_fwd_kernel(const ConvArgs a) {
  using AT = Act<T>;
  const int lane = threadIdx.x & 31;
  const int64_t c = blockIdx.y;
  const int64_t row = (int64_t)blockIdx.z * a.d_inner + c;
  const int64_t t0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * kSpan;
  const int64_t L = a.L;
  if (t0 - lane * kSpan >= L) return;  // whole warp past the end of the row (lane 0 then always has t0 < L)
  const T* xr = static_cast<const T*>(a.x) + row * L;
  const T* sr = a.state0 ? static_cast<const T*>(a.state0) + row * (W - 1) : nullptr;

  // window x̃[t0-8 .. t0+kSpan-1]: win[0..7] the 8 tokens before, win[8..] the thread's own
  float win[kTok + kSpan];
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    const int64_t tv = t0 + v * kTok;
    if (VEC && tv + kTok <= L) {
      load8_vec<T>(xr + tv, win + kTok + v * kTok);
    } else {
#pragma unroll
      for (int i = 0; i < kTok; ++i) win[kTok + v * kTok + i] = (tv + i < L) ? ld_act<T>(xr + tv + i) : 0.f;
    }
  }
  // the 8 tokens before: the last 8 of the lane to the left, or loaded by lane 0
#pragma unroll
  for (int i = 0; i < kTok; ++i) win[i] = __shfl_up_sync(0xffffffffu, win[kSpan + i], 1);
  if (lane == 0) {
    if (t0 >= kTok) {
      if (VEC) {
        load8_vec<T>(xr + t0 - kTok, win);
      } else {
#pragma unroll
        for (int i = 0; i < kTok; ++i) win[i] = ld_act<T>(xr + t0 - kTok + i);
      }
    } else {  // t0 == 0: positions -8..-1 are the carried state (zeros before it)
#pragma unroll
      for (int i = 0; i < kTok; ++i) {
        const int pos = i - kTok;
        win[i] = (sr && pos >= -(W - 1)) ? ld_act<T>(sr + (W - 1) + pos) : 0.f;
      }
    }
  }
  if (t0 >= L) return;

  // out[t0+j] = silu(bias + Σ_k w[k] x̃[t0+j-(W-1)+k]), window index kTok + j - (W-1) + k
  const float* wc = a.w + c * W;
  float wk[W];
#pragma unroll
  for (int k = 0; k < W; ++k) wk[k] = __ldg(wc + k);
  const float b0 = a.bias ? __ldg(a.bias + c) : 0.f;
  T* orow = static_cast<T*>(a.out) + row * L;
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    float y[kTok];
#pragma unroll
    for (int i = 0; i < kTok; ++i) {
      const int j = v * kTok + i;
      float pre = b0;
#pragma unroll
      for (int k = 0; k < W; ++k) pre = fmaf(wk[k], win[kTok + j - (W - 1) + k], pre);  // index >= 1
      y[i] = silu_c<AT::kFast>(pre);
    }
    const int64_t tv = t0 + v * kTok;
    if (VEC && tv + kTok <= L) {
      store8_vec<T>(orow + tv, y);
    } else {
#pragma unroll
      for (int i = 0; i < kTok; ++i)
        if (tv + i < L) orow[tv + i] = AT::from_f(y[i]);
    }
  }
  // final state: x̃[L-(W-1) .. L-1], held in this window by the thread with the last token
  if (a.stateT && t0 + kSpan >= L) {
    T* so = static_cast<T*>(a.stateT) + row * (W - 1);
    // position L-(W-1)+j sits at window index first + j, first = kTok + (L-1-t0) - (W-2)
    const int first = kTok + (int)(L - 1 - t0) - (W - 2);
#pragma unroll
    for (int idx = 0; idx < kTok + kSpan; ++idx) {  // compile-time window index keeps win in registers
      const int j = idx - first;
      if (j >= 0 && j < W - 1) so[j] = AT::from_f(win[idx]);
    }
  }
}

// Grid: x = blocks of kStepItems x 256 channels, y = batch.  A thread takes
// kStepItems channels 256 apart and issues all their loads before any
// arithmetic, so one wave of CTAs keeps enough bytes in flight.
constexpr int kStepItems = 4;

template <typename T, int W>
__global__ void __launch_bounds__(kConvBlock) conv1d_step_kernel(const ConvArgs a) {
  using AT = Act<T>;
  constexpr int S = W > 1 ? W - 1 : 1;  // carried inputs per row (storage for W = 1 unused)
  const int64_t cbase = (int64_t)blockIdx.x * kConvBlock * kStepItems + threadIdx.x;
  const int64_t rbase = (int64_t)blockIdx.y * a.d_inner;
  float st[kStepItems][S], xv[kStepItems], wv[kStepItems][W], bv[kStepItems];
#pragma unroll
  for (int i = 0; i < kStepItems; ++i) {
    const int64_t c = cbase + i * kConvBlock;
    const bool ok = c < a.d_inner;
    const int64_t row = rbase + (ok ? c : 0);
    const T* sp = static_cast<const T*>(a.stateT) + row * (W - 1);
#pragma unroll
    for (int k = 0; k < W - 1; ++k) st[i][k] = ok ? ld_act<T>(sp + k) : 0.f;
    xv[i] = ok ? ld_act<T>(static_cast<const T*>(a.x) + row) : 0.f;
#pragma unroll
    for (int k = 0; k < W; ++k) wv[i][k] = ok ? __ldg(a.w + c * W + k) : 0.f;
    bv[i] = (ok && a.bias) ? __ldg(a.bias + c) : 0.f;
  }
#pragma unroll
  for (int i = 0; i < kStepItems; ++i) {
    const int64_t c = cbase + i * kConvBlock;
    if (c >= a.d_inner) continue;
    const int64_t row = rbase + c;
    float pre = bv[i];
#pragma unroll
    for (int k = 0; k < W; ++k) pre = fmaf(wv[i][k], k == W - 1 ? xv[i] : st[i][k], pre);
    static_cast<T*>(a.out)[row] = AT::from_f(silu_c<AT::kFast>(pre));
    T* sp = static_cast<T*>(a.stateT) + row * (W - 1);
#pragma unroll
    for (int k = 0; k < W - 1; ++k) sp[k] = AT::from_f(k + 1 < W - 1 ? st[i][k + 1] : xv[i]);
  }
}

// Decode step for bf16 and width 4 (Mamba's): a thread owns four consecutive channels of
// one batch row, so that x and out (8 bytes), the carried inputs (24 bytes), the taps
// (64 bytes) and the bias (16 bytes) move as whole vectors; the taps are applied in the
// order of conv1d_step_kernel, so both give the same bits.
__device__ __forceinline__ float bf16_at(const unsigned (&w)[6], int i) {
  return __uint_as_float((i & 1) ? (w[i >> 1] & 0xffff0000u) : (w[i >> 1] << 16));
}
__device__ __forceinline__ unsigned pack2_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<unsigned*>(&h);
}
__global__ void __launch_bounds__(kConvBlock) conv1d_step4_kernel(const ConvArgs a) {
  const int64_t c = 4 * ((int64_t)blockIdx.x * kConvBlock + threadIdx.x);
  if (c >= a.d_inner) return;
  const int64_t row = (int64_t)blockIdx.y * a.d_inner + c;
  const uint2 xw = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(a.x) + row);
  uint2* sp = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.stateT) + row * 3);
  const uint2 s0 = sp[0], s1 = sp[1], s2 = sp[2];  // channel k's three carried inputs: values 3k .. 3k + 2
  const float4* w4 = reinterpret_cast<const float4*>(a.w + c * 4);
  const float4 wq[4] = {__ldg(w4), __ldg(w4 + 1), __ldg(w4 + 2), __ldg(w4 + 3)};
  const float4 bq = a.bias ? __ldg(reinterpret_cast<const float4*>(a.bias + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
  const unsigned sw[6] = {s0.x, s0.y, s1.x, s1.y, s2.x, s2.y};
  const float xs[4] = {__uint_as_float(xw.x << 16), __uint_as_float(xw.x & 0xffff0000u),
                       __uint_as_float(xw.y << 16), __uint_as_float(xw.y & 0xffff0000u)};
  const float bs[4] = {bq.x, bq.y, bq.z, bq.w};
  float y[4], ns[12];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float s_0 = bf16_at(sw, 3 * k), s_1 = bf16_at(sw, 3 * k + 1), s_2 = bf16_at(sw, 3 * k + 2);
    float pre = bs[k];
    pre = fmaf(wq[k].x, s_0, pre);
    pre = fmaf(wq[k].y, s_1, pre);
    pre = fmaf(wq[k].z, s_2, pre);
    pre = fmaf(wq[k].w, xs[k], pre);
    y[k] = silu_c<true>(pre);
    ns[3 * k] = s_1;
    ns[3 * k + 1] = s_2;
    ns[3 * k + 2] = xs[k];
  }
  *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + row) =
      make_uint2(pack2_bf16(y[0], y[1]), pack2_bf16(y[2], y[3]));
  sp[0] = make_uint2(pack2_bf16(ns[0], ns[1]), pack2_bf16(ns[2], ns[3]));
  sp[1] = make_uint2(pack2_bf16(ns[4], ns[5]), pack2_bf16(ns[6], ns[7]));
  sp[2] = make_uint2(pack2_bf16(ns[8], ns[9]), pack2_bf16(ns[10], ns[11]));
}

template <typename T, int W>
cudaError_t fwd_w(const ConvArgs& a, bool vec, cudaStream_t s) {
  // CTA width: enough warps for the row, at most kConvBlock threads
  const int64_t need = (a.L + kSpan - 1) / kSpan;
  const int threads = (int)std::min<int64_t>(kConvBlock, (need + 31) / 32 * 32);
  const int64_t segs = (a.L + (int64_t)threads * kSpan - 1) / ((int64_t)threads * kSpan);
  if (segs > INT32_MAX || a.d_inner > kMaxConvGridYZ || a.rows / a.d_inner > kMaxConvGridYZ)
    return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)segs, (unsigned)a.d_inner, (unsigned)(a.rows / a.d_inner));
  if (vec)
    conv1d_fwd_kernel<T, W, true><<<grid, threads, 0, s>>>(a);
  else
    conv1d_fwd_kernel<T, W, false><<<grid, threads, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t fwd_dt(const ConvArgs& a, bool vec, cudaStream_t s) {
  switch (a.W) {
    case 1: return fwd_w<T, 1>(a, vec, s);
    case 2: return fwd_w<T, 2>(a, vec, s);
    case 3: return fwd_w<T, 3>(a, vec, s);
    case 4: return fwd_w<T, 4>(a, vec, s);
    case 5: return fwd_w<T, 5>(a, vec, s);
    case 6: return fwd_w<T, 6>(a, vec, s);
    case 7: return fwd_w<T, 7>(a, vec, s);
    case 8: return fwd_w<T, 8>(a, vec, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t step_dt(const ConvArgs& a, dim3 grid, cudaStream_t s) {
  switch (a.W) {
    case 1: conv1d_step_kernel<T, 1><<<grid, kConvBlock, 0, s>>>(a); break;
    case 2: conv1d_step_kernel<T, 2><<<grid, kConvBlock, 0, s>>>(a); break;
    case 3: conv1d_step_kernel<T, 3><<<grid, kConvBlock, 0, s>>>(a); break;
    case 4: conv1d_step_kernel<T, 4><<<grid, kConvBlock, 0, s>>>(a); break;
    case 5: conv1d_step_kernel<T, 5><<<grid, kConvBlock, 0, s>>>(a); break;
    case 6: conv1d_step_kernel<T, 6><<<grid, kConvBlock, 0, s>>>(a); break;
    case 7: conv1d_step_kernel<T, 7><<<grid, kConvBlock, 0, s>>>(a); break;
    case 8: conv1d_step_kernel<T, 8><<<grid, kConvBlock, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t conv1d_fwd_launch(const ConvCall& k, cudaStream_t stream) {
  ConvArgs a{};
  a.x = k.x; a.w = k.w; a.bias = k.bias; a.state0 = k.state_in; a.out = k.out; a.stateT = k.state_out;
  a.rows = k.batch * k.d_inner; a.d_inner = k.d_inner; a.L = k.L; a.W = k.W;
  const int esz = k.act == 1 ? 2 : 4;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec = (k.L * esz) % 16 == 0 && a16(k.x) && a16(k.out);
  return k.act == 1 ? fwd_dt<__nv_bfloat16>(a, vec, stream) : fwd_dt<float>(a, vec, stream);
}

cudaError_t conv1d_step_launch(const ConvCall& k, cudaStream_t stream) {
  ConvArgs a{};
  a.x = k.x; a.w = k.w; a.bias = k.bias; a.out = k.out; a.stateT = k.state_out;
  a.rows = k.batch * k.d_inner; a.d_inner = k.d_inner; a.L = 1; a.W = k.W;
  if (k.batch > kMaxConvGridYZ) return cudaErrorInvalidConfiguration;
  auto al = [](const void* q, unsigned n) { return (reinterpret_cast<uintptr_t>(q) & (n - 1u)) == 0; };
  if (k.act == 1 && k.W == 4 && k.d_inner % 4 == 0 && al(k.x, 8) && al(k.out, 8) && al(k.state_out, 8) &&
      al(k.w, 16) && (!k.bias || al(k.bias, 16))) {
    const int64_t per_cta = (int64_t)kConvBlock * 4;
    const dim3 grid((unsigned)((k.d_inner + per_cta - 1) / per_cta), (unsigned)k.batch);
    conv1d_step4_kernel<<<grid, kConvBlock, 0, stream>>>(a);
    return cudaGetLastError();
  }
  const int64_t per_cta = (int64_t)kConvBlock * kStepItems;
  const dim3 grid((unsigned)((k.d_inner + per_cta - 1) / per_cta), (unsigned)k.batch);
  return k.act == 1 ? step_dt<__nv_bfloat16>(a, grid, stream) : step_dt<float>(a, grid, stream);
}

}  // namespace ssm

// Shared device helpers for the GPT-2 training-step kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

typedef __nv_bfloat16 bf16;

// Device error word bits (OR-ed into the handle's error word, read at sync points).
enum : int {
  DEV_ERR_BAD_TOKEN = 1,   // a token id outside [0, V): the read was clamped
  DEV_ERR_TIMEOUT = 2,     // a bounded wait on an mbarrier gave up
  DEV_ERR_BAD_TARGET = 4,  // a target id outside [0, V)
};

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// A 16-byte vector of elements: 4 floats or 8 bf16.
template <typename T> struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  union { uint4 u; T e[N]; };
};

template <typename T>
__device__ __forceinline__ Vec16<T> ld16(const T* p) {
  Vec16<T> v; v.u = *reinterpret_cast<const uint4*>(p); return v;
}
template <typename T>
__device__ __forceinline__ void st16(T* p, const Vec16<T>& v) {
  *reinterpret_cast<uint4*>(p) = v.u;
}
// Streaming (evict-first) variants for data read or written exactly once.
template <typename T>
__device__ __forceinline__ Vec16<T> ld16_cs(const T* p) {
  Vec16<T> v; v.u = __ldcs(reinterpret_cast<const uint4*>(p)); return v;
}
template <typename T>
__device__ __forceinline__ void st16_cs(T* p, const Vec16<T>& v) {
  __stcs(reinterpret_cast<uint4*>(p), v.u);
}

// ------------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------------ exp2 / tanh
// Hardware base-2 exponential (PTX ex2.approx.ftz.f32), used by the online softmax.
// Two bf16 packed in one word (the lower-indexed one in the low half) -> fp32 pair, exactly;
// and an fp32 pair -> two bf16 (round to nearest even) in one word.
__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
__device__ __forceinline__ uint32_t pack2_bf16_rn(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh-approximation GELU, 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), and its
// derivative; tanhf is CUDA's own function.
__device__ __forceinline__ float gelu_tanh(float x) {
  const float k = 0.7978845608028654f;
  float t = tanhf(k * (x + 0.044715f * x * x * x));
  return 0.5f * x * (1.0f + t);
}
__device__ __forceinline__ float gelu_tanh_grad(float x) {
  const float k = 0.7978845608028654f;
  float t = tanhf(k * (x + 0.044715f * x * x * x));
  return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * k * (1.0f + 3.0f * 0.044715f * x * x);
}

// tanh from the hardware approximation (PTX tanh.approx.f32, relative error about 2^-11):
// used where the result is rounded to bf16 (8 significant bits), so the approximation
// error stays well below the rounding step.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// gelu_tanh(x) and, in `grad`, gelu_tanh'(x) from one tanh
__device__ __forceinline__ float2 gelu_tanh_and_grad_fast2(float2 x, float2& grad) {
  const float2 k0 = make_float2(0.7978845608028654f, 0.7978845608028654f);
  const float2 k1 = make_float2(0.044715f * 0.7978845608028654f, 0.044715f * 0.7978845608028654f);
  const float2 k3 = make_float2(3.0f * 0.044715f * 0.7978845608028654f,
                                3.0f * 0.044715f * 0.7978845608028654f);
  const float2 h = make_float2(0.5f, 0.5f), one = make_float2(1.0f, 1.0f);
  const float2 x2 = __fmul2_rn(x, x);
  const float2 u = __fmul2_rn(x, __ffma2_rn(k1, x2, k0));
  const float2 t = make_float2(tanh_approx(u.x), tanh_approx(u.y));
  const float2 nt = make_float2(-t.x, -t.y);
  const float2 hx = __fmul2_rn(h, x);
  // 0.5 (1 + t) + 0.5 x (1 - t^2) (k0 + 3 k1 x^2)
  grad = __ffma2_rn(__fmul2_rn(hx, __ffma2_rn(nt, t, one)), __ffma2_rn(k3, x2, k0),
                    __ffma2_rn(h, t, h));
  return __ffma2_rn(hx, t, hx);
}

__host__ __device__ inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

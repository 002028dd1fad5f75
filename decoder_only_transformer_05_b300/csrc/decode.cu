// Forward-only inference with a KV cache (greedy decoding, one new token per sequence per
// step): the cache store, the one-query attention over the cached keys and values, and a
// gather of the prompt's last positions. The model and the causal scaled softmax attention
// are those of 「从零实现一个最小GPT：代码讲解 + 知识点全解」 (二.3 Head, 三.3); its 三.8
// generation loop re-runs the whole prefix for each new token, whereas here each layer's
// keys and values of earlier positions are kept and only the new position is computed.
#include "common.cuh"
#include "launch.h"

namespace gpt2k {

static cudaError_t last() {
  return cudaGetLastError();
}

// One thread per 16-byte vector of a cached row (2C elements).
template <typename T>
__global__ void kv_store_kernel(T* __restrict__ cache, const T* __restrict__ qkv, int B, int Trows,
                                int pos0, int n, int Tmax, int C) {
  constexpr int VE = 16 / sizeof(T);
  const int vpr = 2 * C / VE;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)B * n * vpr) return;
  const int v = (int)(i % vpr);
  const long long r = i / vpr;
  const int pos = (int)(r % n), b = (int)(r / n);
  const Vec16<T> x = ld16(qkv + ((size_t)b * Trows + pos) * 3 * C + C + (size_t)v * VE);
  st16(cache + ((size_t)b * Tmax + pos0 + pos) * 2 * C + (size_t)v * VE, x);
}

cudaError_t kv_cache_store(DType t, void* cache, const void* qkv, int B, int Trows, int pos0,
                           int n, int Tmax, int C, cudaStream_t s) {
  if (B <= 0 || n <= 0 || pos0 < 0 || pos0 + n > Tmax || n > Trows) return cudaErrorInvalidValue;
  if (t == DType::BF16) {
    const long long total = (long long)B * n * (2 * C / 8);
    kv_store_kernel<bf16><<<ceil_div(total, 256), 256, 0, s>>>((bf16*)cache, (const bf16*)qkv, B,
                                                               Trows, pos0, n, Tmax, C);
  } else {
    const long long total = (long long)B * n * (2 * C / 4);
    kv_store_kernel<float><<<ceil_div(total, 256), 256, 0, s>>>((float*)cache, (const float*)qkv,
                                                                B, Trows, pos0, n, Tmax, C);
  }
  count_launches(1);
  return last();
}

// Block (h, b), four warps. Warp w takes keys w, w + 4, ... <= t; lane l holds dimensions
// l, l + 32, ... of the head (hs <= 128). Each warp keeps an online softmax (running maximum m,
// sum l, weighted value sum) in the log2 domain; the four warps are merged in warp order.
template <typename T>
__global__ void __launch_bounds__(128)
attn_decode_kernel(T* __restrict__ out, const T* __restrict__ qkv, const T* __restrict__ cache,
                   int t, int Tmax, int C, int hs) {
  constexpr float LOG2E = 1.4426950408889634f;
  __shared__ float sm_m[4], sm_l[4];
  __shared__ float sm_o[4][128];
  const int h = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* q = qkv + (size_t)b * 3 * C + h * hs;
  const float sl2 = rsqrtf((float)hs) * LOG2E;
  float qv[4], acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int d = lane + 32 * i;
    qv[i] = d < hs ? to_f32(q[d]) * sl2 : 0.f;
    acc[i] = 0.f;
  }
  const T* kv = cache + (size_t)b * Tmax * 2 * C;
  float m = -INFINITY, l = 0.f;
  for (int j = warp; j <= t; j += 4) {
    const T* kr = kv + (size_t)j * 2 * C + h * hs;
    const T* vr = kr + C;
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int d = lane + 32 * i;
      if (d < hs) part = fmaf(qv[i], to_f32(kr[d]), part);
    }
    const float s = warp_sum(part);
    const float mn = fmaxf(m, s);
    const float alpha = exp2f(m - mn), p = exp2f(s - mn);
    l = l * alpha + p;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int d = lane + 32 * i;
      if (d < hs) acc[i] = acc[i] * alpha + p * to_f32(vr[d]);
    }
    m = mn;
  }
  if (lane == 0) { sm_m[warp] = m; sm_l[warp] = l; }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (lane + 32 * i < hs) sm_o[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  if (warp == 0) {
    float mx = -INFINITY;
    for (int w = 0; w < 4; ++w) mx = fmaxf(mx, sm_m[w]);
    float f[4], L = 0.f;
    for (int w = 0; w < 4; ++w) {   // a warp with no keys has m = -inf and contributes 0
      f[w] = sm_m[w] == -INFINITY ? 0.f : exp2f(sm_m[w] - mx);
      L += sm_l[w] * f[w];
    }
    T* o = out + (size_t)b * C + h * hs;
    for (int d = lane; d < hs; d += 32) {
      float od = 0.f;
      for (int w = 0; w < 4; ++w) od += sm_o[w][d] * f[w];
      o[d] = from_f32<T>(od / L);
    }
  }
}

cudaError_t attention_decode(DType t, void* out, const void* qkv, const void* cache, int B,
                             int t_pos, int Tmax, int C, int H, cudaStream_t s) {
  if (B <= 0 || H <= 0 || C % H || C / H > 128 || t_pos < 0 || t_pos >= Tmax)
    return cudaErrorInvalidValue;
  dim3 grid(H, B);
  if (t == DType::BF16)
    attn_decode_kernel<bf16><<<grid, 128, 0, s>>>((bf16*)out, (const bf16*)qkv,
                                                  (const bf16*)cache, t_pos, Tmax, C, C / H);
  else
    attn_decode_kernel<float><<<grid, 128, 0, s>>>((float*)out, (const float*)qkv,
                                                   (const float*)cache, t_pos, Tmax, C, C / H);
  count_launches(1);
  return last();
}

__global__ void gather_last_kernel(int* out, const int* in, int B, int T) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) out[b] = in[(size_t)b * T + T - 1];
}

cudaError_t gather_last(int* out, const int* in, int B, int T, cudaStream_t s) {
  gather_last_kernel<<<ceil_div(B, 128), 128, 0, s>>>(out, in, B, T);
  count_launches(1);
  return last();
}

}  // namespace gpt2k

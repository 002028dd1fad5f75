// Causal multi-head self-attention, forward and backward.
//
// Math (「从零实现一个最小GPT：代码讲解 + 知识点全解」 三.3-三.4): for head h, q, k, v are
// columns [h*hs, (h+1)*hs) of the Q, K, V thirds of qkv [B, T, 3C];
// s_ij = q_i . k_j / sqrt(hs) for j <= i, p = softmax_j(s), o_i = sum_j p_ij v_j, heads
// concatenated in head order into out [B, T, C]. The T x T weights are never stored:
// the forward keeps lse_i = log sum_j exp(s_ij) per row and the backward recomputes p.
// Backward: D_i = dO_i . O_i; dp_ij = dO_i . v_j; ds_ij = p_ij (dp_ij - D_i);
// dq_i = sum_j ds_ij k_j / sqrt(hs); dk_j = sum_i ds_ij q_i / sqrt(hs); dv_j = sum_i p_ij dO_i.
// dQ and dK/dV come from separate kernels, so no float atomics are needed and the result
// is deterministic.
//
// Two implementations:
//  * fp32: one warp per (batch, head, row), plain FMA (parity path).
//  * bf16, head size 64: the tcgen05 flash-attention kernels of attention_tc.cu; this file
//    keeps the D = rowsum(dO * O) kernel they read.
#include "common.cuh"
#include "launch.h"

namespace gpt2k {

// =====================================================================================
// fp32 path
__global__ void attn_fwd_f32_kernel(float* __restrict__ out, float* __restrict__ lse,
                                    const float* __restrict__ qkv, int B, int T, int C, int H) {
  extern __shared__ float sc_f32[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + wid;
  if (gw >= (long long)B * H * T) return;
  const int i = (int)(gw % T);
  const int h = (int)((gw / T) % H);
  const int b = (int)(gw / ((long long)T * H));
  const int hs = C / H;
  const float scale = 1.0f / sqrtf((float)hs);
  float* s = sc_f32 + (size_t)wid * T;
  const float* base = qkv + (size_t)b * T * 3 * C;
  const float* q = base + (size_t)i * 3 * C + h * hs;
  float mx = -INFINITY;
  for (int j = lane; j <= i; j += 32) {
    const float* k = base + (size_t)j * 3 * C + C + h * hs;
    float d = 0.f;
    for (int e = 0; e < hs; ++e) d = fmaf(q[e], k[e], d);
    s[j] = d * scale;
    mx = fmaxf(mx, s[j]);
  }
  mx = warp_max(mx);
  float sum = 0.f;
  for (int j = lane; j <= i; j += 32) { float p = expf(s[j] - mx); s[j] = p; sum += p; }
  sum = warp_sum(sum);
  __syncwarp();
  for (int d = lane; d < hs; d += 32) {
    float o = 0.f;
    for (int j = 0; j <= i; ++j) o = fmaf(s[j], base[(size_t)j * 3 * C + 2 * C + h * hs + d], o);
    out[((size_t)b * T + i) * C + h * hs + d] = o / sum;
  }
  if (lane == 0) lse[((size_t)b * H + h) * T + i] = mx + logf(sum);
}

// D_i = dO_i . O_i per (b, h, i)
__global__ void attn_bwd_D_f32_kernel(float* __restrict__ Dbuf, const float* __restrict__ dout,
                                      const float* __restrict__ out, int B, int T, int C, int H) {
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= (long long)B * H * T) return;
  const int i = (int)(gw % T), h = (int)((gw / T) % H), b = (int)(gw / ((long long)T * H));
  const int hs = C / H;
  size_t o = ((size_t)b * T + i) * C + h * hs;
  float d = 0.f;
  for (int e = lane; e < hs; e += 32) d = fmaf(dout[o + e], out[o + e], d);
  d = warp_sum(d);
  if (lane == 0) Dbuf[((size_t)b * H + h) * T + i] = d;
}

__global__ void attn_bwd_dq_f32_kernel(float* __restrict__ dqkv, const float* __restrict__ Dbuf,
                                       const float* __restrict__ dout, const float* __restrict__ qkv,
                                       const float* __restrict__ lse, int B, int T, int C, int H) {
  extern __shared__ float sc_f32[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + wid;
  if (gw >= (long long)B * H * T) return;
  const int i = (int)(gw % T), h = (int)((gw / T) % H), b = (int)(gw / ((long long)T * H));
  const int hs = C / H;
  const float scale = 1.0f / sqrtf((float)hs);
  float* ds = sc_f32 + (size_t)wid * T;
  const float* base = qkv + (size_t)b * T * 3 * C;
  const float* q = base + (size_t)i * 3 * C + h * hs;
  const float* dO = dout + ((size_t)b * T + i) * C + h * hs;
  const size_t ri = ((size_t)b * H + h) * T + i;
  const float L = lse[ri], Di = Dbuf[ri];
  for (int j = lane; j <= i; j += 32) {
    const float* k = base + (size_t)j * 3 * C + C + h * hs;
    const float* v = base + (size_t)j * 3 * C + 2 * C + h * hs;
    float s = 0.f, dp = 0.f;
    for (int e = 0; e < hs; ++e) { s = fmaf(q[e], k[e], s); dp = fmaf(dO[e], v[e], dp); }
    float p = expf(s * scale - L);
    ds[j] = p * (dp - Di);
  }
  __syncwarp();
  for (int d = lane; d < hs; d += 32) {
    float a = 0.f;
    for (int j = 0; j <= i; ++j) a = fmaf(ds[j], base[(size_t)j * 3 * C + C + h * hs + d], a);
    dqkv[((size_t)b * T + i) * 3 * C + h * hs + d] = a * scale;
  }
}

__global__ void attn_bwd_dkv_f32_kernel(float* __restrict__ dqkv, const float* __restrict__ Dbuf,
                                        const float* __restrict__ dout,
                                        const float* __restrict__ qkv,
                                        const float* __restrict__ lse, int B, int T, int C, int H) {
  extern __shared__ float sc_f32[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + wid;
  if (gw >= (long long)B * H * T) return;
  const int j = (int)(gw % T), h = (int)((gw / T) % H), b = (int)(gw / ((long long)T * H));
  const int hs = C / H;
  const float scale = 1.0f / sqrtf((float)hs);
  float* P = sc_f32 + (size_t)wid * 2 * T;
  float* dS = P + T;
  const float* base = qkv + (size_t)b * T * 3 * C;
  const float* k = base + (size_t)j * 3 * C + C + h * hs;
  const float* v = base + (size_t)j * 3 * C + 2 * C + h * hs;
  for (int i = j + lane; i < T; i += 32) {
    const float* q = base + (size_t)i * 3 * C + h * hs;
    const float* dO = dout + ((size_t)b * T + i) * C + h * hs;
    const size_t ri = ((size_t)b * H + h) * T + i;
    float s = 0.f, dp = 0.f;
    for (int e = 0; e < hs; ++e) { s = fmaf(q[e], k[e], s); dp = fmaf(dO[e], v[e], dp); }
    float p = expf(s * scale - lse[ri]);
    P[i] = p;
    dS[i] = p * (dp - Dbuf[ri]);
  }
  __syncwarp();
  for (int d = lane; d < hs; d += 32) {
    float av = 0.f, ak = 0.f;
    for (int i = j; i < T; ++i) {
      av = fmaf(P[i], dout[((size_t)b * T + i) * C + h * hs + d], av);
      ak = fmaf(dS[i], base[(size_t)i * 3 * C + h * hs + d], ak);
    }
    size_t o = ((size_t)b * T + j) * 3 * C;
    dqkv[o + C + h * hs + d] = ak * scale;
    dqkv[o + 2 * C + h * hs + d] = av;
  }
}


// =====================================================================================
cudaError_t attention_forward(DType t, void* out, float* lse, const void* qkv, int B, int T, int C,
                              int H, int* err, cudaStream_t s) {
  if (t == DType::BF16) return attention_forward_tc(out, lse, qkv, B, T, C, H, err, s);
  long long warps = (long long)B * H * T;
  attn_fwd_f32_kernel<<<ceil_div(warps, 4), 128, 4 * T * sizeof(float), s>>>(
      (float*)out, lse, (const float*)qkv, B, T, C, H); count_launches(1);
  return cudaGetLastError();
}

cudaError_t attention_backward(DType t, void* dqkv, float* Dbuf, const void* dout,
                               const void* out, const void* qkv, const float* lse, int B, int T,
                               int C, int H, int* err, cudaStream_t s) {
  if (t == DType::BF16) {
    if (C / H != 64 || C % H || T % 4) return cudaErrorInvalidValue;
    return attention_backward_tc(dqkv, Dbuf, dout, out, qkv, lse, B, T, C, H, err, s);
  }
  long long warps = (long long)B * H * T;
  int blocks = ceil_div(warps, 4);
  attn_bwd_D_f32_kernel<<<blocks, 128, 0, s>>>(Dbuf, (const float*)dout, (const float*)out, B, T,
                                               C, H); count_launches(1);
  attn_bwd_dq_f32_kernel<<<blocks, 128, 4 * T * sizeof(float), s>>>(
      (float*)dqkv, Dbuf, (const float*)dout, (const float*)qkv, lse, B, T, C, H); count_launches(1);
  attn_bwd_dkv_f32_kernel<<<blocks, 128, 8 * T * sizeof(float), s>>>(
      (float*)dqkv, Dbuf, (const float*)dout, (const float*)qkv, lse, B, T, C, H); count_launches(1);
  return cudaGetLastError();
}

}  // namespace gpt2k

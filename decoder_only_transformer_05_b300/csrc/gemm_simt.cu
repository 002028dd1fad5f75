// fp32 SIMT GEMM with the training step's fused epilogues. This is the fp32 parity
// path: tf32 tensor cores would not meet the fp32 tolerance, so this path multiplies
// in plain fp32 FMA. 64x64 output tile per 256-thread block, 4x4 outputs per thread.
#include "common.cuh"
#include "launch.h"

namespace gpt2k {

constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16;

template <bool AMN, bool BMN>
__global__ void __launch_bounds__(256) gemm_f32_kernel(GemmArgs g) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Bs[SG_BK][SG_BN + 4];
  const float* A = (const float*)g.A;
  const float* Bm = (const float*)g.B;
  const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += SG_BK) {
    for (int i = threadIdx.x; i < SG_BM * SG_BK; i += 256) {
      int mm, kk;
      if (AMN) { mm = i % SG_BM; kk = i / SG_BM; } else { kk = i % SG_BK; mm = i / SG_BK; }
      int m = m0 + mm, k = k0 + kk;
      float v = 0.f;
      if (m < g.M && k < g.K) v = AMN ? A[(size_t)k * g.lda + m] : A[(size_t)m * g.lda + k];
      As[kk][mm] = v;
    }
    for (int i = threadIdx.x; i < SG_BN * SG_BK; i += 256) {
      int nn, kk;
      if (BMN) { nn = i % SG_BN; kk = i / SG_BN; } else { kk = i % SG_BK; nn = i / SG_BK; }
      int n = n0 + nn, k = k0 + kk;
      float v = 0.f;
      if (n < g.N && k < g.K) v = BMN ? Bm[(size_t)k * g.ldb + n] : Bm[(size_t)n * g.ldb + k];
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int m = m0 + ty * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int n = n0 + tx * 4 + j;
      if (n >= g.N) continue;
      float v = acc[i][j];
      size_t o = (size_t)m * g.ldo + n;
      switch (g.epi) {
        case EPI_STORE:
          if (g.bias) v += ((const float*)g.bias)[n];
          if (g.resid) v += ((const float*)g.resid)[o];
          ((float*)g.out)[o] = v;
          break;
        case EPI_GELU_FWD:
          if (g.bias) v += ((const float*)g.bias)[n];
          ((float*)g.pre)[o] = gelu_tanh_grad(v);
          ((float*)g.out)[o] = gelu_tanh(v);
          break;
        case EPI_GELU_BWD:
          ((float*)g.out)[o] = v * ((const float*)g.aux)[o];
          break;
        case EPI_GELU_FWD_U:
          if (g.bias) v += ((const float*)g.bias)[n];
          ((float*)g.pre)[o] = v;
          ((float*)g.out)[o] = gelu_tanh(v);
          break;
        case EPI_GELU_BWD_U: {
          const float u = ((const float*)g.aux)[o];
          ((float*)g.out)[o] = v * gelu_tanh_grad(u);
          ((float*)g.pre)[o] = gelu_tanh(u);
          break;
        }
        case EPI_ACCUM:
          g.accum[o] += g.scale * v;
          break;
      }
    }
  }
}

cudaError_t gemm_f32(const GemmArgs& g, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return cudaErrorInvalidValue;
  dim3 grid(ceil_div(g.N, SG_BN), ceil_div(g.M, SG_BM));
  if (!g.a_mn && !g.b_mn) { gemm_f32_kernel<false, false><<<grid, 256, 0, s>>>(g); count_launches(1); }
  else if (!g.a_mn && g.b_mn) { gemm_f32_kernel<false, true><<<grid, 256, 0, s>>>(g); count_launches(1); }
  else if (g.a_mn && !g.b_mn) { gemm_f32_kernel<true, false><<<grid, 256, 0, s>>>(g); count_launches(1); }
  else { gemm_f32_kernel<true, true><<<grid, 256, 0, s>>>(g); count_launches(1); }
  return cudaGetLastError();
}

}  // namespace gpt2k

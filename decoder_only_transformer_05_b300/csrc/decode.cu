// Forward-only inference with a KV cache (greedy decoding, one new token per sequence per
// step): the cache store, the one-query attention over the cached keys and values (split over
// key blocks, then combined), the weight-streaming linear layers of the step's few rows (with
// LayerNorm and the cache store fused in), the device-side position counter that lets a
// recorded step be replayed, and a gather of the prompt's last positions. The model and the
// causal scaled softmax attention
// are those of 「从零实现一个最小GPT：代码讲解 + 知识点全解」 (二.3 Head, 三.3); its 三.8
// generation loop re-runs the whole prefix for each new token, whereas here each layer's
// keys and values of earlier positions are kept and only the new position is computed.
#include "common.cuh"
#include "launch.h"

namespace gpt2k {

static cudaError_t last() {
  return cudaGetLastError();
}

// One thread per 16-byte vector of a cached row (2C elements). pos_dev (if not null) holds
// the first position on the device (a replayed decode step reads it there).
template <typename T>
__global__ void kv_store_kernel(T* __restrict__ cache, const T* __restrict__ qkv, int B, int Trows,
                                int pos0, const int* __restrict__ pos_dev, int n, int Tmax, int C) {
  constexpr int VE = 16 / sizeof(T);
  if (pos_dev) pos0 = *pos_dev;
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
                           int n, int Tmax, int C, cudaStream_t s, const int* pos_dev) {
  if (B <= 0 || n <= 0 || pos0 < 0 || pos0 + n > Tmax || n > Trows) return cudaErrorInvalidValue;
  if (t == DType::BF16) {
    const long long total = (long long)B * n * (2 * C / 8);
    kv_store_kernel<bf16><<<ceil_div(total, 256), 256, 0, s>>>((bf16*)cache, (const bf16*)qkv, B,
                                                               Trows, pos0, pos_dev, n, Tmax, C);
  } else {
    const long long total = (long long)B * n * (2 * C / 4);
    kv_store_kernel<float><<<ceil_div(total, 256), 256, 0, s>>>((float*)cache, (const float*)qkv,
                                                                B, Trows, pos0, pos_dev, n, Tmax, C);
  }
  count_launches(1);
  return last();
}

// One query per (batch b, head h) against the cached keys and values of positions 0..t,
// split over the keys: block (h, b, sidx) takes the 128 keys [128 sidx, 128 sidx + 128) ∩
// [0, t], one key per lane (warp w: keys 32 w .. 32 w + 31 of the split), so that a block
// issues all of its key-row and value-row loads at once. Each block writes its partial
// softmax (maximum m and sum l in the log2 domain) and weighted value sum to `part`; the
// combine kernel merges the splits in order. hs <= 128 (a multiple of 8).
constexpr int DEC_KEYS = 128;

template <typename T>
__global__ void __launch_bounds__(128)
attn_decode_split_kernel(float* __restrict__ part, const T* __restrict__ qkv,
                         const T* __restrict__ cache, int t, const int* __restrict__ t_dev,
                         int Tmax, int C, int hs, int S) {
  constexpr float LOG2E = 1.4426950408889634f;
  constexpr int VE = 16 / sizeof(T);
  __shared__ float sq[128];
  __shared__ float sm_m[4], sm_l[4];
  __shared__ float sm_o[4][128];
  if (t_dev) t = *t_dev;
  const int h = blockIdx.x, b = blockIdx.y, sidx = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float sl2 = rsqrtf((float)hs) * LOG2E;
  const T* q = qkv + (size_t)b * 3 * C + h * hs;
  for (int d = threadIdx.x; d < hs; d += 128) sq[d] = to_f32(q[d]) * sl2;
  __syncthreads();
  const int j = sidx * DEC_KEYS + warp * 32 + lane;   // this lane's key
  const bool live = j <= t;
  const T* kv = cache + (size_t)b * Tmax * 2 * C + h * hs;
  // score of the lane's key, 16 bytes of its row at a time
  float sc = -INFINITY;
  if (live) {
    const T* kr = kv + (size_t)j * 2 * C;
    float acc = 0.f;
    for (int d0 = 0; d0 < hs; d0 += VE) {
      const Vec16<T> kk = ld16(kr + d0);
#pragma unroll
      for (int e = 0; e < VE; ++e) acc = fmaf(sq[d0 + e], to_f32(kk.e[e]), acc);
    }
    sc = acc;
  }
  float m = sc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float p = live ? exp2f(sc - m) : 0.f;   // m = -inf only when no key of the warp is live
  float l = p;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  // weighted value sum: lane holds dimensions lane, lane + 32, ...; keys in lane order
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int nk = min(32, t + 1 - (sidx * DEC_KEYS + warp * 32));
  for (int k = 0; k < nk; ++k) {
    const float pk = __shfl_sync(0xffffffffu, p, k);
    const T* vr = kv + (size_t)(sidx * DEC_KEYS + warp * 32 + k) * 2 * C + C;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int d = lane + 32 * i;
      if (d < hs) acc[i] = fmaf(pk, to_f32(vr[d]), acc[i]);
    }
  }
  if (lane == 0) { sm_m[warp] = nk > 0 ? m : -INFINITY; sm_l[warp] = nk > 0 ? l : 0.f; }
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
    float* pp = part + (((size_t)b * gridDim.x + h) * S + sidx) * (hs + 2);
    if (lane == 0) { pp[0] = mx; pp[1] = L; }
    for (int d = lane; d < hs; d += 32) {
      float od = 0.f;
      for (int w = 0; w < 4; ++w) od += sm_o[w][d] * f[w];
      pp[2 + d] = od;
    }
  }
}

// Block (h, b), one warp: merges the splits 0 .. ceil((t + 1) / 128) - 1 in order.
template <typename T>
__global__ void attn_decode_combine_kernel(T* __restrict__ out, const float* __restrict__ part,
                                           int t, const int* __restrict__ t_dev, int C, int hs,
                                           int S) {
  if (t_dev) t = *t_dev;
  const int h = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
  const int ns = (t + DEC_KEYS) / DEC_KEYS;
  const float* pp = part + ((size_t)b * gridDim.x + h) * S * (hs + 2);
  float mx = -INFINITY;
  for (int s2 = 0; s2 < ns; ++s2) mx = fmaxf(mx, pp[s2 * (hs + 2)]);
  float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s2 = 0; s2 < ns; ++s2) {
    const float* q = pp + s2 * (hs + 2);
    const float f = q[0] == -INFINITY ? 0.f : exp2f(q[0] - mx);
    L += q[1] * f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (lane + 32 * i < hs) acc[i] = fmaf(q[2 + lane + 32 * i], f, acc[i]);
  }
  T* o = out + (size_t)b * C + h * hs;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (lane + 32 * i < hs) o[lane + 32 * i] = from_f32<T>(acc[i] / L);
}

size_t attention_decode_scratch_floats(int B, int H, int Tmax, int hs) {
  return (size_t)B * H * ((Tmax + DEC_KEYS - 1) / DEC_KEYS) * (hs + 2);
}

cudaError_t attention_decode(DType t, void* out, const void* qkv, const void* cache, int B,
                             int t_pos, int Tmax, int C, int H, cudaStream_t s, const int* t_dev,
                             float* scratch) {
  if (B <= 0 || H <= 0 || C % H || C / H > 128 || (C / H) % 8 || t_pos < 0 || t_pos >= Tmax ||
      !scratch)
    return cudaErrorInvalidValue;
  const int hs = C / H, S = (Tmax + DEC_KEYS - 1) / DEC_KEYS;
  // with the position on the device (a replayed step), every split up to Tmax runs; the
  // splits past t write an empty partial (m = -inf) that the combine does not read
  const dim3 grid(H, B, t_dev ? S : (t_pos + DEC_KEYS) / DEC_KEYS);
  if (t == DType::BF16) {
    attn_decode_split_kernel<bf16><<<grid, 128, 0, s>>>(scratch, (const bf16*)qkv,
                                                        (const bf16*)cache, t_pos, t_dev, Tmax, C, hs, S);
    attn_decode_combine_kernel<bf16><<<dim3(H, B), 32, 0, s>>>((bf16*)out, scratch, t_pos, t_dev, C, hs, S);
  } else {
    attn_decode_split_kernel<float><<<grid, 128, 0, s>>>(scratch, (const float*)qkv,
                                                         (const float*)cache, t_pos, t_dev, Tmax, C, hs, S);
    attn_decode_combine_kernel<float><<<dim3(H, B), 32, 0, s>>>((float*)out, scratch, t_pos, t_dev, C, hs, S);
  }
  count_launches(2);
  return last();
}

// y[m, n] = sum_k x[m, k] W[n, k] (+ bias[n]) (+ resid[m, n]) for the MM >= M rows of a decode
// step (bf16, K-major W as in Y = X W^T): the step reads every weight once, so this is a
// weight-streaming kernel rather than a tensor-core tile. x sits in shared memory; warp w
// of block i takes the output columns 2 (8 i + w) and 2 (8 i + w) + 1, lane l the 16-byte
// vectors l, l + 32, ... of their two weight rows, and the M dot products per column are
// finished with warp reductions. Epilogues: store, tanh-GELU (gelu(u) to out and gelu'(u),
// or u itself, to pre).
//
// Fused forms for the decode step (GemvFuse): with ln_x set, x is LayerNorm(ln_x; ln_w, ln_b)
// computed here, one warp per row with the lane-to-vector mapping and the operation order of
// ln_fwd_kernel (so the values equal that kernel's bf16 output); with kv_cache set, the
// output columns [C, 3C) of the qkv projection (the new position's keys and values) also go
// to the cache row of position *kv_pos.
template <int MM>
__global__ void __launch_bounds__(256)
gemv_rows_kernel(bf16* __restrict__ out, bf16* __restrict__ pre, const bf16* __restrict__ x,
                 const bf16* __restrict__ W, const bf16* __restrict__ bias,
                 const bf16* __restrict__ resid, int M, int N, int K, long long ldo, int epi,
                 GemvFuse f) {
  extern __shared__ __align__(16) uint8_t gv_smem[];
  uint4* sx = reinterpret_cast<uint4*>(gv_smem);   // [M][K / 8]
  const int kv = K / 8;
  if (f.ln_x) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    for (int m = w; m < M; m += 8) {
      const uint4* xr = reinterpret_cast<const uint4*>((const bf16*)f.ln_x + (size_t)m * K);
      float2 v[12][4];   // up to 12 vectors of 8 per lane (K <= 3072)
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 12; ++j) {
        const int c = j * 32 + l;
        if (c < kv) {
          const uint4 a = xr[c];
          v[j][0] = bf2_to_f2(a.x); v[j][1] = bf2_to_f2(a.y);
          v[j][2] = bf2_to_f2(a.z); v[j][3] = bf2_to_f2(a.w);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) v[j][q] = make_float2(0.f, 0.f);
        }
        if ((j + 1) * 32 <= kv + 31) {
#pragma unroll
          for (int q = 0; q < 4; ++q) s2 = __fadd2_rn(s2, v[j][q]);
        }
      }
      const float mu = warp_sum(s2.x + s2.y) / K;
      const float2 nmu = make_float2(-mu, -mu);
      float2 q2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 12; ++j) {
        if (j * 32 + l < kv) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 d = __fadd2_rn(v[j][q], nmu);
            q2 = __ffma2_rn(d, d, q2);
          }
        }
      }
      const float rs = rsqrtf(warp_sum(q2.x + q2.y) / K + 1e-5f);
      const float2 rs2 = make_float2(rs, rs);
#pragma unroll
      for (int j = 0; j < 12; ++j) {
        const int c = j * 32 + l;
        if (c < kv) {
          const uint4 wq = reinterpret_cast<const uint4*>(f.ln_w)[c];
          const uint4 bq = reinterpret_cast<const uint4*>(f.ln_b)[c];
          const uint32_t ww[4] = {wq.x, wq.y, wq.z, wq.w}, bw[4] = {bq.x, bq.y, bq.z, bq.w};
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 sw = __fmul2_rn(rs2, bf2_to_f2(ww[q]));
            const float2 sh = __ffma2_rn(nmu, sw, bf2_to_f2(bw[q]));
            const float2 r = __ffma2_rn(v[j][q], sw, sh);
            o[q] = pack2_bf16_rn(r.x, r.y);
          }
          sx[m * kv + c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  } else {
    for (int i = threadIdx.x; i < M * kv; i += blockDim.x)
      sx[i] = reinterpret_cast<const uint4*>(x + (size_t)(i / kv) * K)[i % kv];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = 2 * (blockIdx.x * 8 + warp);
  if (n0 >= N) return;
  const uint4* w0 = reinterpret_cast<const uint4*>(W + (size_t)n0 * K);
  const uint4* w1 = reinterpret_cast<const uint4*>(W + (size_t)(n0 + 1) * K);
  float a0[MM], a1[MM];
#pragma unroll
  for (int m = 0; m < MM; ++m) { a0[m] = 0.f; a1[m] = 0.f; }
  for (int v = lane; v < kv; v += 32) {
    const uint4 p = w0[v], q = w1[v];
    const float2 p2[4] = {bf2_to_f2(p.x), bf2_to_f2(p.y), bf2_to_f2(p.z), bf2_to_f2(p.w)};
    const float2 q2[4] = {bf2_to_f2(q.x), bf2_to_f2(q.y), bf2_to_f2(q.z), bf2_to_f2(q.w)};
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      if (m < M) {
        const uint4 xv = sx[m * kv + v];
        const float2 x2[4] = {bf2_to_f2(xv.x), bf2_to_f2(xv.y), bf2_to_f2(xv.z), bf2_to_f2(xv.w)};
        float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s0 = __ffma2_rn(x2[e], p2[e], s0);
          s1 = __ffma2_rn(x2[e], q2[e], s1);
        }
        a0[m] += s0.x + s0.y;
        a1[m] += s1.x + s1.y;
      }
    }
  }
  float r0 = 0.f, r1 = 0.f;   // lane m keeps row m's two sums
#pragma unroll
  for (int m = 0; m < MM; ++m) {
    if (m < M) {
      const float t0 = warp_sum(a0[m]), t1 = warp_sum(a1[m]);
      if (lane == m) { r0 = t0; r1 = t1; }
    }
  }
  if (lane >= M) return;
  const int m = lane;
  float2 u = make_float2(r0, r1);
  if (bias) u = __fadd2_rn(u, bf2_to_f2(*reinterpret_cast<const uint32_t*>(bias + n0)));
  if (resid)
    u = __fadd2_rn(u, bf2_to_f2(*reinterpret_cast<const uint32_t*>(resid + (size_t)m * ldo + n0)));
  uint32_t* o = reinterpret_cast<uint32_t*>(out + (size_t)m * ldo + n0);
  if (epi == EPI_STORE) {
    const uint32_t pk = pack2_bf16_rn(u.x, u.y);
    *o = pk;
    if (f.kv_cache && n0 >= f.kv_C)   // row m = batch element m, at position *kv_pos
      *reinterpret_cast<uint32_t*>((bf16*)f.kv_cache +
                                   ((size_t)m * f.kv_Tmax + *f.kv_pos) * 2 * f.kv_C + (n0 - f.kv_C)) = pk;
  } else {
    float2 d;
    const float2 g = gelu_tanh_and_grad_fast2(u, d);
    *o = pack2_bf16_rn(g.x, g.y);
    *reinterpret_cast<uint32_t*>(pre + (size_t)m * ldo + n0) =
        epi == EPI_GELU_FWD ? pack2_bf16_rn(d.x, d.y) : pack2_bf16_rn(u.x, u.y);
  }
}

template <int MM>
static cudaError_t gemv_launch(const GemmArgs& g, const GemvFuse& f, cudaStream_t s) {
  const size_t smem = (size_t)g.M * g.K * 2;
  static size_t attr = 48 * 1024;
  if (smem > attr) {
    cudaError_t e = cudaFuncSetAttribute(gemv_rows_kernel<MM>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = smem;
  }
  gemv_rows_kernel<MM><<<ceil_div(g.N, 16), 256, smem, s>>>(
      (bf16*)g.out, (bf16*)g.pre, (const bf16*)g.A, (const bf16*)g.B, (const bf16*)g.bias,
      (const bf16*)g.resid, g.M, g.N, g.K, g.ldo, g.epi, f);
  count_launches(1);
  return last();
}

bool gemv_rows_supported(const GemmArgs& g) {
  return g.M >= 1 && g.M <= 16 && !g.a_mn && !g.b_mn && g.lda == g.K && g.ldb == g.K &&
         g.K % 8 == 0 && g.N % 2 == 0 && g.ldo % 2 == 0 && (size_t)g.M * g.K * 2 <= 200 * 1024 &&
         (g.epi == EPI_STORE || g.epi == EPI_GELU_FWD || g.epi == EPI_GELU_FWD_U) &&
         (g.epi == EPI_STORE || g.pre) && ((uintptr_t)g.A & 15u) == 0 && ((uintptr_t)g.B & 15u) == 0;
}

cudaError_t gemv_rows(const GemmArgs& g, cudaStream_t s, const GemvFuse& f) {
  if (!gemv_rows_supported(g)) return cudaErrorInvalidValue;
  if (f.ln_x && (!f.ln_w || !f.ln_b || g.K > 12 * 256 || ((uintptr_t)f.ln_x & 15u) ||
                 ((uintptr_t)f.ln_w & 15u) || ((uintptr_t)f.ln_b & 15u)))
    return cudaErrorInvalidValue;
  if (f.kv_cache && (!f.kv_pos || g.epi != EPI_STORE || g.N != 3 * f.kv_C || f.kv_C % 2))
    return cudaErrorInvalidValue;
  if (g.M <= 1) return gemv_launch<1>(g, f, s);
  if (g.M <= 2) return gemv_launch<2>(g, f, s);
  if (g.M <= 4) return gemv_launch<4>(g, f, s);
  if (g.M <= 8) return gemv_launch<8>(g, f, s);
  return gemv_launch<16>(g, f, s);
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

// *pos = set (set >= 0), else *pos += add: the device copy of the decode position
__global__ void pos_add_kernel(int* pos, int set, int add) {
  if (threadIdx.x == 0 && blockIdx.x == 0) *pos = set >= 0 ? set : *pos + add;
}

cudaError_t decode_position(int* pos_dev, int set, int add, cudaStream_t s) {
  pos_add_kernel<<<1, 32, 0, s>>>(pos_dev, set, add);
  count_launches(1);
  return last();
}

}  // namespace gpt2k

// LayerNorm forward/backward and the deterministic column sums of the training step.
//
// LayerNorm over the rows of [M, C]: y = (x - mean) * rstd * w + b with the biased variance
// and eps 1e-5 (nn.LayerNorm's defaults, the layer of 「从零实现一个最小GPT：代码讲解 +
// 知识点全解」 二.6 Block). Backward (「手写训练脚本：不用框架，从零实现GPT训练流程」 二, the
// hand-derived LayerNorm backward):
//   xhat = (x - mean) rstd,  g = dy w
//   dx = rstd (g - mean_c(g) - xhat mean_c(g xhat));  dres = (accumulate ? dres : 0) + dx
//   dw += sum_rows dy xhat,  db += sum_rows dy
// and, optionally, dproj += sum_rows dres_out: the column sums of the residual-stream
// gradient this kernel writes, which are exactly the bias gradient of the projection
// (attention or MLP output) that fed that residual stream.
//
// Every sum runs in a fixed order: rows are dealt to blocks and warps by a fixed rule,
// each block's warps are combined in warp order, and the per-block partials are added in
// block order by column_reduce, so repeated runs give bit-identical results.
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace gpt2k {

// ------------------------------------------------------------------ async copies
__device__ __forceinline__ uint32_t lsmem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_dyn(int n) {
  // wait until at most n groups of this thread are still in flight (n in 0..2)
  if (n <= 0) asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  else if (n == 1) asm volatile("cp.async.wait_group 1;\n" ::: "memory");
  else asm volatile("cp.async.wait_group 2;\n" ::: "memory");
}

static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// =====================================================================================
// forward: one warp per row, the row in registers (MAXV 16-byte vectors per lane)
template <typename T, int MAXV>
__global__ void ln_fwd_kernel(T* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd,
                              const T* __restrict__ x, const T* __restrict__ w,
                              const T* __restrict__ b, int M, int C) {
  constexpr int VE = 16 / sizeof(T);
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M) return;
  if constexpr (std::is_same<T, bf16>::value) {
    // bf16: pairs of columns as float2 on the packed two-lane fp32 instructions
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * C);
    float2 v[MAXV][4];
    float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int c = j * 32 + lane;
      if (c * 8 < C) {
        const uint4 a = xr[c];
        v[j][0] = bf2_to_f2(a.x); v[j][1] = bf2_to_f2(a.y);
        v[j][2] = bf2_to_f2(a.z); v[j][3] = bf2_to_f2(a.w);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) v[j][q] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) s2 = __fadd2_rn(s2, v[j][q]);
    }
    const float mu = warp_sum(s2.x + s2.y) / C;
    const float2 nmu = make_float2(-mu, -mu);
    float2 q2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      if ((j * 32 + lane) * 8 < C) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 d = __fadd2_rn(v[j][q], nmu);
          q2 = __ffma2_rn(d, d, q2);
        }
      }
    }
    const float rs = rsqrtf(warp_sum(q2.x + q2.y) / C + 1e-5f);
    // y = (v - mu) rs w + b = v (rs w) + (b - mu rs w)
    uint4* yr = reinterpret_cast<uint4*>(y + (size_t)row * C);
    const float2 rs2 = make_float2(rs, rs);
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int c = j * 32 + lane;
      if (c * 8 < C) {
        const uint4 wq = reinterpret_cast<const uint4*>(w)[c];
        const uint4 bq = reinterpret_cast<const uint4*>(b)[c];
        const uint32_t ww[4] = {wq.x, wq.y, wq.z, wq.w}, bw[4] = {bq.x, bq.y, bq.z, bq.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 sw = __fmul2_rn(rs2, bf2_to_f2(ww[q]));
          const float2 sh = __ffma2_rn(nmu, sw, bf2_to_f2(bw[q]));
          const float2 r = __ffma2_rn(v[j][q], sw, sh);
          o[q] = pack2_bf16_rn(r.x, r.y);
        }
        yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    if (lane == 0) { mean[row] = mu; rstd[row] = rs; }
    return;
  }
  const T* xr = x + (size_t)row * C;
  float v[MAXV][VE];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    int c = (j * 32 + lane) * VE;
    if (c < C) {
      Vec16<T> a = ld16(xr + c);
#pragma unroll
      for (int e = 0; e < VE; ++e) { v[j][e] = to_f32(a.e[e]); s += v[j][e]; }
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e) v[j][e] = 0.f;
    }
  }
  const float mu = warp_sum(s) / C;
  float q = 0.f;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    int c = (j * 32 + lane) * VE;
    if (c < C) {
#pragma unroll
      for (int e = 0; e < VE; ++e) { float d = v[j][e] - mu; q += d * d; }
    }
  }
  const float rs = rsqrtf(warp_sum(q) / C + 1e-5f);
  T* yr = y + (size_t)row * C;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    int c = (j * 32 + lane) * VE;
    if (c < C) {
      Vec16<T> wv = ld16(w + c), bv = ld16(b + c), o;
#pragma unroll
      for (int e = 0; e < VE; ++e)
        o.e[e] = from_f32<T>((v[j][e] - mu) * rs * to_f32(wv.e[e]) + to_f32(bv.e[e]));
      st16(yr + c, o);
    }
  }
  if (lane == 0) { mean[row] = mu; rstd[row] = rs; }
}

template <typename T>
static cudaError_t ln_fwd_dispatch(T* y, float* mean, float* rstd, const T* x, const T* w,
                                   const T* b, int M, int C, cudaStream_t s) {
  constexpr int VE = 16 / sizeof(T);
  int vpl = ceil_div(C, 32 * VE);
  dim3 grid(ceil_div(M, 8)), block(256);
  switch (vpl) {
#define LNF_CASE(N) \
  ln_fwd_kernel<T, N><<<grid, block, 0, s>>>(y, mean, rstd, x, w, b, M, C); count_launches(1); break;
    case 1: LNF_CASE(1)
    case 2: LNF_CASE(2)
    case 3: LNF_CASE(3)
    case 4: LNF_CASE(4)
    case 5: case 6: LNF_CASE(6)
    case 7: case 8: LNF_CASE(8)
#undef LNF_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t layernorm_forward(DType t, void* y, float* mean, float* rstd, const void* x,
                              const void* w, const void* b, int M, int C, cudaStream_t s) {
  if (t == DType::BF16) {
    if (C % 8) return cudaErrorInvalidValue;
    return ln_fwd_dispatch<bf16>((bf16*)y, mean, rstd, (const bf16*)x, (const bf16*)w,
                                 (const bf16*)b, M, C, s);
  }
  if (C % 4) return cudaErrorInvalidValue;
  return ln_fwd_dispatch<float>((float*)y, mean, rstd, (const float*)x, (const float*)w,
                                (const float*)b, M, C, s);
}

// =====================================================================================
// backward. Rows come in chunks of LNB_ROWS consecutive rows (one per warp). Block b
// takes chunks b, b + G, b + 2G, ... (G = grid size); the chunk's dy, x (and dres when
// accumulating) rows are copied into shared memory with cp.async, stages - 1 chunks
// ahead of the one being computed (stages = 3 where three fit in LNB_SMEM_BUDGET). Each warp keeps its columns' running sums in
// registers; at the end the block adds its warps in warp order and writes one row of
// partials: [dw (C) | db (C) | dproj (C, when requested)].
constexpr int LNB_THREADS = 256;
constexpr int LNB_ROWS = LNB_THREADS / 32;
constexpr int LNB_MAX_BLOCKS = 2 * 148;
constexpr int LNB_SMEM_BUDGET = 110 * 1024;   // two blocks per SM

int layernorm_backward_blocks(int M) {
  return std::max(1, std::min(ceil_div(M, LNB_ROWS), LNB_MAX_BLOCKS));
}
size_t layernorm_backward_partials_floats(int M, int C, bool dproj) {
  return (size_t)layernorm_backward_blocks(M) * (dproj ? 3 : 2) * (size_t)C;
}
size_t layernorm_deferred_partials_floats(int C, bool dproj) {
  return (size_t)LNB_MAX_BLOCKS * (dproj ? 3 : 2) * (size_t)C;
}

// Two blocks per SM while the per-lane column sums fit in 128 registers (C <= 768 bf16).
template <typename T, int MAXV, bool DPROJ>
__global__ void __launch_bounds__(LNB_THREADS, (MAXV * (int)sizeof(T) <= 6 ? 2 : 1))
ln_bwd_kernel(T* __restrict__ dres, int accumulate, float* __restrict__ partials,
              const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ w,
              const float* __restrict__ mean, const float* __restrict__ rstd, int M, int C,
              int stages, int defer, float pscale) {
  constexpr int VE = 16 / sizeof(T);
  extern __shared__ __align__(16) uint8_t lnb_smem[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int row_bytes = C * (int)sizeof(T);
  const int ntens = accumulate ? 3 : 2;
  const int tens_bytes = LNB_ROWS * row_bytes;
  const int stage_bytes = ntens * tens_bytes;
  const int nchunks = ceil_div(M, LNB_ROWS);
  const uint32_t sbase = lsmem_u32(lnb_smem);

  auto issue = [&](int ci, int st) {
    if (ci < nchunks) {
      const int r0 = ci * LNB_ROWS;
      const int nvec = min(LNB_ROWS, M - r0) * row_bytes / 16;
      const uint32_t dst0 = sbase + st * stage_bytes;
      const char* src[3] = {(const char*)dy, (const char*)x, (const char*)dres};
      for (int t = 0; t < ntens; ++t) {
        const char* s0 = src[t] + (size_t)r0 * row_bytes;
        const uint32_t d0 = dst0 + t * tens_bytes;
        for (int i = threadIdx.x; i < nvec; i += LNB_THREADS) cp_async16(d0 + i * 16, s0 + (size_t)i * 16);
      }
    }
    cp_commit();   // possibly empty: keeps the group count uniform
  };

  // weights, packed, and the running column sums (bf16: as fp32 pairs, so that the
  // arithmetic runs on the packed two-lane fp32 instructions)
  constexpr bool BF = std::is_same<T, bf16>::value;
  Vec16<T> wv[MAXV];
  float dw[MAXV][VE], db[MAXV][VE], dp[MAXV][VE];
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int c = (j * 32 + lane) * VE;
    if (c < C) wv[j] = ld16(w + c);
#pragma unroll
    for (int e = 0; e < VE; ++e) { dw[j][e] = 0.f; db[j][e] = 0.f; dp[j][e] = 0.f; }
  }

  for (int p = 0; p < stages - 1; ++p) issue(blockIdx.x + p * gridDim.x, p);
  int it = 0;
  for (int ci = blockIdx.x; ci < nchunks; ci += gridDim.x, ++it) {
    const int row = ci * LNB_ROWS + wid;
    float mu = 0.f, rs = 0.f;
    if (row < M) { mu = __ldg(mean + row); rs = __ldg(rstd + row); }
    issue(ci + (stages - 1) * gridDim.x, (it + stages - 1) % stages);
    cp_wait_dyn(stages - 1);
    __syncthreads();
    if (BF && row < M) {
      // bf16: a 16-byte vector is 4 words of two bf16 (the lower column in the low half); a
      // bf16 widens to fp32 by a shift or a mask, and pairs of columns run as float2
      const uint8_t* st = lnb_smem + (it % stages) * stage_bytes + wid * row_bytes;
      const uint4* sdy = reinterpret_cast<const uint4*>(st);
      const uint4* sx = reinterpret_cast<const uint4*>(st + tens_bytes);
      const uint4* sres = reinterpret_cast<const uint4*>(st + 2 * tens_bytes);
      const float2 rs2 = make_float2(rs, rs), nmr2 = make_float2(-mu * rs, -mu * rs);
      float2 sg2 = make_float2(0.f, 0.f), sgx2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int v = j * 32 + lane;
        if (v * 8 < C) {
          const uint4 a = sdy[v], b = sx[v];
          const uint4 wq = *reinterpret_cast<const uint4*>(&wv[j]);
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
          const uint32_t ww[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 d = bf2_to_f2(aw[q]);
            const float2 xh = __ffma2_rn(bf2_to_f2(bw[q]), rs2, nmr2);
            const float2 g = __fmul2_rn(d, bf2_to_f2(ww[q]));
            sg2 = __fadd2_rn(sg2, g);
            sgx2 = __ffma2_rn(g, xh, sgx2);
            float2 dwv = make_float2(dw[j][2 * q], dw[j][2 * q + 1]);
            float2 dbv = make_float2(db[j][2 * q], db[j][2 * q + 1]);
            dwv = __ffma2_rn(d, xh, dwv);
            dbv = __fadd2_rn(dbv, d);
            dw[j][2 * q] = dwv.x; dw[j][2 * q + 1] = dwv.y;
            db[j][2 * q] = dbv.x; db[j][2 * q + 1] = dbv.y;
          }
        }
      }
      const float sg = warp_sum(sg2.x + sg2.y), sgx = warp_sum(sgx2.x + sgx2.y);
      // dx = rs (g - mg - xh mgx) = g rs + xh (-rs mgx) + (-rs mg)
      const float mg = sg / C, mgx = sgx / C;
      const float2 kx = make_float2(-rs * mgx, -rs * mgx), k0 = make_float2(-rs * mg, -rs * mg);
      uint4* out = reinterpret_cast<uint4*>(dres + (size_t)row * C);
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int v = j * 32 + lane;
        if (v * 8 < C) {
          const uint4 a = sdy[v], b = sx[v];
          uint4 r = make_uint4(0u, 0u, 0u, 0u);
          if (accumulate) r = sres[v];
          const uint4 wq = *reinterpret_cast<const uint4*>(&wv[j]);
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
          const uint32_t ww[4] = {wq.x, wq.y, wq.z, wq.w}, rw[4] = {r.x, r.y, r.z, r.w};
          uint32_t ow[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 xh = __ffma2_rn(bf2_to_f2(bw[q]), rs2, nmr2);
            const float2 g = __fmul2_rn(bf2_to_f2(aw[q]), bf2_to_f2(ww[q]));
            const float2 dx = __ffma2_rn(xh, kx, __ffma2_rn(g, rs2, k0));
            const float2 o = __fadd2_rn(bf2_to_f2(rw[q]), dx);
            ow[q] = pack2_bf16_rn(o.x, o.y);
            if (DPROJ) {
              const float2 ob = bf2_to_f2(ow[q]);
              dp[j][2 * q] += ob.x;
              dp[j][2 * q + 1] += ob.y;
            }
          }
          out[v] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
      }
    } else if (!BF && row < M) {
      const uint8_t* st = lnb_smem + (it % stages) * stage_bytes + wid * row_bytes;
      const T* sdy = (const T*)st;
      const T* sx = (const T*)(st + tens_bytes);
      const T* sres = (const T*)(st + 2 * tens_bytes);
      float sg = 0.f, sgx = 0.f;
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int c = (j * 32 + lane) * VE;
        if (c < C) {
          Vec16<T> a = ld16(sdy + c), b = ld16(sx + c);
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            const float d = to_f32(a.e[e]);
            const float xh = (to_f32(b.e[e]) - mu) * rs;
            const float g = d * to_f32(wv[j].e[e]);
            sg += g;
            sgx += g * xh;
            dw[j][e] += d * xh;
            db[j][e] += d;
          }
        }
      }
      sg = warp_sum(sg);
      sgx = warp_sum(sgx);
      const float mg = sg / C, mgx = sgx / C;
      T* out = dres + (size_t)row * C;
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int c = (j * 32 + lane) * VE;
        if (c < C) {
          Vec16<T> a = ld16(sdy + c), b = ld16(sx + c), r, o;
          if (accumulate) r = ld16(sres + c);
#pragma unroll
          for (int e = 0; e < VE; ++e) {
            const float xh = (to_f32(b.e[e]) - mu) * rs;
            const float g = to_f32(a.e[e]) * to_f32(wv[j].e[e]);
            const float dx = rs * (g - mg - xh * mgx);
            o.e[e] = from_f32<T>((accumulate ? to_f32(r.e[e]) : 0.f) + dx);
            if (DPROJ) dp[j][e] += to_f32(o.e[e]);
          }
          st16(out + c, o);
        }
      }
    }
    __syncthreads();   // the stage is free for the copy issued next iteration
  }
  cp_wait_dyn(0);
  __syncthreads();

  // warps' sums -> shared [warp][k*C + c], then the block's partial row in warp order
  float* red = reinterpret_cast<float*>(lnb_smem);
  const int nk = DPROJ ? 3 : 2;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int c = (j * 32 + lane) * VE;
    if (c < C) {
      float* r0 = red + (size_t)wid * nk * C + c;
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        r0[e] = dw[j][e];
        r0[C + e] = db[j][e];
        if (DPROJ) r0[2 * C + e] = dp[j][e];
      }
    }
  }
  __syncthreads();
  float* outp = partials + (size_t)blockIdx.x * nk * C;
  for (int c = threadIdx.x; c < nk * C; c += LNB_THREADS) {
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < LNB_ROWS; ++k) s += red[(size_t)k * nk * C + c];
    outp[c] = defer ? outp[c] + pscale * s : s;   // deferred: this block's running sum
  }
}

// out_k[c] += scale * sum_{b < nparts} partials[b * stride + k * N + c]  for the k with
// out_k non-null (and, with clear, the partials are zeroed after being read). Block: 32
// columns x 8 row groups; group g adds parts g, g + 8, ... in order, then the 8 groups
// are added in order.
__global__ void __launch_bounds__(256)
column_reduce_kernel(float* __restrict__ out0, float* __restrict__ out1, float* __restrict__ out2,
                     float* __restrict__ partials, int nparts, int N, int nk, int stride,
                     float scale, int clear, float* __restrict__ nparts_out) {
  __shared__ float sh[8][33];
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
  const int col = blockIdx.x * 32 + lane;   // over nk * N
  float s = 0.f;
  if (col < nk * N) {
    float* p = partials + col;
    int b = g;
    for (; b + 24 < nparts; b += 32) {
      float a0 = p[(size_t)b * stride], a1 = p[(size_t)(b + 8) * stride];
      float a2 = p[(size_t)(b + 16) * stride], a3 = p[(size_t)(b + 24) * stride];
      s += a0; s += a1; s += a2; s += a3;
    }
    for (; b < nparts; b += 8) s += p[(size_t)b * stride];
    if (clear)
      for (b = g; b < nparts; b += 8) p[(size_t)b * stride] = 0.f;
  }
  sh[g][lane] = s;
  __syncthreads();
  float q = 0.f;   // the final values' squares (for the gradient norm)
  if (g == 0 && col < nk * N) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) t += sh[k][lane];
    const int k = col / N, c = col - k * N;
    float* out = k == 0 ? out0 : (k == 1 ? out1 : out2);
    if (out) {
      const float f = out[c] + scale * t;
      out[c] = f;
      q = f * f;
    }
  }
  if (nparts_out && g == 0) {
    q = warp_sum(q);
    if (lane == 0) nparts_out[blockIdx.x] = q;
  }
}

static cudaError_t column_reduce(float* o0, float* o1, float* o2, float* partials,
                                 int nparts, int N, int nk, int stride, float scale,
                                 cudaStream_t s, int clear = 0, float* nparts_out = nullptr) {
  column_reduce_kernel<<<ceil_div((long long)nk * N, 32), 256, 0, s>>>(
      o0, o1, o2, partials, nparts, N, nk, stride, scale, clear, nparts_out);
  count_launches(1);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t ln_bwd_dispatch(T* dres, int acc, float* dw, float* db, float* dproj,
                                   const T* dy, const T* x, const T* w, const float* mean,
                                   const float* rstd, int M, int C, float scale,
                                   float* partials, int defer, cudaStream_t s) {
  constexpr int VE = 16 / sizeof(T);
  if (!aligned16(dres) || !aligned16(dy) || !aligned16(x) || !aligned16(w))
    return cudaErrorInvalidValue;
  const int blocks = layernorm_backward_blocks(M);
  const int stage_bytes = (acc ? 3 : 2) * LNB_ROWS * C * (int)sizeof(T);
  int stages = std::min(3, LNB_SMEM_BUDGET / stage_bytes);
  const int nk = dproj ? 3 : 2;
  size_t smem = std::max((size_t)std::max(stages, 1) * stage_bytes,
                         (size_t)LNB_ROWS * nk * C * sizeof(float));
  if (stages < 1) stages = 1;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  const int vpl = ceil_div(C, 32 * VE);
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<blocks, LNB_THREADS, smem, s>>>(dres, acc, partials, dy, x, w, mean, rstd, M, C,
                                           stages, defer, scale);
    count_launches(1);
    return cudaGetLastError();
  };
  cudaError_t e;
#define LNB_CASE(N)                                                                    \
  e = dproj ? launch(ln_bwd_kernel<T, N, true>) : launch(ln_bwd_kernel<T, N, false>); \
  break;
  switch (vpl) {
    case 1: LNB_CASE(1)
    case 2: LNB_CASE(2)
    case 3: LNB_CASE(3)
    case 4: LNB_CASE(4)
    case 5: case 6: LNB_CASE(6)
    case 7: case 8: LNB_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef LNB_CASE
  if (e != cudaSuccess) return e;
  if (defer) return cudaSuccess;
  return column_reduce(dw, db, dproj, partials, blocks, C, nk, nk * C, scale, s);
}

cudaError_t layernorm_fold(float* dw, float* db, float* dproj, float* partials, int C,
                           cudaStream_t s, float* nparts) {
  const int nk = dproj ? 3 : 2;
  return column_reduce(dw, db, dproj, partials, LNB_MAX_BLOCKS, C, nk, nk * C, 1.0f, s, 1, nparts);
}
int layernorm_fold_norm_parts(int C, bool dproj) { return ceil_div((dproj ? 3 : 2) * C, 32); }

cudaError_t layernorm_backward(DType t, void* dres, int accumulate, float* dw, float* db,
                               float* dproj, const void* dy, const void* x, const void* w,
                               const float* mean, const float* rstd, int M, int C, float scale,
                               float* partials, int defer, cudaStream_t s) {
  if (M <= 0 || C <= 0) return cudaErrorInvalidValue;
  if (t == DType::BF16) {
    if (C % 8) return cudaErrorInvalidValue;
    return ln_bwd_dispatch<bf16>((bf16*)dres, accumulate, dw, db, dproj, (const bf16*)dy,
                                 (const bf16*)x, (const bf16*)w, mean, rstd, M, C, scale,
                                 partials, defer, s);
  }
  if (C % 4) return cudaErrorInvalidValue;
  return ln_bwd_dispatch<float>((float*)dres, accumulate, dw, db, dproj, (const float*)dy,
                                (const float*)x, (const float*)w, mean, rstd, M, C, scale,
                                partials, defer, s);
}

// =====================================================================================
// Bias gradient db[n] += scale * sum_m dy[m, n]. Block (x, y): a strip of 32 * VE columns
// (one 16-byte vector per lane) over the rows of chunk y; warp w adds rows w, w + 8, ...
// of the chunk, the warps are combined in warp order into partials[y], and
// column_reduce adds the chunks in order.
constexpr int COLSUM_THREADS = 256;
constexpr int COLSUM_TARGET_BLOCKS = 4 * 148;

static void colsum_shape(int M, int N, int ve, int* strips, int* chunks, int* rpc) {
  *strips = ceil_div(N, 32 * ve);
  int c = std::max(1, COLSUM_TARGET_BLOCKS / *strips);
  c = std::min(c, std::max(1, ceil_div(M, 64)));
  *rpc = ceil_div(M, c);
  *chunks = ceil_div(M, *rpc);
}

static int colsum_max_chunks(int M, int N) {
  int strips, chunks, rpc, c8;
  colsum_shape(M, N, 8, &strips, &c8, &rpc);
  colsum_shape(M, N, 4, &strips, &chunks, &rpc);
  return std::max(c8, chunks);
}
size_t colsum_partials_floats(int M, int N) { return (size_t)colsum_max_chunks(M, N) * N; }
// chunk counts only shrink with M, so a buffer sized for M_max serves every M <= M_max
size_t colsum_deferred_partials_floats(int M_max, int N) { return colsum_partials_floats(M_max, N); }

template <typename T>
__global__ void __launch_bounds__(COLSUM_THREADS)
colsum_kernel(float* __restrict__ partials, const T* __restrict__ dy, int M, int N, int rpc,
              int defer, float pscale) {
  constexpr int VE = 16 / sizeof(T);
  __shared__ float sh[COLSUM_THREADS / 32][32 * VE];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int c = (blockIdx.x * 32 + lane) * VE;
  const int r0 = blockIdx.y * rpc, r1 = min(M, r0 + rpc);
  float acc[VE];
#pragma unroll
  for (int e = 0; e < VE; ++e) acc[e] = 0.f;
  if (c < N) {
    int r = r0 + wid;
    for (; r + 56 < r1; r += 64) {   // eight rows in flight per thread
      Vec16<T> v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = ld16(dy + (size_t)(r + 8 * k) * N + c);
#pragma unroll
      for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int e = 0; e < VE; ++e) acc[e] += to_f32(v[k].e[e]);
    }
    for (; r + 24 < r1; r += 32) {
      Vec16<T> v0 = ld16(dy + (size_t)r * N + c), v1 = ld16(dy + (size_t)(r + 8) * N + c);
      Vec16<T> v2 = ld16(dy + (size_t)(r + 16) * N + c), v3 = ld16(dy + (size_t)(r + 24) * N + c);
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        acc[e] += to_f32(v0.e[e]); acc[e] += to_f32(v1.e[e]);
        acc[e] += to_f32(v2.e[e]); acc[e] += to_f32(v3.e[e]);
      }
    }
    for (; r < r1; r += 8) {
      Vec16<T> v = ld16(dy + (size_t)r * N + c);
#pragma unroll
      for (int e = 0; e < VE; ++e) acc[e] += to_f32(v.e[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < VE; ++e) sh[wid][lane * VE + e] = acc[e];
  __syncthreads();
  for (int i = threadIdx.x; i < 32 * VE; i += COLSUM_THREADS) {
    const int col = blockIdx.x * 32 * VE + i;
    if (col >= N) continue;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < COLSUM_THREADS / 32; ++k) s += sh[k][i];
    float* o = partials + (size_t)blockIdx.y * N + col;
    *o = defer ? *o + pscale * s : s;   // deferred: this chunk's running sum
  }
}

cudaError_t bias_grad(DType t, float* db, const void* dy, int M, int N, float scale,
                      float* partials, int defer, cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaErrorInvalidValue;
  const int ve = t == DType::BF16 ? 8 : 4;
  if (N % ve || !aligned16(dy)) return cudaErrorInvalidValue;
  int strips, chunks, rpc;
  colsum_shape(M, N, ve, &strips, &chunks, &rpc);
  dim3 grid(strips, chunks);
  if (t == DType::BF16)
    colsum_kernel<bf16><<<grid, COLSUM_THREADS, 0, s>>>(partials, (const bf16*)dy, M, N, rpc,
                                                        defer, scale);
  else
    colsum_kernel<float><<<grid, COLSUM_THREADS, 0, s>>>(partials, (const float*)dy, M, N, rpc,
                                                         defer, scale);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || defer) return e;
  return column_reduce(db, nullptr, nullptr, partials, chunks, N, 1, N, scale, s);
}

cudaError_t bias_grad_fold(float* db, float* partials, int M_max, int N, cudaStream_t s,
                           float* nparts) {
  return column_reduce(db, nullptr, nullptr, partials, colsum_max_chunks(M_max, N), N, 1, N, 1.0f,
                       s, 1, nparts);
}
int bias_grad_fold_norm_parts(int N) { return ceil_div(N, 32); }

}  // namespace gpt2k

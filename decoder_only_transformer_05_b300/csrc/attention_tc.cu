// Causal flash attention on the 5th-generation tensor cores (tcgen05), head size 64, bf16
// in, fp32 accumulation: out = softmax(q k^T / sqrt(64) + causal mask) v per (batch, head),
// heads concatenated, never forming the T x T matrix in global memory (the scaled
// dot-product attention of 「从零实现一个最小GPT：代码讲解 + 知识点全解」 二.3 Head / 三.3,
// with the fused multi-head layout of the qkv projection).
//
// Forward: one block per (batch, head, 128 query rows), 192 threads.
//   warp 0      TMA producer: the Q tile once, then K_j, V_j (128 keys x 64) into a ring
//               of KV_STAGES stages
//   warp 1      MMA issuer: S_j = Q K_j^T (M=128, N=128, K=64) into one of two TMEM score
//               buffers, issued one block ahead; O += P_j V_j (M=128, N=64, K=128) into a
//               TMEM accumulator once the softmax has written P_j
//   warps 2..5  softmax: thread = query row (TMEM lane). Online softmax in registers in
//               the log2 domain: m = running max, l = running sum; P_j = exp2(s - m) as
//               bf16 into a swizzled shared-memory tile (the A operand of P V); when m
//               grows, O is rescaled in tensor memory before P_j V_j is issued. At the end
//               O / l goes out through a TMA store and lse = ln(l) + m ln 2 to memory.
// Rows past T (ragged T) read zeros through the 3-D tensor maps and are never stored.
// Every mbarrier wait is bounded; on timeout the block records DEV_ERR_TIMEOUT and leaves.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace gpt2k {
namespace fatc {

using namespace tc;

constexpr int D = 64;
constexpr int BQ = 128, BKV = 128;
constexpr int THREADS = 192;
constexpr int KV_STAGES = 3;
constexpr int TILE = BQ * D * 2;                 // 16 KB: 128 rows x 128 B
constexpr int SM_Q = 0;
constexpr int SM_KV = SM_Q + TILE;               // stage s: K at +2s*TILE, V at +(2s+1)*TILE
constexpr int SM_P = SM_KV + 2 * KV_STAGES * TILE;   // two 64-key halves of P
constexpr int SM_BAR = SM_P + 2 * TILE;
constexpr int SMEM = SM_BAR + 256 + 1024;
constexpr uint32_t TMEM_COLS = 512;              // S0 [0,128) S1 [128,256) O [256,320)
constexpr uint32_t COL_O = 256;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

struct FwdParams {
  int T, H, C, nqb;
  float* lse;
  int* err;
};

__global__ void __launch_bounds__(THREADS, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_out,
           const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + SM_BAR;
  // barriers: q_full, kv_full[S], kv_empty[S], s_full[2], s_empty[2], p_full, o_done, final
  const uint32_t q_full = bars;
  auto kv_full = [&](int s) { return bars + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bars + 8u * (1 + KV_STAGES + s); };
  auto s_full = [&](int b) { return bars + 8u * (1 + 2 * KV_STAGES + b); };
  auto s_empty = [&](int b) { return bars + 8u * (3 + 2 * KV_STAGES + b); };
  const uint32_t p_full = bars + 8u * (5 + 2 * KV_STAGES);
  const uint32_t o_done = bars + 8u * (6 + 2 * KV_STAGES);
  const uint32_t final_bar = bars + 8u * (7 + 2 * KV_STAGES);
  const uint32_t slot = bars + 8u * (8 + 2 * KV_STAGES);
  volatile uint32_t* slot_ptr = (volatile uint32_t*)(base_ptr + SM_BAR + 8 * (8 + 2 * KV_STAGES));
  volatile int* abort_flag = (volatile int*)(base_ptr + SM_BAR + 8 * (9 + 2 * KV_STAGES));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = p.nqb - 1 - (int)blockIdx.x;     // heavy (late) query blocks first
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int nkv = qb + 1;                          // key blocks 0..qb (BQ == BKV)

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < KV_STAGES; ++s) { mbar_init(kv_full(s), 1); mbar_init(kv_empty(s), 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(s_full(i), 1); mbar_init(s_empty(i), 4); }
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot_ptr;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      bool ok = true;
      mbar_expect_tx(q_full, TILE);
      tma_load_3d(base + SM_Q, &tm_qkv, q_full, h * D, qb * BQ, b);
      int j = 0;
      for (; j < nkv && ok; ++j) {
        const int s = j % KV_STAGES;
        if (!mbar_wait(kv_empty(s), ((uint32_t)(j / KV_STAGES) & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t kdst = base + SM_KV + 2 * s * TILE;
        mbar_expect_tx(kv_full(s), 2 * TILE);
        tma_load_3d(kdst, &tm_qkv, kv_full(s), p.C + h * D, j * BKV, b);
        tma_load_3d(kdst + TILE, &tm_qkv, kv_full(s), 2 * p.C + h * D, j * BKV, b);
      }
      // copies in flight land before the block leaves
      mbar_wait(q_full, 0, abort_flag, nullptr, false);
      for (int i = max(0, j - KV_STAGES); i < j; ++i)
        mbar_wait(kv_full(i % KV_STAGES), (uint32_t)(i / KV_STAGES) & 1u, abort_flag, nullptr,
                  false);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t IDESC_S = make_idesc(BQ, BKV, false, false);
      constexpr uint32_t IDESC_O = make_idesc(BQ, D, false, true);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.err);
      auto issue_s = [&](int j) -> bool {
        const int s = j % KV_STAGES, buf = j & 1;
        if (!mbar_wait(kv_full(s), (uint32_t)(j / KV_STAGES) & 1u, abort_flag, p.err)) return false;
        if (j >= 2 && !mbar_wait(s_empty(buf), (uint32_t)((j >> 1) - 1) & 1u, abort_flag, p.err))
          return false;
        tc_fence_after();
        const uint32_t kb = base + SM_KV + 2 * s * TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_bf16(tmem + buf * BKV, sdesc(base + SM_Q + k * 32, 16, 1024),
                    sdesc(kb + k * 32, 16, 1024), IDESC_S, k > 0 ? 1u : 0u);
        umma_commit(s_full(buf));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nkv && ok; ++j) {
        if (j + 1 < nkv && !issue_s(j + 1)) { ok = false; break; }
        if (!mbar_wait(p_full, (uint32_t)j & 1u, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vb = base + SM_KV + (2 * (j % KV_STAGES) + 1) * TILE;
#pragma unroll
        for (int k = 0; k < BKV / 16; ++k)
          umma_bf16(tmem + COL_O, sdesc(base + SM_P + (k >> 2) * TILE + (k & 3) * 32, 16, 1024),
                    sdesc(vb + k * 2048, 16384, 1024), IDESC_O, (j > 0 || k > 0) ? 1u : 0u);
        umma_commit(o_done);
        umma_commit(kv_empty(j % KV_STAGES));
      }
      umma_commit(final_bar);
      mbar_wait(final_bar, 0, abort_flag, nullptr, false);
    }
  } else {
    // ---------------- softmax warps 2..5: TMEM lane quarter q = warp % 4, one row each
    const int q = warp & 3;
    const int r = q * 32 + lane;                      // row in the tile
    const int query = qb * BQ + r;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const float sl2 = rsqrtf((float)D) * LOG2E;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int buf = j & 1;
      ok = mbar_wait(s_full(buf), (uint32_t)(j >> 1) & 1u, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32_nowait(lane_base + buf * BKV + c * 32, sr[c]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty(buf));
      // scale into the log2 domain and mask the future on the diagonal block
      float mx = -INFINITY;
      const bool diag = (j == qb);
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float v = __uint_as_float(sr[c][e]) * sl2;
          if (diag && (c * 32 + e) > r) v = -INFINITY;
          sr[c][e] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      const float m_new = fmaxf(m, mx);
      const float alpha = fast_exp2(m - m_new);
      m = m_new;
      float sum = 0.f;
      uint32_t pk[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = fast_exp2(__uint_as_float(sr[c][2 * e]) - m_new);
          const float p1 = fast_exp2(__uint_as_float(sr[c][2 * e + 1]) - m_new);
          sum += p0 + p1;
          pk[c][e] = pack2_bf16(p0, p1);
        }
      l = l * alpha + sum;
      if (j > 0) {
        // P_{j-1} V_{j-1} is complete: O is stable and the P tile is free
        ok = mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32_nowait(lane_base + COL_O + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_base + COL_O + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      // P row r: keys 0..63 in the first half-tile, 64..127 in the second; 16-byte unit
      // u of a 128-byte row sits at unit u ^ (r & 7) (128-byte swizzle)
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (c & 1) * 4 + u;
          st_shared16(base + SM_P + (c >> 1) * TILE + r * 128 + ((unit ^ (r & 7)) << 4),
                      make_uint4(pk[c][4 * u], pk[c][4 * u + 1], pk[c][4 * u + 2],
                                 pk[c][4 * u + 3]));
        }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok) ok = mbar_wait(o_done, (uint32_t)(nkv - 1) & 1u, abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      uint32_t o[2][32];
      tmem_ld32_nowait(lane_base + COL_O, o[0]);
      tmem_ld32_nowait(lane_base + COL_O + 32, o[1]);
      tmem_wait_ld();
      const float inv = 1.0f / l;
      // O row into the Q tile's space (free now), 128-byte swizzle, then one TMA store
      const uint32_t stg = base + SM_Q;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t* src = &o[u >> 2][(u & 3) * 8];
        st_shared16(stg + r * 128 + ((u ^ (r & 7)) << 4),
                    make_uint4(pack2_bf16(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv),
                               pack2_bf16(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv),
                               pack2_bf16(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv),
                               pack2_bf16(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv)));
      }
      fence_proxy_async();
      if (query < p.T) p.lse[((size_t)b * p.H + h) * p.T + query] = (m + __log2f(l)) * LN2;
    }
    named_bar_sync(1, 128);
    if (threadIdx.x == 64 && ok) {
      tma_store_3d(&tm_out, base + SM_Q, h * D, qb * BQ, b);
      bulk_commit();
      bulk_wait_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
// [B][T][width] bf16 as a 3-D map {width, T, B}, box {64, 128, 1}, 128-byte swizzle
static bool map_btw(CUtensorMap* m, const void* ptr, int B, int T, int width) {
  auto fn = tensor_map_encoder();
  if (!fn || ((uintptr_t)ptr & 15u) || (width * 2) % 16) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)T * width * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fatc

cudaError_t attention_forward_tc(void* out, float* lse, const void* qkv, int B, int T, int C,
                                 int H, int* err, cudaStream_t s) {
  using namespace fatc;
  if (C / H != D || C % H || C % 64) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap mq, mo;
  if (!map_btw(&mq, qkv, B, T, 3 * C) || !map_btw(&mo, out, B, T, C)) return cudaErrorInvalidValue;
  FwdParams p;
  p.T = T; p.H = H; p.C = C; p.nqb = ceil_div(T, BQ);
  p.lse = lse;
  p.err = err;
  dim3 grid(p.nqb, B * H);
  fwd_kernel<<<grid, THREADS, SMEM, s>>>(mq, mo, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace gpt2k

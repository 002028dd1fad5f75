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

// =====================================================================================
// Backward. With P recomputed from the forward's lse (P = exp2(s sl2 - lse log2 e)) and
// D = rowsum(dO * O), every element is independent: dS = P (dP - D), dP = dO V^T, and
//   dV = P^T dO,  dK = dS^T Q / sqrt(64),  dQ = dS K / sqrt(64).
// Two kernels, each owning its output rows, so no partial sums cross blocks and the
// result is deterministic. 320 threads: warp 0 TMA, warp 1 MMA, warps 2..9 elementwise
// (warp w reads TMEM lane quarter w % 4; warps w and w + 4 take columns 0..63 and 64..127).
constexpr int BWD_THREADS = 320;
constexpr int BWD_STAGES = 2;

struct BwdParams {
  int T, H, C, nqb;
  const float* lse;
  const float* Dbuf;
  int* err;
};

// dK, dV for one block of 128 keys; loops over the query blocks at or after it.
//   S^T = K Q_i^T, dP^T = V dO_i^T (TMEM, 128 + 128 columns), then
//   dV += P^T dO_i, dK += dS^T Q_i (TMEM, 64 + 64 columns) with P^T and dS^T staged as
//   bf16 in shared memory (the A operands).
constexpr int DKV_SM_K = 0;
constexpr int DKV_SM_V = DKV_SM_K + TILE;
constexpr int DKV_SM_QD = DKV_SM_V + TILE;                       // stage s: Q at +2s, dO at +2s+1
constexpr int DKV_SM_PT = DKV_SM_QD + 2 * BWD_STAGES * TILE;     // P^T, two 64-query halves
constexpr int DKV_SM_DST = DKV_SM_PT + 2 * TILE;                 // dS^T
constexpr int DKV_SM_LD = DKV_SM_DST + 2 * TILE;                 // stage s: [lse 128 | D 128]
constexpr int DKV_SM_BAR = DKV_SM_LD + BWD_STAGES * 256 * 4;
constexpr int DKV_SMEM = DKV_SM_BAR + 256 + 1024;

__global__ void __launch_bounds__(BWD_THREADS, 1)
bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dqkv, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + DKV_SM_BAR;
  // barriers: kv_full, qd_full[S], qd_empty[S], s_full, s_empty, p_full, done, final
  const uint32_t kv_full = bars;
  auto qd_full = [&](int s) { return bars + 8u * (1 + s); };
  auto qd_empty = [&](int s) { return bars + 8u * (1 + BWD_STAGES + s); };
  const uint32_t s_full = bars + 8u * (1 + 2 * BWD_STAGES);
  const uint32_t s_empty = bars + 8u * (2 + 2 * BWD_STAGES);
  const uint32_t p_full = bars + 8u * (3 + 2 * BWD_STAGES);
  const uint32_t done = bars + 8u * (4 + 2 * BWD_STAGES);
  const uint32_t final_bar = bars + 8u * (5 + 2 * BWD_STAGES);
  const uint32_t slot = bars + 8u * (6 + 2 * BWD_STAGES);
  volatile uint32_t* slot_ptr = (volatile uint32_t*)(base_ptr + DKV_SM_BAR + 8 * (6 + 2 * BWD_STAGES));
  volatile int* abort_flag = (volatile int*)(base_ptr + DKV_SM_BAR + 8 * (7 + 2 * BWD_STAGES));
  float* sm_ld = reinterpret_cast<float*>(base_ptr + DKV_SM_LD);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = blockIdx.x;                        // key block; query blocks kb..nqb-1
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int n = p.nqb - kb;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < BWD_STAGES; ++s) { mbar_init(qd_full(s), 1); mbar_init(qd_empty(s), 1); }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 8);
    mbar_init(p_full, 8);
    mbar_init(done, 1);
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
  constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 320;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      mbar_expect_tx(kv_full, 2 * TILE);
      tma_load_3d(base + DKV_SM_K, &tm_qkv, kv_full, p.C + h * D, kb * BKV, b);
      tma_load_3d(base + DKV_SM_V, &tm_qkv, kv_full, 2 * p.C + h * D, kb * BKV, b);
      int i = 0;
      for (; i < n && ok; ++i) {
        const int s = i % BWD_STAGES;
        if (!mbar_wait(qd_empty(s), ((uint32_t)(i / BWD_STAGES) & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t dst = base + DKV_SM_QD + 2 * s * TILE;
        const int qbi = kb + i;
        // lse and D of the block's queries ride with the Q / dO tiles (T % 4 == 0, so the
        // row start and the byte count are multiples of 16)
        const uint32_t nb = (uint32_t)min(BQ, p.T - qbi * BQ) * 4u;
        const size_t t0 = (size_t)bh * p.T + (size_t)qbi * BQ;
        mbar_expect_tx(qd_full(s), 2 * TILE + 2 * nb);
        tma_load_3d(dst, &tm_qkv, qd_full(s), h * D, qbi * BQ, b);
        tma_load_3d(dst + TILE, &tm_do, qd_full(s), h * D, qbi * BQ, b);
        const uint32_t ld_dst = base + DKV_SM_LD + s * 1024;
        bulk_load(ld_dst, p.lse + t0, nb, qd_full(s));
        bulk_load(ld_dst + 512, p.Dbuf + t0, nb, qd_full(s));
      }
      mbar_wait(kv_full, 0, abort_flag, nullptr, false);
      for (int k = max(0, i - BWD_STAGES); k < i; ++k)
        mbar_wait(qd_full(k % BWD_STAGES), (uint32_t)(k / BWD_STAGES) & 1u, abort_flag, nullptr,
                  false);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC_S = make_idesc(BKV, BQ, false, false);
      constexpr uint32_t IDESC_G = make_idesc(BKV, D, false, true);
      bool ok = mbar_wait(kv_full, 0, abort_flag, p.err);
      auto issue_s = [&](int i) -> bool {
        const int s = i % BWD_STAGES;
        if (!mbar_wait(qd_full(s), (uint32_t)(i / BWD_STAGES) & 1u, abort_flag, p.err)) return false;
        if (i >= 1 && !mbar_wait(s_empty, (uint32_t)(i - 1) & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t qa = base + DKV_SM_QD + 2 * s * TILE, da = qa + TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          umma_bf16(tmem + COL_S, sdesc(base + DKV_SM_K + k * 32, 16, 1024),
                    sdesc(qa + k * 32, 16, 1024), IDESC_S, k > 0 ? 1u : 0u);
          umma_bf16(tmem + COL_DP, sdesc(base + DKV_SM_V + k * 32, 16, 1024),
                    sdesc(da + k * 32, 16, 1024), IDESC_S, k > 0 ? 1u : 0u);
        }
        umma_commit(s_full);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int i = 0; i < n && ok; ++i) {
        if (i + 1 < n && !issue_s(i + 1)) { ok = false; break; }
        if (!mbar_wait(p_full, (uint32_t)i & 1u, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qa = base + DKV_SM_QD + 2 * (i % BWD_STAGES) * TILE, da = qa + TILE;
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k) {
          const uint32_t off = (k >> 2) * TILE + (k & 3) * 32;
          umma_bf16(tmem + COL_DV, sdesc(base + DKV_SM_PT + off, 16, 1024),
                    sdesc(da + k * 2048, 16384, 1024), IDESC_G, (i > 0 || k > 0) ? 1u : 0u);
          umma_bf16(tmem + COL_DK, sdesc(base + DKV_SM_DST + off, 16, 1024),
                    sdesc(qa + k * 2048, 16384, 1024), IDESC_G, (i > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(done);
        umma_commit(qd_empty(i % BWD_STAGES));
      }
      umma_commit(final_bar);
      mbar_wait(final_bar, 0, abort_flag, nullptr, false);
    }
  } else {
    // ---------------- elementwise warps: key row r, query columns c0 .. c0 + 63
    const int q = warp & 3, half = (warp - 2) >> 2;
    const int r = q * 32 + lane, c0 = half * 64;
    const int key = kb * BKV + r;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const float sl2 = rsqrtf((float)D) * LOG2E;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      // this stage's lse and D (copied with Q_i, dO_i); the stage is not refilled before
      // the MMAs that follow p_full(i) have finished
      const float* ld = sm_ld + (i % BWD_STAGES) * 256;
      ok = mbar_wait(qd_full(i % BWD_STAGES), (uint32_t)(i / BWD_STAGES) & 1u, abort_flag, p.err) &&
           mbar_wait(s_full, (uint32_t)i & 1u, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[2][32], dv[2][32];
      tmem_ld32_nowait(lane_base + COL_S + c0, sv[0]);
      tmem_ld32_nowait(lane_base + COL_S + c0 + 32, sv[1]);
      tmem_ld32_nowait(lane_base + COL_DP + c0, dv[0]);
      tmem_ld32_nowait(lane_base + COL_DP + c0 + 32, dv[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty);
      const int qbase = (kb + i) * BQ + c0;
      uint32_t pk[32], dk[32];
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float pp[2], dd[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int qc = c * 32 + e + u;           // query column within this half
            const int query = qbase + qc;
            float pv = fast_exp2(fmaf(__uint_as_float(sv[c][e + u]), sl2, -ld[c0 + qc] * LOG2E));
            if (query < key || query >= p.T) pv = 0.f;
            pp[u] = pv;
            dd[u] = pv * (__uint_as_float(dv[c][e + u]) - ld[128 + c0 + qc]);
          }
          pk[c * 16 + e / 2] = pack2_bf16(pp[0], pp[1]);
          dk[c * 16 + e / 2] = pack2_bf16(dd[0], dd[1]);
        }
      if (i > 0) {
        ok = mbar_wait(done, (uint32_t)(i - 1) & 1u, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      // rows of P^T and dS^T: this half's 64 queries are one 128-byte swizzled row
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t off = half * TILE + r * 128 + ((u ^ (r & 7)) << 4);
        st_shared16(base + DKV_SM_PT + off,
                    make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]));
        st_shared16(base + DKV_SM_DST + off,
                    make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]));
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok) ok = mbar_wait(done, (uint32_t)(n - 1) & 1u, abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      // this warp's 32 of the 64 head columns of dK and dV, into the (now free) Q/dO stage 0
      uint32_t kv[2][32];
      tmem_ld32_nowait(lane_base + COL_DK + half * 32, kv[0]);
      tmem_ld32_nowait(lane_base + COL_DV + half * 32, kv[1]);
      tmem_wait_ld();
      const float scale = rsqrtf((float)D);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float sc = t == 0 ? scale : 1.0f;
        const uint32_t stg = base + DKV_SM_QD + t * TILE;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t* v = &kv[t][u * 8];
          const int unit = half * 4 + u;
          st_shared16(stg + r * 128 + ((unit ^ (r & 7)) << 4),
                      make_uint4(pack2_bf16(__uint_as_float(v[0]) * sc, __uint_as_float(v[1]) * sc),
                                 pack2_bf16(__uint_as_float(v[2]) * sc, __uint_as_float(v[3]) * sc),
                                 pack2_bf16(__uint_as_float(v[4]) * sc, __uint_as_float(v[5]) * sc),
                                 pack2_bf16(__uint_as_float(v[6]) * sc, __uint_as_float(v[7]) * sc)));
        }
      }
      fence_proxy_async();
    }
    named_bar_sync(1, 256);
    if (threadIdx.x == 64 && ok) {
      tma_store_3d(&tm_dqkv, base + DKV_SM_QD, p.C + h * D, kb * BKV, b);
      tma_store_3d(&tm_dqkv, base + DKV_SM_QD + TILE, 2 * p.C + h * D, kb * BKV, b);
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

// dQ for one block of 128 queries; loops over the key blocks up to the diagonal.
//   S = Q K_j^T, dP = dO V_j^T (TMEM), dS = P (dP - D) as bf16 in shared memory, then
//   dQ += dS K_j (TMEM, 64 columns).
constexpr int DQ_SM_Q = 0;
constexpr int DQ_SM_DO = DQ_SM_Q + TILE;
constexpr int DQ_SM_KV = DQ_SM_DO + TILE;                        // stage s: K at +2s, V at +2s+1
constexpr int DQ_SM_DS = DQ_SM_KV + 2 * BWD_STAGES * TILE;
constexpr int DQ_SM_BAR = DQ_SM_DS + 2 * TILE;
constexpr int DQ_SMEM = DQ_SM_BAR + 256 + 1024;

__global__ void __launch_bounds__(BWD_THREADS, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_dqkv, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + DQ_SM_BAR;
  const uint32_t q_full = bars;
  auto kv_full = [&](int s) { return bars + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bars + 8u * (1 + BWD_STAGES + s); };
  const uint32_t s_full = bars + 8u * (1 + 2 * BWD_STAGES);
  const uint32_t s_empty = bars + 8u * (2 + 2 * BWD_STAGES);
  const uint32_t p_full = bars + 8u * (3 + 2 * BWD_STAGES);
  const uint32_t done = bars + 8u * (4 + 2 * BWD_STAGES);
  const uint32_t final_bar = bars + 8u * (5 + 2 * BWD_STAGES);
  const uint32_t slot = bars + 8u * (6 + 2 * BWD_STAGES);
  volatile uint32_t* slot_ptr = (volatile uint32_t*)(base_ptr + DQ_SM_BAR + 8 * (6 + 2 * BWD_STAGES));
  volatile int* abort_flag = (volatile int*)(base_ptr + DQ_SM_BAR + 8 * (7 + 2 * BWD_STAGES));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = p.nqb - 1 - (int)blockIdx.x;
  const int bh = blockIdx.y, b = bh / p.H, h = bh % p.H;
  const int n = qb + 1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < BWD_STAGES; ++s) { mbar_init(kv_full(s), 1); mbar_init(kv_empty(s), 1); }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 8);
    mbar_init(p_full, 8);
    mbar_init(done, 1);
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
  constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DQ = 256;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      mbar_expect_tx(q_full, 2 * TILE);
      tma_load_3d(base + DQ_SM_Q, &tm_qkv, q_full, h * D, qb * BQ, b);
      tma_load_3d(base + DQ_SM_DO, &tm_do, q_full, h * D, qb * BQ, b);
      int j = 0;
      for (; j < n && ok; ++j) {
        const int s = j % BWD_STAGES;
        if (!mbar_wait(kv_empty(s), ((uint32_t)(j / BWD_STAGES) & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        const uint32_t dst = base + DQ_SM_KV + 2 * s * TILE;
        mbar_expect_tx(kv_full(s), 2 * TILE);
        tma_load_3d(dst, &tm_qkv, kv_full(s), p.C + h * D, j * BKV, b);
        tma_load_3d(dst + TILE, &tm_qkv, kv_full(s), 2 * p.C + h * D, j * BKV, b);
      }
      mbar_wait(q_full, 0, abort_flag, nullptr, false);
      for (int k = max(0, j - BWD_STAGES); k < j; ++k)
        mbar_wait(kv_full(k % BWD_STAGES), (uint32_t)(k / BWD_STAGES) & 1u, abort_flag, nullptr,
                  false);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC_S = make_idesc(BQ, BKV, false, false);
      constexpr uint32_t IDESC_G = make_idesc(BQ, D, false, true);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.err);
      auto issue_s = [&](int j) -> bool {
        const int s = j % BWD_STAGES;
        if (!mbar_wait(kv_full(s), (uint32_t)(j / BWD_STAGES) & 1u, abort_flag, p.err)) return false;
        if (j >= 1 && !mbar_wait(s_empty, (uint32_t)(j - 1) & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t ka = base + DQ_SM_KV + 2 * s * TILE, va = ka + TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          umma_bf16(tmem + COL_S, sdesc(base + DQ_SM_Q + k * 32, 16, 1024),
                    sdesc(ka + k * 32, 16, 1024), IDESC_S, k > 0 ? 1u : 0u);
          umma_bf16(tmem + COL_DP, sdesc(base + DQ_SM_DO + k * 32, 16, 1024),
                    sdesc(va + k * 32, 16, 1024), IDESC_S, k > 0 ? 1u : 0u);
        }
        umma_commit(s_full);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < n && ok; ++j) {
        if (j + 1 < n && !issue_s(j + 1)) { ok = false; break; }
        if (!mbar_wait(p_full, (uint32_t)j & 1u, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t ka = base + DQ_SM_KV + 2 * (j % BWD_STAGES) * TILE;
#pragma unroll
        for (int k = 0; k < BKV / 16; ++k)
          umma_bf16(tmem + COL_DQ, sdesc(base + DQ_SM_DS + (k >> 2) * TILE + (k & 3) * 32, 16, 1024),
                    sdesc(ka + k * 2048, 16384, 1024), IDESC_G, (j > 0 || k > 0) ? 1u : 0u);
        umma_commit(done);
        umma_commit(kv_empty(j % BWD_STAGES));
      }
      umma_commit(final_bar);
      mbar_wait(final_bar, 0, abort_flag, nullptr, false);
    }
  } else {
    // ---------------- elementwise warps: query row r, key columns c0 .. c0 + 63
    const int q = warp & 3, half = (warp - 2) >> 2;
    const int r = q * 32 + lane, c0 = half * 64;
    const int query = qb * BQ + r;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const float sl2 = rsqrtf((float)D) * LOG2E;
    float lse2 = 0.f, Dr = 0.f;
    if (query < p.T) {
      lse2 = __ldg(p.lse + (size_t)bh * p.T + query) * LOG2E;
      Dr = __ldg(p.Dbuf + (size_t)bh * p.T + query);
    }
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = mbar_wait(s_full, (uint32_t)j & 1u, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[2][32], dv[2][32];
      tmem_ld32_nowait(lane_base + COL_S + c0, sv[0]);
      tmem_ld32_nowait(lane_base + COL_S + c0 + 32, sv[1]);
      tmem_ld32_nowait(lane_base + COL_DP + c0, dv[0]);
      tmem_ld32_nowait(lane_base + COL_DP + c0 + 32, dv[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty);
      const int kbase = j * BKV + c0;
      uint32_t dk[32];
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float dd[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int kc = kbase + c * 32 + e + u;
            float pv = fast_exp2(fmaf(__uint_as_float(sv[c][e + u]), sl2, -lse2));
            if (kc > query) pv = 0.f;
            dd[u] = pv * (__uint_as_float(dv[c][e + u]) - Dr);
          }
          dk[c * 16 + e / 2] = pack2_bf16(dd[0], dd[1]);
        }
      if (j > 0) {
        ok = mbar_wait(done, (uint32_t)(j - 1) & 1u, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_shared16(base + DQ_SM_DS + half * TILE + r * 128 + ((u ^ (r & 7)) << 4),
                    make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]));
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok) ok = mbar_wait(done, (uint32_t)(n - 1) & 1u, abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32_nowait(lane_base + COL_DQ + half * 32, v);
      tmem_wait_ld();
      const float sc = rsqrtf((float)D);
      const uint32_t stg = base + DQ_SM_Q;     // Q is no longer read
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t* w = &v[u * 8];
        const int unit = half * 4 + u;
        st_shared16(stg + r * 128 + ((unit ^ (r & 7)) << 4),
                    make_uint4(pack2_bf16(__uint_as_float(w[0]) * sc, __uint_as_float(w[1]) * sc),
                               pack2_bf16(__uint_as_float(w[2]) * sc, __uint_as_float(w[3]) * sc),
                               pack2_bf16(__uint_as_float(w[4]) * sc, __uint_as_float(w[5]) * sc),
                               pack2_bf16(__uint_as_float(w[6]) * sc, __uint_as_float(w[7]) * sc)));
      }
      fence_proxy_async();
    }
    named_bar_sync(1, 256);
    if (threadIdx.x == 64 && ok) {
      tma_store_3d(&tm_dqkv, base + DQ_SM_Q, h * D, qb * BQ, b);
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

cudaError_t attention_backward_tc(void* dqkv, const float* Dbuf, const void* dout,
                                  const void* qkv, const float* lse, int B, int T, int C, int H,
                                  int* err, cudaStream_t s) {
  using namespace fatc;
  if (C / H != D || C % H || C % 64 || T % 4 || ((uintptr_t)lse & 15u) || ((uintptr_t)Dbuf & 15u))
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(bwd_dkv_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, DKV_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DQ_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap mq, md, mg;
  if (!map_btw(&mq, qkv, B, T, 3 * C) || !map_btw(&md, dout, B, T, C) ||
      !map_btw(&mg, dqkv, B, T, 3 * C))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.T = T; p.H = H; p.C = C; p.nqb = ceil_div(T, BQ);
  p.lse = lse; p.Dbuf = Dbuf; p.err = err;
  dim3 grid(p.nqb, B * H);
  bwd_dkv_kernel<<<grid, BWD_THREADS, DKV_SMEM, s>>>(mq, md, mg, p);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_dq_kernel<<<grid, BWD_THREADS, DQ_SMEM, s>>>(mq, md, mg, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace gpt2k

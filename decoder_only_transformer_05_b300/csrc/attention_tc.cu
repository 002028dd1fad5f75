// Causal flash attention on the 5th-generation tensor cores (tcgen05), head size 64, bf16
// in, fp32 accumulation: out = softmax(q k^T / sqrt(64) + causal mask) v per (batch, head),
// heads concatenated, never forming the T x T matrix in global memory (the scaled
// dot-product attention of 「从零实现一个最小GPT：代码讲解 + 知识点全解」 二.3 Head / 三.3,
// with the fused multi-head layout of the qkv projection).
//
// All three kernels are persistent: one 320-thread block per SM walks a fixed list of
// work units (heaviest first, unit c, c + G, c + 2G, ... for block c of G), and the TMA
// rings run on across units so the next unit's tiles load while this one computes.
//   warp 0      TMA producer (Q / K / V / dO tiles of 128 rows x 64, 128-byte swizzle)
//   warp 1      MMA issuer (one thread; tcgen05.mma, fp32 accumulators in tensor memory)
//   warps 2..9  elementwise: warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31
// Each elementwise warp stores its own 32 output rows (a TMA store from its own slice of
// shared memory), so no barrier spans more than one warp. Every mbarrier wait is bounded;
// on timeout the block records DEV_ERR_TIMEOUT and stops.
//
// Forward (unit = one (batch, head) and two consecutive 128-query tiles A, B):
//   S_X = Q_X K_j^T (TMEM, 128 columns per tile), softmax by the tile's four warps (thread =
//   query row) with an online max m and sum l in the log2 domain, P_X = exp2(s - m) as bf16
//   into shared memory, O_X += P_X V_j (TMEM, 64 columns per tile). m only moves when the
//   block's maximum exceeds it by more than 8 (P then stays below 2^8), and O is rescaled in
//   tensor memory when it does. The two tiles' softmax warps run side by side and share
//   every K, V tile; K and V have rings of their own, P is double-buffered per tile, and the
//   MMA thread issues whichever S or P V group is ready (non-blocking probes).
// Backward (P = exp2(s sl2 - lse log2 e), D = rowsum(dO * O)): the dQ kernel runs first;
//   its unit = (batch, head, 128 queries) loads Q, dO and O, computes D for its rows (and
//   writes it for the dK/dV kernel), then S = Q K_j^T, dP = dO V_j^T, dQ += dS K_j with
//   dS = P (dP - D). The dK/dV unit = (batch, head, 128 keys): S^T = K Q_i^T,
//   dP^T = V dO_i^T, then dV += P^T dO_i, dK += dS^T Q_i. Each output row belongs to one
//   unit, so the result is deterministic. The eight elementwise warps split the columns
//   (warps w and w + 4 take 64 each): no row reduction is needed once lse and D are known.
//   P^T, dS^T (dK/dV) and dS (dQ, double-buffered) go back into tensor memory as bf16 pairs
//   and are the A operand of the second-stage MMAs (tcgen05.mma with A in tensor memory), so
//   they never touch shared memory; the Q/dO and K/V rings have four stages.
// Rows past T (ragged T) read zeros through the 3-D tensor maps and are never stored.
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace gpt2k {
namespace fatc {

using namespace tc;

constexpr int D = 64;
constexpr int BQ = 128, BKV = 128;
constexpr int THREADS = 320;
constexpr int TILE = BQ * D * 2;                 // 16 KB: 128 rows x 128 B
constexpr uint32_t TMEM_COLS = 512;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_LOG2 = 8.0f;             // move the running max only past this margin

// phase parity of the n-th completion (n = 0, 1, ...) of a barrier
__device__ __forceinline__ uint32_t par(int n) { return (uint32_t)n & 1u; }

// Row r (0..31 within the warp's slice) of a 32 x 64 bf16 tile, 128 B per row, 128-byte
// swizzle: 16-byte unit u of the row at unit u ^ (r & 7).
__device__ __forceinline__ void stage_row64(uint32_t slice, int r, const float* v, float sc) {
#pragma unroll
  for (int u = 0; u < 8; ++u)
    st_shared16(slice + r * 128 + ((u ^ (r & 7)) << 4),
                make_uint4(pack2_bf16(v[8 * u] * sc, v[8 * u + 1] * sc),
                           pack2_bf16(v[8 * u + 2] * sc, v[8 * u + 3] * sc),
                           pack2_bf16(v[8 * u + 4] * sc, v[8 * u + 5] * sc),
                           pack2_bf16(v[8 * u + 6] * sc, v[8 * u + 7] * sc)));
}
// Row r of a 32 x 32 bf16 tile, 64 B per row, 64-byte swizzle: unit u at u ^ ((r >> 1) & 3).
__device__ __forceinline__ void stage_row32(uint32_t slice, int r, const float* v, float sc) {
#pragma unroll
  for (int u = 0; u < 4; ++u)
    st_shared16(slice + r * 64 + ((u ^ ((r >> 1) & 3)) << 4),
                make_uint4(pack2_bf16(v[8 * u] * sc, v[8 * u + 1] * sc),
                           pack2_bf16(v[8 * u + 2] * sc, v[8 * u + 3] * sc),
                           pack2_bf16(v[8 * u + 4] * sc, v[8 * u + 5] * sc),
                           pack2_bf16(v[8 * u + 6] * sc, v[8 * u + 7] * sc)));
}

struct Params {
  int B, T, H, C, nqb, units;
  float* lse;            // forward output, backward input [B, H, T]
  float* Dbuf;           // backward scratch [2][B, H, T], written by the dQ kernel for the
                         // dK/dV kernel: -D = -rowsum(dO * O), then -lse * log2(e)
  int* err;
};

// consecutive 8-byte mbarriers; after them the TMEM slot and the abort flag
struct Bars {
  uint32_t base;
  __device__ uint32_t operator()(int i) const { return base + 8u * i; }
};

// =====================================================================================
// forward
//   unit = (batch, head, query tiles A = 2 pair and B = 2 pair + 1 of 128 queries each);
//   keys in blocks of 128.
//   shared memory: Q_A, Q_B of two units (double-buffered: the next unit's queries load while
//   this one runs) | K ring | V ring | output staging (8 warps x 32 rows x 128 B)
//   tensor memory: S_A, S_B (fp32, 128 columns each) | P_A, P_B (bf16 pairs, 64 columns
//   each: the A operand of O += P V, read by the MMA from tensor memory) | O_A, O_B (fp32)
constexpr int F_RING = 4;
constexpr int F_SM_Q = 0;                                  // [buf][tile]
constexpr int F_SM_K = F_SM_Q + 4 * TILE;                  // K ring
constexpr int F_SM_V = F_SM_K + F_RING * TILE;             // V ring
constexpr int F_SM_STG = F_SM_V + F_RING * TILE;           // 8 warps x 4 KB
constexpr int F_SM_BAR = F_SM_STG + 8 * 4096;
constexpr int F_SMEM = F_SM_BAR + 512 + 1024;
constexpr uint32_t F_COL_S = 0, F_COL_P = 256, F_COL_O = 384;
enum {
  FB_QFULL = 0,                  // [buf]
  FB_QEMPTY = 2,                 // [buf]
  FB_KFULL = 4,                  // [F_RING]
  FB_KEMPTY = FB_KFULL + F_RING,
  FB_VFULL = FB_KEMPTY + F_RING,
  FB_VEMPTY = FB_VFULL + F_RING,
  FB_SFULL = FB_VEMPTY + F_RING,   // [tile]: S_x computed
  FB_SEMPTY = FB_SFULL + 2,        // [tile]: S_x read out by the tile's four softmax warps
  FB_PFULL = FB_SEMPTY + 2,        // [tile]: P_x written
  FB_ODONE = FB_PFULL + 2,         // [tile]: O_x += P_x V done (P_x free, O_x stable)
  FB_OFREE = FB_ODONE + 2,         // [tile]: the unit's O_x read out
  FB_FINAL = FB_OFREE + 2,
  FB_COUNT
};
static_assert(8 * FB_COUNT + 16 <= 512, "forward barrier area");

struct FwdUnit {
  int b, h, qa, nA, nB;      // tile A = query block qa, tile B = qa + 1 (nB = 0: absent)
};
__device__ __forceinline__ FwdUnit fwd_unit(const Params& p, int u) {
  const int BH = p.B * p.H, npairs = (p.nqb + 1) / 2;
  const int pair = npairs - 1 - u / BH, bh = u % BH;
  FwdUnit w;
  w.b = bh / p.H;
  w.h = bh % p.H;
  w.qa = 2 * pair;
  w.nA = w.qa + 1;
  w.nB = (w.qa + 1 < p.nqb) ? w.qa + 2 : 0;
  return w;
}

// 11 warps: warp 0 TMA producer, warp 1 + x the MMA issuer of query tile x (each tile's
// chain of S, softmax and P V then never waits on the other tile's), warps 3..10 softmax
constexpr int F_THREADS = 352;

__global__ void __launch_bounds__(F_THREADS, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_out,
           const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const Bars bar{base + F_SM_BAR};
  volatile uint32_t* slot_ptr = (volatile uint32_t*)(base_ptr + F_SM_BAR + 8 * FB_COUNT);
  volatile int* abort_flag = (volatile int*)(base_ptr + F_SM_BAR + 8 * FB_COUNT + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // Q, K and V stages are released by both MMA issuers (one commit each)
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(FB_QFULL + i), 1);
      mbar_init(bar(FB_QEMPTY + i), 2);
    }
    for (int s = 0; s < F_RING; ++s) {
      mbar_init(bar(FB_KFULL + s), 1);
      mbar_init(bar(FB_KEMPTY + s), 2);
      mbar_init(bar(FB_VFULL + s), 1);
      mbar_init(bar(FB_VEMPTY + s), 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(FB_SFULL + x), 1);
      mbar_init(bar(FB_SEMPTY + x), 4);
      mbar_init(bar(FB_PFULL + x), 4);
      mbar_init(bar(FB_ODONE + x), 1);
      mbar_init(bar(FB_OFREE + x), 4);
    }
    mbar_init(bar(FB_FINAL), 2);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(bar(FB_COUNT), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot_ptr;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: Q_A, Q_B per unit (double-buffered), then K_j, V_j on
      // their rings
      bool ok = true;
      int uc = 0, kv = 0;
      int nq = 0, nk = 0, nv = 0;   // copies issued per barrier (what an abort waits for)
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++uc) {
        const FwdUnit w = fwd_unit(p, u);
        const int qb = uc & 1;
        if (uc >= 2 && !mbar_wait(bar(FB_QEMPTY + qb), par((uc >> 1) - 1), abort_flag, p.err)) {
          ok = false;
          break;
        }
        ++nq;
        const uint32_t qdst = base + F_SM_Q + 2 * qb * TILE;
        mbar_expect_tx(bar(FB_QFULL + qb), (w.nB ? 2 : 1) * TILE);
        tma_load_3d(qdst, &tm_qkv, bar(FB_QFULL + qb), w.h * D, w.qa * BQ, w.b);
        if (w.nB)
          tma_load_3d(qdst + TILE, &tm_qkv, bar(FB_QFULL + qb), w.h * D, (w.qa + 1) * BQ, w.b);
        const int nkv = w.nB ? w.nB : w.nA;
        for (int j = 0; j < nkv && ok; ++j, ++kv) {
          const int s = kv % F_RING;
          const uint32_t ph = par(kv / F_RING) ^ 1u;
          if (!mbar_wait(bar(FB_KEMPTY + s), ph, abort_flag, p.err)) { ok = false; break; }
          ++nk;
          mbar_expect_tx(bar(FB_KFULL + s), TILE);
          tma_load_3d(base + F_SM_K + s * TILE, &tm_qkv, bar(FB_KFULL + s), p.C + w.h * D, j * BKV, w.b);
          if (!mbar_wait(bar(FB_VEMPTY + s), ph, abort_flag, p.err)) { ok = false; break; }
          ++nv;
          mbar_expect_tx(bar(FB_VFULL + s), TILE);
          tma_load_3d(base + F_SM_V + s * TILE, &tm_qkv, bar(FB_VFULL + s), 2 * p.C + w.h * D, j * BKV, w.b);
        }
      }
      if (!ok) {   // let issued copies land before the block leaves
        for (int i = max(0, nq - 2); i < nq; ++i)
          mbar_wait(bar(FB_QFULL + (i & 1)), par(i >> 1), abort_flag, nullptr, false);
        for (int k = max(0, nk - F_RING); k < nk; ++k)
          mbar_wait(bar(FB_KFULL + k % F_RING), par(k / F_RING), abort_flag, nullptr, false);
        for (int k = max(0, nv - F_RING); k < nv; ++k)
          mbar_wait(bar(FB_VFULL + k % F_RING), par(k / F_RING), abort_flag, nullptr, false);
      }
    }
  } else if (warp <= 2) {
    // ---------------- MMA issuer of tile x (the whole warp runs the loop; one elected lane
    // issues), per key block j: S_x(j) = Q_x K_j^T, then O_x += P_x(j-1) V_{j-1} (P_x read
    // from tensor memory). Every K, V and Q stage gets one release commit from each issuer,
    // also for blocks this tile does not use.
    const int x = warp - 1;
    // every lane waits; the result is made warp-uniform so the lanes never diverge
    auto wait_u = [&](uint32_t b, uint32_t ph) {
      return __all_sync(0xffffffffu, mbar_wait(b, ph, abort_flag, p.err));
    };
    constexpr uint32_t IDESC_S = make_idesc(BQ, BKV, false, false);
    constexpr uint32_t IDESC_O = make_idesc(BQ, D, false, true);
    bool ok = true;
    int uc = 0, kv = 0, gs = 0, gp = 0, uo = 0;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++uc) {
      const FwdUnit w = fwd_unit(p, u);
      const int n = x == 0 ? w.nA : w.nB;
      const int nkv = w.nB ? w.nB : w.nA;
      const int qb = uc & 1;
      if (n > 0 && !wait_u(bar(FB_QFULL + qb), par(uc >> 1))) {
        ok = false;
        break;
      }
      const uint64_t qd = sdesc(base + F_SM_Q + (2 * qb + x) * TILE, 16, 1024);
      for (int j = 0; j <= nkv && ok; ++j) {
        if (j < nkv) {
          const int kb = kv + j, s = kb % F_RING;
          if (j < n) {
            // S_x's columns are free once the softmax warps have read the previous S_x
            if (!wait_u(bar(FB_KFULL + s), par(kb / F_RING)) ||
                (gs > 0 && !wait_u(bar(FB_SEMPTY + x), par(gs - 1)))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t kd = sdesc(base + F_SM_K + s * TILE, 16, 1024);
            if (elect_one()) {
#pragma unroll
              for (int k = 0; k < D / 16; ++k)   // a k step of 16 columns adds 32 bytes (2 units)
                umma_bf16(tmem + F_COL_S + x * BKV, qd + 2 * k, kd + 2 * k, IDESC_S, k > 0 ? 1u : 0u);
              umma_commit(bar(FB_SFULL + x));
            }
            __syncwarp();
            ++gs;
          }
          if (elect_one()) {
            umma_commit(bar(FB_KEMPTY + s));
            if (j == nkv - 1) umma_commit(bar(FB_QEMPTY + qb));
          }
          __syncwarp();
        }
        if (j >= 1) {
          const int jp = j - 1, vb = kv + jp, s = vb % F_RING;
          if (jp < n) {
            if (!wait_u(bar(FB_VFULL + s), par(vb / F_RING)) ||
                !wait_u(bar(FB_PFULL + x), par(gp)) ||
                (jp == 0 && uo > 0 && !wait_u(bar(FB_OFREE + x), par(uo - 1)))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t vd = sdesc(base + F_SM_V + s * TILE, 16384, 1024);
            if (elect_one()) {
#pragma unroll
              for (int k = 0; k < BKV / 16; ++k)   // a k step of 16 keys adds 2048 bytes
                umma_bf16_ts(tmem + F_COL_O + x * D, tmem + F_COL_P + x * 64 + k * 8, vd + 128 * k,
                             IDESC_O, (jp > 0 || k > 0) ? 1u : 0u);
              umma_commit(bar(FB_ODONE + x));
            }
            __syncwarp();
            ++gp;
          }
          if (elect_one()) umma_commit(bar(FB_VEMPTY + s));
          __syncwarp();
        }
      }
      if (!ok) break;
      kv += nkv;
      if (n > 0) ++uo;
    }
    if (elect_one()) {
      umma_commit(bar(FB_FINAL));
      mbar_wait(bar(FB_FINAL), 0, abort_flag, nullptr, false);
    }
    __syncwarp();
  } else {
    // ---------------- softmax: tile x = 0 (warps 3..6) or 1 (warps 7..10); thread = query row
    const int x = (warp - 3) >> 2, q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t s_col = F_COL_S + x * BKV, p_col = F_COL_P + x * 64, o_col = F_COL_O + x * D;
    const uint32_t slice = base + F_SM_STG + (warp - 3) * 4096;
    const float sl2 = rsqrtf((float)D) * LOG2E;
    int g = 0;                                          // S / P blocks of this tile so far
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      const FwdUnit w = fwd_unit(p, u);
      const int n = x == 0 ? w.nA : w.nB;
      if (n == 0) continue;
      const int qblk = w.qa + x;
      const int query = qblk * BQ + r;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j, ++g) {
        ok = mbar_wait(bar(FB_SFULL + x), par(g), abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        // the block's score row (one tensor-memory round trip), then its maximum (causal
        // mask on the diagonal block only) in eight independent chains
        const bool diag = (j == qblk);
        uint32_t sr[4][32];
#pragma unroll
        tmem_ld64_nowait(lane_base + s_col, *reinterpret_cast<uint32_t (*)[64]>(&sr[0][0]));
        tmem_ld64_nowait(lane_base + s_col + 64, *reinterpret_cast<uint32_t (*)[64]>(&sr[2][0]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(FB_SEMPTY + x));
        float mxp[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) mxp[t] = -INFINITY;
        if (diag) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e <= r) mxp[e & 7] = fmaxf(mxp[e & 7], __uint_as_float(sr[c][e]));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) mxp[e & 7] = fmaxf(mxp[e & 7], __uint_as_float(sr[c][e]));
        }
        float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                         fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
        mx *= sl2;
        float alpha = 1.0f;
        if (mx > m + RESCALE_LOG2) {
          alpha = fast_exp2(m - mx);
          m = mx;
        }
        // P_x and O_x are free once the previous O_x += P_x V has completed (it was issued
        // when this tile's previous P was written, so it has had the S wait, the load and the
        // maximum to run)
        if (g >= 1) {
          ok = mbar_wait(bar(FB_ODONE + x), par(g - 1), abort_flag, p.err);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
        }
        // P = exp2(s sl2 - m) as bf16 pairs straight into tensor memory, 32 keys at a time
        // (the scaling on packed fp32 pairs); the row sum in two packed partials
        const float2 sl2x2 = make_float2(sl2, sl2), nm2 = make_float2(-m, -m);
        float2 sp2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 a = __ffma2_rn(make_float2(__uint_as_float(sr[c][2 * e]),
                                                    __uint_as_float(sr[c][2 * e + 1])),
                                        sl2x2, nm2);
            float2 pv = make_float2(fast_exp2(a.x), fast_exp2(a.y));
            if (diag) {
              if (c * 32 + 2 * e > r) pv.x = 0.f;
              if (c * 32 + 2 * e + 1 > r) pv.y = 0.f;
            }
            sp2[e & 1] = __fadd2_rn(sp2[e & 1], pv);
            pk[e] = pack2_bf16(pv.x, pv.y);
          }
          tmem_st16(lane_base + p_col + c * 16, pk);
        }
        l = l * alpha + ((sp2[0].x + sp2[1].x) + (sp2[0].y + sp2[1].y));
        // a moved maximum rescales O (which holds the sum up to the previous block)
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32_nowait(lane_base + o_col + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_base + o_col + c * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(FB_PFULL + x));
      }
      if (!ok) break;
      // the unit's last O_x += P_x V is done: O is final
      ok = mbar_wait(bar(FB_ODONE + x), par(g - 1), abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t o[2][32];
      tmem_ld64_nowait(lane_base + o_col, *reinterpret_cast<uint32_t (*)[64]>(&o[0][0]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(FB_OFREE + x));
      // O / l through this warp's staging slice (free once its previous store has read it),
      // one TMA store of the warp's 32 rows
      if (lane == 0) bulk_wait_read();
      __syncwarp();
      stage_row64(slice, lane, reinterpret_cast<const float*>(o), 1.0f / l);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tm_out, slice, w.h * D, qblk * BQ + q * 32, w.b);
        bulk_commit();
      }
      if (query < p.T) p.lse[((size_t)w.b * p.H + w.h) * p.T + query] = (m + __log2f(l)) * LN2;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
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
// backward: dK, dV
constexpr int K_QD_STAGES = 4;
constexpr int K_SM_KV = 0;                                  // [2 units]: K, V
constexpr int K_SM_QD = K_SM_KV + 4 * TILE;                 // stage s: Q at 2s, dO at 2s+1
constexpr int K_SM_STG = K_SM_QD + 2 * K_QD_STAGES * TILE;  // 8 warps x 2 KB output staging
constexpr int K_SM_LD = K_SM_STG + TILE;                    // stage s: lse[128], D[128]
constexpr int K_SM_BAR = K_SM_LD + K_QD_STAGES * 1024;
constexpr int K_SMEM = K_SM_BAR + 256 + 1024;
enum {
  KB_KVFULL = 0,    // [2]
  KB_KVEMPTY = 2,   // [2]
  KB_QDFULL = 4,    // [K_QD_STAGES]
  KB_QDEMPTY = 4 + K_QD_STAGES,
  KB_SFULL = 4 + 2 * K_QD_STAGES,
  KB_SEMPTY,
  KB_PFULL,
  KB_DONE,
  KB_ACCFREE,
  KB_FINAL,
  KB_COUNT
};

__device__ __forceinline__ void dkv_unit(const Params& p, int u, int& b, int& h, int& kb, int& n) {
  const int BH = p.B * p.H;
  kb = u / BH;                       // ascending: key block 0 has the most query blocks
  const int bh = u % BH;
  b = bh / p.H;
  h = bh % p.H;
  n = p.nqb - kb;
}

// 10 warps: one SM sub-partition holds three of them, so at most 168 registers
__global__ void __launch_bounds__(THREADS, 1)
bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dqkv, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const Bars bar{base + K_SM_BAR};
  volatile uint32_t* slot_ptr = (volatile uint32_t*)(base_ptr + K_SM_BAR + 8 * KB_COUNT);
  volatile int* abort_flag = (volatile int*)(base_ptr + K_SM_BAR + 8 * KB_COUNT + 8);
  const float* sm_ld = reinterpret_cast<const float*>(base_ptr + K_SM_LD);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(KB_KVFULL + i), 1);
      mbar_init(bar(KB_KVEMPTY + i), 1);
    }
    for (int i = 0; i < K_QD_STAGES; ++i) {
      mbar_init(bar(KB_QDFULL + i), 1);
      mbar_init(bar(KB_QDEMPTY + i), 1);
    }
    mbar_init(bar(KB_SFULL), 1);
    mbar_init(bar(KB_SEMPTY), 8);
    mbar_init(bar(KB_PFULL), 8);
    mbar_init(bar(KB_DONE), 1);
    mbar_init(bar(KB_ACCFREE), 8);
    mbar_init(bar(KB_FINAL), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(bar(KB_COUNT), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot_ptr;
  // S^T, dP^T fp32; the dV, dK accumulators; P^T, dS^T as bf16 pairs (the A operands of
  // the dV, dK MMAs, read from tensor memory)
  constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 320, COL_PT = 384,
                     COL_DST = 448;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      int uc = 0, it = 0, nkv = 0;   // nkv: K / V copies issued (what an abort waits for)
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++uc) {
        int b, h, kb, n;
        dkv_unit(p, u, b, h, kb, n);
        const int kbuf = uc & 1;
        if (uc >= 2 && !mbar_wait(bar(KB_KVEMPTY + kbuf), par((uc >> 1) - 1), abort_flag, p.err)) {
          ok = false;
          break;
        }
        ++nkv;
        const uint32_t kdst = base + K_SM_KV + kbuf * 2 * TILE;
        mbar_expect_tx(bar(KB_KVFULL + kbuf), 2 * TILE);
        tma_load_3d(kdst, &tm_qkv, bar(KB_KVFULL + kbuf), p.C + h * D, kb * BKV, b);
        tma_load_3d(kdst + TILE, &tm_qkv, bar(KB_KVFULL + kbuf), 2 * p.C + h * D, kb * BKV, b);
        const size_t bh_t = ((size_t)b * p.H + h) * p.T;
        for (int i = 0; i < n; ++i, ++it) {
          const int s = it % K_QD_STAGES;
          if (!mbar_wait(bar(KB_QDEMPTY + s), par(it / K_QD_STAGES) ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const int qbi = kb + i;
          // lse and D of the block's queries ride with the Q / dO tiles (T % 4 == 0: the
          // row start and the byte count are multiples of 16)
          const uint32_t nb = (uint32_t)min(BQ, p.T - qbi * BQ) * 4u;
          const uint32_t dst = base + K_SM_QD + 2 * s * TILE;
          mbar_expect_tx(bar(KB_QDFULL + s), 2 * TILE + 2 * nb);
          tma_load_3d(dst, &tm_qkv, bar(KB_QDFULL + s), h * D, qbi * BQ, b);
          tma_load_3d(dst + TILE, &tm_do, bar(KB_QDFULL + s), h * D, qbi * BQ, b);
          const size_t bht = (size_t)p.B * p.H * p.T;
          bulk_load(base + K_SM_LD + s * 1024, p.Dbuf + bht + bh_t + (size_t)qbi * BQ, nb,
                    bar(KB_QDFULL + s));
          bulk_load(base + K_SM_LD + s * 1024 + 512, p.Dbuf + bh_t + (size_t)qbi * BQ, nb,
                    bar(KB_QDFULL + s));
        }
      }
      if (!ok) {
        for (int i = max(0, nkv - 2); i < nkv; ++i)
          mbar_wait(bar(KB_KVFULL + (i & 1)), par(i >> 1), abort_flag, nullptr, false);
        for (int k = max(0, it - K_QD_STAGES); k < it; ++k)
          mbar_wait(bar(KB_QDFULL + k % K_QD_STAGES), par(k / K_QD_STAGES), abort_flag, nullptr,
                    false);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: the whole warp runs the loop (waits made warp-uniform, so
    // the operand descriptors stay uniform) and one elected lane issues
    auto wait_u = [&](uint32_t b, uint32_t ph) {
      return __all_sync(0xffffffffu, mbar_wait(b, ph, abort_flag, p.err));
    };
    constexpr uint32_t IDESC_S = make_idesc(BKV, BQ, false, false);
    constexpr uint32_t IDESC_G = make_idesc(BKV, D, false, true);
    bool ok = true;
    int uc = 0, it = 0, gs = 0, gp = 0;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++uc) {
      int b, h, kb, n;
      dkv_unit(p, u, b, h, kb, n);
      const int kbuf = uc & 1;
      const uint64_t kd = sdesc(base + K_SM_KV + kbuf * 2 * TILE, 16, 1024);
      const uint64_t vd = kd + (TILE >> 4);
      if (!wait_u(bar(KB_KVFULL + kbuf), par(uc >> 1))) { ok = false; break; }
      for (int i = 0; i <= n && ok; ++i) {
        // S^T, dP^T of block i (one block ahead of dV, dK of block i - 1)
        if (i < n) {
          const int s = (it + i) % K_QD_STAGES;
          if (!wait_u(bar(KB_QDFULL + s), par((it + i) / K_QD_STAGES)) ||
              (gs >= 1 && !wait_u(bar(KB_SEMPTY), par(gs - 1)))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t qd = sdesc(base + K_SM_QD + 2 * s * TILE, 16, 1024);
          const uint64_t dd = qd + (TILE >> 4);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {   // a k step of 16 columns adds 32 bytes
              umma_bf16(tmem + COL_S, kd + 2 * k, qd + 2 * k, IDESC_S, k > 0 ? 1u : 0u);
              umma_bf16(tmem + COL_DP, vd + 2 * k, dd + 2 * k, IDESC_S, k > 0 ? 1u : 0u);
            }
            umma_commit(bar(KB_SFULL));
          }
          __syncwarp();
          ++gs;
        }
        if (i >= 1) {
          const int ib = i - 1, s = (it + ib) % K_QD_STAGES;
          if (!wait_u(bar(KB_PFULL), par(gp)) ||
              (ib == 0 && uc >= 1 && !wait_u(bar(KB_ACCFREE), par(uc - 1)))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t qg = sdesc(base + K_SM_QD + 2 * s * TILE, 16384, 1024);
          const uint64_t dg = qg + (TILE >> 4);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < BQ / 16; ++k) {   // a k step of 16 queries adds 2048 bytes
              umma_bf16_ts(tmem + COL_DV, tmem + COL_PT + k * 8, dg + 128 * k, IDESC_G,
                           (ib > 0 || k > 0) ? 1u : 0u);
              umma_bf16_ts(tmem + COL_DK, tmem + COL_DST + k * 8, qg + 128 * k, IDESC_G,
                           (ib > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit(bar(KB_DONE));
            umma_commit(bar(KB_QDEMPTY + s));
          }
          __syncwarp();
          ++gp;
        }
      }
      if (!ok) break;
      it += n;
      if (elect_one()) umma_commit(bar(KB_KVEMPTY + kbuf));
      __syncwarp();
    }
    if (elect_one()) {
      umma_commit(bar(KB_FINAL));
      mbar_wait(bar(KB_FINAL), 0, abort_flag, nullptr, false);
    }
    __syncwarp();
  } else {
    // ---------------- elementwise: key row r, query columns c0 .. c0 + 63
    const int q = warp & 3, half = (warp - 2) >> 2;
    const int r = q * 32 + lane, c0 = half * 64;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    // this warp's output staging slice (32 rows x 32 columns bf16), dK then dV
    const uint32_t slice = base + K_SM_STG + (warp - 2) * 2048;
    const float sl2 = rsqrtf((float)D) * LOG2E;
    int it = 0, g = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      int b, h, kb, n;
      dkv_unit(p, u, b, h, kb, n);
      const int key = kb * BKV + r;
      for (int i = 0; i < n; ++i, ++it, ++g) {
        const int s = it % K_QD_STAGES;
        ok = mbar_wait(bar(KB_QDFULL + s), par(it / K_QD_STAGES), abort_flag, p.err) &&
             mbar_wait(bar(KB_SFULL), par(g), abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const float4* lse4 = reinterpret_cast<const float4*>(sm_ld + s * 256 + c0);
        const float4* D4 = reinterpret_cast<const float4*>(sm_ld + s * 256 + 128 + c0);
        const int q0 = (kb + i) * BQ + c0;              // first query of these columns
        // P^T and dS^T of 64 query columns, 32 at a time (S^T, dP^T released after the
        // second load), each chunk stored as soon as it is computed; the mask (causal on
        // the diagonal block, past T on the last) only in the blocks that need it
        uint32_t sv[2][32], dv[2][32];
        tmem_ld64_nowait(lane_base + COL_S + c0, *reinterpret_cast<uint32_t (*)[64]>(&sv[0][0]));
        tmem_ld64_nowait(lane_base + COL_DP + c0, *reinterpret_cast<uint32_t (*)[64]>(&dv[0][0]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KB_SEMPTY));
        // per query column: -lse log2(e) and -D (stored pre-negated by the dQ kernel), so
        // P = exp2(s sl2 - lse log2 e) is one fma and dS = P (dP - D) an add and a multiply,
        // each on packed fp32 pairs
        auto chunk = [&](int c, auto masked_tag) -> bool {
          constexpr bool MASKED = decltype(masked_tag)::value;
          uint32_t pk[16], dk[16];
          const float2 sl2x2 = make_float2(sl2, sl2);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 L = lse4[c * 8 + e4], Dd = D4[c * 8 + e4];
            const float2 lv[2] = {make_float2(L.x, L.y), make_float2(L.z, L.w)};
            const float2 dd[2] = {make_float2(Dd.x, Dd.y), make_float2(Dd.z, Dd.w)};
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int e = e4 * 4 + 2 * t;
              const float2 a = __ffma2_rn(
                  make_float2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), sl2x2, lv[t]);
              float2 pv = make_float2(fast_exp2(a.x), fast_exp2(a.y));
              float2 dsv = __fmul2_rn(
                  pv, __fadd2_rn(make_float2(__uint_as_float(dv[c][e]), __uint_as_float(dv[c][e + 1])),
                                 dd[t]));
              if (MASKED) {
                // past T the lse / D entries were never loaded: zero both results outright
                const int query = q0 + c * 32 + e;
                if (query < key || query >= p.T) { pv.x = 0.f; dsv.x = 0.f; }
                if (query + 1 < key || query + 1 >= p.T) { pv.y = 0.f; dsv.y = 0.f; }
              }
              pk[e4 * 2 + t] = pack2_bf16(pv.x, pv.y);
              dk[e4 * 2 + t] = pack2_bf16(dsv.x, dsv.y);
            }
          }
          if (c == 0) {
            // the previous block's dV, dK MMAs have read P^T, dS^T from tensor memory (for
            // the first block of a unit, the previous unit's last block)
            if (g >= 1) {
              const bool w_ok = mbar_wait(bar(KB_DONE), par(g - 1), abort_flag, p.err);
              if (!__all_sync(0xffffffffu, w_ok)) return false;
            }
          }
          tmem_st16(lane_base + COL_PT + half * 32 + c * 16, pk);
          tmem_st16(lane_base + COL_DST + half * 32 + c * 16, dk);
          return true;
        };
        if (i == 0 || q0 + 64 > p.T) {
          ok = chunk(0, std::true_type{}) && chunk(1, std::true_type{});
        } else {
          ok = chunk(0, std::false_type{}) && chunk(1, std::false_type{});
        }
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(KB_PFULL));
      }
      if (!ok) break;
      ok = mbar_wait(bar(KB_DONE), par(g - 1), abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t kv2[2][32];
      tmem_ld32_nowait(lane_base + COL_DK + half * 32, kv2[0]);
      tmem_ld32_nowait(lane_base + COL_DV + half * 32, kv2[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(KB_ACCFREE));
      // dK, then dV, through the warp's 2 KB slice (free once the previous store read it)
      const int row = kb * BKV + q * 32;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (lane == 0) bulk_wait_read();
        __syncwarp();
        stage_row32(slice, lane, reinterpret_cast<const float*>(kv2[t]),
                    t == 0 ? rsqrtf((float)D) : 1.0f);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tm_dqkv, slice, (t == 0 ? p.C : 2 * p.C) + h * D + half * 32, row, b);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
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
// backward: dQ (and D)
constexpr int Q_KV_STAGES = 4;
constexpr int Q_SM_QD = 0;                                   // [2 units]: Q, dO
constexpr int Q_SM_KV = Q_SM_QD + 4 * TILE;                  // stage s: K at 2s, V at 2s+1
constexpr int Q_SM_STG = Q_SM_KV + 2 * Q_KV_STAGES * TILE;   // 8 warps x 2 KB output staging
constexpr int Q_SM_O = Q_SM_STG + TILE;                      // the unit's O rows (for D)
constexpr int Q_SM_BAR = Q_SM_O + TILE;
constexpr int Q_SMEM = Q_SM_BAR + 256 + 1024;
enum {
  QB_QFULL = 0,     // [2]
  QB_QEMPTY = 2,    // [2]
  QB_KVFULL = 4,    // [Q_KV_STAGES]
  QB_KVEMPTY = 4 + Q_KV_STAGES,
  QB_SFULL = 4 + 2 * Q_KV_STAGES,
  QB_SEMPTY,
  QB_PFULL,
  QB_DONE,          // [2]: one per dS buffer
  QB_ACCFREE = QB_DONE + 2,
  QB_FINAL,
  QB_OFULL,
  QB_OEMPTY,
  QB_COUNT
};

__device__ __forceinline__ void dq_unit(const Params& p, int u, int& b, int& h, int& qb, int& n) {
  const int BH = p.B * p.H;
  qb = p.nqb - 1 - u / BH;           // descending: the last query block has the most keys
  const int bh = u % BH;
  b = bh / p.H;
  h = bh % p.H;
  n = qb + 1;
}

// 10 warps: one SM sub-partition holds three of them, so at most 168 registers
__global__ void __launch_bounds__(THREADS, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_dqkv,
              const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const Bars bar{base + Q_SM_BAR};
  volatile uint32_t* slot_ptr = (volatile uint32_t*)(base_ptr + Q_SM_BAR + 8 * QB_COUNT);
  volatile int* abort_flag = (volatile int*)(base_ptr + Q_SM_BAR + 8 * QB_COUNT + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) { mbar_init(bar(QB_QFULL + i), 1); mbar_init(bar(QB_QEMPTY + i), 1); }
    for (int s = 0; s < Q_KV_STAGES; ++s) {
      mbar_init(bar(QB_KVFULL + s), 1);
      mbar_init(bar(QB_KVEMPTY + s), 1);
    }
    mbar_init(bar(QB_SFULL), 1);
    mbar_init(bar(QB_SEMPTY), 8);
    mbar_init(bar(QB_PFULL), 8);
    mbar_init(bar(QB_DONE), 1);
    mbar_init(bar(QB_DONE + 1), 1);
    mbar_init(bar(QB_ACCFREE), 8);
    mbar_init(bar(QB_FINAL), 1);
    mbar_init(bar(QB_OFULL), 1);
    mbar_init(bar(QB_OEMPTY), 8);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(bar(QB_COUNT), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot_ptr;
  // S, dP fp32; the dQ accumulator; dS as bf16 pairs, double-buffered (the A operand of the
  // dQ MMA, read from tensor memory)
  constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DQ = 256, COL_DS = 320;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      int uc = 0, kv = 0, n_q = 0, n_o = 0;   // n_q, n_o: Q / dO and O copies issued
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++uc) {
        int b, h, qb, n;
        dq_unit(p, u, b, h, qb, n);
        const int qbuf = uc & 1;
        if (uc >= 2 && !mbar_wait(bar(QB_QEMPTY + qbuf), par((uc >> 1) - 1), abort_flag, p.err)) {
          ok = false;
          break;
        }
        ++n_q;
        const uint32_t qdst = base + Q_SM_QD + qbuf * 2 * TILE;
        mbar_expect_tx(bar(QB_QFULL + qbuf), 2 * TILE);
        tma_load_3d(qdst, &tm_qkv, bar(QB_QFULL + qbuf), h * D, qb * BQ, b);
        tma_load_3d(qdst + TILE, &tm_do, bar(QB_QFULL + qbuf), h * D, qb * BQ, b);
        // O rows of the unit (D), once the elementwise warps have read the previous unit's
        if (uc >= 1 && !mbar_wait(bar(QB_OEMPTY), par(uc - 1), abort_flag, p.err)) {
          ok = false;
          break;
        }
        mbar_expect_tx(bar(QB_OFULL), TILE);
        tma_load_3d(base + Q_SM_O, &tm_o, bar(QB_OFULL), h * D, qb * BQ, b);
        ++n_o;
        for (int j = 0; j < n; ++j, ++kv) {
          const int s = kv % Q_KV_STAGES;
          if (!mbar_wait(bar(QB_KVEMPTY + s), par(kv / Q_KV_STAGES) ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t dst = base + Q_SM_KV + 2 * s * TILE;
          mbar_expect_tx(bar(QB_KVFULL + s), 2 * TILE);
          tma_load_3d(dst, &tm_qkv, bar(QB_KVFULL + s), p.C + h * D, j * BKV, b);
          tma_load_3d(dst + TILE, &tm_qkv, bar(QB_KVFULL + s), 2 * p.C + h * D, j * BKV, b);
        }
      }
      if (!ok) {
        for (int i = max(0, n_q - 2); i < n_q; ++i)   // the last two units' Q / dO copies
          mbar_wait(bar(QB_QFULL + (i & 1)), par(i >> 1), abort_flag, nullptr, false);
        if (n_o > 0) mbar_wait(bar(QB_OFULL), par(n_o - 1), abort_flag, nullptr, false);
        for (int k = max(0, kv - Q_KV_STAGES); k < kv; ++k)
          mbar_wait(bar(QB_KVFULL + k % Q_KV_STAGES), par(k / Q_KV_STAGES), abort_flag, nullptr,
                    false);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: the whole warp runs the loop (waits made warp-uniform, so
    // the operand descriptors stay uniform) and one elected lane issues
    auto wait_u = [&](uint32_t b, uint32_t ph) {
      return __all_sync(0xffffffffu, mbar_wait(b, ph, abort_flag, p.err));
    };
    constexpr uint32_t IDESC_S = make_idesc(BQ, BKV, false, false);
    constexpr uint32_t IDESC_G = make_idesc(BQ, D, false, true);
    bool ok = true;
    int uc = 0, kv = 0, gs = 0, gp = 0;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++uc) {
      int b, h, qb, n;
      dq_unit(p, u, b, h, qb, n);
      const int qbuf = uc & 1;
      const uint64_t qd = sdesc(base + Q_SM_QD + qbuf * 2 * TILE, 16, 1024);
      const uint64_t dd = qd + (TILE >> 4);
      if (!wait_u(bar(QB_QFULL + qbuf), par(uc >> 1))) { ok = false; break; }
      for (int j = 0; j <= n && ok; ++j) {
        if (j < n) {
          const int s = (kv + j) % Q_KV_STAGES;
          if (!wait_u(bar(QB_KVFULL + s), par((kv + j) / Q_KV_STAGES)) ||
              (gs >= 1 && !wait_u(bar(QB_SEMPTY), par(gs - 1)))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = sdesc(base + Q_SM_KV + 2 * s * TILE, 16, 1024);
          const uint64_t vd = kd + (TILE >> 4);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {   // a k step of 16 columns adds 32 bytes
              umma_bf16(tmem + COL_S, qd + 2 * k, kd + 2 * k, IDESC_S, k > 0 ? 1u : 0u);
              umma_bf16(tmem + COL_DP, dd + 2 * k, vd + 2 * k, IDESC_S, k > 0 ? 1u : 0u);
            }
            umma_commit(bar(QB_SFULL));
          }
          __syncwarp();
          ++gs;
        }
        if (j >= 1) {
          const int jb = j - 1, s = (kv + jb) % Q_KV_STAGES;
          if (!wait_u(bar(QB_PFULL), par(gp)) ||
              (jb == 0 && uc >= 1 && !wait_u(bar(QB_ACCFREE), par(uc - 1)))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kg = sdesc(base + Q_SM_KV + 2 * s * TILE, 16384, 1024);
          const uint32_t ds = tmem + COL_DS + (uint32_t)(gp & 1) * 64;
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < BKV / 16; ++k)   // a k step of 16 keys adds 2048 bytes
              umma_bf16_ts(tmem + COL_DQ, ds + k * 8, kg + 128 * k, IDESC_G,
                           (jb > 0 || k > 0) ? 1u : 0u);
            umma_commit(bar(QB_DONE + (gp & 1)));
            umma_commit(bar(QB_KVEMPTY + s));
          }
          __syncwarp();
          ++gp;
        }
      }
      if (!ok) break;
      kv += n;
      if (elect_one()) umma_commit(bar(QB_QEMPTY + qbuf));
      __syncwarp();
    }
    if (elect_one()) {
      umma_commit(bar(QB_FINAL));
      mbar_wait(bar(QB_FINAL), 0, abort_flag, nullptr, false);
    }
    __syncwarp();
  } else {
    // ---------------- elementwise: query row r, key columns c0 .. c0 + 63
    const int q = warp & 3, half = (warp - 2) >> 2;
    const int r = q * 32 + lane, c0 = half * 64;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t slice = base + Q_SM_STG + (warp - 2) * 2048;   // output staging
    const float sl2 = rsqrtf((float)D) * LOG2E;
    int g = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++uc) {
      int b, h, qb, n;
      dq_unit(p, u, b, h, qb, n);
      const int query = qb * BQ + r;
      const size_t t = ((size_t)b * p.H + h) * p.T + query;
      const float nlse2 = query < p.T ? -__ldg(p.lse + t) * LOG2E : 0.f;
      // D = rowsum(dO * O) of this thread's query row, from the unit's dO and O tiles
      // (rows past T were loaded as zeros); both warps of a row compute the same value
      const int qbuf = uc & 1;
      ok = mbar_wait(bar(QB_QFULL + qbuf), par(uc >> 1), abort_flag, p.err) &&
           mbar_wait(bar(QB_OFULL), par(uc), abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      float Dr = 0.f;
      {
        const uint32_t drow = base + Q_SM_QD + (2 * qbuf + 1) * TILE + r * 128;
        const uint32_t orow = base + Q_SM_O + r * 128;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint32_t off = (uint32_t)((v ^ (r & 7)) << 4);
          const uint4 x = ld_shared16(drow + off), y = ld_shared16(orow + off);
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 a = bf2_to_f2(xs[e]), c = bf2_to_f2(ys[e]);
            Dr = fmaf(a.x, c.x, Dr);
            Dr = fmaf(a.y, c.y, Dr);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(QB_OEMPTY));
      if (half == 0 && query < p.T) {   // for the dK/dV kernel, pre-negated
        p.Dbuf[t] = -Dr;
        p.Dbuf[(size_t)p.B * p.H * p.T + t] = nlse2;
      }
      for (int j = 0; j < n; ++j, ++g) {
        ok = mbar_wait(bar(QB_SFULL), par(g), abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[2][32], dv[2][32];
        tmem_ld64_nowait(lane_base + COL_S + c0, *reinterpret_cast<uint32_t (*)[64]>(&sv[0][0]));
        tmem_ld64_nowait(lane_base + COL_DP + c0, *reinterpret_cast<uint32_t (*)[64]>(&dv[0][0]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_SEMPTY));
        const int k0 = j * BKV + c0;
        uint32_t dk[32];
        // dS = exp2(s sl2 - lse log2 e) (dP - D) on packed fp32 pairs; the causal mask on
        // the diagonal block only
        const float2 sl2x2 = make_float2(sl2, sl2), nl2 = make_float2(nlse2, nlse2);
        const float2 nD2 = make_float2(-Dr, -Dr);
        auto compute = [&](auto masked_tag) {
          constexpr bool MASKED = decltype(masked_tag)::value;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 a = __ffma2_rn(
                  make_float2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), sl2x2, nl2);
              float2 pv = make_float2(fast_exp2(a.x), fast_exp2(a.y));
              if (MASKED) {
                if (k0 + c * 32 + e > query) pv.x = 0.f;
                if (k0 + c * 32 + e + 1 > query) pv.y = 0.f;
              }
              const float2 ds = __fmul2_rn(
                  pv, __fadd2_rn(make_float2(__uint_as_float(dv[c][e]), __uint_as_float(dv[c][e + 1])),
                                 nD2));
              dk[c * 16 + e / 2] = pack2_bf16(ds.x, ds.y);
            }
          }
        };
        if (j == qb) compute(std::true_type{});
        else compute(std::false_type{});
        // dS buffer g & 1 was last read by the dQ MMAs of block g - 2
        if (g >= 2) {
          ok = mbar_wait(bar(QB_DONE + (g & 1)), par((g >> 1) - 1), abort_flag, p.err);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        }
        {
          const uint32_t dst = lane_base + COL_DS + (uint32_t)(g & 1) * 64 + half * 32;
          uint32_t lo[16], hi[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) { lo[e] = dk[e]; hi[e] = dk[16 + e]; }
          tmem_st16(dst, lo);
          tmem_st16(dst + 16, hi);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QB_PFULL));
      }
      if (!ok) break;
      ok = mbar_wait(bar(QB_DONE + ((g - 1) & 1)), par((g - 1) >> 1), abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32_nowait(lane_base + COL_DQ + half * 32, v);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(QB_ACCFREE));
      if (lane == 0) bulk_wait_read();   // the slice's previous store has read it
      __syncwarp();
      stage_row32(slice, lane, reinterpret_cast<const float*>(v), rsqrtf((float)D));
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tm_dqkv, slice, h * D + half * 32, qb * BQ + q * 32, b);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
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
// [B][T][width] bf16 as a 3-D map {width, T, B}, box {box_w, box_rows, 1}
static bool map_btw(CUtensorMap* m, const void* ptr, int B, int T, int width, int box_w,
                    int box_rows, CUtensorMapSwizzle swz) {
  auto fn = tensor_map_encoder();
  if (!fn || ((uintptr_t)ptr & 15u) || (width * 2) % 16) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)T * width * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_w, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

}  // namespace fatc

cudaError_t attention_forward_tc(void* out, float* lse, const void* qkv, int B, int T, int C,
                                 int H, int* err, cudaStream_t s) {
  using namespace fatc;
  if (C / H != D || C % H || C % 64 || B <= 0 || T <= 0) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         F_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap mq, mo;
  if (!map_btw(&mq, qkv, B, T, 3 * C, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !map_btw(&mo, out, B, T, C, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  Params p;
  p.B = B; p.T = T; p.H = H; p.C = C; p.nqb = ceil_div(T, BQ);
  p.units = B * H * ((p.nqb + 1) / 2);
  p.lse = lse; p.Dbuf = nullptr; p.err = err;
  const int grid = std::min(p.units, num_sms());
  fwd_kernel<<<grid, F_THREADS, F_SMEM, s>>>(mq, mo, p);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t attention_backward_tc(void* dqkv, float* Dbuf, const void* dout, const void* out,
                                  const void* qkv, const float* lse, int B, int T, int C, int H,
                                  int* err, cudaStream_t s) {
  using namespace fatc;
  if (C / H != D || C % H || C % 64 || B <= 0 || T <= 0 || T % 4 || ((uintptr_t)lse & 15u) ||
      ((uintptr_t)Dbuf & 15u))
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(bwd_dkv_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, K_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Q_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap mq, md, mo, mg;
  if (!map_btw(&mq, qkv, B, T, 3 * C, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !map_btw(&md, dout, B, T, C, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !map_btw(&mo, out, B, T, C, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !map_btw(&mg, dqkv, B, T, 3 * C, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  Params p;
  p.B = B; p.T = T; p.H = H; p.C = C; p.nqb = ceil_div(T, BQ);
  p.units = B * H * p.nqb;
  p.lse = const_cast<float*>(lse); p.Dbuf = Dbuf; p.err = err;
  const int grid = std::min(p.units, num_sms());
  // dQ first: it computes D = rowsum(dO * O), which the dK/dV kernel reads
  bwd_dq_kernel<<<grid, THREADS, Q_SMEM, s>>>(mq, md, mo, mg, p);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_dkv_kernel<<<grid, THREADS, K_SMEM, s>>>(mq, md, mg, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace gpt2k

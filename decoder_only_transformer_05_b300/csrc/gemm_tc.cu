// bf16 GEMM on the 5th-generation tensor cores (tcgen05) for sm_103a, with the training
// step's fused epilogues (bias, residual add, tanh-GELU and its derivative, fp32
// gradient accumulation).
//
// C(m, n) = sum_k A(m, k) B(n, k); each operand is K-major (k contiguous) or MN-major
// (m or n contiguous). Forward GEMMs are K-major x K-major, dgrad GEMMs K-major x
// MN-major, wgrad GEMMs MN-major x MN-major.
//
// Structure (one persistent block of 320 threads per SM, blocks paired in clusters of 2; a
// work unit is two vertically adjacent 128 x BN output tiles, one per block):
//   warp 0      TMA producer (both blocks): the block's 128 x 64 rows of A and its half
//               (BN/2 x 64) of the B tile, 128-byte swizzle, into a ring of shared-memory
//               stages; both blocks' bytes complete on the even block's full barrier.
//   warp 1      MMA issuer (one thread of the even block): tcgen05.mma.cta_group::2 with
//               M = 256, N = BN, K = 16 reads the A rows and the B half each block holds and
//               writes each block's 128 rows of the fp32 accumulator into that block's
//               tensor memory; its commits free a stage, or hand over an accumulator, in both
//               blocks at once. Two accumulators alternate so the epilogue of one tile
//               overlaps the main loop of the next. Each block holds only half of B, which
//               cuts the shared-memory operand bytes per FLOP by a third against one block
//               per tile.
//   warps 2..9  epilogue (both blocks): warp w reads TMEM lanes 32*(w%4).. (the rows of its
//               quarter), warps w and w+4 take alternate 64-column steps of the tile. Per
//               step: the bias and input rows (loaded first), one tcgen05.ld of 64 columns,
//               the epilogue arithmetic on packed fp32 pairs in two 32-column halves, the
//               result into a swizzled shared-memory staging slot (128-byte rows), then one
//               TMA bulk-tensor store per output (for gradient accumulation, two 32-column
//               TMA bulk-tensor reduce-adds). The epilogue warps of both blocks arrive on
//               the even block's barrier when an accumulator is free again.
// Every mbarrier wait is bounded: on timeout the block records DEV_ERR_TIMEOUT, stops
// issuing work, waits for its own copies and MMAs and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace gpt2k {
namespace tc {

constexpr int BM = 128, BK = 64;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;

// XS: the epilogue has a second bf16 output or a TMA-loaded input, so each epilogue warp
// stages 2 x 4 KB (and the operand ring has one stage fewer)
template <int BN, bool XS> struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;         // 16 KB: this block's 128 rows of A
  static constexpr int B_BYTES = (BN / 2) * BK * 2;   // this block's half of the B tile
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? (XS ? 5 : 6) : (XS ? 6 : 8);   // 144-192 KB in flight
  static constexpr int STG = XS ? 8192 : 4096;        // per epilogue warp: 32 rows x 128 B (x 2)
  static constexpr int TMEM_COLS = 2 * BN;            // two accumulators
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = STAGES * STAGE + EPI_WARPS * STG + 1024 + BAR_BYTES;
};

struct Params {
  int M, N, K;
  int num_m, num_n, splits, kb_per_split, num_kb;
  int epi;
  int n_fast;     // unit order: column tile fastest (few column tiles: the tiles that share
                  // a row block of A run at the same time, so A streams from DRAM once)
  int defer;      // split partials: 0 = summed into accum after the kernel, 1 = added into
                  // the workspace, which the caller folds in later
  long long ldo;
  const bf16* bias; const bf16* resid; const bf16* aux;
  float scale;
  int* err;
  int vocab; float* ce_part;    // EPI_LOGITS_CE
  unsigned long long wait_ns;   // limit of every bounded wait (normally TIMEOUT_NS)
  int drop_first_signal;        // test hook: the first accumulator of each block pair is
                                // never signalled ready, so its epilogue wait runs out
};

// ------------------------------------------------------------------ epilogue
// One step of an epilogue warp: its 32 rows (thread = row0 + lane) x 64 columns
// [col0, col0 + 64); `acc` holds the 64 accumulator values of the row (the tensor-memory load
// complete). The two 32-column halves are handled in turn (bias, input rows, arithmetic on
// packed fp32 pairs, staging); then lane 0 stores the step with one TMA store per output
// (a 32 x 64 bf16 box, 128-byte rows), or, for gradient accumulation, two fp32 32 x 32
// reduce-adds through the slot one after the other.
struct EpiMaps {
  CUtensorMap out;   // bf16 [M, N] (box 64 x 32, 128-byte swizzle) or fp32 [M, N] / [splits, M, N] (box 32 x 32)
  CUtensorMap pre;   // bf16 [M, N]: the second output of EPI_GELU_FWD / _FWD_U / _BWD_U
  CUtensorMap in;    // bf16 [M, N] gelu'(u) rows, EPI_GELU_BWD only
};

// 16-byte units 4h .. 4h+3 of row r of a 32 x 64 bf16 tile (128 B per row), laid out for a TMA
// map with 128-byte swizzle: unit j of row r at unit j ^ (r & 7).
__device__ __forceinline__ void stage_half_bf16(uint32_t buf, int r, int h, const uint32_t (&w)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared16(buf + r * 128 + (((4 * h + j) ^ (r & 7)) << 4),
                make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]));
}

// stg: the warp's staging slot (out in the first 4 KB, the second output in the second).
// inr: the row's 64 input values (residual, gelu'(u) or u; zeros if none) and bia: the 64
// bias values, both loaded before the accumulator so that their latency overlaps it.
__device__ __forceinline__ void epilogue_step(const Params& p, const EpiMaps& maps, int row0,
                                              int col0, int split, uint32_t stg,
                                              const uint32_t (&acc)[64], const uint32_t (&inr)[32],
                                              const uint4 (&bia)[8], float& ce_m, float& ce_s) {
  const int lane = threadIdx.x & 31;
  if (p.epi == EPI_ACCUM) {
    const float s = (p.splits == 1 || p.defer) ? p.scale : 1.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (lane == 0) bulk_wait_read();   // the slot's previous stores have read it
      __syncwarp();
      float f[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(acc[32 * h + i]);
      stage_row_f32(stg, lane, f, s);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        if (row0 < p.M) {   // stores start in range; TMA clips the rest
          if (p.splits == 1) tma_reduce_add_2d(&maps.out, stg, col0 + 32 * h, row0);
          else if (p.defer) tma_reduce_add_3d(&maps.out, stg, col0 + 32 * h, row0, split);
          else tma_store_3d(&maps.out, stg, col0 + 32 * h, row0, split);
        }
        bulk_commit();
      }
    }
    return;
  }
  const bool two = p.epi == EPI_GELU_FWD || p.epi == EPI_GELU_FWD_U || p.epi == EPI_GELU_BWD_U;
  const bool src = p.epi == EPI_GELU_BWD || p.epi == EPI_GELU_BWD_U || (p.epi == EPI_STORE && p.resid);
  if (lane == 0) bulk_wait_read();   // the slot's previous stores have read it
  __syncwarp();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c0 = col0 + 32 * h;
    float2 v[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      v[e] = make_float2(__uint_as_float(acc[32 * h + 2 * e]), __uint_as_float(acc[32 * h + 2 * e + 1]));
    if (p.bias) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 b4 = bia[4 * h + i];
        v[4 * i] = __fadd2_rn(v[4 * i], bf2_to_f2(b4.x));
        v[4 * i + 1] = __fadd2_rn(v[4 * i + 1], bf2_to_f2(b4.y));
        v[4 * i + 2] = __fadd2_rn(v[4 * i + 2], bf2_to_f2(b4.z));
        v[4 * i + 3] = __fadd2_rn(v[4 * i + 3], bf2_to_f2(b4.w));
      }
    }
    uint32_t in[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) in[e] = inr[16 * h + e];
    uint32_t w[16];
    if (p.epi == EPI_STORE || p.epi == EPI_LOGITS_CE) {
      if (src) {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __fadd2_rn(v[e], bf2_to_f2(in[e]));
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = pack2_bf16(v[e].x, v[e].y);
      if (p.epi == EPI_LOGITS_CE) {
        // softmax statistics of the rounded logits of this half's columns < vocab, merged
        // into the running (ce_m, ce_s) of the thread's row (log2 domain); the column mask
        // only in a half that reaches past vocab
        constexpr float L2E = 1.4426950408889634f;
        float2 z[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) z[e] = bf2_to_f2(w[e]);
        if (c0 + 32 > p.vocab) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            if (c0 + 2 * e >= p.vocab) z[e].x = -INFINITY;
            if (c0 + 2 * e + 1 >= p.vocab) z[e].y = -INFINITY;
          }
        }
        float zm0 = fmaxf(z[0].x, z[0].y), zm1 = fmaxf(z[1].x, z[1].y);
#pragma unroll
        for (int e = 2; e < 16; e += 2) {
          zm0 = fmaxf(zm0, fmaxf(z[e].x, z[e].y));
          zm1 = fmaxf(zm1, fmaxf(z[e + 1].x, z[e + 1].y));
        }
        const float zm = fmaxf(zm0, zm1);
        if (zm != -INFINITY) {
          const float cm = zm * L2E;
          const float2 l2e2 = make_float2(L2E, L2E), ncm = make_float2(-cm, -cm);
          float2 cs2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 a = __ffma2_rn(z[e], l2e2, ncm);
            cs2 = __fadd2_rn(cs2, make_float2(fast_exp2(a.x), fast_exp2(a.y)));
          }
          const float cs = cs2.x + cs2.y;
          const float mn = fmaxf(ce_m, cm);
          ce_s = ce_s * fast_exp2(ce_m - mn) + cs * fast_exp2(cm - mn);
          ce_m = mn;
        }
      }
    } else if (p.epi == EPI_GELU_FWD) {
      uint32_t u[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float2 d;
        const float2 g = gelu_tanh_and_grad_fast2(v[e], d);
        u[e] = pack2_bf16(d.x, d.y);
        w[e] = pack2_bf16(g.x, g.y);
      }
      stage_half_bf16(stg + 4096, lane, h, u);
    } else if (p.epi == EPI_GELU_FWD_U) {   // keep u itself for the recomputing backward
      uint32_t u[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float2 d;
        const float2 g = gelu_tanh_and_grad_fast2(v[e], d);
        u[e] = pack2_bf16(v[e].x, v[e].y);
        w[e] = pack2_bf16(g.x, g.y);
      }
      stage_half_bf16(stg + 4096, lane, h, u);
    } else if (p.epi == EPI_GELU_BWD_U) {   // gelu'(u) and gelu(u) recomputed from u
      uint32_t gu[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float2 d;
        const float2 g = gelu_tanh_and_grad_fast2(bf2_to_f2(in[e]), d);
        const float2 o = __fmul2_rn(v[e], d);
        w[e] = pack2_bf16(o.x, o.y);
        gu[e] = pack2_bf16(g.x, g.y);
      }
      stage_half_bf16(stg + 4096, lane, h, gu);
    } else {   // EPI_GELU_BWD
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float2 g = __fmul2_rn(v[e], bf2_to_f2(in[e]));
        w[e] = pack2_bf16(g.x, g.y);
      }
    }
    stage_half_bf16(stg, lane, h, w);
  }
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    if (row0 < p.M) {   // stores start in range; TMA clips the rest
      tma_store_2d(&maps.out, stg, col0, row0);
      if (two) tma_store_2d(&maps.pre, stg + 4096, col0, row0);
    }
    bulk_commit();
  }
}

// ------------------------------------------------------------------ kernel
template <int BN, bool AMN, bool BMN, bool XS>
__global__ void __launch_bounds__(THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ EpiMaps maps, const Params p) {
  using Cf = Cfg<BN, XS>;
  // the pair MMA: M = 256 (128 rows per block), N = BN
  constexpr uint32_t IDESC = make_idesc(2 * BM, BN, AMN, BMN);
  constexpr uint16_t PAIR = 0x3;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t staging = base + Cf::STAGES * Cf::STAGE;
  const uint32_t bars = staging + EPI_WARPS * Cf::STG;
  uint8_t* bars_ptr = base_ptr + Cf::STAGES * Cf::STAGE + EPI_WARPS * Cf::STG;
  // barrier layout (the same in both blocks): full[S] empty[S] tfull[2] tempty[2] final,
  // then the tmem slot and the abort flag. full, tempty and final are used in the even
  // (MMA-issuing) block only.
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (Cf::STAGES + s); };
  auto tfull = [&](int a) { return bars + 8u * (2 * Cf::STAGES + a); };
  auto tempty = [&](int a) { return bars + 8u * (2 * Cf::STAGES + 2 + a); };
  const uint32_t final_bar = bars + 8u * (2 * Cf::STAGES + 4);
  auto in_bar = [&](int ew) { return bars + 8u * (2 * Cf::STAGES + 7 + ew); };   // epilogue inputs
  const uint32_t slot = bars + 8u * (2 * Cf::STAGES + 5);
  volatile uint32_t* slot_ptr = (volatile uint32_t*)(bars_ptr + 8 * (2 * Cf::STAGES + 5));
  volatile int* abort_flag = (volatile int*)(bars_ptr + 8 * (2 * Cf::STAGES + 6));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cf::STAGES; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(tfull(a), 1); mbar_init(tempty(a), 2 * EPI_WARPS); }
    mbar_init(final_bar, 1);
    for (int e = 0; e < EPI_WARPS; ++e) mbar_init(in_bar(e), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {   // one warp of each block, collectively
    tmem_alloc_pair(slot, Cf::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();   // both blocks' barriers and tensor memory exist before either is used
  tc_fence_after();
  const uint32_t tmem_base = *slot_ptr;

  // work unit = a pair of vertically adjacent 128 x BN tiles; this block takes row tile
  // 2 mp + rank (past the last row tile when num_m is odd: its loads read zeros and
  // nothing is stored)
  const int num_mp = (p.num_m + 1) / 2;
  const int units = num_mp * p.num_n * p.splits;
  const int first = blockIdx.x >> 1, stride = gridDim.x >> 1;
  auto decode = [&](int unit, int& mb, int& nb, int& sp) {
    int r;
    if (p.n_fast) {
      nb = unit % p.num_n;
      r = unit / p.num_n;
      mb = 2 * (r % num_mp) + (int)rank;
      sp = r / num_mp;
    } else {
      mb = 2 * (unit % num_mp) + (int)rank;
      r = unit / num_mp;
      nb = r % p.num_n;
      sp = r / p.num_n;
    }
  };

  // Producer and MMA issuer loops run on whole warps: waits are made warp-uniform (so the
  // coordinates and operand descriptors stay uniform) and one elected lane issues.
  auto wait_u = [&](uint32_t b, uint32_t ph) {
    return __all_sync(0xffffffffu, mbar_wait(b, ph, abort_flag, p.err, true, p.wait_ns));
  };
  if (warp == 0) {
    // ---------------- TMA producer (both blocks): this block's rows of A and its half
    // of the B columns, completing on the even block's full barrier
    int it = 0;
    bool ok = true;
    for (int unit = first; unit < units && ok; unit += stride) {
      int mb, nb, sp;
      decode(unit, mb, nb, sp);
      const int m0 = mb * BM, n0 = nb * BN + (int)rank * (BN / 2);
      const int kb0 = sp * p.kb_per_split, kb1 = min(p.num_kb, kb0 + p.kb_per_split);
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = it % Cf::STAGES;
        const uint32_t ph = (uint32_t)(it / Cf::STAGES) & 1u;
        if (!wait_u(empty(s), ph ^ 1u)) { ok = false; break; }
        const uint32_t a_dst = base + s * Cf::STAGE, b_dst = a_dst + Cf::A_BYTES;
        const uint32_t fb = mapa_shared(full(s), 0);
        if (elect_one()) {
          if (leader) mbar_expect_tx(full(s), 2 * Cf::STAGE);   // both blocks' bytes
          if (AMN) {
            tma_load_2d_pair(a_dst, &tmA, fb, m0, kb * BK);
            tma_load_2d_pair(a_dst + 8192, &tmA, fb, m0 + 64, kb * BK);
          } else {
            tma_load_2d_pair(a_dst, &tmA, fb, kb * BK, m0);
          }
          if (BMN) {
#pragma unroll
            for (int i = 0; i < BN / 128; ++i)
              tma_load_2d_pair(b_dst + i * 8192, &tmB, fb, n0 + i * 64, kb * BK);
          } else {
            tma_load_2d_pair(b_dst, &tmB, fb, kb * BK, n0);
          }
        }
        __syncwarp();
      }
    }
    if (!ok && leader && lane == 0) {
      // let the copies already issued land before the block exits
      for (int j = max(0, it - Cf::STAGES); j < it; ++j)
        mbar_wait(full(j % Cf::STAGES), (uint32_t)(j / Cf::STAGES) & 1u, abort_flag, nullptr, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (leader) {
      // ---------------- MMA issuer (even block): M = 256 MMAs over both blocks' stages
      int it = 0, tcount = 0;
      bool ok = true;
      for (int unit = first; unit < units && ok; unit += stride, ++tcount) {
        int mb, nb, sp;
        decode(unit, mb, nb, sp);
        const int kb0 = sp * p.kb_per_split, kb1 = min(p.num_kb, kb0 + p.kb_per_split);
        const int acc = tcount & 1;
        const uint32_t aph = (uint32_t)(tcount >> 1) & 1u;
        if (!wait_u(tempty(acc), aph ^ 1u)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % Cf::STAGES;
          const uint32_t ph = (uint32_t)(it / Cf::STAGES) & 1u;
          if (!wait_u(full(s), ph)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_base = base + s * Cf::STAGE, b_base = a_base + Cf::A_BYTES;
          // a k step of 16 adds 32 bytes along K (K-major) or 2048 bytes (MN-major)
          const uint64_t ad0 = AMN ? sdesc(a_base, 8192, 1024) : sdesc(a_base, 16, 1024);
          const uint64_t bd0 = BMN ? sdesc(b_base, 8192, 1024) : sdesc(b_base, 16, 1024);
          constexpr uint64_t ASTEP = AMN ? 128 : 2, BSTEP = BMN ? 128 : 2;
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              umma_bf16_pair(d, ad0 + ASTEP * k, bd0 + BSTEP * k, IDESC,
                             (kb > kb0 || k > 0) ? 1u : 0u);
            umma_commit_pair_mc(empty(s), PAIR);   // the stage is free in both blocks
          }
          __syncwarp();
        }
        if (!ok) break;
        if (elect_one() && !(p.drop_first_signal && tcount == 0))
          umma_commit_pair_mc(tfull(acc), PAIR);   // both blocks' accumulators are ready
        __syncwarp();
      }
      // all issued MMAs complete before tensor memory is released
      if (elect_one()) {
        umma_commit_pair(final_bar);
        mbar_wait(final_bar, 0, abort_flag, nullptr, false);
      }
      __syncwarp();
    }
  } else {
    // ---------------- epilogue warps 2..9 of both blocks; warp % 4 selects the TMEM lane
    // quarter, and warps w, w + 4 split the tile's 64-column steps between them
    const int q = warp & 3, ew = warp - 2, half = ew >> 2;
    const uint32_t stg = staging + ew * Cf::STG;
    if ((p.epi == EPI_GELU_FWD || p.epi == EPI_GELU_FWD_U || p.epi == EPI_GELU_BWD_U) &&
        lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"((unsigned long long)&maps.pre) : "memory");
    }
    // EPI_GELU_BWD: the gelu'(u) rows of a step come by TMA into the second half of the warp's
    // staging slot, one step ahead: step k + 1's copy is issued as soon as step k's rows are
    // in registers.
    const bool has_in = XS && p.epi == EPI_GELU_BWD;
    const uint32_t in_buf = stg + 4096, ibar = in_bar(ew);
    int n_in = 0;   // input copies consumed (their barrier phases)
    bool in_pending = false;
    const bf16* rsrc = p.epi == EPI_GELU_BWD_U ? p.aux : (p.epi == EPI_STORE ? p.resid : nullptr);
    // the warp's step after (unit, c): (unit, c + 2) in the same tile, else the first of the
    // next unit in which the warp has a step
    auto next_step = [&](int& unit, int& c) -> bool {
      int mb, nb, sp;
      decode(unit, mb, nb, sp);
      if (c + 2 < BN / 64 && nb * BN + (c + 2) * 64 < p.N) { c += 2; return true; }
      c = half;
      for (unit += stride; unit < units; unit += stride) {
        decode(unit, mb, nb, sp);
        if (nb * BN + half * 64 < p.N) return true;
      }
      return false;
    };
    auto issue_in = [&](int unit, int c) {
      int mb, nb, sp;
      decode(unit, mb, nb, sp);
      if (lane == 0) {
        mbar_expect_tx(ibar, 4096);
        tma_load_2d(in_buf, &maps.in, ibar, nb * BN + c * 64, mb * BM + q * 32);
      }
      in_pending = true;
    };
    if (has_in && first < units) {
      int u0 = first, c0 = half;
      int mb, nb, sp;
      decode(u0, mb, nb, sp);
      if (nb * BN + half * 64 < p.N || next_step(u0, c0)) issue_in(u0, c0);
    }
    int tcount = 0;
    for (int unit = first; unit < units; unit += stride, ++tcount) {
      int mb, nb, sp;
      decode(unit, mb, nb, sp);
      const int acc = tcount & 1;
      const uint32_t aph = (uint32_t)(tcount >> 1) & 1u;
      bool ok = mbar_wait(tfull(acc), aph, abort_flag, p.err, true, p.wait_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int row0 = mb * BM + q * 32;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      float ce_m = -INFINITY, ce_s = 0.f;   // EPI_LOGITS_CE: this row's stats over the tile half
#pragma unroll 1
      for (int c = half; c < BN / 64; c += 2) {
        const int col0 = nb * BN + c * 64;
        if (col0 >= p.N) break;
        uint4 bia[8];
        if (p.bias && p.epi != EPI_ACCUM) {
#pragma unroll
          for (int j = 0; j < 8; ++j) bia[j] = __ldg(reinterpret_cast<const uint4*>(p.bias + col0) + j);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) bia[j] = make_uint4(0u, 0u, 0u, 0u);
        }
        uint32_t inr[32];
        if (has_in) {
          ok = __all_sync(0xffffffffu, mbar_wait(ibar, (uint32_t)n_in & 1u, abort_flag, p.err, true, p.wait_ns));
          if (!ok) break;
          ++n_in;
          in_pending = false;
          // row `lane` of the 32 x 64 tile, 128-byte swizzle: 16-byte unit j at j ^ (lane & 7)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 t = ld_shared16(in_buf + lane * 128 + ((j ^ (lane & 7)) << 4));
            inr[4 * j] = t.x; inr[4 * j + 1] = t.y; inr[4 * j + 2] = t.z; inr[4 * j + 3] = t.w;
          }
          __syncwarp();
          fence_proxy_async();
          int nu = unit, nc = c;
          if (next_step(nu, nc)) issue_in(nu, nc);
        } else if (rsrc && row0 + lane < p.M) {   // rows past M are computed, never stored
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 t = __ldg(reinterpret_cast<const uint4*>(rsrc + (size_t)(row0 + lane) * p.ldo + col0) + j);
            inr[4 * j] = t.x; inr[4 * j + 1] = t.y; inr[4 * j + 2] = t.z; inr[4 * j + 3] = t.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) inr[j] = 0u;
        }
        uint32_t r[64];
        tmem_ld64(taddr + c * 64, r);
        epilogue_step(p, maps, row0, col0, sp, stg, r, inr, bia, ce_m, ce_s);
      }
      if (!ok) break;
      if (p.epi == EPI_LOGITS_CE && row0 + lane < p.M)   // rows past M are never stored
        reinterpret_cast<float2*>(p.ce_part)[(size_t)(2 * nb + half) * p.M + row0 + lane] =
            make_float2(ce_m, ce_s);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty(acc), 0));
    }
    // an input copy issued for a step the loop did not reach (abort) lands before exit
    if (has_in && in_pending && lane == 0)
      mbar_wait(ibar, (uint32_t)n_in & 1u, abort_flag, nullptr, false);
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  // neither block leaves (or frees tensor memory) while the pair's MMAs, copies or
  // arrivals may still reach it
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cf::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
// Test hook for the bounded waits (gpt2_debug_gemm_waits): a wait limit other than
// TIMEOUT_NS and a dropped accumulator signal, read at every launch. Off by default.
static std::atomic<long long> g_gemm_wait_ns{0};
static std::atomic<int> g_gemm_drop_signal{0};

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  });
  return fn;
}

// Tensor map over a row-major matrix (rank 2) or a stack of them (rank 3): `inner`
// contiguous elements per row, `outer` rows `ld` elements apart, `depth` matrices `dstride`
// elements apart; box = box_inner x box_outer (x 1); out-of-range elements read as zero
// and are not written.
static bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* ptr,
                     uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                     uint32_t box_outer, CUtensorMapSwizzle swz, uint64_t depth = 0,
                     uint64_t dstride = 0) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  if (((uintptr_t)ptr & 15u) || (ld * esize) % 16 || (depth && (dstride * esize) % 16))
    return false;
  const cuuint32_t rank = depth ? 3 : 2;
  cuuint64_t dims[3] = {inner, outer, depth};
  cuuint64_t strides[2] = {ld * esize, dstride * esize};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, dt, rank, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
static bool make_map_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                          uint64_t ld, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, inner, outer, ld, box_inner,
                  box_outer, swz);
}

template <int BN, bool AMN, bool BMN, bool XS>
static cudaError_t launch(const GemmArgs& g, int num_sms, cudaStream_t s) {
  using Cf = Cfg<BN, XS>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, AMN, BMN, XS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  CUtensorMap ma, mb;
  bool ok = AMN ? make_map_bf16(&ma, g.A, g.M, g.K, g.lda, 64, 64)
                : make_map_bf16(&ma, g.A, g.K, g.M, g.lda, 64, BM);
  ok = ok && (BMN ? make_map_bf16(&mb, g.B, g.N, g.K, g.ldb, 64, 64)
                  : make_map_bf16(&mb, g.B, g.K, g.N, g.ldb, 64, BN / 2));
  if (!ok) return cudaErrorInvalidValue;
  Params p;
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.num_m = ceil_div(g.M, BM);
  p.num_n = ceil_div(g.N, BN);
  p.num_kb = ceil_div(g.K, BK);   // a ragged last k-block reads zeros past K
  p.splits = (g.epi == EPI_ACCUM && g.splits > 1) ? g.splits : 1;
  p.kb_per_split = ceil_div(p.num_kb, p.splits);
  p.n_fast = p.num_n <= 4;
  p.splits = ceil_div(p.num_kb, p.kb_per_split);
  p.epi = g.epi;
  p.defer = g.defer_partials;
  p.ldo = g.ldo;
  p.bias = (const bf16*)g.bias; p.resid = (const bf16*)g.resid;
  p.aux = (const bf16*)g.aux;
  p.scale = g.scale;
  p.err = g.err;
  p.vocab = g.vocab;
  p.ce_part = g.ce_part;
  {
    const long long w = g_gemm_wait_ns.load(std::memory_order_relaxed);
    p.wait_ns = w > 0 ? (unsigned long long)w : TIMEOUT_NS;
    p.drop_first_signal = g_gemm_drop_signal.load(std::memory_order_relaxed);
  }
  if (p.splits > 1 && !g.workspace) return cudaErrorInvalidValue;
  if ((g.bias && ((uintptr_t)g.bias & 15u)) || (g.resid && ((uintptr_t)g.resid & 15u)) ||
      (g.aux && ((uintptr_t)g.aux & 15u)) || (g.ldo % 8))
    return cudaErrorInvalidValue;
  EpiMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (g.epi == EPI_LOGITS_CE &&
      (BN != 256 || !g.ce_part || ((uintptr_t)g.ce_part & 7u) || g.bias || g.resid))
    return cudaErrorInvalidValue;
  if (g.epi == EPI_ACCUM) {
    if (p.splits == 1)
      ok = make_map(&maps.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.accum, g.N, g.M, g.ldo, 32,
                    32, CU_TENSOR_MAP_SWIZZLE_128B);
    else
      ok = make_map(&maps.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.workspace, g.N, g.M, g.N,
                    32, 32, CU_TENSOR_MAP_SWIZZLE_128B, (uint64_t)p.splits,
                    (uint64_t)g.M * g.N);
  } else {
    if ((g.epi == EPI_GELU_BWD || g.epi == EPI_GELU_BWD_U) && !g.aux) return cudaErrorInvalidValue;
    ok = make_map_bf16(&maps.out, g.out, g.N, g.M, g.ldo, 64, 32);
    const void* in = g.epi == EPI_GELU_BWD ? g.aux : nullptr;
    if (ok && in) ok = make_map_bf16(&maps.in, in, g.N, g.M, g.ldo, 64, 32);
    if (ok && (g.epi == EPI_GELU_FWD || g.epi == EPI_GELU_FWD_U || g.epi == EPI_GELU_BWD_U))
      ok = g.pre && make_map_bf16(&maps.pre, g.pre, g.N, g.M, g.ldo, 64, 32);
  }
  if (!ok) return cudaErrorInvalidValue;
  // clusters of two blocks; as many as can be resident at once (persistent)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Cf::SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters = 0;
  if (!max_clusters) {
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cudaError_t e = cudaOccupancyMaxActiveClusters(&max_clusters, gemm_kernel<BN, AMN, BMN, XS>, &cfg);
    if (e != cudaSuccess) return e;
    if (max_clusters <= 0) return cudaErrorInvalidConfiguration;
  }
  const int units = ceil_div(p.num_m, 2) * p.num_n * p.splits;
  cfg.gridDim = dim3(2 * std::min(units, max_clusters));
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_kernel<BN, AMN, BMN, XS>, ma, mb, maps, p);
  count_launches(1);
  if (e != cudaSuccess) return e;
  if (p.splits > 1 && !p.defer)
    return splitk_reduce(g.accum, g.workspace, p.splits, (long long)g.M * g.N, g.scale, s);
  return cudaSuccess;
}

}  // namespace tc

void gemm_tc_debug_waits(long long wait_limit_ns, int drop_first_signal) {
  tc::g_gemm_wait_ns.store(wait_limit_ns > 0 ? wait_limit_ns : 0);
  tc::g_gemm_drop_signal.store(drop_first_signal ? 1 : 0);
}

int gemm_tc_num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// 256-wide tiles unless the columns a partial last tile wastes exceed 1/16 of N (the
// padded vocabulary, 50304 = 196.5 x 256, keeps 256; N = 384 takes 128).
static int pick_bn(int N) {
  const int waste = (256 - N % 256) % 256;
  return waste * 16 <= N ? 256 : 128;
}

int gemm_ce_parts(int N) { return 2 * ceil_div(N, 256); }

int gemm_tc_pick_splits(int M, int N, int K, int num_sms) {
  const int bn = pick_bn(N);
  const int tiles = ceil_div(M, tc::BM) * ceil_div(N, bn);
  const int nkb = ceil_div(K, tc::BK);
  if (tiles >= num_sms) return 1;
  int s = num_sms / tiles;
  while (s > 1 && nkb / s < 8) --s;
  return s < 1 ? 1 : s;
}

cudaError_t gemm_bf16_tc(const GemmArgs& g, cudaStream_t s) {
  // N: whole 64-column epilogue steps. Any K: a K that is not a multiple of 64 ends in
  // a block that reads zeros past K (the tensor maps check the 16-byte row pitches).
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.N % 64) return cudaErrorInvalidValue;
  const int sms = gemm_tc_num_sms();
  GemmArgs a = g;
  if (a.epi == EPI_ACCUM && a.splits <= 0) a.splits = gemm_tc_pick_splits(a.M, a.N, a.K, sms);
  const int bn = a.epi == EPI_LOGITS_CE ? 256 : pick_bn(a.N);
  // a second bf16 output (the GELU epilogues) or a TMA-loaded input needs the wide staging
  const bool xs = a.epi == EPI_GELU_FWD || a.epi == EPI_GELU_FWD_U || a.epi == EPI_GELU_BWD ||
                  a.epi == EPI_GELU_BWD_U;
#define GEMM_TC_DISPATCH(BN_, XS_)                                                 \
  if (!a.a_mn && !a.b_mn) return tc::launch<BN_, false, false, XS_>(a, sms, s);    \
  if (!a.a_mn && a.b_mn) return tc::launch<BN_, false, true, XS_>(a, sms, s);      \
  if (a.a_mn && a.b_mn) return tc::launch<BN_, true, true, XS_>(a, sms, s);        \
  return tc::launch<BN_, true, false, XS_>(a, sms, s);
  if (xs) {
    if (a.a_mn) return cudaErrorInvalidValue;   // the GELU epilogues' A operand is K-major
    if (bn == 256) {
      if (a.b_mn) return tc::launch<256, false, true, true>(a, sms, s);
      return tc::launch<256, false, false, true>(a, sms, s);
    }
    if (a.b_mn) return tc::launch<128, false, true, true>(a, sms, s);
    return tc::launch<128, false, false, true>(a, sms, s);
  }
  if (bn == 256) { GEMM_TC_DISPATCH(256, false) }
  GEMM_TC_DISPATCH(128, false)
#undef GEMM_TC_DISPATCH
}

}  // namespace gpt2k

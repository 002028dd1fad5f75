// Memory-bound kernels of the GPT-2 training step: embedding gather and its
// deterministic scatter-add backward, the fused softmax-cross-entropy classifier,
// split-K reduction, global gradient norm and AdamW (LayerNorm and the column sums are
// in layernorm.cu).
//
// Every reduction runs in a fixed order (fixed partitions, fixed combine order), so two
// runs on the same inputs give bit-identical results.
#include "common.cuh"
#include "launch.h"

namespace gpt2k {

static inline cudaError_t last() { return cudaGetLastError(); }

long long& launch_counter() {
  static long long n = 0;
  return n;
}

// =====================================================================================
// Embedding: x[b, t] = wte[tok[b, t]] + wpe[t]
// (「从零实现一个最小GPT：代码讲解 + 知识点全解」 二.7 MiniGPT.forward, step 1)
template <typename T>
__global__ void encoder_fwd_kernel(T* __restrict__ x, const int* __restrict__ tokens,
                                   const T* __restrict__ wte, const T* __restrict__ wpe,
                                   int M, int T_, int C, int V, int* err, int pos0,
                                   const int* __restrict__ pos_dev) {
  constexpr int VE = 16 / sizeof(T);
  if (pos_dev) pos0 = *pos_dev;
  const int vpr = C / VE;
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)M * vpr) return;
  int p = (int)(i / vpr);
  int c = (int)(i % vpr) * VE;
  int tok = tokens[p];
  if (tok < 0 || tok >= V) {
    atomicOr(err, DEV_ERR_BAD_TOKEN);
    tok = tok < 0 ? 0 : V - 1;
  }
  int t = pos0 + p % T_;
  Vec16<T> a = ld16(wte + (size_t)tok * C + c);
  Vec16<T> b = ld16(wpe + (size_t)t * C + c);
  Vec16<T> o;
#pragma unroll
  for (int e = 0; e < VE; ++e) o.e[e] = from_f32<T>(to_f32(a.e[e]) + to_f32(b.e[e]));
  st16(x + (size_t)p * C + c, o);
}

cudaError_t encoder_forward(DType t, void* x, const int* tokens, const void* wte, const void* wpe,
                            int B, int T_, int C, int V, int* err, cudaStream_t s, int pos0,
                            const int* pos_dev) {
  int M = B * T_;
  if (t == DType::BF16) {
    long long n = (long long)M * (C / 8);
    encoder_fwd_kernel<bf16><<<ceil_div(n, 256), 256, 0, s>>>(
        (bf16*)x, tokens, (const bf16*)wte, (const bf16*)wpe, M, T_, C, V, err, pos0, pos_dev); count_launches(1);
  } else {
    long long n = (long long)M * (C / 4);
    encoder_fwd_kernel<float><<<ceil_div(n, 256), 256, 0, s>>>(
        (float*)x, tokens, (const float*)wte, (const float*)wpe, M, T_, C, V, err, pos0, pos_dev); count_launches(1);
  }
  return last();
}

// -------------------------------------------------------------------------------------
// Embedding backward.
// Stage 1 (one block): stable LSD radix sort of the positions by token id, 8 bits per
// pass. Each warp owns a contiguous slice of positions; within a warp, equal digits are
// ranked by lane order (match.any), across warps by warp order, so the sort is stable
// and the result does not depend on scheduling. Then segment starts (first position of
// each distinct id) are found with a block scan.
// Stage 2 (one block per segment): the rows of one id are summed in position order
// (each warp a fixed contiguous share of the rows, warps combined in warp order) and
// added, times scale, to dwte[id].
// Stage 3: dwpe[t] += scale * sum_b dx[b, t], b in increasing order.
constexpr int SORT_THREADS = 1024;
constexpr int SORT_WARPS = SORT_THREADS / 32;

// Segments (runs of one token id in the sorted order) longer than ENC_BIG rows are summed by a
// wider block of their own (the frequent ids of a skewed stream have hundreds of rows).
constexpr int ENC_BIG = 64;
constexpr int ENC_BIG_THREADS = 512;
struct EncScratch {
  int* key0; int* pos0; int* key1; int* pos1; int* seg_start; int* nseg; int* big;
};
static int enc_max_big(int M) { return M / (ENC_BIG + 1) + 1; }
static EncScratch enc_scratch(void* base, int M) {
  char* p = (char*)base;
  auto take = [&](size_t bytes) { char* r = p; p += (bytes + 255) / 256 * 256; return (int*)r; };
  EncScratch s;
  s.key0 = take(sizeof(int) * M); s.pos0 = take(sizeof(int) * M);
  s.key1 = take(sizeof(int) * M); s.pos1 = take(sizeof(int) * M);
  s.seg_start = take(sizeof(int) * (M + 1)); s.nseg = take(sizeof(int) * 4);
  s.big = take(sizeof(int) * enc_max_big(M));
  return s;
}
size_t encoder_backward_scratch_bytes(int M, int Vp) {
  (void)Vp;
  size_t a = ((size_t)M * 4 + 255) / 256 * 256;
  size_t b = ((size_t)(M + 1) * 4 + 255) / 256 * 256;
  size_t c = ((size_t)enc_max_big(M) * 4 + 255) / 256 * 256;
  return 4 * a + b + 256 + c;
}

// Exclusive scan of one int per thread over the block; returns the total in *total.
__device__ int block_exclusive_scan(int v, int* sh, int* total) {
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
    int xs = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, xs, o);
      if (lane >= o) xs += y;
    }
    sh[lane] = xs - s;           // exclusive prefix of warp totals
    if (lane == 31) sh[32] = xs; // block total
  }
  __syncthreads();
  int r = sh[w] + x - v;
  *total = sh[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(SORT_THREADS, 1)
encoder_sort_kernel(const int* __restrict__ tokens, int M, int Vp, EncScratch sc, int packed) {
  __shared__ int hist[256][SORT_WARPS + 1];
  __shared__ int scan_sh[40];
  extern __shared__ uint32_t srt[];   // packed: [2][M] of (key << 16 | position)
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int per_warp = (M + SORT_WARPS - 1) / SORT_WARPS;
  const int lo = min(M, w * per_warp), hi = min(M, lo + per_warp);
  if (packed) {
    // M <= 65536 and Vp <= 65536: key and position share one word and both radix passes run
    // in shared memory (the same stable per-warp counting, scan and scatter as below)
    uint32_t* a = srt;
    uint32_t* b = srt + M;
    for (int i = threadIdx.x; i < M; i += blockDim.x) {
      int t = tokens[i];
      t = t < 0 ? 0 : (t >= Vp ? Vp - 1 : t);
      a[i] = ((uint32_t)t << 16) | (uint32_t)i;
    }
    int kbits = 0;
    while ((1 << kbits) < Vp) kbits += 8;
    for (int shift = 16; shift < 16 + kbits; shift += 8) {
      for (int i = threadIdx.x; i < 256 * (SORT_WARPS + 1); i += blockDim.x)
        (&hist[0][0])[i] = 0;
      __syncthreads();
      for (int base = lo; base < hi; base += 32) {
        const int i = base + lane;
        const bool valid = i < hi;
        const int d = valid ? (int)((a[i] >> shift) & 255u) : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        if (valid && lane == __ffs(peers) - 1) hist[d][w] += __popc(peers);
        __syncwarp();
      }
      __syncthreads();
      {
        const int cells = 256 * SORT_WARPS;
        const int per = cells / SORT_THREADS;
        const int c0 = threadIdx.x * per;
        int local = 0;
        for (int j = 0; j < per; ++j) { const int c = c0 + j; local += hist[c / SORT_WARPS][c % SORT_WARPS]; }
        int total;
        int run = block_exclusive_scan(local, scan_sh, &total);
        for (int j = 0; j < per; ++j) {
          const int c = c0 + j;
          const int v = hist[c / SORT_WARPS][c % SORT_WARPS];
          hist[c / SORT_WARPS][c % SORT_WARPS] = run;
          run += v;
        }
      }
      __syncthreads();
      for (int base = lo; base < hi; base += 32) {
        const int i = base + lane;
        const bool valid = i < hi;
        const uint32_t k = valid ? a[i] : 0u;
        const int d = valid ? (int)((k >> shift) & 255u) : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        const int leader = __ffs(peers) - 1;
        const int basepos = valid ? hist[d][w] : 0;
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (valid) b[basepos + rank] = k;
        __syncwarp();
        if (valid && lane == leader) hist[d][w] = basepos + __popc(peers);
        __syncwarp();
      }
      __syncthreads();
      uint32_t* t = a; a = b; b = t;
    }
    for (int i = threadIdx.x; i < M; i += blockDim.x) {
      sc.key0[i] = (int)(a[i] >> 16);
      sc.pos0[i] = (int)(a[i] & 0xffffu);
    }
    __syncthreads();
  }
  // load keys (clamped ids) and positions
  for (int i = threadIdx.x; !packed && i < M; i += blockDim.x) {
    int t = tokens[i];
    t = t < 0 ? 0 : (t >= Vp ? Vp - 1 : t);
    sc.key0[i] = t;
    sc.pos0[i] = i;
  }
  __syncthreads();
  int bits = 0;
  while (!packed && (1 << bits) < Vp) bits += 8;   // packed: already sorted
  int* kin = sc.key0; int* pin = sc.pos0; int* kout = sc.key1; int* pout = sc.pos1;
  for (int shift = 0; shift < bits; shift += 8) {
    for (int i = threadIdx.x; i < 256 * (SORT_WARPS + 1); i += blockDim.x)
      (&hist[0][0])[i] = 0;
    __syncthreads();
    // per-warp digit counts
    for (int base = lo; base < hi; base += 32) {
      int i = base + lane;
      bool valid = i < hi;
      int d = valid ? (kin[i] >> shift) & 255 : -1 - lane;
      unsigned peers = __match_any_sync(0xffffffffu, d);
      if (valid && lane == __ffs(peers) - 1) hist[d][w] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    // exclusive offsets in (digit, warp) order: each thread owns 8 (digit, warp) cells
    {
      const int cells = 256 * SORT_WARPS;   // 8192
      const int per = cells / SORT_THREADS; // 8
      int c0 = threadIdx.x * per;
      int local = 0;
      for (int j = 0; j < per; ++j) { int c = c0 + j; local += hist[c / SORT_WARPS][c % SORT_WARPS]; }
      int total;
      int run = block_exclusive_scan(local, scan_sh, &total);
      for (int j = 0; j < per; ++j) {
        int c = c0 + j;
        int v = hist[c / SORT_WARPS][c % SORT_WARPS];
        hist[c / SORT_WARPS][c % SORT_WARPS] = run;
        run += v;
      }
    }
    __syncthreads();
    // stable scatter
    for (int base = lo; base < hi; base += 32) {
      int i = base + lane;
      bool valid = i < hi;
      int k = valid ? kin[i] : 0;
      int d = valid ? (k >> shift) & 255 : -1 - lane;
      unsigned peers = __match_any_sync(0xffffffffu, d);
      int leader = __ffs(peers) - 1;
      int basepos = valid ? hist[d][w] : 0;
      int rank = __popc(peers & ((1u << lane) - 1u));
      if (valid) { kout[basepos + rank] = k; pout[basepos + rank] = pin[i]; }
      __syncwarp();
      if (valid && lane == leader) hist[d][w] = basepos + __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    int* t0 = kin; kin = kout; kout = t0;
    int* t1 = pin; pin = pout; pout = t1;
  }
  // sorted keys/positions are now in kin/pin; make sure they sit in key0/pos0
  if (kin != sc.key0) {
    for (int i = threadIdx.x; i < M; i += blockDim.x) { sc.key0[i] = kin[i]; sc.pos0[i] = pin[i]; }
    __syncthreads();
  }
  // segment starts: i where key changes
  int nseg_total = 0;
  for (int base = 0; base < M; base += blockDim.x) {
    int i = base + threadIdx.x;
    int flag = (i < M) && (i == 0 || sc.key0[i] != sc.key0[i - 1]);
    int total;
    int off = block_exclusive_scan(flag, scan_sh, &total);
    if (flag) sc.seg_start[nseg_total + off] = i;
    nseg_total += total;
  }
  if (threadIdx.x == 0) { sc.seg_start[nseg_total] = M; sc.nseg[0] = nseg_total; }
  __syncthreads();
  // the long segments, in segment order
  int nbig = 0;
  for (int base = 0; base < nseg_total; base += blockDim.x) {
    const int g = base + threadIdx.x;
    const int flag = g < nseg_total && sc.seg_start[g + 1] - sc.seg_start[g] > ENC_BIG;
    int total;
    const int off = block_exclusive_scan(flag, scan_sh, &total);
    if (flag) sc.big[nbig + off] = g;
    nbig += total;
  }
  if (threadIdx.x == 0) sc.nseg[1] = nbig;
}

// One warp per segment of at most ENC_BIG rows: the warp sums the segment's rows in order
// (four per step when registers permit, all loads issued before the adds) and adds the sum to
// that token's row of dwte, of which it is the only writer.
template <typename T, int MAXV>
__global__ void __launch_bounds__(256)
encoder_segsum_kernel(float* __restrict__ dwte, const T* __restrict__ dx, int C, float scale,
                      EncScratch sc) {
  constexpr int VE = 16 / sizeof(T);
  const int lane = threadIdx.x & 31;
  const int seg = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (seg >= sc.nseg[0]) return;
  const int start = sc.seg_start[seg], end = sc.seg_start[seg + 1];
  if (end - start > ENC_BIG) return;   // encoder_bigseg_kernel
  const int id = sc.key0[start];
  float acc[MAXV][VE];
#pragma unroll
  for (int j = 0; j < MAXV; ++j)
#pragma unroll
    for (int e = 0; e < VE; ++e) acc[j][e] = 0.f;
  int r = start;
  constexpr int RB = MAXV <= 4 ? 4 : 1;
  for (; r + RB <= end; r += RB) {
    int pos[RB];
#pragma unroll
    for (int k = 0; k < RB; ++k) pos[k] = sc.pos0[r + k];
    Vec16<T> v[RB][MAXV];
#pragma unroll
    for (int k = 0; k < RB; ++k)
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int c = (j * 32 + lane) * VE;
        if (c < C) v[k][j] = ld16(dx + (size_t)pos[k] * C + c);
      }
#pragma unroll
    for (int k = 0; k < RB; ++k)
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int c = (j * 32 + lane) * VE;
        if (c < C) {
#pragma unroll
          for (int e = 0; e < VE; ++e) acc[j][e] += to_f32(v[k][j].e[e]);
        }
      }
  }
  for (; r < end; ++r) {
    const T* row = dx + (size_t)sc.pos0[r] * C;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int c = (j * 32 + lane) * VE;
      if (c < C) {
        Vec16<T> v = ld16(row + c);
#pragma unroll
        for (int e = 0; e < VE; ++e) acc[j][e] += to_f32(v.e[e]);
      }
    }
  }
  float* out = dwte + (size_t)id * C;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int c = (j * 32 + lane) * VE;
    if (c < C) {
#pragma unroll
      for (int e = 0; e < VE; ++e) out[c + e] += scale * acc[j][e];
    }
  }
}

// One block of 16 warps per long segment: warp w sums its fixed share of the segment's rows
// (four rows per step, in row order) into shared memory; thread c then adds the 16 warp rows
// of column c in warp order: a fixed order, so the result is bit-reproducible.
template <typename T, int MAXV>
__global__ void __launch_bounds__(ENC_BIG_THREADS)
encoder_bigseg_kernel(float* __restrict__ dwte, const T* __restrict__ dx, int C, float scale,
                      EncScratch sc) {
  constexpr int VE = 16 / sizeof(T);
  constexpr int NW = ENC_BIG_THREADS / 32;
  extern __shared__ float bpart[];   // [NW][C]
  if ((int)blockIdx.x >= sc.nseg[1]) return;
  const int seg = sc.big[blockIdx.x];
  const int start = sc.seg_start[seg], end = sc.seg_start[seg + 1];
  const int id = sc.key0[start];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int n = end - start;
  const int per = (n + NW - 1) / NW;
  const int r0 = start + min(n, w * per), r1 = start + min(n, (w + 1) * per);
  float acc[MAXV][VE];
#pragma unroll
  for (int j = 0; j < MAXV; ++j)
#pragma unroll
    for (int e = 0; e < VE; ++e) acc[j][e] = 0.f;
  int r = r0;
  constexpr int RB = MAXV <= 4 ? 4 : 1;   // rows per step (registers permitting)
  for (; r + RB <= r1; r += RB) {
    int pos[RB];
#pragma unroll
    for (int k = 0; k < RB; ++k) pos[k] = sc.pos0[r + k];
    Vec16<T> v[RB][MAXV];
#pragma unroll
    for (int k = 0; k < RB; ++k)
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int c = (j * 32 + lane) * VE;
        if (c < C) v[k][j] = ld16(dx + (size_t)pos[k] * C + c);
      }
#pragma unroll
    for (int k = 0; k < RB; ++k)
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int c = (j * 32 + lane) * VE;
        if (c < C) {
#pragma unroll
          for (int e = 0; e < VE; ++e) acc[j][e] += to_f32(v[k][j].e[e]);
        }
      }
  }
  for (; r < r1; ++r) {
    const T* row = dx + (size_t)sc.pos0[r] * C;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int c = (j * 32 + lane) * VE;
      if (c < C) {
        Vec16<T> v = ld16(row + c);
#pragma unroll
        for (int e = 0; e < VE; ++e) acc[j][e] += to_f32(v.e[e]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int c = (j * 32 + lane) * VE;
    if (c < C) {
#pragma unroll
      for (int e = 0; e < VE; ++e) bpart[(size_t)w * C + c + e] = acc[j][e];
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < C; c += blockDim.x) {
    float t = 0.f;
#pragma unroll 8
    for (int k = 0; k < NW; ++k) t += bpart[(size_t)k * C + c];
    dwte[(size_t)id * C + c] += scale * t;
  }
}

template <typename T>
__global__ void encoder_wpe_kernel(float* __restrict__ dwpe, const T* __restrict__ dx, int B,
                                   int T_, int C, float scale) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)T_ * C) return;
  float s = 0.f;
  for (int b = 0; b < B; ++b) s += to_f32(dx[(size_t)b * T_ * C + i]);
  dwpe[i] += scale * s;
}

// The segment sums and the position-embedding column sums for one element type and row width.
template <typename T, int MAXV>
static cudaError_t encoder_sums(float* dwte, float* dwpe, const void* dx, int B, int T_, int C,
                                float scale, EncScratch sc, cudaStream_t s) {
  const int M = B * T_;
  const T* x = (const T*)dx;
  encoder_segsum_kernel<T, MAXV><<<ceil_div(M, 8), 256, 0, s>>>(dwte, x, C, scale, sc);
  count_launches(1);
  const size_t smem = (size_t)(ENC_BIG_THREADS / 32) * C * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(encoder_bigseg_kernel<T, MAXV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  encoder_bigseg_kernel<T, MAXV><<<enc_max_big(M), ENC_BIG_THREADS, smem, s>>>(dwte, x, C, scale,
                                                                               sc);
  count_launches(1);
  encoder_wpe_kernel<T><<<ceil_div((long long)T_ * C, 256), 256, 0, s>>>(dwpe, x, B, T_, C, scale);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t encoder_backward(DType t, float* dwte, float* dwpe, const void* dx, const int* tokens,
                             int B, int T_, int C, int Vp, float scale, void* scratch,
                             cudaStream_t s) {
  const int M = B * T_;
  EncScratch sc = enc_scratch(scratch, M);
  // keys and positions packed in one word and sorted in shared memory where they fit
  const int packed = M <= 65536 && Vp <= 65536 && (size_t)M * 8 <= 180 * 1024;
  const size_t smem = packed ? (size_t)M * 8 : 0;
  if (packed) {
    static size_t attr = 0;
    if (smem > attr) {
      cudaError_t e = cudaFuncSetAttribute(encoder_sort_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr = smem;
    }
  }
  encoder_sort_kernel<<<1, SORT_THREADS, smem, s>>>(tokens, M, Vp, sc, packed);
  count_launches(1);
  // MAXV 16-byte vectors per lane cover the row: 8 bf16 or 4 fp32 each, 32 lanes
  if (t == DType::BF16) {
    if (C > 2048 || C % 8) return cudaErrorInvalidValue;
    if (C <= 256) return encoder_sums<bf16, 1>(dwte, dwpe, dx, B, T_, C, scale, sc, s);
    if (C <= 512) return encoder_sums<bf16, 2>(dwte, dwpe, dx, B, T_, C, scale, sc, s);
    if (C <= 1024) return encoder_sums<bf16, 4>(dwte, dwpe, dx, B, T_, C, scale, sc, s);
    return encoder_sums<bf16, 8>(dwte, dwpe, dx, B, T_, C, scale, sc, s);
  }
  if (C > 1024 || C % 4) return cudaErrorInvalidValue;
  if (C <= 128) return encoder_sums<float, 1>(dwte, dwpe, dx, B, T_, C, scale, sc, s);
  if (C <= 256) return encoder_sums<float, 2>(dwte, dwpe, dx, B, T_, C, scale, sc, s);
  if (C <= 512) return encoder_sums<float, 4>(dwte, dwpe, dx, B, T_, C, scale, sc, s);
  return encoder_sums<float, 8>(dwte, dwpe, dx, B, T_, C, scale, sc, s);
}

// =====================================================================================
// Fused classifier (「从零实现一个最小GPT」 二.7 forward step 4, F.cross_entropy with mean
// reduction): one block per row. Pass 1 reads the row once with a running (max, sum of
// exp) per thread over the first V columns; the block combines them into lse and the
// row loss lse - z[y]. Pass 2 re-reads the row (from L2) and writes, in place,
// dlogits = (exp(z - lse) - [v == y]) / M, and 0 in the padded columns [V, Vp).
constexpr int CLS_THREADS = 512;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ void online_merge(float& m, float& s, float m2, float s2) {
  float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  s = s * fast_exp2(m - mn) + s2 * fast_exp2(m2 - mn);
  m = mn;
}

template <typename T>
__global__ void __launch_bounds__(CLS_THREADS)
classifier_kernel(T* __restrict__ logits, float* __restrict__ losses,
                  const int* __restrict__ targets, int V, int Vp, float inv_M, int* err) {
  constexpr int VE = 16 / sizeof(T);
  __shared__ float sm_m[CLS_THREADS / 32], sm_s[CLS_THREADS / 32];
  __shared__ float sh_lse;
  const int row = blockIdx.x;
  T* z = logits + (size_t)row * Vp;
  int y = targets[row];
  if (y < 0 || y >= V) {
    if (threadIdx.x == 0) atomicOr(err, DEV_ERR_BAD_TARGET);
    y = y < 0 ? 0 : V - 1;
  }
  // pass 1 (log2 domain): running max m and sum s of 2^(z*log2e - m)
  float m = -INFINITY, s = 0.f;
  const int nvec = Vp / VE;
  auto consume = [&](const Vec16<T>& v, int i) {
    float a[VE];
    float lm = -INFINITY;
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      a[e] = (i * VE + e < V) ? to_f32(v.e[e]) * LOG2E : -INFINITY;
      lm = fmaxf(lm, a[e]);
    }
    if (lm == -INFINITY) return;
    float ls = 0.f;
#pragma unroll
    for (int e = 0; e < VE; ++e) ls += fast_exp2(a[e] - lm);
    online_merge(m, s, lm, ls);
  };
  // two vectors per step, both loads issued first (more bytes in flight per thread)
  int i = threadIdx.x;
  for (; i + CLS_THREADS < nvec; i += 2 * CLS_THREADS) {
    const Vec16<T> v0 = ld16(z + (size_t)i * VE), v1 = ld16(z + (size_t)(i + CLS_THREADS) * VE);
    consume(v0, i);
    consume(v1, i + CLS_THREADS);
  }
  if (i < nvec) consume(ld16(z + (size_t)i * VE), i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    online_merge(m, s, m2, s2);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) { sm_m[wid] = m; sm_s[wid] = s; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M0 = sm_m[0], S0 = sm_s[0];
    for (int k = 1; k < CLS_THREADS / 32; ++k) online_merge(M0, S0, sm_m[k], sm_s[k]);
    float lse2 = M0 + __log2f(S0);     // log2-domain lse
    sh_lse = lse2;
    losses[row] = lse2 * LN2 - to_f32(z[y]);
  }
  __syncthreads();
  const float lse2 = sh_lse;
  for (int i = threadIdx.x; i < nvec; i += CLS_THREADS) {
    Vec16<T> v = ld16(z + (size_t)i * VE), o;
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      int col = i * VE + e;
      float d = 0.f;
      if (col < V) {
        d = fast_exp2(to_f32(v.e[e]) * LOG2E - lse2);
        if (col == y) d -= 1.0f;
        d *= inv_M;
      }
      o.e[e] = from_f32<T>(d);
    }
    st16_cs(z + (size_t)i * VE, o);
  }
}

cudaError_t classifier(DType t, void* logits, float* losses, const int* targets, int M, int V,
                       int Vp, int* err, cudaStream_t s) {
  float inv = 1.0f / (float)M;
  if (t == DType::BF16)
    classifier_kernel<bf16><<<M, CLS_THREADS, 0, s>>>((bf16*)logits, losses, targets, V, Vp, inv, err);
  else
    classifier_kernel<float><<<M, CLS_THREADS, 0, s>>>((float*)logits, losses, targets, V, Vp, inv, err);
  count_launches(1);
  return last();
}

// ------------------------------------------------------------------ cross-entropy from the
// lm_head's softmax statistics (EPI_LOGITS_CE): the row's partials (float2 (m, s) at
// ce_part[part * M + row], log2 domain) merged into lse2 = m + log2(s). Block: 32 rows (the
// lanes, so every load of a warp is 32 consecutive rows) x 8 warps; warp g merges the parts
// g, g + 8, ... in order, then the 8 results are merged in warp order. Then one block per row
// writes the loss and the dlogits in a single streaming pass.
constexpr int CEC_WARPS = 8;
__global__ void __launch_bounds__(32 * CEC_WARPS)
ce_combine_kernel(float* __restrict__ lse2_out, const float2* __restrict__ part, int nparts,
                  int M) {
  __shared__ float sm[CEC_WARPS][32], ss[CEC_WARPS][32];
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
  const int row = blockIdx.x * 32 + lane;
  float m = -INFINITY, s = 0.f;
  if (row < M) {
    int k = g;
    for (; k + 3 * CEC_WARPS < nparts; k += 4 * CEC_WARPS) {   // four loads in flight
      float2 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = part[(size_t)(k + i * CEC_WARPS) * M + row];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (v[i].x != -INFINITY) online_merge(m, s, v[i].x, v[i].y);   // -inf: no column < V
    }
    for (; k < nparts; k += CEC_WARPS) {
      const float2 v = part[(size_t)k * M + row];
      if (v.x != -INFINITY) online_merge(m, s, v.x, v.y);
    }
  }
  sm[g][lane] = m;
  ss[g][lane] = s;
  __syncthreads();
  if (g == 0 && row < M) {
    float mm = -INFINITY, sum = 0.f;
#pragma unroll
    for (int w = 0; w < CEC_WARPS; ++w)
      if (sm[w][lane] != -INFINITY) online_merge(mm, sum, sm[w][lane], ss[w][lane]);
    lse2_out[row] = mm + __log2f(sum);
  }
}

template <typename T>
__global__ void __launch_bounds__(CLS_THREADS)
ce_finish_kernel(T* __restrict__ logits, float* __restrict__ losses, const float* __restrict__ lse2s,
                 const int* __restrict__ targets, int V, int Vp, float inv_M, int* err) {
  constexpr int VE = 16 / sizeof(T);
  const int row = blockIdx.x;
  T* z = logits + (size_t)row * Vp;
  int y = targets[row];
  if (y < 0 || y >= V) {
    if (threadIdx.x == 0) atomicOr(err, DEV_ERR_BAD_TARGET);
    y = y < 0 ? 0 : V - 1;
  }
  const float lse2 = lse2s[row];
  if (threadIdx.x == 0) losses[row] = lse2 * LN2 - to_f32(z[y]);
  __syncthreads();   // z[y] is read before any thread overwrites it
  const int nvec = Vp / VE;
  auto emit = [&](const Vec16<T>& v, int i) {
    Vec16<T> o;
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      const int col = i * VE + e;
      float d = 0.f;
      if (col < V) {
        d = fast_exp2(to_f32(v.e[e]) * LOG2E - lse2);
        if (col == y) d -= 1.0f;
        d *= inv_M;
      }
      o.e[e] = from_f32<T>(d);
    }
    st16_cs(z + (size_t)i * VE, o);
  };
  // two vectors per step, both loads issued first
  int i = threadIdx.x;
  for (; i + CLS_THREADS < nvec; i += 2 * CLS_THREADS) {
    const Vec16<T> v0 = ld16_cs(z + (size_t)i * VE), v1 = ld16_cs(z + (size_t)(i + CLS_THREADS) * VE);
    emit(v0, i);
    emit(v1, i + CLS_THREADS);
  }
  if (i < nvec) emit(ld16_cs(z + (size_t)i * VE), i);
}

cudaError_t ce_from_partials(DType t, void* logits, float* losses, const float* ce_part,
                             int nparts, const int* targets, int M, int V, int Vp, float* lse_tmp,
                             int* err, cudaStream_t s) {
  if (t != DType::BF16 || M <= 0 || nparts <= 0) return cudaErrorInvalidValue;
  ce_combine_kernel<<<ceil_div(M, 32), 32 * CEC_WARPS, 0, s>>>(lse_tmp, (const float2*)ce_part,
                                                                nparts, M);
  count_launches(1);
  ce_finish_kernel<bf16><<<M, CLS_THREADS, 0, s>>>((bf16*)logits, losses, lse_tmp, targets, V, Vp,
                                                  1.0f / (float)M, err);
  count_launches(1);
  return last();
}

__global__ void mean_loss_kernel(float* out, const float* __restrict__ losses, int M) {
  __shared__ double sh[1024];
  double a = 0.0;
  for (int i = threadIdx.x; i < M; i += blockDim.x) a += (double)losses[i];
  sh[threadIdx.x] = a;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[0] = (float)(sh[0] / M);
}

cudaError_t mean_loss(float* loss_out, const float* losses, int M, cudaStream_t s) {
  mean_loss_kernel<<<1, 1024, 0, s>>>(loss_out, losses, M); count_launches(1);
  return last();
}

template <typename T, bool VEC>
__global__ void argmax_kernel(int* out, const T* __restrict__ logits, int V, int Vp) {
  // one block per row; thread i scans the 16-byte vectors i, i + blockDim, ... (single
  // elements when the row pitch is not a multiple of 16 bytes; columns increase within a
  // thread, so its first maximum is kept), then the lowest index among equal maxima wins
  // across threads
  constexpr int VE = VEC ? 16 / sizeof(T) : 1;
  __shared__ float sv[32];
  __shared__ int si[32];
  const T* z = logits + (size_t)blockIdx.x * Vp;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int c0 = threadIdx.x * VE; c0 < V; c0 += blockDim.x * VE) {
    alignas(16) T a[VE];
    if constexpr (VEC) *reinterpret_cast<uint4*>(a) = *reinterpret_cast<const uint4*>(z + c0);
    else a[0] = z[c0];
#pragma unroll
    for (int e = 0; e < VE; ++e) {
      const float v = to_f32(a[e]);
      if (c0 + e < V && v > best) { best = v; bi = c0 + e; }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, best, o);
    int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (v2 > best || (v2 == best && i2 < bi)) { best = v2; bi = i2; }
  }
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) { sv[w] = best; si[w] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < (int)(blockDim.x >> 5); ++k)
      if (sv[k] > best || (sv[k] == best && si[k] < bi)) { best = sv[k]; bi = si[k]; }
    out[blockIdx.x] = bi;
  }
}

cudaError_t argmax_rows(DType t, int* out, const void* logits, int M, int V, int Vp,
                        cudaStream_t s) {
  // rows as 16-byte vectors where the row pitch keeps them aligned
  const bool al = ((uintptr_t)logits & 15u) == 0;
  if (t == DType::BF16) {
    if (al && Vp % 8 == 0) argmax_kernel<bf16, true><<<M, 1024, 0, s>>>(out, (const bf16*)logits, V, Vp);
    else argmax_kernel<bf16, false><<<M, 1024, 0, s>>>(out, (const bf16*)logits, V, Vp);
  } else {
    if (al && Vp % 4 == 0) argmax_kernel<float, true><<<M, 1024, 0, s>>>(out, (const float*)logits, V, Vp);
    else argmax_kernel<float, false><<<M, 1024, 0, s>>>(out, (const float*)logits, V, Vp);
  }
  count_launches(1);
  return last();
}

// =====================================================================================
__global__ void splitk_reduce_kernel(float* __restrict__ accum, const float* __restrict__ ws,
                                     int splits, long long n4, long long n, float scale) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  float4 a = reinterpret_cast<float4*>(accum)[i];
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < splits; ++k) {
    float4 w = reinterpret_cast<const float4*>(ws + (size_t)k * n)[i];
    s.x += w.x; s.y += w.y; s.z += w.z; s.w += w.w;
  }
  a.x += scale * s.x; a.y += scale * s.y; a.z += scale * s.z; a.w += scale * s.w;
  reinterpret_cast<float4*>(accum)[i] = a;
}

cudaError_t splitk_reduce(float* accum, const float* ws, int splits, long long n, float scale,
                          cudaStream_t s) {
  if (n % 4) return cudaErrorInvalidValue;
  long long n4 = n / 4;
  splitk_reduce_kernel<<<ceil_div(n4, 256), 256, 0, s>>>(accum, ws, splits, n4, n, scale); count_launches(1);
  return last();
}

// accum += sum_k ws[k] in k order, then ws = 0
// (all of a thread's loads are issued before its first store, so they overlap)
template <int S>
__global__ void splitk_fold_kernel(float* __restrict__ accum, float* __restrict__ ws, int splits,
                                   long long n4, long long n) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  float4 a = reinterpret_cast<float4*>(accum)[i];
  for (int k0 = 0; k0 < splits; k0 += S) {
    float4 w[S];
#pragma unroll
    for (int k = 0; k < S; ++k)
      if (k0 + k < splits) w[k] = __ldcs(reinterpret_cast<const float4*>(ws + (size_t)(k0 + k) * n) + i);
#pragma unroll
    for (int k = 0; k < S; ++k)
      if (k0 + k < splits) {
        a.x += w[k].x; a.y += w[k].y; a.z += w[k].z; a.w += w[k].w;
        __stcs(reinterpret_cast<float4*>(ws + (size_t)(k0 + k) * n) + i, make_float4(0.f, 0.f, 0.f, 0.f));
      }
  }
  reinterpret_cast<float4*>(accum)[i] = a;
}

cudaError_t splitk_fold(float* accum, float* ws, int splits, long long n, cudaStream_t s) {
  if (n % 4) return cudaErrorInvalidValue;
  long long n4 = n / 4;
  splitk_fold_kernel<8><<<ceil_div(n4, 256), 256, 0, s>>>(accum, ws, splits, n4, n); count_launches(1);
  return last();
}

// The same fold, each block also writing the sum of squares of the final values it wrote to
// nparts[blockIdx.x] (fold_norm_parts(n) blocks): the gradient norm's share of this tensor,
// produced while the final values pass by.
int fold_norm_parts(long long n) { return ceil_div(n / 4, 256); }

template <int S>
__global__ void __launch_bounds__(256)
splitk_fold_norm_kernel(float* __restrict__ accum, float* __restrict__ ws, int splits,
                        long long n4, long long n, float* __restrict__ nparts) {
  __shared__ float sh[8];
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  float q = 0.f;
  if (i < n4) {
    float4 a = reinterpret_cast<float4*>(accum)[i];
    for (int k0 = 0; k0 < splits; k0 += S) {
      float4 w[S];
#pragma unroll
      for (int k = 0; k < S; ++k)
        if (k0 + k < splits) w[k] = __ldcs(reinterpret_cast<const float4*>(ws + (size_t)(k0 + k) * n) + i);
#pragma unroll
      for (int k = 0; k < S; ++k)
        if (k0 + k < splits) {
          a.x += w[k].x; a.y += w[k].y; a.z += w[k].z; a.w += w[k].w;
          __stcs(reinterpret_cast<float4*>(ws + (size_t)(k0 + k) * n) + i, make_float4(0.f, 0.f, 0.f, 0.f));
        }
    }
    reinterpret_cast<float4*>(accum)[i] = a;
    q = a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
  }
  q = warp_sum(q);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = q;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int k = 0; k < 8; ++k) t += sh[k];
    nparts[blockIdx.x] = t;
  }
}

cudaError_t splitk_fold_norm(float* accum, float* ws, int splits, long long n, float* nparts,
                             cudaStream_t s) {
  if (n % 4) return cudaErrorInvalidValue;
  splitk_fold_norm_kernel<8><<<fold_norm_parts(n), 256, 0, s>>>(accum, ws, splits, n / 4, n,
                                                                 nparts);
  count_launches(1);
  return last();
}

// =====================================================================================
// Global gradient norm and clip coefficient, on device (no host sync):
// out[0] = ||g||_2, out[1] = max_norm > 0 ? min(1, max_norm / (||g|| + 1e-6)) : 1.
constexpr int NORM_BLOCKS = 592;   // 4 x 148 SMs
int norm_partials_count() { return NORM_BLOCKS; }

__global__ void __launch_bounds__(256)
sumsq_kernel(float* __restrict__ partials, const float* __restrict__ g, long long n) {
  __shared__ float sh[8];
  long long n4 = n / 4;
  long long per = (n4 + gridDim.x - 1) / gridDim.x;
  long long b0 = blockIdx.x * per, b1 = min(n4, b0 + per);
  float a = 0.f;
  for (long long i = b0 + threadIdx.x; i < b1; i += blockDim.x) {
    float4 v = __ldcs(reinterpret_cast<const float4*>(g) + i);
    a += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  if (blockIdx.x == gridDim.x - 1)
    for (long long i = n4 * 4 + threadIdx.x; i < n; i += blockDim.x) a += g[i] * g[i];
  a = warp_sum(a);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int k = 0; k < 8; ++k) t += sh[k];
    partials[blockIdx.x] = t;
  }
}

__global__ void norm_finish_kernel(float* out, const float* __restrict__ partials, int np,
                                   float max_norm) {
  if (threadIdx.x != 0) return;
  double s = 0.0;
  for (int k = 0; k < np; ++k) s += (double)partials[k];
  float nrm = (float)sqrt(s);
  out[0] = nrm;
  out[1] = max_norm > 0.f ? fminf(1.0f, max_norm / (nrm + 1e-6f)) : 1.0f;
}

// The same over many partials: thread i adds partials i, i + 1024, ... in order (double),
// then a fixed tree; deterministic.
__global__ void __launch_bounds__(1024)
norm_finish_many_kernel(float* out, const float* __restrict__ partials, int np, float max_norm) {
  __shared__ double sh[1024];
  double a = 0.0;
  for (int k = threadIdx.x; k < np; k += 1024) a += (double)partials[k];
  sh[threadIdx.x] = a;
  __syncthreads();
  for (int o = 512; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const float nrm = (float)sqrt(sh[0]);
    out[0] = nrm;
    out[1] = max_norm > 0.f ? fminf(1.0f, max_norm / (nrm + 1e-6f)) : 1.0f;
  }
}

// Sums of squares over a list of [offset, offset + count) ranges of g, one block per range
// (ranges of at most a few hundred thousand elements), into partials[block].
__global__ void __launch_bounds__(256)
sumsq_ranges_kernel(float* __restrict__ partials, const float* __restrict__ g,
                    const long long* __restrict__ ranges) {
  __shared__ float sh[8];
  const long long off = ranges[2 * blockIdx.x], cnt = ranges[2 * blockIdx.x + 1];
  float a = 0.f;
  for (long long i = threadIdx.x; i < cnt; i += blockDim.x) {
    const float v = __ldcs(g + off + i);
    a += v * v;
  }
  a = warp_sum(a);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int k = 0; k < 8; ++k) t += sh[k];
    partials[blockIdx.x] = t;
  }
}

cudaError_t grad_norm_finish(float* out, const float* partials, int np, const float* g,
                             const long long* d_ranges, int nranges, float* range_parts,
                             float max_norm, cudaStream_t s) {
  if (nranges > 0) {
    sumsq_ranges_kernel<<<nranges, 256, 0, s>>>(range_parts, g, d_ranges);
    count_launches(1);
  }
  norm_finish_many_kernel<<<1, 1024, 0, s>>>(out, partials, np, max_norm);
  count_launches(1);
  return last();
}

cudaError_t grad_norm(float* out, float* partials, const float* g, long long n, float max_norm,
                      cudaStream_t s) {
  sumsq_kernel<<<NORM_BLOCKS, 256, 0, s>>>(partials, g, n); count_launches(1);
  norm_finish_kernel<<<1, 32, 0, s>>>(out, partials, NORM_BLOCKS, max_norm); count_launches(1);
  return last();
}

// AdamW, decoupled weight decay (「从零实现一个最小GPT」 三.9), PyTorch's formulation:
// p *= 1 - lr wd; m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
// p -= lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
__global__ void __launch_bounds__(256)
adamw_kernel(float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
             float* __restrict__ v, bf16* __restrict__ pb, long long n4, float lr, float b1,
             float b2, float eps, float decay, float inv_bc1, float inv_bc2,
             const float* __restrict__ coef) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float c = coef ? coef[1] : 1.0f;
  float4 pp = reinterpret_cast<float4*>(p)[i];
  float4 gg = __ldcs(reinterpret_cast<const float4*>(g) + i);
  float4 mm = reinterpret_cast<float4*>(m)[i];
  float4 vv = reinterpret_cast<float4*>(v)[i];
  float* P = &pp.x; float* G = &gg.x; float* Mv = &mm.x; float* Vv = &vv.x;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float gr = G[e] * c;
    Mv[e] = b1 * Mv[e] + (1.0f - b1) * gr;
    Vv[e] = b2 * Vv[e] + (1.0f - b2) * gr * gr;
    float pv = P[e] * decay;
    P[e] = pv - lr * (Mv[e] * inv_bc1) / (sqrtf(Vv[e] * inv_bc2) + eps);
  }
  reinterpret_cast<float4*>(p)[i] = pp;
  reinterpret_cast<float4*>(m)[i] = mm;
  reinterpret_cast<float4*>(v)[i] = vv;
  if (pb) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(pp.x, pp.y), hi = __floats2bfloat162_rn(pp.z, pp.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(pb)[i] = u;
  }
}

cudaError_t adamw(float* p, const float* g, float* m, float* v, void* p_bf16, long long n,
                  float lr, float beta1, float beta2, float eps, float weight_decay, int t,
                  const float* coef, cudaStream_t s) {
  if (n % 4) return cudaErrorInvalidValue;
  double bc1 = 1.0 - pow((double)beta1, (double)t), bc2 = 1.0 - pow((double)beta2, (double)t);
  long long n4 = n / 4;
  adamw_kernel<<<ceil_div(n4, 256), 256, 0, s>>>(p, g, m, v, (bf16*)p_bf16, n4, lr, beta1, beta2,
                                                 eps, 1.0f - lr * weight_decay,
                                                 (float)(1.0 / bc1), (float)(1.0 / bc2), coef); count_launches(1);
  return last();
}

__global__ void to_bf16_kernel(bf16* __restrict__ dst, const float* __restrict__ src, long long n) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = __float2bfloat16_rn(src[i]);
}

cudaError_t to_bf16(void* dst, const float* src, long long n, cudaStream_t s) {
  to_bf16_kernel<<<ceil_div(n, 256), 256, 0, s>>>((bf16*)dst, src, n); count_launches(1);
  return last();
}

}  // namespace gpt2k

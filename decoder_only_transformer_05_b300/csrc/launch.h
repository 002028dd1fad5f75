// Host-side launchers for every kernel of the training step. Each launcher enqueues on
// `stream`, never synchronises and never allocates; it returns the launch status.
#pragma once
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace gpt2k {

// Number of kernels this library has launched (every launcher adds its own count).
long long& launch_counter();
inline void count_launches(int n) { launch_counter() += n; }

enum class DType : int { F32 = 0, BF16 = 1 };

// ---------------------------------------------------------------- GEMM
// C(m, n) = sum_k A(m, k) * B(n, k), with
//   A(m, k) = a_mn ? A[k * lda + m] : A[m * lda + k]
//   B(n, k) = b_mn ? B[k * ldb + n] : B[n * ldb + k]
// and one of these epilogues on the fp32 accumulator v = C(m, n):
enum GemmEpi : int {
  EPI_STORE = 0,     // out = v (+ bias[n]) (+ resid[m, n])
  EPI_GELU_FWD = 1,  // u = v + bias[n]; out = gelu_tanh(u); pre = gelu_tanh'(u)
  EPI_GELU_BWD = 2,  // out = v * aux[m, n]  (aux: the pre of EPI_GELU_FWD)
  EPI_ACCUM = 3,     // accum[m, n] += scale * v   (fp32; wgrad into the grad buffer)
  // activation recomputation: the forward keeps the pre-activation u instead of gelu'(u),
  // the backward recomputes gelu'(u) and gelu(u) from it
  EPI_GELU_FWD_U = 4,  // u = v + bias[n]; out = gelu_tanh(u); pre = u
  EPI_GELU_BWD_U = 5,  // u = aux[m, n]; out = v * gelu_tanh'(u); pre = gelu_tanh(u)
  // lm_head with the cross-entropy's softmax statistics: out = v (the logits, rounded to the
  // activation type); per row and per 128 columns (a tile half) of the first `vocab`
  // columns, the log2-domain maximum m and sum of 2^(z log2 e - m) of the rounded logits,
  // written as float2 to ce_part[part * M + row], part = 2 * column tile + half
  EPI_LOGITS_CE = 6,
};

struct GemmArgs {
  int M = 0, N = 0, K = 0;
  const void* A = nullptr; long long lda = 0; bool a_mn = false;
  const void* B = nullptr; long long ldb = 0; bool b_mn = false;
  int epi = EPI_STORE;
  void* out = nullptr; long long ldo = 0;   // element type = the path's activation type
  const void* bias = nullptr;               // [N], activation type
  const void* resid = nullptr;              // [M, ldo]
  void* pre = nullptr;                      // EPI_GELU_FWD: gelu'(pre-activation) [M, ldo]
  const void* aux = nullptr;                // EPI_GELU_BWD: that gelu' [M, ldo]
  float* accum = nullptr;                   // EPI_ACCUM target [M, ldo] fp32
  float scale = 1.0f;
  int splits = 1;                           // EPI_ACCUM split-K count (tensor-core path)
  float* workspace = nullptr;               // splits * M * N fp32 when splits > 1
  // split-K partials of EPI_ACCUM: 0 = summed into accum right after the kernel (workspace
  // contents overwritten); 1 = scaled and added into the workspace, which holds the running
  // sums until the caller folds them in with splitk_fold (which also clears them)
  int defer_partials = 0;
  int* err = nullptr;                       // device error word
  int vocab = 0;                            // EPI_LOGITS_CE: columns that enter the softmax
  float* ce_part = nullptr;                 // EPI_LOGITS_CE: [ce_parts(N)][M] float2
};

// fp32 SIMT GEMM (all operands float).
cudaError_t gemm_f32(const GemmArgs& g, cudaStream_t s);
// bf16 tcgen05 GEMM (A, B, out, bias, resid, pre, aux bf16; accum fp32).
// Needs M, N, K > 0, N % 64 == 0, 16-byte aligned pointers and leading
// dimensions that are multiples of 8 elements.
cudaError_t gemm_bf16_tc(const GemmArgs& g, cudaStream_t s);
// Largest split-K factor gemm_bf16_tc would choose for an EPI_ACCUM call of this shape.
int gemm_tc_pick_splits(int M, int N, int K, int num_sms);
// Sum of split-K partials into the fp32 accumulator: accum += scale * sum_s ws[s].
cudaError_t splitk_reduce(float* accum, const float* ws, int splits, long long n,
                          float scale, cudaStream_t s);
// accum += sum_s ws[s] (fixed order), then ws = 0: folds deferred split-K partials.
cudaError_t splitk_fold(float* accum, float* ws, int splits, long long n, cudaStream_t s);
// The same, also writing fold_norm_parts(n) sums of squares of the final values to nparts.
cudaError_t splitk_fold_norm(float* accum, float* ws, int splits, long long n, float* nparts,
                             cudaStream_t s);
int fold_norm_parts(long long n);
int gemm_tc_num_sms();
// Number of softmax-statistics partials per row that EPI_LOGITS_CE writes for N columns.
int gemm_ce_parts(int N);
// Test hook of the bounded waits: later GEMM launches use wait_limit_ns (<= 0: the default
// 2 s) as every wait's limit, and with drop_first_signal the first accumulator of each
// block pair is never signalled ready (its epilogue wait runs out and reports
// DEV_ERR_TIMEOUT).
void gemm_tc_debug_waits(long long wait_limit_ns, int drop_first_signal);

// ---------------------------------------------------------------- elementwise
// x[b, t] = wte[tokens[b, t]] + wpe[pos0 + t]; pos0 read from pos_dev on the device if given
cudaError_t encoder_forward(DType t, void* x, const int* tokens, const void* wte, const void* wpe,
                            int B, int T, int C, int V, int* err, cudaStream_t s, int pos0 = 0,
                            const int* pos_dev = nullptr);
// Deterministic embedding backward: counting sort of positions by token id, then a
// per-id segmented sum in position order. scratch: encoder_backward_scratch_bytes(M, Vp).
size_t encoder_backward_scratch_bytes(int M, int Vp);
cudaError_t encoder_backward(DType t, float* dwte, float* dwpe, const void* dx, const int* tokens,
                             int B, int T, int C, int Vp, float scale, void* scratch,
                             cudaStream_t s);

cudaError_t layernorm_forward(DType t, void* y, float* mean, float* rstd, const void* x,
                              const void* w, const void* b, int M, int C, cudaStream_t s);
// dres (+)= dx of LayerNorm; dw, db += scale * column sums of dy*xhat and dy; when dproj
// is non-null, dproj += scale * column sums of the dres this call writes (the bias
// gradient of the projection that produced the residual stream). Two deterministic
// stages; partials: layernorm_backward_partials_floats(M, C, dproj != nullptr) floats.
// defer = 1 leaves the scaled per-block sums added into `partials` (which must start at
// zero and have room for LNB_MAX_BLOCKS blocks) for a later layernorm_fold.
int layernorm_backward_blocks(int M);
size_t layernorm_backward_partials_floats(int M, int C, bool dproj);
size_t layernorm_deferred_partials_floats(int C, bool dproj);
cudaError_t layernorm_backward(DType t, void* dres, int accumulate, float* dw, float* db,
                               float* dproj, const void* dy, const void* x, const void* w,
                               const float* mean, const float* rstd, int M, int C, float scale,
                               float* partials, int defer, cudaStream_t s);
// dw += sum of the deferred partials' first C columns, db the next C, dproj (if non-null)
// the last C; the partials are cleared.
// With nparts, also writes layernorm_fold_norm_parts(C, dproj) sums of squares of the
// final values (for the gradient norm), one per block.
cudaError_t layernorm_fold(float* dw, float* db, float* dproj, float* partials, int C,
                           cudaStream_t s, float* nparts = nullptr);
int layernorm_fold_norm_parts(int C, bool dproj);

// Fused classifier over the logits rows: per row loss = lse - z[y] over the first V
// columns; in place, logits become dlogits = (softmax - onehot) / M (0 in pad columns).
cudaError_t classifier(DType t, void* logits, float* losses, const int* targets, int M, int V,
                       int Vp, int* err, cudaStream_t s);
// The cross-entropy after an EPI_LOGITS_CE lm_head: per row, the partials combined in part
// order into lse; losses[row] = lse - z[y]; then, in place over the logits,
// dlogits = (softmax - onehot) / M over the first V columns and 0 in [V, Vp).
cudaError_t ce_from_partials(DType t, void* logits, float* losses, const float* ce_part,
                             int nparts, const int* targets, int M, int V, int Vp, float* lse_tmp,
                             int* err, cudaStream_t s);
// loss_out[0] = mean(losses[0..M))  (one block, fixed order)
cudaError_t mean_loss(float* loss_out, const float* losses, int M, cudaStream_t s);
// argmax over the first V columns of each row (lowest index on ties)
cudaError_t argmax_rows(DType t, int* out, const void* logits, int M, int V, int Vp,
                        cudaStream_t s);

// Bias gradient: db[n] += scale * sum_m dy[m, n] (two deterministic stages);
// partials: colsum_partials_floats(M, N) floats. defer = 1 leaves the scaled chunk sums
// added into `partials` (zero-initialised, colsum_deferred_partials_floats(M_max, N)
// floats) for a later bias_grad_fold.
size_t colsum_partials_floats(int M, int N);
size_t colsum_deferred_partials_floats(int M_max, int N);
cudaError_t bias_grad(DType t, float* db, const void* dy, int M, int N, float scale,
                      float* partials, int defer, cudaStream_t s);
cudaError_t bias_grad_fold(float* db, float* partials, int M_max, int N, cudaStream_t s,
                           float* nparts = nullptr);
int bias_grad_fold_norm_parts(int N);

// ---------------------------------------------------------------- attention
// qkv [B, T, 3C] -> out [B, T, C], lse [B, H, T] (natural log). The bf16 path runs the
// tcgen05 kernel (head size 64; err, when non-null, receives DEV_ERR_TIMEOUT).
cudaError_t attention_forward(DType t, void* out, float* lse, const void* qkv, int B, int T, int C,
                              int H, int* err, cudaStream_t s);
cudaError_t attention_forward_tc(void* out, float* lse, const void* qkv, int B, int T, int C,
                                 int H, int* err, cudaStream_t s);
// dout [B, T, C] -> dqkv [B, T, 3C]; Dbuf [B, H, T] scratch. The bf16 path runs the tcgen05
// dQ kernel (which also computes D = rowsum(dout * out) into Dbuf) and then the dK/dV
// kernel (needs T % 4 == 0).
cudaError_t attention_backward(DType t, void* dqkv, float* Dbuf, const void* dout,
                               const void* out, const void* qkv, const float* lse, int B, int T,
                               int C, int H, int* err, cudaStream_t s);
cudaError_t attention_backward_tc(void* dqkv, float* Dbuf, const void* dout, const void* out,
                                  const void* qkv, const float* lse, int B, int T, int C, int H,
                                  int* err, cudaStream_t s);

// ---------------------------------------------------------------- inference (KV cache)
// cache [Bmax][Tmax][2C] (K then V of each position): rows i < n of batch b of qkv
// ([B * Trows, 3C]) go to positions pos0 + i of the cache (pos0 read from pos_dev on the
// device if given; the host pos0 is then the value it will hold, for the bounds check)
cudaError_t kv_cache_store(DType t, void* cache, const void* qkv, int B, int Trows, int pos0,
                           int n, int Tmax, int C, cudaStream_t s, const int* pos_dev = nullptr);
// One query per (batch, head) at position t: q from qkv row b ([B, 3C], Q third), keys and
// values of positions 0..t from the cache; out [B, C] (heads concatenated); head size <= 128.
// t read from t_dev on the device if given (t_pos: the value it will hold, for the check).
// scratch: attention_decode_scratch_floats(B, H, Tmax, C / H) floats (the per-split partials).
cudaError_t attention_decode(DType t, void* out, const void* qkv, const void* cache, int B,
                             int t_pos, int Tmax, int C, int H, cudaStream_t s,
                             const int* t_dev, float* scratch);
size_t attention_decode_scratch_floats(int B, int H, int Tmax, int hs);
// out[b] = in[b * T + T - 1]
cudaError_t gather_last(int* out, const int* in, int B, int T, cudaStream_t s);
// bf16 Y = X W^T (+ bias, + residual, tanh-GELU epilogues) for at most 16 rows: the decode
// step's linear layers, streaming each weight once (gemv_rows_supported says which GemmArgs
// it takes: K-major operands, N and ldo even, K % 8 == 0, epilogues store / GELU forward)
bool gemv_rows_supported(const GemmArgs& g);
// Optional fusions of the decode step: ln_x set -> X = LayerNorm(ln_x; ln_w, ln_b) (eps 1e-5)
// computed inside (K <= 3072); kv_cache set (qkv projection, EPI_STORE, N = 3 kv_C) -> the
// K and V columns also go to cache[(m Tmax + *kv_pos) 2C + (n - C)].
struct GemvFuse {   // bf16 pointers
  const void* ln_x = nullptr; const void* ln_w = nullptr; const void* ln_b = nullptr;
  void* kv_cache = nullptr; int kv_Tmax = 0; int kv_C = 0; const int* kv_pos = nullptr;
};
cudaError_t gemv_rows(const GemmArgs& g, cudaStream_t s, const GemvFuse& f = GemvFuse());
// the device copy of the decode position: *pos_dev = set if set >= 0, else *pos_dev += add
cudaError_t decode_position(int* pos_dev, int set, int add, cudaStream_t s);

// ---------------------------------------------------------------- optimiser
// partials: norm_partials_count() floats; out[0] = ||g||, out[1] = clip coefficient
int norm_partials_count();
// ||g|| from partial sums of squares already written (partials[0, np)) plus those of the
// ranges d_ranges[2i], d_ranges[2i + 1] (offset, count) of g, which go to range_parts
// (inside partials[0, np)); out as grad_norm's.
cudaError_t grad_norm_finish(float* out, const float* partials, int np, const float* g,
                             const long long* d_ranges, int nranges, float* range_parts,
                             float max_norm, cudaStream_t s);
cudaError_t grad_norm(float* out, float* partials, const float* g, long long n, float max_norm,
                      cudaStream_t s);
// One AdamW step over n elements (t counts from 1). The gradient is multiplied by
// coef[0] (device, from grad_norm) when coef is non-null. p_bf16 (optional) receives the
// bf16 copy of the updated parameters.
cudaError_t adamw(float* p, const float* g, float* m, float* v, void* p_bf16, long long n,
                  float lr, float beta1, float beta2, float eps, float weight_decay, int t,
                  const float* coef, cudaStream_t s);
// dst[i] = bf16(src[i]) (round to nearest even)
cudaError_t to_bf16(void* dst, const float* src, long long n, cudaStream_t s);

}  // namespace gpt2k

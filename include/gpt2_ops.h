/*
 * gpt2_ops.h — single-kernel entry points of libgpt2, on caller-owned device buffers.
 * They run exactly the kernels gpt2_forward / gpt2_backward use and exist so that each
 * step of the training step can be checked on its own. Same conventions as gpt2.h:
 * int return (GPT2_OK or GPT2_ERR_*), work queued on `stream` (a cudaStream_t, NULL =
 * legacy default stream), no synchronisation, no allocation. `precision` selects the
 * element type of the activation operands: GPT2_FP32 (float) or GPT2_BF16 (bf16).
 */
#ifndef GPT2_OPS_H
#define GPT2_OPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  GPT2_EPI_STORE = 0,    /* out = v (+ bias[n]) (+ resid[m, n]) */
  GPT2_EPI_GELU_FWD = 1, /* u = v + bias[n]; out = gelu_tanh(u); pre = gelu_tanh'(u) */
  GPT2_EPI_GELU_BWD = 2, /* out = v * aux[m, n] (aux: the pre of GPT2_EPI_GELU_FWD) */
  GPT2_EPI_ACCUM = 3,    /* accum[m, n] += scale * v (fp32) */
  /* for activation recomputation (gpt2_config.recompute): */
  GPT2_EPI_GELU_FWD_U = 4, /* u = v + bias[n]; out = gelu_tanh(u); pre = u */
  GPT2_EPI_GELU_BWD_U = 5  /* u = aux[m, n]; out = v * gelu_tanh'(u); pre = gelu_tanh(u) */
};

/*
 * C(m, n) = sum_k A(m, k) B(n, k) for m < M, n < N, k < K, with
 *   A(m, k) = a_mn ? A[k*lda + m] : A[m*lda + k],  B(n, k) = b_mn ? B[k*ldb + n] : B[n*ldb + k]
 * followed by the epilogue `epi` on v = C(m, n); outputs are row-major with leading
 * dimension ldo (out, pre, aux, resid, accum). This is every Linear layer of the model:
 * forward Y = X W^T (K-major x K-major), dgrad dX = dY W (K-major x MN-major), wgrad
 * dW += dY^T X (MN-major x MN-major). GPT2_BF16 runs the tcgen05 tensor-core kernel and
 * needs N % 64 == 0 (any K), 16-byte aligned pointers and leading dimensions that
 * are multiples of 8; GPT2_EPI_ACCUM may then split K (splits = 0: automatic, needs
 * `workspace` of splits * M * N floats; 1: no split).
 */
int gpt2_op_gemm(int precision, int M, int N, int K, const void* A, int64_t lda, int a_mn,
                 const void* B, int64_t ldb, int b_mn, int epi, void* out, int64_t ldo,
                 const void* bias, const void* resid, void* pre, const void* aux, float* accum,
                 float scale, int splits, float* workspace, size_t workspace_bytes,
                 void* stream);

/* Causal attention over qkv [B, T, 3C] (Q, K, V thirds; head h = columns h*hs..) ->
   out [B, T, C] (heads concatenated) and lse [B, H, T] fp32 (natural log).
   GPT2_BF16 needs head size 64. */
int gpt2_op_attention_forward(int precision, void* out, float* lse, const void* qkv, int B,
                              int T, int C, int H, void* stream);
/* dout [B, T, C] -> dqkv [B, T, 3C]; Dbuf is fp32 scratch of 2 * B * H * T floats (its
   contents on return are unspecified). */
int gpt2_op_attention_backward(int precision, void* dqkv, float* Dbuf, const void* dout,
                               const void* out, const void* qkv, const float* lse, int B,
                               int T, int C, int H, void* stream);

/* y = LN(x) over rows of C (biased variance, eps 1e-5); mean, rstd fp32 [M]. */
int gpt2_op_layernorm_forward(int precision, void* y, float* mean, float* rstd, const void* x,
                              const void* w, const void* b, int M, int C, void* stream);
/* dres = (accumulate ? dres : 0) + dx; dw, db += scale * column sums (fp32).
   partials: gpt2_op_layernorm_partials_floats(M, C) floats of scratch. */
size_t gpt2_op_layernorm_partials_floats(int M, int C);
int gpt2_op_layernorm_backward(int precision, void* dres, int accumulate, float* dw, float* db,
                               const void* dy, const void* x, const void* w, const float* mean,
                               const float* rstd, int M, int C, float scale, float* partials,
                               void* stream);

/*
 * gpt2_op_layernorm_backward without a scratch argument and without any allocation. The
 * paper has no counterpart to this call; it exists for callers that cannot allocate device memory
 * once they run (a host whose memory manager reserved the device's memory for its own
 * pool at start-up, a plug-in interface that hands over only inputs and outputs, a loop
 * that must never reach cudaMalloc/cudaFree because they can synchronise the device).
 * Same arguments and results as gpt2_op_layernorm_backward minus `partials`.
 *   - Scratch: one fixed array of 2^20 floats (4 MiB) built into the library's device
 *     code. Every GPU that loads the library holds it until the process exits.
 *   - Limit: gpt2_op_layernorm_partials_floats(M, C) must be <= 2^20 (true for C <= 1771
 *     at any M, e.g. C = 768 or 1024); larger shapes return GPT2_ERR_ARG with a message
 *     and launch nothing.
 *   - Set-up: the first call on each device (made with that device current) looks up the
 *     array's device address with cudaGetSymbolAddress, and so does the first call after
 *     that device's CUDA context changed (cudaDeviceReset, a driver-API context); make
 *     those calls before any stream capture on that device.
 *   - Sharing: every call uses the same array. Calls whose work overlaps on the GPU (two
 *     streams, or two host threads) race on it; serialise them. Nothing in the array needs
 *     to start at zero: each call overwrites the partial sums it reads.
 */
int gpt2_op_layernorm_backward_noalloc(int precision, void* dres, int accumulate, float* dw,
                                       float* db, const void* dy, const void* x,
                                       const void* w, const float* mean, const float* rstd,
                                       int M, int C, float scale, void* stream);

/* Per row of logits [M, Vp]: losses[row] = logsumexp(z[:V]) - z[target]; logits become,
   in place, (softmax - onehot) / M over the first V columns and 0 in [V, Vp).
   err: device int, OR-ed with 4 when a target is out of range. */
int gpt2_op_classifier(int precision, void* logits, float* losses, const int32_t* targets,
                       int M, int V, int Vp, int* err, void* stream);

/*
 * The tied lm_head with the cross-entropy fused into it (bf16 only): logits = x wte^T
 * ([M, C] x [Vp, C]^T, rounded to bf16), whose GEMM epilogue also produces every row's
 * softmax statistics (maximum and sum of exponentials per 128 columns of the first V), then
 * one streaming pass: losses[row] = logsumexp(z[:V]) - z[target] and, in place over the
 * logits, dlogits = (softmax - onehot) / M in [0, V) and 0 in [V, Vp) (the loss and its
 * gradient of 「从零实现一个最小GPT」 三.7, F.cross_entropy with the mean over rows).
 * scratch: gpt2_op_lmhead_ce_scratch_bytes(M, Vp) bytes, 16-byte aligned. Vp % 64 == 0.
 * err: device int, OR-ed with 4 when a target is outside [0, V).
 */
size_t gpt2_op_lmhead_ce_scratch_bytes(int M, int Vp);
int gpt2_op_lmhead_cross_entropy(int M, int C, int V, int Vp, const void* x, const void* wte,
                                 const int32_t* targets, void* logits, float* losses,
                                 void* scratch, size_t scratch_bytes, int* err, void* stream);

/*
 * Test hook for failure detection; the pages have no counterpart. Every mbarrier wait in the
 * tensor-core GEMM is bounded: when one runs out, the kernel sets GPT2_ERR_TIMEOUT in the
 * device error word it was given (a handle's word: reported by its next gpt2_sync /
 * gpt2_get_loss), stops issuing work, lets its own copies and MMAs finish, frees its tensor
 * memory and returns, so the context and the handle stay usable. This call changes, for the
 * GEMM launches that follow it in this process, the limit of those waits (wait_limit_ns;
 * <= 0 restores the default of 2 s) and, with drop_first_signal = 1, withholds the signal
 * that the first accumulator of each block pair is ready, so that its epilogue's wait runs
 * out. Launches already recorded into a CUDA graph keep the settings they were recorded
 * with. Off by default; (0, 0) turns it off.
 */
int gpt2_debug_gemm_waits(int64_t wait_limit_ns, int drop_first_signal);

#ifdef __cplusplus
}
#endif

#endif /* GPT2_OPS_H */

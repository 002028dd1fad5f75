/*
 * gpt2.h — C ABI of libgpt2: one GPT-2 training step (forward, backward, global-norm
 * clip + AdamW) on one NVIDIA B300 (sm_103a).
 *
 * The model is the decoder-only transformer of 「从零实现一个最小GPT：代码讲解 + 知识点全解」
 * (sections 二.3-二.7, 三.3-三.7): token + position embedding, pre-LN blocks
 * x += proj(attn(LN1 x)); x += fcproj(gelu(fc(LN2 x))), causal softmax attention scaled by
 * 1/sqrt(head_size), a final LayerNorm, an lm_head and a mean next-token cross-entropy.
 * With these choices where that page and the GPT-2 pages differ:
 *   - the Q, K, V projections of all heads form one fused [3C, C] weight (rows: the Q,
 *     K, V thirds, heads in order within each third);
 *   - the GELU is the tanh approximation (「两小时手搓GPT-2」, section on the GELU
 *     approximation), not the exact erf form;
 *   - the lm_head is tied to the token embedding wte; logits are computed over a padded
 *     vocabulary Vp and the columns [V, Vp) are masked out of the softmax;
 *   - dropout is 0; LayerNorm has gamma and beta, eps 1e-5, biased variance; the bias
 *     flag covers the Linear layers only.
 * All parameters, gradients and AdamW moments live in one contiguous device buffer
 * (「手写训练脚本：不用框架，从零实现GPT训练流程」 section 二: one flat array that every
 * weight points into).
 *
 * Conventions for every call:
 *   - returns GPT2_OK (0) or a negative GPT2_ERR_* code; gpt2_last_error() gives a
 *     thread-local message for the last failure;
 *   - device pointers ("d_") are caller-owned and must stay valid until the work queued
 *     on the handle's stream has finished; host pointers ("h_") are read or written
 *     before the call returns;
 *   - work is queued on the stream given to gpt2_set_stream (default: the legacy default
 *     stream). Calls never synchronise unless they write a host result (h_loss,
 *     h_grad_norm, gpt2_get_loss, gpt2_copy_region);
 *   - no device memory is allocated after gpt2_create;
 *   - after any error the handle can still be passed to gpt2_destroy.
 */
#ifndef GPT2_H
#define GPT2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  GPT2_OK = 0,
  GPT2_ERR_INVALID_CONFIG = -1, /* sizes <= 0, C % H != 0, Vp < V, unsupported shape */
  GPT2_ERR_OOM = -2,            /* device allocation failed in gpt2_create */
  GPT2_ERR_CUDA = -3,           /* a CUDA call or kernel launch failed */
  GPT2_ERR_BAD_TOKEN = -4,      /* a token or target id outside [0, V) (reads clamped) */
  GPT2_ERR_SEQ_TOO_LONG = -5,   /* T > block_size or B > batch_size */
  GPT2_ERR_TIMEOUT = -6,        /* a bounded device-side wait gave up */
  GPT2_ERR_STATE = -7,          /* call out of order, e.g. backward without a forward */
  GPT2_ERR_ARG = -8             /* null handle/pointer, bad region, bad size */
};

enum { GPT2_FP32 = 0, GPT2_BF16 = 1 };

/* Regions of device memory that gpt2_copy_region / gpt2_region_ptr expose. */
enum {
  GPT2_REGION_PARAMS = 0,      /* fp32 master parameters, [num_params_padded] */
  GPT2_REGION_GRADS = 1,       /* fp32 gradients, same layout */
  GPT2_REGION_M = 2,           /* AdamW first moments, same layout */
  GPT2_REGION_V = 3,           /* AdamW second moments, same layout */
  GPT2_REGION_PARAMS_BF16 = 4, /* bf16 copy of the parameters (GPT2_BF16 only) */
  GPT2_REGION_LOGITS = 5,      /* [B*T, Vp] activation dtype; after a forward with
                                  targets it holds dlogits (written in place) */
  GPT2_REGION_LOSSES = 6,      /* fp32 per-position losses of the last forward [B*T] */
  GPT2_REGION_ENCODED = 7,     /* embedding output x0 [B*T, C], activation dtype */
  GPT2_REGION_ARGMAX = 8       /* int32 [B*T]: argmax over the first V logits of each
                                  position, written by a forward without targets */
};

typedef struct gpt2* gpt2_handle;

typedef struct {
  int32_t vocab_size;        /* V */
  int32_t padded_vocab_size; /* Vp >= V, multiple of 64 for GPT2_BF16; 0: V rounded up to 128 */
  int32_t block_size;        /* maximum sequence length T */
  int32_t n_layer;           /* L (>= 0) */
  int32_t n_head;            /* H */
  int32_t n_embd;            /* C, divisible by H */
  int32_t bias;              /* 1: Linear layers have biases */
  int32_t precision;         /* GPT2_FP32 or GPT2_BF16 (bf16 activations, fp32 master) */
  int32_t batch_size;        /* maximum B; sizes the activation memory */
  int32_t init;              /* 1: initialise weights from seed (see below); 0: all zero */
  uint64_t seed;
  int32_t recompute;         /* 1: activation recomputation (see below); 0: keep them all */
} gpt2_config;

/*
 * Create a handle: one device allocation for [params | grads | m | v | bf16 params] (the
 * flat array of 「手写训练脚本」 section 二, which every weight tensor indexes into), one
 * for activations and scratch. The initialisation with init = 1 follows the _init_weights
 * of 「从零实现一个最小GPT」 section 三.7 (normal(0, 0.02) weights, zero biases).
 * With recompute = 1 the activation memory holds, per layer, the MLP pre-activation u
 * instead of gelu(u) and gelu'(u), and no LayerNorm outputs: the backward recomputes both
 * LayerNorm outputs of a layer (from the kept residual streams, means and inverse standard
 * deviations) and gelu(u), gelu'(u) (from u, in the fc-proj input-gradient GEMM) where it
 * needs them. Per layer that is 2 [B*T, C] + [B*T, 4C] activation elements fewer, for a
 * few more kernels (memory relief, not speed). The forward's results are unchanged; the
 * gradients differ from recompute = 0 only by the rounding of u to the activation type. With init = 1 weights are N(0, 0.02) (residual
 * projections attnproj and fcproj N(0, 0.02/sqrt(2L))), Linear biases 0, LayerNorm
 * gamma 1 and beta 0, padded vocabulary rows 0, drawn with SplitMix64 in counter mode
 * (tensor i of the full table draws from stream draw(seed, i); normals by Box-Muller).
 * Grads, m and v start at zero and the AdamW step counter at 0.
 * GPT2_BF16 needs C/H == 64, C % 64 == 0 and Vp % 64 == 0.
 */
int gpt2_create(const gpt2_config* cfg, gpt2_handle* out);

/*
 * Host-only: write the initial flat parameter buffer gpt2_create would upload for this
 * config (init = 1) into h_out[0..n), n = the layout's element count (the n_buffer of
 * gpt2_num_params). Needs no GPU.
 */
int gpt2_host_init(const gpt2_config* cfg, float* h_out, size_t n);
/* Host-only: the parameter counts gpt2_num_params would report for this config. */
int gpt2_host_num_params(const gpt2_config* cfg, size_t* n_model, size_t* n_buffer);

/* Queue all later work on this cudaStream_t (NULL: the legacy default stream). */
int gpt2_set_stream(gpt2_handle h, void* cuda_stream);

/*
 * Forward pass on d_tokens [B, T] (int32, row-major, device): the model's forward(idx,
 * targets) of 「从零实现一个最小GPT」 sections 二.7 and 三.7 (embeddings, L blocks, final
 * LayerNorm, lm_head, mean cross-entropy). T <= block_size, B <= batch_size
 * (GPT2_ERR_SEQ_TOO_LONG otherwise).
 * With d_targets [B, T] (the next tokens): computes the mean cross-entropy over all B*T
 * positions and overwrites the logits with dlogits = (softmax - onehot)/(B*T), ready
 * for gpt2_backward. If h_loss is non-NULL the call waits and writes the loss there;
 * otherwise it stays on the device (gpt2_get_loss).
 * Without targets: keeps the logits and writes the argmax region.
 */
int gpt2_forward(gpt2_handle h, const int32_t* d_tokens, const int32_t* d_targets, int32_t B,
                 int32_t T, float* h_loss);

/*
 * Backward pass of the last forward (which must have had targets): the loss.backward() of
 * the training loop in 「从零实现一个最小GPT」 section 三.9, every layer's gradient written out
 * by hand (the chain rule through the same steps as the forward, in reverse). Adds
 * loss_scale * d(mean loss)/d(param) to the gradients (gradients accumulate, as in
 * PyTorch; use loss_scale = 1/accum for gradient accumulation). The bf16 path needs
 * T % 4 == 0 (GPT2_ERR_ARG otherwise).
 * Some contributions (the LayerNorm and bias gradients' per-block sums, the split-K
 * partial sums of the weight gradients) are kept in library-owned buffers across calls and
 * folded into GPT2_REGION_GRADS, in a fixed order, when the gradients are next read:
 * gpt2_adamw_step, gpt2_copy_region / gpt2_region_ptr of GPT2_REGION_GRADS. Read the
 * gradients through those calls, not through a pointer obtained before a backward.
 */
int gpt2_backward(gpt2_handle h, float loss_scale);

/*
 * One micro-batch of the gradient-accumulation loop of 「4.1 GPT-2 (124M) 复现」 section 2.3
 * (the caller sums accum of these with loss_scale = 1/accum before gpt2_adamw_step):
 * gpt2_forward with targets, then gpt2_backward(loss_scale), with the same
 * results and the same state afterwards (the loss stays on the device for gpt2_get_loss).
 * tokens and targets [B, T] int32 may be device or host pointers: they are copied with
 * cudaMemcpyAsync into library-owned buffers on the handle's stream (pinned host memory
 * keeps the copy asynchronous). Not in the pages: it is the host-side launch machinery.
 * Graph mode (the default, gpt2_set_graph_mode): the first call for a given
 * (B, T, loss_scale) runs eagerly and then records the forward and backward launches into a
 * CUDA graph on a private stream; later calls with the same triple replay that graph on the
 * handle's stream. Up to 8 graphs are kept (least recently created dropped first);
 * instantiating one takes driver resources but no device buffer. While profiling is enabled
 * (gpt2_profile_enable with a non-zero mask) the call runs eagerly so the events can
 * bracket each launch. Errors as gpt2_forward / gpt2_backward; a capture or instantiation
 * failure returns GPT2_ERR_CUDA after the micro-batch itself has run.
 */
int gpt2_forward_backward(gpt2_handle h, const int32_t* tokens, const int32_t* targets,
                          int32_t B, int32_t T, float loss_scale);
/*
 * Forward-only inference with a key/value cache and greedy (argmax) decoding: the
 * generation loop of 「从零实现一个最小GPT」 三.8, where each new token's logits come from
 * the last position, with the keys and values of earlier positions kept per layer instead
 * of recomputed. Tokens are device int32; sampling is not provided.
 * gpt2_prefill: runs the forward over the prompt d_tokens [B, T0] (B <= batch_size,
 *   T0 <= block_size), stores every layer's keys and values of the T0 positions in the
 *   handle's cache (sized at create for batch_size x block_size) and writes to d_next[B]
 *   the argmax over the first V logits of each row's last position (lowest index on ties).
 *   The logits region then holds all B*T0 rows' logits.
 * gpt2_decode_step: appends d_tokens[B] (one token per row, at position t = the current
 *   length) to the cached sequences: computes that position through every layer (its
 *   attention reads the cached keys and values of positions 0..t), stores its keys and
 *   values, and writes the argmax of its logits to d_next[B]; the logits region holds the
 *   B rows of logits. GPT2_ERR_STATE without a prefill, GPT2_ERR_ARG if B differs from the
 *   prefill's, GPT2_ERR_SEQ_TOO_LONG once t = block_size.
 * Any gpt2_forward / gpt2_forward_backward discards the cache (length 0).
 */
int gpt2_prefill(gpt2_handle h, const int32_t* d_tokens, int32_t B, int32_t T0, int32_t* d_next);
int gpt2_decode_step(gpt2_handle h, const int32_t* d_tokens, int32_t B, int32_t* d_next);
/* Current length of the cached sequences (0: no cache). */
int gpt2_decode_length(gpt2_handle h, int32_t* length);

/* Turn graph recording and replay in gpt2_forward_backward on (1) or off (0: every call
 * runs eagerly; the recorded graphs are destroyed). */
int gpt2_set_graph_mode(gpt2_handle h, int enabled);

/* Set every gradient (and every pending partial sum) to zero: the zero_grad of the training
   loop in 「从零实现一个最小GPT」 section 三.9. */
int gpt2_zero_grad(gpt2_handle h);

/*
 * One optimiser step over the whole flat buffer: the optimizer.step() of the training loop
 * in 「从零实现一个最小GPT」 section 三.9 (AdamW; the learning rate is the caller's, e.g. the
 * warm-up + cosine schedule whose numbers 「4.1 GPT-2 (124M) 复现」 section 2.3 lists). That
 * loop has no clipping step; the one here is the usual global-norm clip: if grad_clip > 0
 * the gradients are scaled by min(1, grad_clip / (||g||_2 + 1e-6)), computed on the
 * device; then AdamW
 * (decoupled weight decay applied to every parameter, bias-corrected moments, step
 * counter t incremented first, t = 1 on the first call). Gradients are left as they are.
 * If h_grad_norm is non-NULL the call waits and writes ||g||_2 (before clipping).
 */
int gpt2_adamw_step(gpt2_handle h, float lr, float beta1, float beta2, float eps,
                    float weight_decay, float grad_clip, float* h_grad_norm);

/* Wait for the stream and read the mean loss of the last forward with targets. Also
   reports GPT2_ERR_BAD_TOKEN / GPT2_ERR_TIMEOUT raised by device code since the last
   check. */
int gpt2_get_loss(gpt2_handle h, float* h_loss);

/* Wait for the stream and report (then clear) device-side errors. */
int gpt2_sync(gpt2_handle h);

/* Parameter table: number of tensors, and for tensor i its name, element offset in the
   flat buffer (each tensor starts on a 256-byte boundary), rank and shape (<= 3 dims). */
int gpt2_num_tensors(gpt2_handle h);
int gpt2_tensor_info(gpt2_handle h, int i, const char** name, size_t* offset, int* ndim,
                     int64_t* shape);
/* Parameter counts: unpadded (the model's own count, the tied wte counted once) and the
   number of elements of the flat buffer (padding included). */
int gpt2_num_params(gpt2_handle h, size_t* n_model, size_t* n_buffer);

/*
 * Copy `bytes` bytes between host memory and a region, starting `offset` bytes into the
 * region (to_device = 0: region -> h_buf; 1: h_buf -> region). Waits for the stream.
 * Writing GPT2_REGION_PARAMS also refreshes the bf16 copy.
 */
int gpt2_copy_region(gpt2_handle h, int region, size_t offset, void* h_buf, size_t bytes,
                     int to_device);
/* Device address and size in bytes of a region (no copy, no wait; for GPT2_REGION_GRADS
   the pending partial sums are first folded in, queued on the stream). */
int gpt2_region_ptr(gpt2_handle h, int region, void** d_ptr, size_t* bytes);

/* AdamW step counter (for checkpoint/resume together with PARAMS, M and V). */
int gpt2_get_step(gpt2_handle h, int64_t* t);
int gpt2_set_step(gpt2_handle h, int64_t t);

/*
 * Optional per-kernel-class timing with CUDA events recorded on the handle's stream
 * around every launch of the selected classes (bit mask of GPT2_PROF_*; 0 = off). The
 * events are created by gpt2_profile_enable (capacity pairs); launches beyond the
 * capacity are not timed until the next reset.
 * gpt2_profile_read waits for the stream and returns, per class, the number of launches
 * and their total duration in ms since the last reset, plus the algorithmic FLOPs
 * (GEMM classes) or bytes (others) those launches processed.
 */
enum {
  GPT2_PROF_GEMM = 1 << 0,
  GPT2_PROF_ATTENTION = 1 << 1,
  GPT2_PROF_LAYERNORM = 1 << 2,
  GPT2_PROF_CLASSIFIER = 1 << 3,
  GPT2_PROF_ENCODER = 1 << 4,
  GPT2_PROF_OPTIMIZER = 1 << 5,
  GPT2_PROF_OTHER = 1 << 6,
  GPT2_PROF_NUM_CLASSES = 7
};
int gpt2_profile_enable(gpt2_handle h, int class_mask, int capacity /* event pairs */);
int gpt2_profile_read(gpt2_handle h, int cls, int64_t* launches, double* total_ms,
                      double* work, int reset);

/* Number of CUDA kernels this library has launched in this process so far. */
int64_t gpt2_kernel_launches(void);

/* Device memory the handle holds, in bytes: the flat parameter block (params, grads, m, v,
   bf16 copy) and everything else (activations, scratch, deferred gradient partials). */
int gpt2_memory_bytes(gpt2_handle h, size_t* param_bytes, size_t* other_bytes);

/* Message of the last failed call on this thread ("" if none). */
const char* gpt2_last_error(void);

/* Release everything the handle owns. NULL-safe. */
void gpt2_destroy(gpt2_handle h);

#ifdef __cplusplus
}
#endif

#endif /* GPT2_H */

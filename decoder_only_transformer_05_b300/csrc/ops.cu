// Single-kernel entry points (include/gpt2_ops.h): thin wrappers over launch.h.
#include "../../include/gpt2.h"
#include "../../include/gpt2_ops.h"
#include "launch.h"

using namespace gpt2k;

int gpt2_set_error(int code, const char* msg);   // gpt2.cu

static int status(cudaError_t e) {
  if (e == cudaSuccess) return GPT2_OK;
  if (e == cudaErrorInvalidValue)
    return gpt2_set_error(GPT2_ERR_ARG, "unsupported shape, alignment or argument");
  return gpt2_set_error(GPT2_ERR_CUDA, cudaGetErrorString(e));
}
static DType dtype(int precision) { return precision == GPT2_BF16 ? DType::BF16 : DType::F32; }

extern "C" int gpt2_op_gemm(int precision, int M, int N, int K, const void* A, int64_t lda,
                            int a_mn, const void* B, int64_t ldb, int b_mn, int epi, void* out,
                            int64_t ldo, const void* bias, const void* resid, void* pre,
                            const void* aux, float* accum, float scale, int splits,
                            float* workspace, size_t workspace_bytes, void* stream) {
  if (epi < 0 || epi > 5) return gpt2_set_error(GPT2_ERR_ARG, "bad epilogue (the lm_head cross-entropy has its own entry point)");
  GemmArgs g;
  g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = lda; g.a_mn = a_mn != 0;
  g.B = B; g.ldb = ldb; g.b_mn = b_mn != 0;
  g.epi = epi; g.out = out; g.ldo = ldo;
  g.bias = bias; g.resid = resid; g.pre = pre; g.aux = aux;
  g.accum = accum; g.scale = scale;
  g.splits = splits; g.workspace = workspace;
  cudaStream_t s = (cudaStream_t)stream;
  if (precision != GPT2_BF16) return status(gemm_f32(g, s));
  if (epi == EPI_ACCUM) {
    int sp = splits > 0 ? splits : gemm_tc_pick_splits(M, N, K, gemm_tc_num_sms());
    if (sp > 1 && (!workspace || workspace_bytes < (size_t)sp * M * N * sizeof(float)))
      return gpt2_set_error(GPT2_ERR_ARG, "split-K workspace missing or too small");
    g.splits = sp;
  }
  return status(gemm_bf16_tc(g, s));
}

extern "C" int gpt2_op_attention_forward(int precision, void* out, float* lse, const void* qkv,
                                         int B, int T, int C, int H, void* stream) {
  return status(attention_forward(dtype(precision), out, lse, qkv, B, T, C, H, nullptr,
                                  (cudaStream_t)stream));
}

extern "C" int gpt2_op_attention_backward(int precision, void* dqkv, float* Dbuf,
                                          const void* dout, const void* out, const void* qkv,
                                          const float* lse, int B, int T, int C, int H,
                                          void* stream) {
  return status(attention_backward(dtype(precision), dqkv, Dbuf, dout, out, qkv, lse, B, T, C,
                                   H, nullptr, (cudaStream_t)stream));
}

extern "C" int gpt2_op_layernorm_forward(int precision, void* y, float* mean, float* rstd,
                                         const void* x, const void* w, const void* b, int M,
                                         int C, void* stream) {
  return status(layernorm_forward(dtype(precision), y, mean, rstd, x, w, b, M, C,
                                  (cudaStream_t)stream));
}

extern "C" size_t gpt2_op_layernorm_partials_floats(int M, int C) {
  return layernorm_backward_partials_floats(M, C, false);
}

extern "C" int gpt2_op_layernorm_backward(int precision, void* dres, int accumulate, float* dw,
                                          float* db, const void* dy, const void* x,
                                          const void* w, const float* mean, const float* rstd,
                                          int M, int C, float scale, float* partials,
                                          void* stream) {
  return status(layernorm_backward(dtype(precision), dres, accumulate, dw, db, nullptr, dy, x,
                                   w, mean, rstd, M, C, scale, partials, 0, (cudaStream_t)stream));
}

extern "C" int gpt2_op_classifier(int precision, void* logits, float* losses,
                                  const int32_t* targets, int M, int V, int Vp, int* err,
                                  void* stream) {
  return status(classifier(dtype(precision), logits, losses, targets, M, V, Vp, err,
                           (cudaStream_t)stream));
}

extern "C" int gpt2_debug_gemm_waits(int64_t wait_limit_ns, int drop_first_signal) {
  gemm_tc_debug_waits((long long)wait_limit_ns, drop_first_signal);
  return GPT2_OK;
}

extern "C" size_t gpt2_op_lmhead_ce_scratch_bytes(int M, int Vp) {
  if (M <= 0 || Vp <= 0) return 0;
  return (size_t)gemm_ce_parts(Vp) * M * 8 + (size_t)M * 4 + 256;
}

extern "C" int gpt2_op_lmhead_cross_entropy(int M, int C, int V, int Vp, const void* x,
                                            const void* wte, const int32_t* targets,
                                            void* logits, float* losses, void* scratch,
                                            size_t scratch_bytes, int* err, void* stream) {
  if (M <= 0 || C <= 0 || V <= 0 || Vp < V || !scratch || ((uintptr_t)scratch & 15u))
    return gpt2_set_error(GPT2_ERR_ARG, "bad size or scratch");
  if (scratch_bytes < gpt2_op_lmhead_ce_scratch_bytes(M, Vp))
    return gpt2_set_error(GPT2_ERR_ARG, "scratch too small");
  cudaStream_t s = (cudaStream_t)stream;
  const size_t part_bytes = (size_t)gemm_ce_parts(Vp) * M * 8;
  float* part = (float*)scratch;
  float* lse = (float*)((char*)scratch + (part_bytes + 255) / 256 * 256);
  GemmArgs g;
  g.M = M; g.N = Vp; g.K = C;
  g.A = x; g.lda = C; g.a_mn = false;
  g.B = wte; g.ldb = C; g.b_mn = false;
  g.epi = EPI_LOGITS_CE; g.out = logits; g.ldo = Vp;
  g.vocab = V; g.ce_part = part; g.err = err;
  int rc = status(gemm_bf16_tc(g, s));
  if (rc) return rc;
  return status(ce_from_partials(DType::BF16, logits, losses, part, gemm_ce_parts(Vp), targets, M,
                                 V, Vp, lse, err, s));
}

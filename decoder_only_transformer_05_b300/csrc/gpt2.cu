// libgpt2: the C ABI declared in include/gpt2.h. Owns the flat parameter buffer
// [params | grads | m | v | bf16 params], the activation arena and scratch, and queues
// the training step's kernels (launch.h) on the caller's stream.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "../../include/gpt2.h"
#include "common.cuh"
#include "launch.h"

using namespace gpt2k;

// ------------------------------------------------------------------ errors
static thread_local std::string g_last_error;

static int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int gpt2_set_error(int code, const char* msg) { return fail(code, "%s", msg); }

#define CK(x)                                                                               \
  do {                                                                                      \
    cudaError_t e_ = (x);                                                                   \
    if (e_ != cudaSuccess)                                                                  \
      return fail(GPT2_ERR_CUDA, "%s failed: %s", #x, cudaGetErrorString(e_));              \
  } while (0)

// ------------------------------------------------------------------ init (SplitMix64)
// Counter-mode SplitMix64 (Steele, Lea, Flood, OOPSLA 2014):
// draw(k, i) = mix(k + (i + 1) * 0x9E3779B97F4A7C15); stream j of seed s has key draw(s, j);
// uniforms are (draw >> 11) * 2^-53; normals are Box-Muller pairs over consecutive uniforms.
static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
static inline uint64_t sm64_draw(uint64_t key, uint64_t i) {
  return sm64_mix(key + (i + 1) * 0x9E3779B97F4A7C15ull);
}
static inline double sm64_uniform(uint64_t key, uint64_t i) {
  return (double)(sm64_draw(key, i) >> 11) * (1.0 / 9007199254740992.0);
}
// element i of the normal stream with this key
static void fill_normal(float* dst, size_t n, uint64_t key, double std) {
  const unsigned nth = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
  std::vector<std::thread> pool;
  const size_t pairs = (n + 1) / 2;
  for (unsigned t = 0; t < nth; ++t) {
    pool.emplace_back([=] {
      size_t p0 = pairs * t / nth, p1 = pairs * (t + 1) / nth;
      for (size_t pr = p0; pr < p1; ++pr) {
        double u0 = sm64_uniform(key, 2 * pr), u1 = sm64_uniform(key, 2 * pr + 1);
        double r = std::sqrt(-2.0 * std::log1p(-u0));
        double a = 2.0 * M_PI * u1;
        size_t i = 2 * pr;
        dst[i] = (float)(std * (r * std::cos(a)));
        if (i + 1 < n) dst[i + 1] = (float)(std * (r * std::sin(a)));
      }
    });
  }
  for (auto& th : pool) th.join();
}

// ------------------------------------------------------------------ handle
enum TensorId {
  T_WTE, T_WPE, T_LN1W, T_LN1B, T_QKVW, T_QKVB, T_ATTPROJW, T_ATTPROJB, T_LN2W, T_LN2B,
  T_FCW, T_FCB, T_FCPROJW, T_FCPROJB, T_LNFW, T_LNFB, T_COUNT
};
static const char* kTensorNames[T_COUNT] = {
    "wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
    "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb"};

struct TensorInfo {
  int id;
  size_t offset, numel;
  int ndim;
  int64_t shape[3];
};

struct ProfPair { cudaEvent_t a, b; int cls; double work; };

struct gpt2 {
  gpt2_config cfg{};
  int V = 0, Vp = 0, T = 0, L = 0, H = 0, C = 0, Bmax = 0;
  bool is_bf16 = false, bias = false, recompute = false;
  DType dt = DType::F32;
  size_t es = 4;   // activation element size
  cudaStream_t stream = nullptr;

  std::vector<TensorInfo> tensors;
  int index[T_COUNT];
  size_t P = 0, n_model = 0;

  char* pmem = nullptr;   // params block
  size_t pmem_bytes = 0;
  float *params = nullptr, *grads = nullptr, *m = nullptr, *v = nullptr;
  bf16* params_bf16 = nullptr;
  char* amem = nullptr;   // activations + scratch
  size_t amem_bytes = 0;

  // activations (element type per path). With recompute, ln1[l] and ln2[l] all point at one
  // shared LayerNorm-output buffer and fcg[l] at one shared GELU-output buffer, and fch[l]
  // holds the pre-activation u (otherwise gelu'(u)).
  std::vector<void*> x;   // L+1 residual streams
  std::vector<void*> ln1, qkv, att, xmid, ln2, fch, fcg;
  std::vector<float*> ln1_mean, ln1_rstd, ln2_mean, ln2_rstd, lse;
  void *lnf = nullptr, *logits = nullptr;
  float *lnf_mean = nullptr, *lnf_rstd = nullptr, *losses = nullptr;
  int* argmax = nullptr;
  // inference: per layer the keys and values of every position so far, [Bmax][T][2C]
  void* kvcache = nullptr;
  int dec_B = 0, dec_len = 0;   // batch and length of the cached sequences (0: none)
  void* kv(int layer) { return (char*)kvcache + (size_t)layer * Bmax * T * 2 * C * es; }
  // backward scratch
  void *dres = nullptr, *dln = nullptr, *datt = nullptr, *dqkv = nullptr, *dfch = nullptr;
  float* Dbuf = nullptr;
  float* splitk_ws = nullptr;
  float* norm_partials = nullptr;
  float* ce_part = nullptr;   // bf16 lm_head cross-entropy: softmax-statistics partials
  float* ce_lse = nullptr;    // and the per-row log2-domain lse
  void* enc_scratch = nullptr;
  int* d_err = nullptr;
  float* d_loss = nullptr;
  float* d_norm = nullptr;

  // Deferred gradient partial sums. The backward adds each micro-batch's per-block or
  // per-split sums into these buffers (each element receives one addition per micro-batch,
  // so the result does not depend on scheduling); flush_grads() folds them into the flat
  // gradient buffer and clears them, once per optimiser step or when gradients are read.
  struct DefWgrad { float* grad; float* ws; int splits; size_t n; };   // split-K weight grads
  struct DefLN { float* dw; float* db; float* dproj; float* part; };   // LayerNorm (+ bias)
  struct DefCol { float* db; float* part; int N; };                    // bias column sums
  std::vector<DefWgrad> def_wg;   // [layer * 4 + kind], kinds: qkv, attproj, fc, fcproj
  std::vector<DefLN> def_ln;      // LN1 [0, L), LN2 [L, 2L), lnf 2L
  std::vector<DefCol> def_col;    // fc bias [0, L), qkv bias [L, 2L)
  char* dmem = nullptr;
  size_t dmem_bytes = 0;
  bool grads_pending = false;
  // Gradient norm from the folds: when gpt2_adamw_step itself folds the pending partials,
  // each fold also writes sums of squares of the final values it writes (norm_slots, in
  // fold order), and only the gradient ranges no fold finalises (wte, wpe, weights without
  // split partials) are read again for the norm, as items of at most 256K elements.
  float* norm_slots = nullptr;
  int norm_fold_slots = 0, norm_items = 0;
  long long* norm_ranges = nullptr;   // device: [norm_items][offset, count]

  // gpt2_forward_backward: token/target copies and one CUDA graph of the micro-batch per
  // (B, T, loss scale)
  int32_t *mb_tok = nullptr, *mb_tgt = nullptr;
  struct MicroGraph { int B, T; float scale; cudaGraphExec_t exec; long long launches; };
  std::vector<MicroGraph> graphs;
  bool graph_mode = true;
  cudaStream_t cap_stream = nullptr;
  // gpt2_decode_step: the position on the device (read by the replayed kernels) and one
  // CUDA graph of the step for the current decode batch
  int* d_pos = nullptr;
  cudaGraphExec_t dec_exec = nullptr;
  int dec_exec_B = 0;
  long long dec_exec_launches = 0;

  // state
  int last_B = 0, last_T = 0;
  bool have_targets = false;
  const int* last_tokens = nullptr;
  int64_t step = 0;

  // profiling
  int prof_mask = 0;
  std::vector<ProfPair> prof;
  size_t prof_used = 0;
  int64_t prof_launches[GPT2_PROF_NUM_CLASSES] = {};
  double prof_ms[GPT2_PROF_NUM_CLASSES] = {}, prof_work[GPT2_PROF_NUM_CLASSES] = {};

  // weight as the path consumes it: the bf16 copy (bf16 path) or the fp32 master
  const void* pw(int id, int layer = 0) {
    const TensorInfo& t = tensors[index[id]];
    size_t per = layer ? t.numel / L : 0;
    if (is_bf16) return params_bf16 + t.offset + per * layer;
    return params + t.offset + per * layer;
  }
  float* gw(int id, int layer = 0) {
    const TensorInfo& t = tensors[index[id]];
    size_t per = layer ? t.numel / L : 0;
    return grads + t.offset + per * layer;
  }
  bool has(int id) const { return index[id] >= 0; }
};

// ------------------------------------------------------------------ profiling helpers
static size_t prof_begin(gpt2* h, int cls) {
  if (!(h->prof_mask & (1 << cls)) || h->prof_used >= h->prof.size()) return (size_t)-1;
  size_t i = h->prof_used++;
  h->prof[i].cls = cls;
  cudaEventRecord(h->prof[i].a, h->stream);
  return i;
}
static void prof_end(gpt2* h, size_t i, double work) {
  if (i == (size_t)-1) return;
  h->prof[i].work = work;
  cudaEventRecord(h->prof[i].b, h->stream);
}
enum { PC_GEMM = 0, PC_ATTN = 1, PC_LN = 2, PC_CLS = 3, PC_ENC = 4, PC_OPT = 5, PC_OTHER = 6 };

// ------------------------------------------------------------------ layout
static int build_layout(gpt2* h) {
  const int64_t V = h->V, Vp = h->Vp, T = h->T, L = h->L, C = h->C;
  struct Row { int id; int ndim; int64_t s[3]; };
  std::vector<Row> rows = {
      {T_WTE, 2, {Vp, C, 0}},        {T_WPE, 2, {T, C, 0}},
      {T_LN1W, 2, {L, C, 0}},        {T_LN1B, 2, {L, C, 0}},
      {T_QKVW, 3, {L, 3 * C, C}},    {T_QKVB, 2, {L, 3 * C, 0}},
      {T_ATTPROJW, 3, {L, C, C}},    {T_ATTPROJB, 2, {L, C, 0}},
      {T_LN2W, 2, {L, C, 0}},        {T_LN2B, 2, {L, C, 0}},
      {T_FCW, 3, {L, 4 * C, C}},     {T_FCB, 2, {L, 4 * C, 0}},
      {T_FCPROJW, 3, {L, C, 4 * C}}, {T_FCPROJB, 2, {L, C, 0}},
      {T_LNFW, 1, {C, 0, 0}},        {T_LNFB, 1, {C, 0, 0}}};
  size_t off = 0;
  for (int i = 0; i < T_COUNT; ++i) h->index[i] = -1;
  h->n_model = 0;
  for (auto& r : rows) {
    bool is_bias = r.id == T_QKVB || r.id == T_ATTPROJB || r.id == T_FCB || r.id == T_FCPROJB;
    if (is_bias && !h->bias) continue;
    TensorInfo t;
    t.id = r.id;
    t.ndim = r.ndim;
    t.numel = 1;
    for (int d = 0; d < 3; ++d) t.shape[d] = d < r.ndim ? r.s[d] : 0;
    for (int d = 0; d < r.ndim; ++d) t.numel *= (size_t)r.s[d];
    t.offset = off;
    off += (t.numel + 63) / 64 * 64;   // 256-byte aligned starts (fp32)
    h->index[r.id] = (int)h->tensors.size();
    h->tensors.push_back(t);
    h->n_model += t.numel;
  }
  h->n_model -= (size_t)(Vp - V) * C;
  h->P = off;
  return GPT2_OK;
}

static size_t align256(size_t b) { return (b + 255) / 256 * 256; }


// Initial parameters into a host buffer of h->P floats (zeros where nothing is drawn).
static void fill_init(const gpt2* h, float* host) {
  for (auto& t : h->tensors) {
    float* dst = host + t.offset;
    switch (t.id) {
      case T_LN1W: case T_LN2W: case T_LNFW:
        for (size_t i = 0; i < t.numel; ++i) dst[i] = 1.0f;
        break;
      case T_WTE: case T_WPE: case T_QKVW: case T_FCW: case T_ATTPROJW: case T_FCPROJW: {
        double std = 0.02;
        if (t.id == T_ATTPROJW || t.id == T_FCPROJW) std = 0.02 / std::sqrt(2.0 * h->L);
        size_t n = t.id == T_WTE ? (size_t)h->V * h->C : t.numel;
        fill_normal(dst, n, sm64_draw(h->cfg.seed, (uint64_t)t.id), std);
        break;
      }
      default: break;   // biases and LayerNorm betas stay 0
    }
  }
}

static int validate(gpt2_config& cfg) {
  if (cfg.padded_vocab_size == 0) cfg.padded_vocab_size = (cfg.vocab_size + 127) / 128 * 128;
  if (cfg.vocab_size <= 0 || cfg.block_size <= 0 || cfg.n_layer < 0 || cfg.n_head <= 0 ||
      cfg.n_embd <= 0 || cfg.batch_size <= 0 || cfg.n_embd % cfg.n_head ||
      cfg.padded_vocab_size < cfg.vocab_size ||
      (cfg.precision != GPT2_FP32 && cfg.precision != GPT2_BF16))
    return fail(GPT2_ERR_INVALID_CONFIG, "invalid configuration");
  if (cfg.precision == GPT2_BF16 &&
      (cfg.n_embd / cfg.n_head != 64 || cfg.n_embd % 64 || cfg.padded_vocab_size % 64))
    return fail(GPT2_ERR_INVALID_CONFIG,
                "bf16 path needs head size 64, n_embd %% 64 == 0 and padded vocab %% 64 == 0");
  if (cfg.precision == GPT2_FP32 && cfg.n_embd % 4)
    return fail(GPT2_ERR_INVALID_CONFIG, "fp32 path needs n_embd %% 4 == 0");
  if (cfg.n_embd > 2048) return fail(GPT2_ERR_INVALID_CONFIG, "n_embd > 2048 unsupported");
  return GPT2_OK;
}

static void setup_shape(gpt2* h, const gpt2_config& cfg) {
  h->cfg = cfg;
  h->V = cfg.vocab_size; h->Vp = cfg.padded_vocab_size; h->T = cfg.block_size;
  h->L = cfg.n_layer; h->H = cfg.n_head; h->C = cfg.n_embd; h->Bmax = cfg.batch_size;
  h->is_bf16 = cfg.precision == GPT2_BF16;
  h->bias = cfg.bias != 0;
  h->recompute = cfg.recompute != 0;
  h->dt = h->is_bf16 ? DType::BF16 : DType::F32;
  h->es = h->is_bf16 ? 2 : 4;
  build_layout(h);
}

extern "C" int gpt2_host_num_params(const gpt2_config* cfg_in, size_t* n_model,
                                    size_t* n_buffer) {
  if (!cfg_in) return fail(GPT2_ERR_ARG, "null argument");
  gpt2_config cfg = *cfg_in;
  int rc = validate(cfg);
  if (rc) return rc;
  gpt2 tmp;
  setup_shape(&tmp, cfg);
  if (n_model) *n_model = tmp.n_model;
  if (n_buffer) *n_buffer = tmp.P;
  return GPT2_OK;
}

extern "C" int gpt2_host_init(const gpt2_config* cfg_in, float* h_out, size_t n) {
  if (!cfg_in || !h_out) return fail(GPT2_ERR_ARG, "null argument");
  gpt2_config cfg = *cfg_in;
  int rc = validate(cfg);
  if (rc) return rc;
  gpt2 tmp;
  setup_shape(&tmp, cfg);
  if (n != tmp.P) return fail(GPT2_ERR_ARG, "buffer has %zu elements, layout needs %zu", n, tmp.P);
  std::fill(h_out, h_out + n, 0.0f);
  fill_init(&tmp, h_out);
  return GPT2_OK;
}

static int plan_norm(gpt2* h, std::vector<long long>& items);

// ------------------------------------------------------------------ create / destroy
extern "C" int gpt2_create(const gpt2_config* cfg_in, gpt2_handle* out) {
  if (!cfg_in || !out) return fail(GPT2_ERR_ARG, "null argument");
  *out = nullptr;
  gpt2_config cfg = *cfg_in;
  int vrc = validate(cfg);
  if (vrc) return vrc;
  gpt2* h = new gpt2();
  setup_shape(h, cfg);

  // ---- parameter block
  const size_t P = h->P;
  size_t pbytes = 4 * align256(P * 4) + (h->is_bf16 ? align256(P * 2) : 0);
  h->pmem_bytes = pbytes;
  if (cudaError_t e = cudaMalloc(&h->pmem, pbytes); e != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return fail(e == cudaErrorMemoryAllocation ? GPT2_ERR_OOM : GPT2_ERR_CUDA,
                "cudaMalloc of %zu bytes for parameters failed: %s", pbytes,
                cudaGetErrorString(e));
  }
  h->params = (float*)h->pmem;
  h->grads = (float*)(h->pmem + align256(P * 4));
  h->m = (float*)(h->pmem + 2 * align256(P * 4));
  h->v = (float*)(h->pmem + 3 * align256(P * 4));
  if (h->is_bf16) h->params_bf16 = (bf16*)(h->pmem + 4 * align256(P * 4));

  // ---- activation arena
  const size_t M = (size_t)h->Bmax * h->T, C = h->C, L = h->L, es = h->es;
  const size_t BHT = (size_t)h->Bmax * h->H * h->T;
  size_t need = 0;
  auto plan = [&](size_t bytes) { size_t o = need; need += align256(bytes); return o; };
  std::vector<size_t> o_x(L + 1), o_ln1(L), o_qkv(L), o_att(L), o_xmid(L), o_ln2(L), o_fch(L),
      o_fcg(L), o_m1(L), o_r1(L), o_m2(L), o_r2(L), o_lse(L);
  for (size_t l = 0; l <= L; ++l) o_x[l] = plan(M * C * es);
  const size_t o_ln_shared = h->recompute ? plan(M * C * es) : 0;
  const size_t o_g_shared = h->recompute ? plan(M * 4 * C * es) : 0;
  for (size_t l = 0; l < L; ++l) {
    o_ln1[l] = h->recompute ? o_ln_shared : plan(M * C * es);
    o_qkv[l] = plan(M * 3 * C * es); o_att[l] = plan(M * C * es);
    o_xmid[l] = plan(M * C * es);
    o_ln2[l] = h->recompute ? o_ln_shared : plan(M * C * es);
    o_fch[l] = plan(M * 4 * C * es);
    o_fcg[l] = h->recompute ? o_g_shared : plan(M * 4 * C * es);
    o_m1[l] = plan(M * 4); o_r1[l] = plan(M * 4); o_m2[l] = plan(M * 4); o_r2[l] = plan(M * 4);
    o_lse[l] = plan(BHT * 4);
  }
  size_t o_lnf = plan(M * C * es), o_lnfm = plan(M * 4), o_lnfr = plan(M * 4);
  size_t o_logits = plan(M * (size_t)h->Vp * es), o_losses = plan(M * 4), o_argmax = plan(M * 4);
  size_t o_dres = plan(M * C * es), o_dln = plan(M * C * es), o_datt = plan(M * C * es);
  size_t o_dqkv = plan(M * 3 * C * es), o_dfch = plan(M * 4 * C * es);
  // the attention backward's -D, -lse log2e rows; greedy decoding's attention partials
  size_t o_D = plan(std::max((size_t)(2 * BHT * 4),
                             attention_decode_scratch_floats((int)h->Bmax, (int)h->H, (int)h->T,
                                                             (int)(C / h->H)) * 4));
  // split-K workspace for a tied lm_head gradient that needed one (it does not at these
  // shapes; the per-layer weight gradients use the deferred buffers below)
  size_t ws = 0;
  if (h->is_bf16) {
    int sp = gemm_tc_pick_splits(h->Vp, (int)C, (int)M, gemm_tc_num_sms());
    if (sp > 1) ws = (size_t)sp * h->Vp * C * 4;
  }
  size_t o_ws = plan(ws + 256);
  size_t o_np = plan((size_t)norm_partials_count() * 4);
  size_t o_enc = plan(encoder_backward_scratch_bytes((int)M, h->Vp));
  size_t o_err = plan(64), o_loss = plan(64), o_norm = plan(64);
  size_t o_mbtok = plan(M * 4), o_mbtgt = plan(M * 4), o_pos = plan(256);
  size_t o_kv = plan(L * M * 2 * C * es);
  const size_t ce_parts = h->is_bf16 ? (size_t)gemm_ce_parts(h->Vp) : 0;
  size_t o_cep = plan(ce_parts * M * 8 + 16), o_cel = plan(M * 4);
  h->amem_bytes = need;
  if (cudaError_t e = cudaMalloc(&h->amem, need); e != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->pmem);
    delete h;
    return fail(e == cudaErrorMemoryAllocation ? GPT2_ERR_OOM : GPT2_ERR_CUDA,
                "cudaMalloc of %zu bytes for activations failed: %s", need,
                cudaGetErrorString(e));
  }
  char* a = h->amem;
  for (size_t l = 0; l <= L; ++l) h->x.push_back(a + o_x[l]);
  for (size_t l = 0; l < L; ++l) {
    h->ln1.push_back(a + o_ln1[l]); h->qkv.push_back(a + o_qkv[l]); h->att.push_back(a + o_att[l]);
    h->xmid.push_back(a + o_xmid[l]); h->ln2.push_back(a + o_ln2[l]);
    h->fch.push_back(a + o_fch[l]); h->fcg.push_back(a + o_fcg[l]);
    h->ln1_mean.push_back((float*)(a + o_m1[l])); h->ln1_rstd.push_back((float*)(a + o_r1[l]));
    h->ln2_mean.push_back((float*)(a + o_m2[l])); h->ln2_rstd.push_back((float*)(a + o_r2[l]));
    h->lse.push_back((float*)(a + o_lse[l]));
  }
  h->lnf = a + o_lnf; h->lnf_mean = (float*)(a + o_lnfm); h->lnf_rstd = (float*)(a + o_lnfr);
  h->logits = a + o_logits; h->losses = (float*)(a + o_losses); h->argmax = (int*)(a + o_argmax);
  h->dres = a + o_dres; h->dln = a + o_dln; h->datt = a + o_datt; h->dqkv = a + o_dqkv;
  h->dfch = a + o_dfch; h->Dbuf = (float*)(a + o_D);
  h->splitk_ws = (float*)(a + o_ws); h->norm_partials = (float*)(a + o_np);
  h->enc_scratch = a + o_enc;
  h->d_err = (int*)(a + o_err); h->d_loss = (float*)(a + o_loss); h->d_norm = (float*)(a + o_norm);
  h->mb_tok = (int32_t*)(a + o_mbtok); h->mb_tgt = (int32_t*)(a + o_mbtgt);
  h->d_pos = (int*)(a + o_pos);
  h->kvcache = a + o_kv;
  h->ce_part = (float*)(a + o_cep); h->ce_lse = (float*)(a + o_cel);

  // ---- deferred gradient partials (zeroed; see the handle)
  std::vector<long long> norm_items;
  {
    size_t dneed = 0;
    auto dplan = [&](size_t floats) { size_t o = dneed; dneed += align256(floats * 4); return o; };
    struct WgPlan { int id; int N, K; };
    const WgPlan kinds[4] = {{T_QKVW, 3 * (int)C, (int)C}, {T_ATTPROJW, (int)C, (int)C},
                             {T_FCW, 4 * (int)C, (int)C}, {T_FCPROJW, (int)C, 4 * (int)C}};
    std::vector<size_t> o_wg(4 * L, 0), o_ln(2 * L + 1), o_col(2 * L, 0);
    std::vector<int> sp_wg(4 * L, 1);
    for (size_t l = 0; l < L; ++l)
      for (int k = 0; k < 4; ++k) {
        int sp = h->is_bf16 ? gemm_tc_pick_splits(kinds[k].N, kinds[k].K, (int)M, gemm_tc_num_sms()) : 1;
        sp_wg[l * 4 + k] = sp;
        if (sp > 1) o_wg[l * 4 + k] = dplan((size_t)sp * kinds[k].N * kinds[k].K);
      }
    for (size_t i = 0; i < 2 * L + 1; ++i) o_ln[i] = dplan(layernorm_deferred_partials_floats((int)C, true));
    if (h->bias)
      for (size_t l = 0; l < L; ++l) {
        o_col[l] = dplan(colsum_deferred_partials_floats((int)M, 4 * (int)C));
        o_col[L + l] = dplan(colsum_deferred_partials_floats((int)M, 3 * (int)C));
      }
    // gradient-norm slots and range list (upper bounds; plan_norm fills them once the
    // deferred buffers below exist)
    const size_t max_slots = (size_t)L * (fold_norm_parts(3 * C * C) + fold_norm_parts(C * C) +
                                          2 * fold_norm_parts(4 * C * C)) +
                             (2 * L + 1) * (size_t)layernorm_fold_norm_parts((int)C, true) +
                             2 * L * (size_t)bias_grad_fold_norm_parts(4 * (int)C);
    const size_t max_items = P / 262144 + 4 * L + 8;
    const size_t o_nslots = dplan(max_slots + max_items + 64);
    const size_t o_nranges = dplan(max_items * 4 + 64);   // long long pairs
    h->dmem_bytes = dneed + 256;
    if (cudaError_t e = cudaMalloc(&h->dmem, h->dmem_bytes); e != cudaSuccess) {
      cudaGetLastError();
      cudaFree(h->amem);
      cudaFree(h->pmem);
      delete h;
      return fail(e == cudaErrorMemoryAllocation ? GPT2_ERR_OOM : GPT2_ERR_CUDA,
                  "cudaMalloc of %zu bytes for gradient partials failed: %s", dneed,
                  cudaGetErrorString(e));
    }
    char* d = h->dmem;
    h->norm_slots = (float*)(d + o_nslots);
    h->norm_ranges = (long long*)(d + o_nranges);
    for (size_t l = 0; l < L; ++l)
      for (int k = 0; k < 4; ++k) {
        const int i = (int)(l * 4 + k);
        h->def_wg.push_back({h->gw(kinds[k].id, (int)l), sp_wg[i] > 1 ? (float*)(d + o_wg[i]) : nullptr,
                             sp_wg[i], (size_t)kinds[k].N * kinds[k].K});
      }
    auto bias_or_null = [&](int id, int layer) -> float* {
      return (h->bias && layer >= 0) ? h->gw(id, layer) : nullptr;
    };
    for (size_t l = 0; l < L; ++l)   // LN1 of layer l feeds fcproj's bias of layer l - 1
      h->def_ln.push_back({h->gw(T_LN1W, (int)l), h->gw(T_LN1B, (int)l),
                           bias_or_null(T_FCPROJB, (int)l - 1), (float*)(d + o_ln[l])});
    for (size_t l = 0; l < L; ++l)   // LN2 of layer l feeds attproj's bias of layer l
      h->def_ln.push_back({h->gw(T_LN2W, (int)l), h->gw(T_LN2B, (int)l),
                           bias_or_null(T_ATTPROJB, (int)l), (float*)(d + o_ln[L + l])});
    h->def_ln.push_back({h->gw(T_LNFW), h->gw(T_LNFB), bias_or_null(T_FCPROJB, (int)L - 1),
                         (float*)(d + o_ln[2 * L])});
    if (h->bias) {
      for (size_t l = 0; l < L; ++l)
        h->def_col.push_back({h->gw(T_FCB, (int)l), (float*)(d + o_col[l]), 4 * (int)C});
      for (size_t l = 0; l < L; ++l)
        h->def_col.push_back({h->gw(T_QKVB, (int)l), (float*)(d + o_col[L + l]), 3 * (int)C});
    }
    h->norm_fold_slots = plan_norm(h, norm_items);
    h->norm_items = (int)(norm_items.size() / 2);
    if ((size_t)h->norm_fold_slots > max_slots || (size_t)h->norm_items > max_items)
      h->norm_items = -1;   // the fold norm is then not used (never expected)
  }

  // ---- initial values
  int rc = GPT2_OK;
  if (cudaMemset(h->pmem, 0, pbytes) != cudaSuccess || cudaMemset(h->amem, 0, need) != cudaSuccess ||
      cudaMemset(h->dmem, 0, h->dmem_bytes) != cudaSuccess)
    rc = fail(GPT2_ERR_CUDA, "cudaMemset failed");
  if (rc == GPT2_OK && h->norm_items > 0 &&
      cudaMemcpy(h->norm_ranges, norm_items.data(), norm_items.size() * sizeof(long long),
                 cudaMemcpyHostToDevice) != cudaSuccess)
    rc = fail(GPT2_ERR_CUDA, "norm range upload failed");
  if (rc == GPT2_OK && cfg.init) {
    std::vector<float> host(P, 0.0f);
    fill_init(h, host.data());
    if (cudaMemcpy(h->params, host.data(), P * 4, cudaMemcpyHostToDevice) != cudaSuccess)
      rc = fail(GPT2_ERR_CUDA, "parameter upload failed");
  }
  if (rc == GPT2_OK && h->is_bf16) {
    if (to_bf16(h->params_bf16, h->params, (long long)P, 0) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      rc = fail(GPT2_ERR_CUDA, "bf16 copy failed");
  }
  if (rc != GPT2_OK) {
    cudaFree(h->dmem);
    cudaFree(h->amem);
    cudaFree(h->pmem);
    delete h;
    return rc;
  }
  *out = h;
  return GPT2_OK;
}

extern "C" void gpt2_destroy(gpt2_handle h) {
  if (!h) return;
  for (auto& p : h->prof) { cudaEventDestroy(p.a); cudaEventDestroy(p.b); }
  for (auto& g : h->graphs) cudaGraphExecDestroy(g.exec);
  if (h->dec_exec) cudaGraphExecDestroy(h->dec_exec);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->dmem) cudaFree(h->dmem);
  if (h->amem) cudaFree(h->amem);
  if (h->pmem) cudaFree(h->pmem);
  delete h;
}

extern "C" int gpt2_set_stream(gpt2_handle h, void* s) {
  if (!h) return fail(GPT2_ERR_ARG, "null handle");
  h->stream = (cudaStream_t)s;
  return GPT2_OK;
}

// ------------------------------------------------------------------ helpers
static int check_device_errors(gpt2* h) {
  int err = 0;
  CK(cudaMemcpyAsync(&err, h->d_err, sizeof(int), cudaMemcpyDeviceToHost, h->stream));
  CK(cudaStreamSynchronize(h->stream));
  if (err) {
    CK(cudaMemsetAsync(h->d_err, 0, sizeof(int), h->stream));
    CK(cudaStreamSynchronize(h->stream));
    if (err & DEV_ERR_TIMEOUT) return fail(GPT2_ERR_TIMEOUT, "a device-side wait timed out");
    if (err & (DEV_ERR_BAD_TOKEN | DEV_ERR_BAD_TARGET))
      return fail(GPT2_ERR_BAD_TOKEN, "token or target id outside [0, vocab_size)");
  }
  return GPT2_OK;
}

static cudaError_t run_gemm(gpt2* h, GemmArgs g, const gpt2::DefWgrad* def = nullptr) {
  g.err = h->d_err;
  size_t pi = prof_begin(h, PC_GEMM);
  cudaError_t e;
  if (h->is_bf16) {
    if (g.epi == EPI_ACCUM) {
      if (def && def->splits > 1) {   // partial sums stay in the layer's own workspace
        g.splits = def->splits;
        g.workspace = def->ws;
        g.defer_partials = 1;
      } else {
        g.splits = 0;
        g.workspace = h->splitk_ws;
      }
    }
    // a handful of rows (the decode step) streams the weights instead of filling 128-row tiles
    e = g.M <= 16 && gemv_rows_supported(g) ? gemv_rows(g, h->stream) : gemm_bf16_tc(g, h->stream);
  } else {
    e = gemm_f32(g, h->stream);
  }
  prof_end(h, pi, 2.0 * g.M * g.N * g.K);
  return e;
}

// Y[M, N] = X[M, K] W[N, K]^T with an epilogue
static GemmArgs linear_fwd(int M, int N, int K, const void* X, const void* W, void* Y) {
  GemmArgs g;
  g.M = M; g.N = N; g.K = K;
  g.A = X; g.lda = K; g.a_mn = false;
  g.B = W; g.ldb = K; g.b_mn = false;
  g.out = Y; g.ldo = N;
  return g;
}
// dX[M, K] = dY[M, N] W[N, K]
static GemmArgs linear_dgrad(int M, int N, int K, const void* dY, const void* W, void* dX) {
  GemmArgs g;
  g.M = M; g.N = K; g.K = N;
  g.A = dY; g.lda = N; g.a_mn = false;
  g.B = W; g.ldb = K; g.b_mn = true;
  g.out = dX; g.ldo = K;
  return g;
}
// dW[N, K] += scale * dY[M, N]^T X[M, K]
static GemmArgs linear_wgrad(int M, int N, int K, const void* dY, const void* X, float* dW,
                             float scale) {
  GemmArgs g;
  g.M = N; g.N = K; g.K = M;
  g.A = dY; g.lda = N; g.a_mn = true;
  g.B = X; g.ldb = K; g.b_mn = true;
  g.epi = EPI_ACCUM; g.accum = dW; g.ldo = K; g.scale = scale;
  return g;
}

// Fold the deferred partial sums into the gradient buffer (and clear them). With norm, each
// fold also writes its sums of squares into the next norm_slots (the order and counts of
// plan_norm).
static cudaError_t flush_grads(gpt2* h, bool norm = false) {
  if (!h->grads_pending) return cudaSuccess;
  cudaStream_t s = h->stream;
  cudaError_t e = cudaSuccess;
  float* slot = h->norm_slots;
  for (auto& d : h->def_wg)
    if (e == cudaSuccess && d.splits > 1) {
      if (norm) {
        e = splitk_fold_norm(d.grad, d.ws, d.splits, (long long)d.n, slot, s);
        slot += fold_norm_parts((long long)d.n);
      } else {
        e = splitk_fold(d.grad, d.ws, d.splits, (long long)d.n, s);
      }
    }
  for (auto& d : h->def_ln)
    if (e == cudaSuccess) {
      e = layernorm_fold(d.dw, d.db, d.dproj, d.part, h->C, s, norm ? slot : nullptr);
      if (norm) slot += layernorm_fold_norm_parts(h->C, d.dproj != nullptr);
    }
  for (auto& d : h->def_col)
    if (e == cudaSuccess) {
      e = bias_grad_fold(d.db, d.part, h->Bmax * h->T, d.N, s, norm ? slot : nullptr);
      if (norm) slot += bias_grad_fold_norm_parts(d.N);
    }
  if (e == cudaSuccess) h->grads_pending = false;
  return e;
}

// The slots the folds write and the gradient ranges they leave to a separate read, as host
// data; returns the number of fold slots, the range items in `items`.
static int plan_norm(gpt2* h, std::vector<long long>& items) {
  int slots = 0;
  for (auto& d : h->def_wg) if (d.splits > 1) slots += fold_norm_parts((long long)d.n);
  for (auto& d : h->def_ln) slots += layernorm_fold_norm_parts(h->C, d.dproj != nullptr);
  for (auto& d : h->def_col) slots += bias_grad_fold_norm_parts(d.N);
  // elements no fold finalises: wte, wpe, and the layer weights whose gradient has no
  // split partials (written whole by their weight-gradient GEMM)
  std::vector<std::pair<size_t, size_t>> ranges;
  auto add = [&](size_t off, size_t n) {
    if (!ranges.empty() && ranges.back().first + ranges.back().second == off) ranges.back().second += n;
    else ranges.push_back({off, n});
  };
  const TensorInfo& te = h->tensors[h->index[T_WTE]];
  add(te.offset, te.numel);
  const TensorInfo& tp = h->tensors[h->index[T_WPE]];
  add(tp.offset, tp.numel);
  const int kinds[4] = {T_QKVW, T_ATTPROJW, T_FCW, T_FCPROJW};
  for (int l = 0; l < h->L; ++l)
    for (int k = 0; k < 4; ++k) {
      const gpt2::DefWgrad& d = h->def_wg[l * 4 + k];
      if (d.splits > 1) continue;
      add((size_t)(h->gw(kinds[k], l) - h->grads), d.n);
    }
  constexpr size_t ITEM = 262144;
  for (auto& r : ranges)
    for (size_t o = 0; o < r.second; o += ITEM) {
      items.push_back((long long)(r.first + o));
      items.push_back((long long)std::min(ITEM, r.second - o));
    }
  return slots;
}

#define CKL(x)                                                                              \
  do {                                                                                      \
    cudaError_t e_ = (x);                                                                   \
    if (e_ != cudaSuccess) return fail(GPT2_ERR_CUDA, "%s: %s", #x, cudaGetErrorString(e_)); \
  } while (0)

// ------------------------------------------------------------------ forward
extern "C" int gpt2_forward(gpt2_handle h, const int32_t* tokens, const int32_t* targets,
                            int32_t B, int32_t T, float* h_loss) {
  if (!h || !tokens) return fail(GPT2_ERR_ARG, "null argument");
  if (B <= 0 || T <= 0) return fail(GPT2_ERR_ARG, "B and T must be positive");
  if (T > h->T || B > h->Bmax)
    return fail(GPT2_ERR_SEQ_TOO_LONG, "T=%d > block_size=%d or B=%d > batch_size=%d", T, h->T,
                B, h->Bmax);
  const int M = B * T, C = h->C, L = h->L, H = h->H, Vp = h->Vp;
  const DType dt = h->dt;
  cudaStream_t s = h->stream;
  h->have_targets = false;
  h->last_B = B; h->last_T = T; h->last_tokens = tokens;
  h->dec_len = 0;   // the activations no longer match a decode cache
  const double es = (double)h->es;

  size_t pi = prof_begin(h, PC_ENC);
  CKL(encoder_forward(dt, h->x[0], tokens, h->pw(T_WTE), h->pw(T_WPE), B, T, C, h->V, h->d_err, s));
  prof_end(h, pi, (double)M * C * es * 3);
  for (int l = 0; l < L; ++l) {
    pi = prof_begin(h, PC_LN);
    CKL(layernorm_forward(dt, h->ln1[l], h->ln1_mean[l], h->ln1_rstd[l], h->x[l],
                          h->pw(T_LN1W, l), h->pw(T_LN1B, l), M, C, s));
    prof_end(h, pi, (double)M * C * es * 2);
    GemmArgs g = linear_fwd(M, 3 * C, C, h->ln1[l], h->pw(T_QKVW, l), h->qkv[l]);
    if (h->bias) g.bias = h->pw(T_QKVB, l);
    CKL(run_gemm(h, g));
    pi = prof_begin(h, PC_ATTN);
    CKL(attention_forward(dt, h->att[l], h->lse[l], h->qkv[l], B, T, C, H, h->d_err, s));
    prof_end(h, pi, 2.0 * 2.0 * B * H * (double)T * (T + 1) / 2 * (C / H));
    g = linear_fwd(M, C, C, h->att[l], h->pw(T_ATTPROJW, l), h->xmid[l]);
    if (h->bias) g.bias = h->pw(T_ATTPROJB, l);
    g.resid = h->x[l];
    CKL(run_gemm(h, g));
    pi = prof_begin(h, PC_LN);
    CKL(layernorm_forward(dt, h->ln2[l], h->ln2_mean[l], h->ln2_rstd[l], h->xmid[l],
                          h->pw(T_LN2W, l), h->pw(T_LN2B, l), M, C, s));
    prof_end(h, pi, (double)M * C * es * 2);
    g = linear_fwd(M, 4 * C, C, h->ln2[l], h->pw(T_FCW, l), h->fcg[l]);
    if (h->bias) g.bias = h->pw(T_FCB, l);
    g.epi = h->recompute ? EPI_GELU_FWD_U : EPI_GELU_FWD;   // keeps u or gelu'(u)
    g.pre = h->fch[l];
    CKL(run_gemm(h, g));
    g = linear_fwd(M, C, 4 * C, h->fcg[l], h->pw(T_FCPROJW, l), h->x[l + 1]);
    if (h->bias) g.bias = h->pw(T_FCPROJB, l);
    g.resid = h->xmid[l];
    CKL(run_gemm(h, g));
  }
  pi = prof_begin(h, PC_LN);
  CKL(layernorm_forward(dt, h->lnf, h->lnf_mean, h->lnf_rstd, h->x[L], h->pw(T_LNFW),
                        h->pw(T_LNFB), M, C, s));
  prof_end(h, pi, (double)M * C * es * 2);
  if (targets && h->is_bf16) {
    // the lm_head GEMM also writes each row's softmax statistics; one streaming pass then
    // writes the losses and the dlogits in place
    GemmArgs g = linear_fwd(M, Vp, C, h->lnf, h->pw(T_WTE), h->logits);
    g.epi = EPI_LOGITS_CE;
    g.vocab = h->V;
    g.ce_part = h->ce_part;
    CKL(run_gemm(h, g));
    pi = prof_begin(h, PC_CLS);
    CKL(ce_from_partials(dt, h->logits, h->losses, h->ce_part, gemm_ce_parts(Vp), targets, M,
                         h->V, Vp, h->ce_lse, h->d_err, s));
    prof_end(h, pi, (double)M * Vp * es * 2);
  } else {
    CKL(run_gemm(h, linear_fwd(M, Vp, C, h->lnf, h->pw(T_WTE), h->logits)));
  }
  if (targets) {
    if (!h->is_bf16) {
      pi = prof_begin(h, PC_CLS);
      CKL(classifier(dt, h->logits, h->losses, targets, M, h->V, Vp, h->d_err, s));
      prof_end(h, pi, (double)M * Vp * es * 2);
    }
    CKL(mean_loss(h->d_loss, h->losses, M, s));
    h->have_targets = true;
  } else {
    CKL(argmax_rows(dt, h->argmax, h->logits, M, h->V, Vp, s));
  }
  if (h_loss) {
    if (!targets) return fail(GPT2_ERR_STATE, "h_loss needs targets");
    int rc = check_device_errors(h);
    if (rc) return rc;
    CK(cudaMemcpy(h_loss, h->d_loss, sizeof(float), cudaMemcpyDeviceToHost));
  }
  return GPT2_OK;
}

// ------------------------------------------------------------------ backward
extern "C" int gpt2_backward(gpt2_handle h, float loss_scale) {
  if (!h) return fail(GPT2_ERR_ARG, "null handle");
  if (!h->have_targets) return fail(GPT2_ERR_STATE, "backward needs a forward with targets");
  if (h->is_bf16 && h->last_T % 4)
    return fail(GPT2_ERR_ARG, "the bf16 backward needs T %% 4 == 0 (T = %d)", h->last_T);
  const int B = h->last_B, T = h->last_T, M = B * T, C = h->C, L = h->L, H = h->H, Vp = h->Vp;
  const DType dt = h->dt;
  cudaStream_t s = h->stream;
  const float sc = loss_scale;
  const double es = (double)h->es;
  size_t pi;

  // lm_head (tied): dlnf = dlogits wte ; dwte += sc dlogits^T lnf
  CKL(run_gemm(h, linear_dgrad(M, Vp, C, h->logits, h->pw(T_WTE), h->dln)));
  CKL(run_gemm(h, linear_wgrad(M, Vp, C, h->logits, h->lnf, h->gw(T_WTE), sc)));
  // The column sums of each residual-stream gradient that a LayerNorm backward writes are
  // the bias gradient of the projection that fed that stream: lnf -> fcproj of layer L-1,
  // LN2 of layer l -> attproj of layer l, LN1 of layer l -> fcproj of layer l-1 (the
  // def_ln entries carry those targets). LayerNorm, bias and split weight-gradient sums
  // go to the deferred partial buffers.
  h->grads_pending = true;
  auto ln_bwd = [&](int i, int acc, const void* x, int wid, int layer, const float* mean,
                    const float* rstd) -> cudaError_t {
    const gpt2::DefLN& d = h->def_ln[i];
    return layernorm_backward(dt, h->dres, acc, d.dw, d.db, d.dproj, h->dln, x, h->pw(wid, layer),
                              mean, rstd, M, C, sc, d.part, 1, s);
  };
  auto wg = [&](int layer, int kind) { return &h->def_wg[layer * 4 + kind]; };
  pi = prof_begin(h, PC_LN);
  CKL(ln_bwd(2 * L, 0, h->x[L], T_LNFW, 0, h->lnf_mean, h->lnf_rstd));
  prof_end(h, pi, (double)M * C * es * 3);
  for (int l = L - 1; l >= 0; --l) {
    // x[l+1] = xmid + gelu(u) Wp^T + bp with u the fc pre-activation, whose derivative
    // gelu'(u) the forward kept in fch  (bp's gradient came with dres, above)
    GemmArgs g = linear_dgrad(M, C, 4 * C, h->dres, h->pw(T_FCPROJW, l), h->dfch);
    g.epi = EPI_GELU_BWD;
    g.aux = h->fch[l];
    if (h->recompute) {   // gelu'(u) from u, and gelu(u) into the shared buffer for the wgrad
      g.epi = EPI_GELU_BWD_U;
      g.pre = h->fcg[l];
    }
    CKL(run_gemm(h, g));
    CKL(run_gemm(h, linear_wgrad(M, C, 4 * C, h->dres, h->fcg[l], h->gw(T_FCPROJW, l), sc), wg(l, 3)));
    // fch = ln2 Wfc^T + bfc
    if (h->recompute) {   // LN2's output, recomputed from the kept residual stream
      pi = prof_begin(h, PC_LN);
      CKL(layernorm_forward(dt, h->ln2[l], h->ln2_mean[l], h->ln2_rstd[l], h->xmid[l],
                            h->pw(T_LN2W, l), h->pw(T_LN2B, l), M, C, s));
      prof_end(h, pi, (double)M * C * es * 2);
    }
    CKL(run_gemm(h, linear_dgrad(M, 4 * C, C, h->dfch, h->pw(T_FCW, l), h->dln)));
    CKL(run_gemm(h, linear_wgrad(M, 4 * C, C, h->dfch, h->ln2[l], h->gw(T_FCW, l), sc), wg(l, 2)));
    if (h->bias) {
      pi = prof_begin(h, PC_OTHER);
      CKL(bias_grad(dt, h->gw(T_FCB, l), h->dfch, M, 4 * C, sc, h->def_col[l].part, 1, s));
      prof_end(h, pi, (double)M * 4 * C * es);
    }
    pi = prof_begin(h, PC_LN);
    CKL(ln_bwd(L + l, 1, h->xmid[l], T_LN2W, l, h->ln2_mean[l], h->ln2_rstd[l]));
    prof_end(h, pi, (double)M * C * es * 4);
    // xmid = x + att Wo^T + bo  (bo's gradient came with dres, above)
    CKL(run_gemm(h, linear_dgrad(M, C, C, h->dres, h->pw(T_ATTPROJW, l), h->datt)));
    CKL(run_gemm(h, linear_wgrad(M, C, C, h->dres, h->att[l], h->gw(T_ATTPROJW, l), sc), wg(l, 1)));
    pi = prof_begin(h, PC_ATTN);
    CKL(attention_backward(dt, h->dqkv, h->Dbuf, h->datt, h->att[l], h->qkv[l], h->lse[l], B, T,
                           C, H, h->d_err, s));
    prof_end(h, pi, 2.5 * 2.0 * 2.0 * B * H * (double)T * (T + 1) / 2 * (C / H));
    // qkv = ln1 Wqkv^T + bqkv
    if (h->recompute) {   // LN1's output, recomputed from the kept residual stream
      pi = prof_begin(h, PC_LN);
      CKL(layernorm_forward(dt, h->ln1[l], h->ln1_mean[l], h->ln1_rstd[l], h->x[l],
                            h->pw(T_LN1W, l), h->pw(T_LN1B, l), M, C, s));
      prof_end(h, pi, (double)M * C * es * 2);
    }
    CKL(run_gemm(h, linear_dgrad(M, 3 * C, C, h->dqkv, h->pw(T_QKVW, l), h->dln)));
    CKL(run_gemm(h, linear_wgrad(M, 3 * C, C, h->dqkv, h->ln1[l], h->gw(T_QKVW, l), sc), wg(l, 0)));
    if (h->bias) {
      pi = prof_begin(h, PC_OTHER);
      CKL(bias_grad(dt, h->gw(T_QKVB, l), h->dqkv, M, 3 * C, sc, h->def_col[L + l].part, 1, s));
      prof_end(h, pi, (double)M * 3 * C * es);
    }
    pi = prof_begin(h, PC_LN);
    CKL(ln_bwd(l, 1, h->x[l], T_LN1W, l, h->ln1_mean[l], h->ln1_rstd[l]));
    prof_end(h, pi, (double)M * C * es * 4);
  }
  pi = prof_begin(h, PC_ENC);
  CKL(encoder_backward(dt, h->gw(T_WTE), h->gw(T_WPE), h->dres, h->last_tokens, B, T, C, Vp, sc,
                       h->enc_scratch, s));
  prof_end(h, pi, (double)M * C * es * 2);
  return GPT2_OK;
}

// ------------------------------------------------------------------ micro-batch as a graph
// The ~275 launches of a forward + backward are recorded once per (B, T, loss scale) into
// a CUDA graph on a private capturing stream and replayed on the handle's stream, which
// removes the per-launch host work and most of the gaps between dependent kernels. The
// graph reads tokens and targets from the handle's own buffers, so every replay works on
// whatever the caller copied in last; all other buffers have fixed addresses.
static int microbatch_eager(gpt2* h, int B, int T, float scale) {
  int rc = gpt2_forward(h, h->mb_tok, h->mb_tgt, B, T, nullptr);
  return rc ? rc : gpt2_backward(h, scale);
}

static int microbatch_capture(gpt2* h, int B, int T, float scale) {
  if (!h->cap_stream) CK(cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking));
  const long long n0 = launch_counter();
  cudaStream_t user = h->stream;
  h->stream = h->cap_stream;
  CK(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
  const int rc = microbatch_eager(h, B, T, scale);   // recorded, not executed
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(h->cap_stream, &graph);
  h->stream = user;
  const long long launches = launch_counter() - n0;
  launch_counter() = n0;
  if (rc || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    if (rc) return rc;
    return fail(GPT2_ERR_CUDA, "stream capture of the micro-batch failed: %s",
                cudaGetErrorString(e));
  }
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess)
    return fail(GPT2_ERR_CUDA, "cudaGraphInstantiate: %s", cudaGetErrorString(ei));
  if (h->graphs.size() >= 8) {
    cudaGraphExecDestroy(h->graphs.front().exec);
    h->graphs.erase(h->graphs.begin());
  }
  h->graphs.push_back({B, T, scale, exec, launches});
  return GPT2_OK;
}

extern "C" int gpt2_forward_backward(gpt2_handle h, const int32_t* tokens,
                                     const int32_t* targets, int32_t B, int32_t T,
                                     float loss_scale) {
  if (!h || !tokens || !targets) return fail(GPT2_ERR_ARG, "null argument");
  if (B <= 0 || T <= 0) return fail(GPT2_ERR_ARG, "B and T must be positive");
  if (T > h->T || B > h->Bmax)
    return fail(GPT2_ERR_SEQ_TOO_LONG, "T=%d > block_size=%d or B=%d > batch_size=%d", T, h->T,
                B, h->Bmax);
  if (h->is_bf16 && T % 4)
    return fail(GPT2_ERR_ARG, "the bf16 backward needs T %% 4 == 0 (T = %d)", T);
  const size_t bytes = (size_t)B * T * sizeof(int32_t);
  CK(cudaMemcpyAsync(h->mb_tok, tokens, bytes, cudaMemcpyDefault, h->stream));
  CK(cudaMemcpyAsync(h->mb_tgt, targets, bytes, cudaMemcpyDefault, h->stream));
  // timed launches (gpt2_profile_enable) need the events between kernels: run eagerly
  if (!h->graph_mode || h->prof_mask) return microbatch_eager(h, B, T, loss_scale);
  for (const auto& g : h->graphs) {
    if (g.B != B || g.T != T || g.scale != loss_scale) continue;
    CK(cudaGraphLaunch(g.exec, h->stream));
    count_launches((int)g.launches);
    // host-side state the recorded forward and backward leave behind
    h->dec_len = 0;
    h->have_targets = true;
    h->last_B = B; h->last_T = T; h->last_tokens = h->mb_tok;
    h->grads_pending = true;
    return GPT2_OK;
  }
  // first call with this shape: run it, then record it for the next calls
  int rc = microbatch_eager(h, B, T, loss_scale);
  return rc ? rc : microbatch_capture(h, B, T, loss_scale);
}

// ------------------------------------------------------------------ inference (KV cache)
extern "C" int gpt2_prefill(gpt2_handle h, const int32_t* tokens, int32_t B, int32_t T0,
                            int32_t* next) {
  if (!h || !tokens || !next) return fail(GPT2_ERR_ARG, "null argument");
  int rc = gpt2_forward(h, tokens, nullptr, B, T0, nullptr);
  if (rc) return rc;
  cudaStream_t s = h->stream;
  for (int l = 0; l < h->L; ++l)
    CKL(kv_cache_store(h->dt, h->kv(l), h->qkv[l], B, T0, 0, T0, h->T, h->C, s));
  CKL(gather_last(next, h->argmax, B, T0, s));
  CKL(decode_position(h->d_pos, T0, 0, s));
  h->dec_B = B;
  h->dec_len = T0;
  return GPT2_OK;
}

// The launches of one decode step for B rows at position t: the new tokens come from
// mb_tok, the position from d_pos (incremented at the end), so that the same launches,
// recorded once, serve every later position.
static int decode_launches(gpt2* h, int B, int t) {
  const int C = h->C, L = h->L, Vp = h->Vp;
  const DType dt = h->dt;
  cudaStream_t s = h->stream;
  // the new position's activations use rows 0..B-1 of the forward's buffers
  CKL(encoder_forward(dt, h->x[0], h->mb_tok, h->pw(T_WTE), h->pw(T_WPE), B, 1, C, h->V,
                      h->d_err, s, t, h->d_pos));
  // bf16, at most 16 rows: the weight-streaming kernel also computes LN1 / LN2 itself and
  // writes the new keys and values into the cache (fewer dependent launches per layer)
  const bool fuse = h->is_bf16 && B <= 16;
  for (int l = 0; l < L; ++l) {
    GemmArgs g = linear_fwd(B, 3 * C, C, h->ln1[l], h->pw(T_QKVW, l), h->qkv[l]);
    if (h->bias) g.bias = h->pw(T_QKVB, l);
    if (fuse) {
      GemvFuse f;
      f.ln_x = h->x[l]; f.ln_w = h->pw(T_LN1W, l); f.ln_b = h->pw(T_LN1B, l);
      f.kv_cache = h->kv(l); f.kv_Tmax = h->T; f.kv_C = C; f.kv_pos = h->d_pos;
      CKL(gemv_rows(g, s, f));
    } else {
      CKL(layernorm_forward(dt, h->ln1[l], h->ln1_mean[l], h->ln1_rstd[l], h->x[l],
                            h->pw(T_LN1W, l), h->pw(T_LN1B, l), B, C, s));
      CKL(run_gemm(h, g));
      CKL(kv_cache_store(dt, h->kv(l), h->qkv[l], B, 1, t, 1, h->T, C, s, h->d_pos));
    }
    CKL(attention_decode(dt, h->att[l], h->qkv[l], h->kv(l), B, t, h->T, C, h->H, s, h->d_pos,
                         h->Dbuf));
    g = linear_fwd(B, C, C, h->att[l], h->pw(T_ATTPROJW, l), h->xmid[l]);
    if (h->bias) g.bias = h->pw(T_ATTPROJB, l);
    g.resid = h->x[l];
    CKL(run_gemm(h, g));
    g = linear_fwd(B, 4 * C, C, h->ln2[l], h->pw(T_FCW, l), h->fcg[l]);
    if (h->bias) g.bias = h->pw(T_FCB, l);
    g.epi = h->recompute ? EPI_GELU_FWD_U : EPI_GELU_FWD;
    g.pre = h->fch[l];
    if (fuse) {
      GemvFuse f;
      f.ln_x = h->xmid[l]; f.ln_w = h->pw(T_LN2W, l); f.ln_b = h->pw(T_LN2B, l);
      CKL(gemv_rows(g, s, f));
    } else {
      CKL(layernorm_forward(dt, h->ln2[l], h->ln2_mean[l], h->ln2_rstd[l], h->xmid[l],
                            h->pw(T_LN2W, l), h->pw(T_LN2B, l), B, C, s));
      CKL(run_gemm(h, g));
    }
    g = linear_fwd(B, C, 4 * C, h->fcg[l], h->pw(T_FCPROJW, l), h->x[l + 1]);
    if (h->bias) g.bias = h->pw(T_FCPROJB, l);
    g.resid = h->xmid[l];
    CKL(run_gemm(h, g));
  }
  CKL(layernorm_forward(dt, h->lnf, h->lnf_mean, h->lnf_rstd, h->x[L], h->pw(T_LNFW),
                        h->pw(T_LNFB), B, C, s));
  CKL(run_gemm(h, linear_fwd(B, Vp, C, h->lnf, h->pw(T_WTE), h->logits)));
  CKL(argmax_rows(dt, h->argmax, h->logits, B, h->V, Vp, s));
  CKL(decode_position(h->d_pos, -1, 1, s));
  return GPT2_OK;
}

static int decode_capture(gpt2* h, int B, int t) {
  if (!h->cap_stream) CK(cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking));
  const long long n0 = launch_counter();
  cudaStream_t user = h->stream;
  h->stream = h->cap_stream;
  CK(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
  const int rc = decode_launches(h, B, t);   // recorded, not executed
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(h->cap_stream, &graph);
  h->stream = user;
  const long long launches = launch_counter() - n0;
  launch_counter() = n0;
  if (rc || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    if (rc) return rc;
    return fail(GPT2_ERR_CUDA, "stream capture of the decode step failed: %s",
                cudaGetErrorString(e));
  }
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess)
    return fail(GPT2_ERR_CUDA, "cudaGraphInstantiate: %s", cudaGetErrorString(ei));
  if (h->dec_exec) cudaGraphExecDestroy(h->dec_exec);
  h->dec_exec = exec;
  h->dec_exec_B = B;
  h->dec_exec_launches = launches;
  return GPT2_OK;
}

extern "C" int gpt2_decode_step(gpt2_handle h, const int32_t* tokens, int32_t B, int32_t* next) {
  if (!h || !tokens || !next) return fail(GPT2_ERR_ARG, "null argument");
  if (h->dec_len <= 0) return fail(GPT2_ERR_STATE, "decode_step needs a prefill first");
  if (B != h->dec_B) return fail(GPT2_ERR_ARG, "B=%d differs from the prefill's B=%d", B, h->dec_B);
  const int t = h->dec_len;
  if (t >= h->T) return fail(GPT2_ERR_SEQ_TOO_LONG, "position %d >= block_size %d", t, h->T);
  cudaStream_t s = h->stream;
  CK(cudaMemcpyAsync(h->mb_tok, tokens, (size_t)B * sizeof(int32_t), cudaMemcpyDefault, s));
  if (h->graph_mode && !h->prof_mask && h->dec_exec && h->dec_exec_B == B) {
    CK(cudaGraphLaunch(h->dec_exec, s));
    count_launches((int)h->dec_exec_launches);
  } else {
    int rc = decode_launches(h, B, t);
    // the first step for this batch runs eagerly, then is recorded for the later ones
    if (!rc && h->graph_mode && !h->prof_mask) rc = decode_capture(h, B, t);
    if (rc) return rc;
  }
  h->have_targets = false;
  h->last_B = B; h->last_T = 1; h->last_tokens = h->mb_tok;
  CK(cudaMemcpyAsync(next, h->argmax, (size_t)B * sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
  h->dec_len = t + 1;
  return GPT2_OK;
}

extern "C" int gpt2_decode_length(gpt2_handle h, int32_t* length) {
  if (!h || !length) return fail(GPT2_ERR_ARG, "null argument");
  *length = h->dec_len;
  return GPT2_OK;
}

extern "C" int gpt2_set_graph_mode(gpt2_handle h, int enabled) {
  if (!h) return fail(GPT2_ERR_ARG, "null handle");
  h->graph_mode = enabled != 0;
  if (!h->graph_mode) {
    for (auto& g : h->graphs) cudaGraphExecDestroy(g.exec);
    h->graphs.clear();
    if (h->dec_exec) cudaGraphExecDestroy(h->dec_exec);
    h->dec_exec = nullptr;
    h->dec_exec_B = 0;
  }
  return GPT2_OK;
}

extern "C" int gpt2_zero_grad(gpt2_handle h) {
  if (!h) return fail(GPT2_ERR_ARG, "null handle");
  CK(cudaMemsetAsync(h->grads, 0, h->P * 4, h->stream));
  if (h->grads_pending) CK(cudaMemsetAsync(h->dmem, 0, h->dmem_bytes, h->stream));
  h->grads_pending = false;
  return GPT2_OK;
}

// ------------------------------------------------------------------ optimiser
extern "C" int gpt2_adamw_step(gpt2_handle h, float lr, float beta1, float beta2, float eps,
                               float weight_decay, float grad_clip, float* h_grad_norm) {
  if (!h) return fail(GPT2_ERR_ARG, "null handle");
  const bool norm = grad_clip > 0.f || h_grad_norm;
  // when this call folds the pending partials, the folds also produce the norm's sums of
  // squares of what they finalise, and only the rest of the gradients is read again
  const bool fold_norm = norm && h->grads_pending && h->norm_items >= 0;
  CKL(flush_grads(h, fold_norm));
  h->step += 1;
  cudaStream_t s = h->stream;
  size_t pi = prof_begin(h, PC_OPT);
  if (fold_norm) {
    CKL(grad_norm_finish(h->d_norm, h->norm_slots, h->norm_fold_slots + h->norm_items, h->grads,
                         h->norm_ranges, h->norm_items, h->norm_slots + h->norm_fold_slots,
                         grad_clip, s));
  } else if (norm) {
    CKL(grad_norm(h->d_norm, h->norm_partials, h->grads, (long long)h->P, grad_clip, s));
  }
  prof_end(h, pi, (double)h->P * 4);
  pi = prof_begin(h, PC_OPT);
  CKL(adamw(h->params, h->grads, h->m, h->v, h->is_bf16 ? (void*)h->params_bf16 : nullptr,
            (long long)h->P, lr, beta1, beta2, eps, weight_decay, (int)h->step,
            grad_clip > 0.f ? h->d_norm : nullptr, s));
  prof_end(h, pi, (double)h->P * (h->is_bf16 ? 30 : 28));
  if (h_grad_norm) {
    int rc = check_device_errors(h);
    if (rc) return rc;
    CK(cudaMemcpy(h_grad_norm, h->d_norm, sizeof(float), cudaMemcpyDeviceToHost));
  }
  return GPT2_OK;
}

extern "C" int gpt2_get_loss(gpt2_handle h, float* h_loss) {
  if (!h || !h_loss) return fail(GPT2_ERR_ARG, "null argument");
  int rc = check_device_errors(h);
  if (rc) return rc;
  CK(cudaMemcpyAsync(h_loss, h->d_loss, sizeof(float), cudaMemcpyDeviceToHost, h->stream));
  CK(cudaStreamSynchronize(h->stream));
  return GPT2_OK;
}

extern "C" int gpt2_sync(gpt2_handle h) {
  if (!h) return fail(GPT2_ERR_ARG, "null handle");
  return check_device_errors(h);
}

// ------------------------------------------------------------------ introspection
extern "C" int gpt2_num_tensors(gpt2_handle h) {
  if (!h) return fail(GPT2_ERR_ARG, "null handle");
  return (int)h->tensors.size();
}

extern "C" int gpt2_tensor_info(gpt2_handle h, int i, const char** name, size_t* offset,
                                int* ndim, int64_t* shape) {
  if (!h || i < 0 || i >= (int)h->tensors.size()) return fail(GPT2_ERR_ARG, "bad tensor index");
  const TensorInfo& t = h->tensors[i];
  if (name) *name = kTensorNames[t.id];
  if (offset) *offset = t.offset;
  if (ndim) *ndim = t.ndim;
  if (shape) for (int d = 0; d < 3; ++d) shape[d] = t.shape[d];
  return GPT2_OK;
}

extern "C" int gpt2_num_params(gpt2_handle h, size_t* n_model, size_t* n_buffer) {
  if (!h) return fail(GPT2_ERR_ARG, "null handle");
  if (n_model) *n_model = h->n_model;
  if (n_buffer) *n_buffer = h->P;
  return GPT2_OK;
}

static int region(gpt2* h, int r, void** p, size_t* bytes) {
  const size_t M = (size_t)(h->last_B ? h->last_B * h->last_T : h->Bmax * h->T);
  if (r == GPT2_REGION_GRADS) {
    cudaError_t e = flush_grads(h);
    if (e != cudaSuccess) return fail(GPT2_ERR_CUDA, "gradient fold failed: %s", cudaGetErrorString(e));
  }
  switch (r) {
    case GPT2_REGION_PARAMS: *p = h->params; *bytes = h->P * 4; return GPT2_OK;
    case GPT2_REGION_GRADS: *p = h->grads; *bytes = h->P * 4; return GPT2_OK;
    case GPT2_REGION_M: *p = h->m; *bytes = h->P * 4; return GPT2_OK;
    case GPT2_REGION_V: *p = h->v; *bytes = h->P * 4; return GPT2_OK;
    case GPT2_REGION_PARAMS_BF16:
      if (!h->is_bf16) return fail(GPT2_ERR_ARG, "no bf16 copy in the fp32 path");
      *p = h->params_bf16; *bytes = h->P * 2; return GPT2_OK;
    case GPT2_REGION_LOGITS: *p = h->logits; *bytes = M * h->Vp * h->es; return GPT2_OK;
    case GPT2_REGION_LOSSES: *p = h->losses; *bytes = M * 4; return GPT2_OK;
    case GPT2_REGION_ENCODED: *p = h->x[0]; *bytes = M * h->C * h->es; return GPT2_OK;
    case GPT2_REGION_ARGMAX: *p = h->argmax; *bytes = M * 4; return GPT2_OK;
  }
  return fail(GPT2_ERR_ARG, "unknown region %d", r);
}

extern "C" int gpt2_region_ptr(gpt2_handle h, int r, void** d_ptr, size_t* bytes) {
  if (!h || !d_ptr || !bytes) return fail(GPT2_ERR_ARG, "null argument");
  return region(h, r, d_ptr, bytes);
}

extern "C" int gpt2_copy_region(gpt2_handle h, int r, size_t offset, void* h_buf, size_t bytes,
                                int to_device) {
  if (!h || (!h_buf && bytes)) return fail(GPT2_ERR_ARG, "null argument");
  void* p = nullptr;
  size_t n = 0;
  int rc = region(h, r, &p, &n);
  if (rc) return rc;
  if (offset > n || bytes > n - offset) return fail(GPT2_ERR_ARG, "copy out of range");
  char* d = (char*)p + offset;
  if (to_device) {
    CK(cudaMemcpyAsync(d, h_buf, bytes, cudaMemcpyHostToDevice, h->stream));
    if (r == GPT2_REGION_PARAMS && h->is_bf16)
      CK(to_bf16(h->params_bf16, h->params, (long long)h->P, h->stream));
  } else {
    CK(cudaMemcpyAsync(h_buf, d, bytes, cudaMemcpyDeviceToHost, h->stream));
  }
  CK(cudaStreamSynchronize(h->stream));
  return GPT2_OK;
}

extern "C" int gpt2_get_step(gpt2_handle h, int64_t* t) {
  if (!h || !t) return fail(GPT2_ERR_ARG, "null argument");
  *t = h->step;
  return GPT2_OK;
}
extern "C" int gpt2_set_step(gpt2_handle h, int64_t t) {
  if (!h || t < 0) return fail(GPT2_ERR_ARG, "bad argument");
  h->step = t;
  return GPT2_OK;
}

// ------------------------------------------------------------------ profiling
extern "C" int gpt2_profile_enable(gpt2_handle h, int mask, int capacity) {
  if (!h || capacity < 0) return fail(GPT2_ERR_ARG, "bad argument");
  if ((size_t)capacity > h->prof.size()) {
    for (size_t i = h->prof.size(); i < (size_t)capacity; ++i) {
      ProfPair p{};
      CK(cudaEventCreate(&p.a));
      CK(cudaEventCreate(&p.b));
      h->prof.push_back(p);
    }
  }
  h->prof_mask = mask;
  return GPT2_OK;
}

extern "C" int gpt2_profile_read(gpt2_handle h, int cls, int64_t* launches, double* total_ms,
                                 double* work, int reset) {
  if (!h || cls < 0 || cls >= GPT2_PROF_NUM_CLASSES) return fail(GPT2_ERR_ARG, "bad argument");
  if (h->prof_used) {
    CK(cudaStreamSynchronize(h->stream));
    for (size_t i = 0; i < h->prof_used; ++i) {
      float ms = 0.f;
      CK(cudaEventElapsedTime(&ms, h->prof[i].a, h->prof[i].b));
      int c = h->prof[i].cls;
      h->prof_launches[c] += 1;
      h->prof_ms[c] += ms;
      h->prof_work[c] += h->prof[i].work;
    }
    h->prof_used = 0;
  }
  if (launches) *launches = h->prof_launches[cls];
  if (total_ms) *total_ms = h->prof_ms[cls];
  if (work) *work = h->prof_work[cls];
  if (reset) {
    for (int c = 0; c < GPT2_PROF_NUM_CLASSES; ++c) {
      h->prof_launches[c] = 0; h->prof_ms[c] = 0; h->prof_work[c] = 0;
    }
  }
  return GPT2_OK;
}

extern "C" int gpt2_memory_bytes(gpt2_handle h, size_t* param_bytes, size_t* other_bytes) {
  if (!h) return fail(GPT2_ERR_ARG, "null handle");
  if (param_bytes) *param_bytes = h->pmem_bytes;
  if (other_bytes) *other_bytes = h->amem_bytes + h->dmem_bytes;
  return GPT2_OK;
}

extern "C" const char* gpt2_last_error(void) { return g_last_error.c_str(); }

extern "C" int64_t gpt2_kernel_launches(void) { return (int64_t)launch_counter(); }

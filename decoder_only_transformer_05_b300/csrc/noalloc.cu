// LayerNorm backward without any device allocation (declared in include/gpt2_ops.h).
//
// The ordinary entry point, gpt2_op_layernorm_backward, asks the caller for a buffer of
// per-block partial column sums. Some callers cannot provide one: a host whose memory
// manager reserved the device's memory for its own pool when it started, so that
// cudaMalloc either fails or steals from that pool; a plug-in interface that passes the
// library its inputs and outputs and nothing else; or a loop that must never reach
// cudaMalloc/cudaFree, which can synchronise the whole device. For them this variant keeps
// the scratch in one fixed array that is part of the library's device image: it is
// reserved when the library's device code is loaded on a GPU and stays reserved until the
// process exits, on every GPU that loads it.
#include <cuda.h>
#include <cstdio>
#include <mutex>

#include "../../include/gpt2.h"
#include "../../include/gpt2_ops.h"
#include "launch.h"

using namespace gpt2k;

int gpt2_set_error(int code, const char* msg);   // gpt2.cu

namespace {

// 4 MiB of fp32 partial sums: enough for C = 768 or 1024 at any M (the partial buffer
// holds at most 296 blocks x 2C floats), and for C up to 1771 in general.
constexpr size_t kScratchFloats = size_t(1) << 20;
static __device__ __align__(256) float g_ln_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Per device: the scratch address and the CUDA context it was looked up in. A device reset
// (cudaDeviceReset) or a context made through the driver API gives the device another
// context, in which the old address means nothing; the lookup is then made again.
struct ScratchEntry { float* ptr; CUcontext ctx; };
ScratchEntry g_scratch[kMaxDevices] = {};

// cuCtxGetCurrent from the driver, looked up once through the runtime (no -lcuda).
CUresult (*ctx_get_current())(CUcontext*) {
  static CUresult (*fn)(CUcontext*) = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CUresult (*)(CUcontext*)>(f);
  });
  return fn;
}

// Device address of g_ln_scratch on the current device. In host code the symbol itself
// is only a host-side handle, so the address is looked up with cudaGetSymbolAddress,
// once per device (and again after that device's context changed), while that device is
// current.
int scratch_on_current_device(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gpt2_set_error(GPT2_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return gpt2_set_error(GPT2_ERR_ARG, "device index beyond the scratch table");
  // the current context (null before the runtime has made the device's context; the
  // lookup below makes it, and the entry records the context it ran in)
  CUcontext ctx = nullptr;
  auto get = ctx_get_current();
  if (!get || get(&ctx) != CUDA_SUCCESS)
    return gpt2_set_error(GPT2_ERR_CUDA, "cuCtxGetCurrent is not available");
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchEntry& ent = g_scratch[dev];
  if (!ent.ptr || ent.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ln_scratch);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the built-in scratch failed: %s",
               cudaGetErrorString(e));
      return gpt2_set_error(GPT2_ERR_CUDA, msg);
    }
    if (get(&ctx) != CUDA_SUCCESS) return gpt2_set_error(GPT2_ERR_CUDA, "cuCtxGetCurrent failed");
    ent.ptr = static_cast<float*>(p);
    ent.ctx = ctx;
  }
  *out = ent.ptr;
  return GPT2_OK;
}

}  // namespace

extern "C" int gpt2_op_layernorm_backward_noalloc(int precision, void* dres, int accumulate,
                                                  float* dw, float* db, const void* dy,
                                                  const void* x, const void* w,
                                                  const float* mean, const float* rstd, int M,
                                                  int C, float scale, void* stream) {
  if (M <= 0 || C <= 0) return gpt2_set_error(GPT2_ERR_ARG, "M and C must be positive");
  const size_t need = layernorm_backward_partials_floats(M, C, false);
  if (need > kScratchFloats) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "M=%d, C=%d needs %zu floats of LayerNorm-backward scratch; the built-in array "
             "holds %zu (use gpt2_op_layernorm_backward with a caller buffer)",
             M, C, need, kScratchFloats);
    return gpt2_set_error(GPT2_ERR_ARG, msg);
  }
  float* scratch = nullptr;
  int rc = scratch_on_current_device(&scratch);
  if (rc != GPT2_OK) return rc;
  // Every block of the backward kernel writes its whole row of partial sums before the
  // reduction reads it, so the previous call's contents never need clearing.
  cudaError_t e = layernorm_backward(precision == GPT2_BF16 ? DType::BF16 : DType::F32, dres,
                                     accumulate, dw, db, nullptr, dy, x, w, mean, rstd, M, C,
                                     scale, scratch, 0, (cudaStream_t)stream);
  if (e == cudaSuccess) return GPT2_OK;
  if (e == cudaErrorInvalidValue)
    return gpt2_set_error(GPT2_ERR_ARG, "unsupported shape, alignment or argument");
  return gpt2_set_error(GPT2_ERR_CUDA, cudaGetErrorString(e));
}

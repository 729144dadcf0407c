// grpo_loss_fwd_static: grpo_loss_fwd for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the loss:
// code running inside a memory pool or allocator that must not be re-entered,
// plugin hosts that hand out only the tensors they own, or runtimes that
// forbid allocation after start-up.  They can still pass inputs and outputs,
// but not the workspace grpo_loss_fwd needs.  This entry point uses instead a
// scratch array that lives in the library itself: a file-scope __device__
// array, which every GPU that loads the library holds until the process
// exits.  It allocates nothing and calls grpo_loss_fwd with that array as its
// workspace; everything else is identical.
#include <mutex>

#include "common.cuh"
#include "grpo.h"

namespace grpo {
namespace {

// Largest batch the static scratch covers, and the scratch size: the
// workspace layout for 4096 completions fits in 64 KiB.
constexpr int64_t kStaticMaxN = 4096;
constexpr size_t kStaticScratchBytes = 64 * 1024;

// In host code this name is only a stand-in for the device array: its device
// address comes from cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mutex;
void* g_addr[64] = {};  // device address of g_static_scratch, per device ordinal

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_mutex);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);  // `dev` is current here
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace grpo

extern "C" grpo_status grpo_loss_fwd_static(const void* logits, grpo_dtype dtype, int64_t N,
                                            int64_t P, int64_t C, int64_t V,
                                            const int64_t* input_ids, const int32_t* len,
                                            const float* adv, const float* old_logp,
                                            const float* ref_logp, float eps, float beta,
                                            float norm, float* logp, float* lse, float* w,
                                            float* loss, grpo_stream_t stream) {
  using namespace grpo;
  if (N > kStaticMaxN) return GRPO_ERR_UNSUPPORTED;  // the static scratch is too small
  if (N < 0) return GRPO_ERR_INVALID_ARG;
  if (ws_layout(N).total > kStaticScratchBytes) return GRPO_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return GRPO_ERR_CUDA;
  // grpo_loss_fwd's first kernel resets the scratch header (error flags and
  // the reduction counter); everything else it reads it writes first.
  return grpo_loss_fwd(logits, dtype, N, P, C, V, input_ids, len, adv, old_logp, ref_logp, eps,
                       beta, norm, logp, lse, w, loss, scratch, kStaticScratchBytes, stream);
}

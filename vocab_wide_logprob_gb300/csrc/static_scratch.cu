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
#include "host_ctx.cuh"

namespace grpo {
namespace {

// Largest batch the static scratch covers, and the scratch size: the
// workspace layout for 4096 completions fits in 64 KiB.
constexpr int64_t kStaticMaxN = 4096;
constexpr size_t kStaticScratchBytes = 64 * 1024;

// In host code this name is only a stand-in for the device array: its device
// address comes from cudaGetSymbolAddress below, once per device context.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The array's device address belongs to a CUDA context: a device reset or a
// non-primary context on the same device gives the same symbol another
// address.  The cache is therefore keyed on the current context's unique id.
struct CachedAddress {
  unsigned long long ctx_id;
  void* addr;
};

std::mutex g_mutex;
constexpr int kCacheSlots = 64;
CachedAddress g_cache[kCacheSlots] = {};
int g_cache_used = 0;
int g_cache_next = 0;  // slot replaced next once every slot is taken

// Device address of g_static_scratch in the calling thread's current context
// (the current device's primary context unless the caller made another one
// current).  The first call in a context looks it up with cudaGetSymbolAddress.
cudaError_t scratch_address(void** out) {
  unsigned long long id = 0;
  cudaError_t e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(g_mutex);
  for (int k = 0; k < g_cache_used; ++k) {
    if (g_cache[k].ctx_id == id) {
      *out = g_cache[k].addr;
      return cudaSuccess;
    }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);  // in the current context
  if (e != cudaSuccess) return e;
  int slot;
  if (g_cache_used < kCacheSlots) {
    slot = g_cache_used++;
  } else {
    slot = g_cache_next;
    g_cache_next = (g_cache_next + 1) % kCacheSlots;
  }
  g_cache[slot] = CachedAddress{id, p};
  *out = p;
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

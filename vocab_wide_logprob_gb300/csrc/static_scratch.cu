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
// address comes from cudaGetSymbolAddress below, once per device context.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The array's device address belongs to a CUDA context: a device reset or a
// non-primary context on the same device gives the same symbol another
// address.  The cache is therefore keyed on the current context's unique id
// (cuCtxGetId: ids are never reused within a process), resolved through the
// runtime's driver entry points so the library needs no link to libcuda.
using CtxGetCurrentFn = int (*)(void** ctx);
using CtxGetIdFn = int (*)(void* ctx, unsigned long long* id);

struct CachedAddress {
  unsigned long long ctx_id;
  void* addr;
};

std::mutex g_mutex;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
constexpr int kCacheSlots = 64;
CachedAddress g_cache[kCacheSlots] = {};
int g_cache_used = 0;
int g_cache_next = 0;  // slot replaced next once every slot is taken

cudaError_t resolve_driver_calls() {
  if (g_ctx_get_current != nullptr && g_ctx_get_id != nullptr) return cudaSuccess;
  void* a = nullptr;
  void* b = nullptr;
  cudaDriverEntryPointQueryResult qa, qb;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000,
                                                   cudaEnableDefault, &qa);
  if (e != cudaSuccess) return e;
  e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb);
  if (e != cudaSuccess) return e;
  if (qa != cudaDriverEntryPointSuccess || qb != cudaDriverEntryPointSuccess || !a || !b)
    return cudaErrorNotSupported;
  g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
  g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
  return cudaSuccess;
}

// Device address of g_static_scratch in the calling thread's current context
// (the current device's primary context unless the caller made another one
// current).  The first call in a context looks it up with cudaGetSymbolAddress.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(g_mutex);
  e = resolve_driver_calls();
  if (e != cudaSuccess) return e;
  void* ctx = nullptr;
  if (g_ctx_get_current(&ctx) != 0) return cudaErrorDeviceUninitialized;
  if (ctx == nullptr) {
    // no context current yet: make the device's primary context current
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (g_ctx_get_current(&ctx) != 0 || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  unsigned long long id = 0;
  if (g_ctx_get_id(ctx, &id) != 0) return cudaErrorDeviceUninitialized;
  for (int k = 0; k < g_cache_used; ++k) {
    if (g_cache[k].ctx_id == id) {
      *out = g_cache[k].addr;
      return cudaSuccess;
    }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);  // `ctx` is current here
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

// Host helpers tied to the calling thread's current CUDA context.
#include <map>
#include <mutex>
#include <utility>

#include "host_ctx.cuh"

namespace grpo {
namespace {

// cuCtxGetCurrent and cuCtxGetId, resolved through the runtime's driver entry
// points so the library needs no link to libcuda.
using CtxGetCurrentFn = int (*)(void** ctx);
using CtxGetIdFn = int (*)(void* ctx, unsigned long long* id);

std::mutex g_fn_mutex;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

cudaError_t resolve_driver_calls() {
  std::lock_guard<std::mutex> g(g_fn_mutex);
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

// (context id, kernel) -> the dynamic shared-memory limit set there
std::mutex g_smem_mutex;
std::map<std::pair<unsigned long long, const void*>, int> g_smem;

}  // namespace

cudaError_t current_context_id(unsigned long long* id) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
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
  return g_ctx_get_id(ctx, id) == 0 ? cudaSuccess : cudaErrorDeviceUninitialized;
}

cudaError_t ensure_dynamic_smem(const void* kern, int bytes) {
  unsigned long long id = 0;
  cudaError_t e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(g_smem_mutex);
  const auto key = std::make_pair(id, kern);
  const auto it = g_smem.find(key);
  if (it != g_smem.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  g_smem[key] = bytes;
  return cudaSuccess;
}

}  // namespace grpo

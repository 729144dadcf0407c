// Device-to-device copy with 16-byte loads and streaming stores: the HBM
// ceiling the streaming kernels of this library are compared with (one read
// and one write per byte, the same access pattern as the backward pass).
#include "common.cuh"

namespace grpo {

__global__ void __launch_bounds__(kThreads) copy_kernel(uint4* __restrict__ dst,
                                                        const uint4* __restrict__ src,
                                                        int64_t nvec) {
  constexpr int U = 4;
  pdl_wait();
  pdl_trigger();
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t k0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; k0 < nvec; k0 += stride * U) {
    uint4 d[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (k0 + u * stride < nvec) d[u] = ld_stream(src + k0 + u * stride);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (k0 + u * stride < nvec) st_stream(dst + k0 + u * stride, d[u]);
  }
}

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, const DeviceInfo& d,
                        cudaStream_t st) {
  const int64_t nvec = (int64_t)(bytes / 16);
  if (nvec == 0) return cudaSuccess;
  // oversubscribed grid-stride grid: faster than a persistent one for streams
  int64_t grid = (int64_t)grid_mult("GRPO_COPY_GRID", 256) * d.sms;
  const int64_t need = (nvec + kThreads - 1) / kThreads;
  if (grid > need) grid = need;
  return launch_pdl(copy_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, 1,
                    static_cast<uint4*>(dst), static_cast<const uint4*>(src), nvec);
}

}  // namespace grpo

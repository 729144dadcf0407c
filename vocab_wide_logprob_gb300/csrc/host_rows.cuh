// Internal header: copy of the scored logits rows from mapped host memory.
#pragma once

#include "common.cuh"

namespace grpo {

// After launch_prep: rows P-1+t (t < len_i) of every sequence i of the
// [N, P+C, V] logits at `src` (a device address of page-locked host memory)
// to the same rows of `dst` (device memory of the same shape).
cudaError_t launch_gather_host_rows(const void* src, void* dst, size_t esize, const FwdArgs& a,
                                    const DeviceInfo& d, cudaStream_t st);

// After launch_prep: the fused forward + backward (lse_grad_kernel) reading
// the scored rows from `a.logits`, the device mapping of page-locked host
// logits, and writing them to the same rows of `staging` on the way (device
// memory of the logits' shape).  The host rows, staging and b.dlogits share
// their 16-byte phase.  Same results, bit for bit, as launch_lse_grad on the
// logits in device memory.
cudaError_t launch_lse_grad_host(const FwdArgs& a, const BwdArgs& b, void* staging,
                                 const DeviceInfo& d, cudaStream_t st);

}  // namespace grpo

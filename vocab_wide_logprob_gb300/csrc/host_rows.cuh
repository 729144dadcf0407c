// Internal header: copy of the scored logits rows from mapped host memory.
#pragma once

#include "common.cuh"

namespace grpo {

// After launch_prep: rows P-1+t (t < len_i) of every sequence i of the
// [N, P+C, V] logits at `src` (a device address of page-locked host memory)
// to the same rows of `dst` (device memory of the same shape).
cudaError_t launch_gather_host_rows(const void* src, void* dst, size_t esize, const FwdArgs& a,
                                    const DeviceInfo& d, cudaStream_t st);

}  // namespace grpo

// Host helpers tied to the calling thread's current CUDA context.  Internal
// header.
#pragma once

#include <cuda_runtime.h>

namespace grpo {

// Unique id of the calling thread's current context (the current device's
// primary context, made current first, when none is); ids are never reused
// within a process, so a device reset or another context on the same device
// gives a new one.
cudaError_t current_context_id(unsigned long long* id);

// Raises `kern`'s dynamic shared-memory limit to at least `bytes` in the
// current context, once per (context, kernel), thread-safe.  (The runtime
// also carries a limit it was given into contexts it loads the kernel in
// later; the library does not depend on that.)
cudaError_t ensure_dynamic_smem(const void* kern, int bytes);

}  // namespace grpo

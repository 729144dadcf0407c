// Internal header: the bounded-wait self-test kernel (grpo_selftest_timeout).
#pragma once

#include "common.cuh"

namespace grpo {

// One CTA waits on a shared-memory barrier that nothing completes; after the
// wait limit it sets kFlagTimeout in the workspace header and exits.
cudaError_t launch_selftest_timeout(void* workspace, cudaStream_t st);

}  // namespace grpo

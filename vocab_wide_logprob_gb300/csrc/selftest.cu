// grpo_selftest_timeout: runs the library's bounded wait against a barrier
// that nothing completes, so that a caller (or a test) can check that the
// wait ends by itself and reports through the workspace, with the context
// left usable.  Every wait of the library's kernels on a transaction or
// arrival barrier goes through the same mbar_wait(): after kWaitLimitNs it
// gives up, the kernel records kFlagTimeout in the workspace header and
// stops issuing work.  Nothing faults, traps or hangs.
#include "selftest.cuh"

namespace grpo {
namespace {

__global__ void __launch_bounds__(32) selftest_timeout_kernel(WsHeader* hdr) {
  __shared__ __align__(8) uint64_t s_bar;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x != 0) return;
  const uint32_t bar = smem_u32(&s_bar);
  mbar_init(bar, 1);  // one arrival expected; none is ever made
  mbar_init_fence();
  if (!mbar_wait(bar, 0)) atomicOr(&hdr->flags, kFlagTimeout);
}

}  // namespace
}  // namespace grpo

namespace grpo {

cudaError_t launch_selftest_timeout(void* workspace, cudaStream_t st) {
  return launch_pdl(selftest_timeout_kernel, dim3(1), dim3(32), 0, st, 1,
                    static_cast<WsHeader*>(workspace));
}

}  // namespace grpo

// Completion mask and group advantage.
//
// mask_kernel restates "The completion mask" of "Making Dr GRPO go brrr"
// (salahadawi.com): 1 up to and including the first EOS of the completion,
// 0 after it, and a completion with no EOS entirely valid.  It finds the
// first EOS as a minimum over positions rather than with argmax, so the
// "argmax returns 0 when there is no True" trap cannot arise.
//
// advantage_kernel restates section "Dr. GRPO": A_i = R_i - mu of the group,
// with no division by sigma, one warp per group with a shuffle reduction.
#include "common.cuh"

namespace grpo {

// One CTA per completion.  Each thread scans positions tid, tid+256, ...
// without an early exit (so its loads are independent and overlap), keeps the
// smallest EOS position it saw, and the CTA takes the minimum of those.
__global__ void __launch_bounds__(kThreads) mask_kernel(const int64_t* __restrict__ ids,
                                                        int64_t T, int64_t P, int64_t C,
                                                        int64_t eos, uint8_t* __restrict__ mask,
                                                        int32_t* __restrict__ len) {
  __shared__ int64_t warp_min[kWarps];
  pdl_wait();
  pdl_trigger();
  const int64_t i = blockIdx.x;
  const int64_t* comp = ids + i * T + P;
  int64_t first = C;  // C stands for "no EOS"
#pragma unroll 4
  for (int64_t j = threadIdx.x; j < C; j += kThreads)
    if (comp[j] == eos && j < first) first = j;
  for (int o = 16; o > 0; o >>= 1) {
    const int64_t other = __shfl_xor_sync(0xffffffffu, first, o);
    first = other < first ? other : first;
  }
  if ((threadIdx.x & 31) == 0) warp_min[threadIdx.x >> 5] = first;
  __syncthreads();
  first = warp_min[0];
#pragma unroll
  for (int k = 1; k < kWarps; ++k) first = warp_min[k] < first ? warp_min[k] : first;
  // positions <= first EOS are real; no EOS (first == C) keeps all C
  const int64_t n_valid = first < C ? first + 1 : C;
  if (threadIdx.x == 0) len[i] = (int32_t)n_valid;
  if (mask != nullptr) {
    uint8_t* m = mask + i * C;
    for (int64_t j = threadIdx.x; j < C; j += kThreads) m[j] = (uint8_t)(j < n_valid);
  }
}

cudaError_t launch_mask(const int64_t* ids, int64_t N, int64_t P, int64_t C, int64_t eos,
                        uint8_t* mask, int32_t* len, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  return launch_pdl(mask_kernel, dim3((unsigned)N), dim3(kThreads), 0, st, 1, ids, P + C, P, C,
                    eos, mask, len);
}

// One warp per group.  Lane l sums rewards l, l+32, ... of the group in that
// order; a butterfly of shuffles then leaves the same total in every lane
// (each step adds the same two operands in both partner lanes).
//   mode 0 (Dr. GRPO):      A = R - mu
//   mode 1 (original GRPO): A = (R - mu) / (sigma + std_eps), sigma over the G
//                           rewards (dividing by G), IEEE sqrt and division
// n_contrast (optional) counts the groups whose rewards are not all equal.
__device__ __forceinline__ void advantage_group(const float* __restrict__ R, int64_t B, int64_t G,
                                                int mode, float std_eps, float* __restrict__ adv,
                                                int32_t* __restrict__ n_contrast) {
  const int64_t b = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const float* r = R + b * G;
  float sum = 0.f;
  for (int64_t g = lane; g < G; g += 32) sum += r[g];
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  // IEEE division: k/G is exact for binary rewards and power-of-two G
  const float mu = __fdiv_rn(sum, (float)G);
  float scale = 1.f;
  if (mode == 1) {
    float ss = 0.f;
    for (int64_t g = lane; g < G; g += 32) ss += (r[g] - mu) * (r[g] - mu);
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    scale = __fadd_rn(__fsqrt_rn(__fdiv_rn(ss, (float)G)), std_eps);
  }
  for (int64_t g = lane; g < G; g += 32)
    adv[b * G + g] = mode == 1 ? __fdiv_rn(r[g] - mu, scale) : r[g] - mu;
  if (n_contrast != nullptr) {
    bool differs = false;
    for (int64_t g = lane; g < G; g += 32) differs |= r[g] != r[0];
    if (__any_sync(0xffffffffu, differs) && lane == 0) atomicAdd(n_contrast, 1);
  }
}

// after_mask: the preceding kernel is grpo_mask's, which reads the ids and
// writes the mask and lengths only (everything before it has completed), so
// the rewards and advantages are touched without waiting on it; thread 0 of
// CTA 0 waits before it exits, so this kernel still completes after it.
__global__ void __launch_bounds__(kThreads) advantage_kernel(const float* __restrict__ R,
                                                             int64_t B, int64_t G, int mode,
                                                             float std_eps,
                                                             float* __restrict__ adv,
                                                             int32_t* __restrict__ n_contrast,
                                                             int after_mask) {
  if (!after_mask) pdl_wait();
  pdl_trigger();
  advantage_group(R, B, G, mode, std_eps, adv, n_contrast);
  if (after_mask && blockIdx.x == 0 && threadIdx.x == 0) pdl_wait();
}

cudaError_t launch_advantage(const float* R, int64_t B, int64_t G, int mode, float std_eps,
                             float* adv, int32_t* n_contrast, cudaStream_t st, bool after_mask) {
  if (B == 0) return n_contrast ? cudaMemsetAsync(n_contrast, 0, sizeof(int32_t), st) : cudaSuccess;
  if (n_contrast != nullptr) {
    cudaError_t e = cudaMemsetAsync(n_contrast, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
    after_mask = false;  // the memset now comes between the two kernels
  }
  const unsigned blocks = (unsigned)((B + kWarps - 1) / kWarps);
  return launch_pdl(advantage_kernel, dim3(blocks), dim3(kThreads), 0, st, 1, R, B, G, mode,
                    std_eps, adv, n_contrast, after_mask ? 1 : 0);
}

}  // namespace grpo

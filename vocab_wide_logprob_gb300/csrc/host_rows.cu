// Scored logits rows from page-locked host memory: the loss reads logits row
// P-1+t of sequence i only for t < len_i ("compute_logprobs" shifts by one
// and the completion mask zeroes the rest, "Making Dr GRPO go brrr",
// salahadawi.com), so when the logits sit in host memory only those rows have
// to cross the host link.  This kernel reads them through the buffer's device
// mapping and writes them to the same rows of a device buffer of the logits'
// shape; the other rows of that buffer are left as they are (nothing reads
// them).
#include "host_rows.cuh"

namespace grpo {
namespace {

// Row of the n-th scored token: binary search of the completion over the
// exclusive prefix sums of the clamped lengths.
__device__ __forceinline__ int64_t scored_row(const int32_t* __restrict__ off, int64_t N,
                                              int64_t T, int64_t P, int64_t r) {
  int lo = 0, hi = (int)N;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= r)
      lo = mid;
    else
      hi = mid;
  }
  return (int64_t)lo * T + P - 1 + (r - off[lo]);
}

// U: the unit copied per access (16 bytes when a row is a whole number of
// 16-byte vectors and both buffers are 16-byte aligned, else one element).
// Each thread keeps kGatherUnroll loads in flight (the host link's latency is
// microseconds), so a grid of a few CTAs per SM fills the link and leaves
// the SMs' other slots to a kernel running beside this one.
constexpr int kGatherUnroll = 4;

template <typename U>
__global__ void __launch_bounds__(kThreads) gather_host_rows_kernel(const U* __restrict__ src,
                                                                    U* __restrict__ dst,
                                                                    const int32_t* __restrict__ off,
                                                                    int64_t N, int64_t T, int64_t P,
                                                                    int64_t units_per_row) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)off[N] * units_per_row;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t k0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; k0 < total;
       k0 += stride * kGatherUnroll) {
    U v[kGatherUnroll];
    int64_t e[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      const int64_t k = k0 + u * stride;
      e[u] = -1;
      if (k < total) {
        const int64_t r = k / units_per_row, c = k - r * units_per_row;
        e[u] = scored_row(off, N, T, P, r) * units_per_row + c;
        if constexpr (sizeof(U) == 16)
          v[u] = ld_stream(src + e[u]);
        else
          v[u] = src[e[u]];
      }
    }
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u) {
      if (e[u] < 0) continue;
      if constexpr (sizeof(U) == 16)
        st_stream(dst + e[u], v[u]);
      else
        dst[e[u]] = v[u];
    }
  }
}

}  // namespace

cudaError_t launch_gather_host_rows(const void* src, void* dst, size_t esize, const FwdArgs& a,
                                    const DeviceInfo& d, cudaStream_t st) {
  const WsLayout l = ws_layout(a.N);
  const int32_t* off =
      reinterpret_cast<const int32_t*>(static_cast<const char*>(a.ws) + l.offsets);
  const int64_t T = a.P + a.C;
  const size_t row_bytes = (size_t)a.V * esize;
  const bool vec = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(dst) % 16 == 0;
  // bound by the host link, not by the SMs: a few CTAs per SM
  const int64_t grid = (int64_t)grid_mult("GRPO_HOST_GRID", 4) * d.sms;
  if (vec)
    return launch_pdl(gather_host_rows_kernel<uint4>, dim3((unsigned)grid), dim3(kThreads), 0, st,
                      1, static_cast<const uint4*>(src), static_cast<uint4*>(dst), off, a.N, T,
                      a.P, (int64_t)(row_bytes / 16));
  if (esize == 4)
    return launch_pdl(gather_host_rows_kernel<uint32_t>, dim3((unsigned)grid), dim3(kThreads), 0,
                      st, 1, static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), off,
                      a.N, T, a.P, a.V);
  return launch_pdl(gather_host_rows_kernel<uint16_t>, dim3((unsigned)grid), dim3(kThreads), 0, st,
                    1, static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), off, a.N, T,
                    a.P, a.V);
}

}  // namespace grpo

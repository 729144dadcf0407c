// Shifted log-softmax + gather over the vocabulary ("compute_logprobs" of
// "Making Dr GRPO go brrr", salahadawi.com): for every valid completion token
// t of sequence i, with y = input_ids[i, P+t] and z = logits row P-1+t
// ("logits at position t predict the token at t+1"),
//     lse  = log sum_v exp(z_v),    logp = z_y - lse.
// The page materialises log_softmax over [B*G, C, V] and gathers one column;
// here one streaming pass over each valid row keeps only a running
// (max, sum of exp) per thread, and the target logit is picked out of the
// same loads.  Rows past the first EOS are not read at all.
//
// Layout of the work: each valid row is split over the K CTAs of a thread
// block cluster (split-V).  CTA k streams its 1/K of the row with 16-byte
// loads, reduces its (max, sum) over its 256 threads, and sends the partial
// to CTA 0 of the cluster through distributed shared memory; CTA 0 merges
// the K partials in rank order (deterministic) and writes logp and lse.
// The grid is persistent: as many clusters as fit on the GPU at once, each
// looping over valid rows r = cluster, cluster + #clusters, ... The row of
// valid token r is found by binary search in the prefix sums of the lengths
// that prep_kernel writes.
#include <stdlib.h>

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"

namespace grpo {

// Prefix-sum table entries kept in shared memory (larger N searches global).
constexpr int kSmemOffsets = 4096;

// ---------------------------------------------------------------------------
// prep: clamp lengths, exclusive prefix sums, reset the workspace header
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(1024) prep_kernel(const int32_t* __restrict__ len, int64_t N,
                                                    int64_t C, WsHeader* hdr,
                                                    int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ lens_c) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  __shared__ uint32_t flags;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry = 0;
    flags = 0;
  }
  __syncthreads();
  for (int64_t base = 0; base < N; base += 1024) {
    const int64_t i = base + tid;
    int32_t L = 0;
    if (i < N) {
      const int32_t raw = len[i];
      L = raw < 0 ? 0 : (raw > C ? (int32_t)C : raw);
      if (L != raw) atomicOr(&flags, kFlagLengthRange);
      lens_c[i] = L;
    }
    int32_t x = L;  // inclusive scan within the warp
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int32_t tw = warp_tot[lane];
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, tw, o);
        if (lane >= o) tw += y;
      }
      warp_tot[lane] = tw;  // inclusive over the warps of this chunk
    }
    __syncthreads();
    if (i < N) offsets[i] = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - L;
    __syncthreads();
    if (tid == 0) carry += warp_tot[31];
    __syncthreads();
  }
  if (tid == 0) {
    offsets[N] = carry;
    hdr->flags = flags;
    hdr->ticket = 0;
  }
}

cudaError_t launch_prep(const FwdArgs& a, cudaStream_t st) {
  const WsLayout l = ws_layout(a.N);
  char* ws = static_cast<char*>(a.ws);
  prep_kernel<<<1, 1024, 0, st>>>(a.len, a.N, a.C, reinterpret_cast<WsHeader*>(ws),
                                  reinterpret_cast<int32_t*>(ws + l.offsets),
                                  reinterpret_cast<int32_t*>(ws + l.lens));
  return cudaGetLastError();
}

template <typename T>
struct LseParams {
  const T* logits;
  int64_t T_len, P, C, V, N;
  const int64_t* ids;
  const int32_t* offsets;  // [N+1] exclusive prefix sums of the clamped lengths
  float* logp;
  float* lse;
  WsHeader* hdr;
  int64_t chunk;  // elements of a row per CTA of the cluster (multiple of kPerVec)
};

// Online update of a thread's running (m, s0..s3) with one value.
__device__ __forceinline__ void online1(float x, float& m, float& s0, float& s1, float& s2,
                                        float& s3) {
  if (x > m) {
    const float sc = ex2((m - x) * kLog2e);
    s0 *= sc;
    s1 *= sc;
    s2 *= sc;
    s3 *= sc;
    m = x;
  }
  if (m != -INFINITY) s0 += ex2(fmaf(x, kLog2e, -m * kLog2e));
}

template <typename T, int K>
__global__ void __launch_bounds__(kThreads) lse_gather_kernel(const LseParams<T> p) {
  using E = Elt<T>;
  constexpr int EPV = E::kPerVec;
  constexpr int U = E::kUnroll;
  extern __shared__ int32_t s_off_dyn[];
  __shared__ float4 s_part[2][K];     // CTA 0: partial (m, s, z_y, has z_y) of each rank
  __shared__ float2 s_red[2][kWarps];  // per-warp (m, s)
  __shared__ float s_zy[2];
  __shared__ int64_t s_found[2];       // row whose target logit this CTA picked up
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = K > 1 ? cluster_ctarank() : 0u;
  const int64_t q = K > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
  const int64_t nq = K > 1 ? (int64_t)nclusters_x() : (int64_t)gridDim.x;

  const int32_t* off = p.offsets;
  if (p.N + 1 <= kSmemOffsets) {
    for (int64_t k = tid; k <= p.N; k += kThreads) s_off_dyn[k] = p.offsets[k];
    off = s_off_dyn;
  }
  if (tid < 2) s_found[tid] = -1;
  // every CTA of the cluster is running (and has initialised its shared
  // memory) before any distributed-shared-memory store
  if (K > 1)
    cluster_sync();
  else
    __syncthreads();

  const int64_t tv = off[p.N];  // number of valid tokens
  const int64_t v0 = (int64_t)rank * p.chunk;
  const int64_t v1 = min(p.V, v0 + p.chunk);
  int par = 0;
  for (int64_t r = q; r < tv; r += nq, par ^= 1) {
    // completion i holding valid token r: off[i] <= r < off[i+1]
    int lo = 0, hi = (int)p.N;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (off[mid] <= r)
        lo = mid;
      else
        hi = mid;
    }
    const int64_t i = lo, t = r - off[lo];
    const T* row = p.logits + (i * p.T_len + (p.P - 1 + t)) * p.V;
    const int64_t y = p.ids[i * p.T_len + p.P + t];

    float m = -INFINITY, s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    float zy = 0.f;
    bool found = false;
    if (v0 < v1) {
      // 16-byte aligned interior [a, b) of the slice [v0, v1)
      const uintptr_t addr = reinterpret_cast<uintptr_t>(row + v0);
      const int64_t skip = (int64_t)(((16u - (unsigned)(addr & 15u)) & 15u) / sizeof(T));
      const int64_t a = min(v0 + skip, v1);
      const int64_t nvec = (v1 - a) / EPV;
      const int64_t b = a + nvec * EPV;
      const uint4* vp = reinterpret_cast<const uint4*>(row + a);
      const int64_t ky = (y >= a && y < b) ? (y - a) / EPV : -1;
      const int ey = ky >= 0 ? (int)((y - a) % EPV) : 0;
      for (int64_t k0 = tid; k0 < nvec; k0 += (int64_t)kThreads * U) {
        uint4 d[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t k = k0 + (int64_t)u * kThreads;
          d[u] = k < nvec ? ld_stream(vp + k)
                          : make_uint4(E::kNegInf, E::kNegInf, E::kNegInf, E::kNegInf);
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (k0 + (int64_t)u * kThreads == ky) {
            zy = E::extract(d[u], ey);
            found = true;
          }
        float x[U * EPV];
#pragma unroll
        for (int u = 0; u < U; ++u) E::unpack(d[u], x + u * EPV);
        float bm = x[0];
#pragma unroll
        for (int k = 1; k < U * EPV; ++k) bm = fmaxf(bm, x[k]);
        if (bm > m) {
          const float sc = ex2((m - bm) * kLog2e);
          s0 *= sc;
          s1 *= sc;
          s2 *= sc;
          s3 *= sc;
          m = bm;
        }
        if (m != -INFINITY) {
          const float mL = m * kLog2e;
#pragma unroll
          for (int k = 0; k < U * EPV; k += 4) {
            s0 += ex2(fmaf(x[k + 0], kLog2e, -mL));
            s1 += ex2(fmaf(x[k + 1], kLog2e, -mL));
            s2 += ex2(fmaf(x[k + 2], kLog2e, -mL));
            s3 += ex2(fmaf(x[k + 3], kLog2e, -mL));
          }
        }
      }
      // ragged head [v0, a) and tail [b, v1): fewer than EPV elements each
      int64_t e = -1;
      if (tid < a - v0)
        e = v0 + tid;
      else if (tid >= 32 && tid - 32 < v1 - b)
        e = b + (tid - 32);
      if (e >= 0) {
        const float xv = E::load1(row + e);
        if (e == y) {
          zy = xv;
          found = true;
        }
        online1(xv, m, s0, s1, s2, s3);
      }
    }
    float s = (s0 + s1) + (s2 + s3);
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2b = __shfl_xor_sync(0xffffffffu, s, o);
      lse_merge(m, s, m2, s2b);
    }
    if (lane == 0) s_red[par][warp] = make_float2(m, s);
    if (found) {
      s_zy[par] = zy;
      s_found[par] = r;
    }
    __syncthreads();
    if (tid == 0) {
      float cm = s_red[par][0].x, cs = s_red[par][0].y;
#pragma unroll
      for (int k = 1; k < kWarps; ++k) lse_merge(cm, cs, s_red[par][k].x, s_red[par][k].y);
      const bool has = s_found[par] == r;
      const float4 part = make_float4(cm, cs, has ? s_zy[par] : 0.f, has ? 1.f : 0.f);
      if (K > 1)
        st_cluster_f32x4(map_to_rank(smem_u32(&s_part[par][rank]), 0), part);
      else
        s_part[par][0] = part;
    }
    if (K > 1) cluster_sync();
    if (rank == 0 && tid == 0) {
      float4 pk = s_part[par][0];
      float cm = pk.x, cs = pk.y, z = pk.z;
      bool has = pk.w != 0.f;
#pragma unroll
      for (int k = 1; k < K; ++k) {
        pk = s_part[par][k];
        lse_merge(cm, cs, pk.x, pk.y);
        if (pk.w != 0.f) {
          z = pk.z;
          has = true;
        }
      }
      const float l = cm + logf(cs);
      const int64_t o = i * p.C + t;
      if (has) {
        p.logp[o] = z - l;
        p.lse[o] = l;
      } else {  // y outside [0, V): no CTA saw it
        p.logp[o] = __int_as_float(0x7fc00000);
        p.lse[o] = __int_as_float(0x7fc00000);
        atomicOr(&p.hdr->flags, kFlagTokenRange);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------

namespace {

std::mutex g_occ_mutex;
std::map<std::tuple<int, int, int, int>, int> g_occ;  // (device, dtype, K, smem) -> clusters

template <typename T, int K>
cudaError_t launch_k(const FwdArgs& a, const DeviceInfo& d, cudaStream_t st) {
  constexpr int EPV = Elt<T>::kPerVec;
  const WsLayout l = ws_layout(a.N);
  char* ws = static_cast<char*>(a.ws);
  LseParams<T> p;
  p.logits = static_cast<const T*>(a.logits);
  p.T_len = a.P + a.C;
  p.P = a.P;
  p.C = a.C;
  p.V = a.V;
  p.N = a.N;
  p.ids = a.ids;
  p.offsets = reinterpret_cast<const int32_t*>(ws + l.offsets);
  p.logp = a.logp;
  p.lse = a.lse;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.chunk = ((a.V + K - 1) / K + EPV - 1) / EPV * EPV;

  const size_t smem = a.N + 1 <= kSmemOffsets ? sizeof(int32_t) * (size_t)(a.N + 1) : 0;
  auto kern = lse_gather_kernel<T, K>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = K;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = K > 1 ? 1 : 0;

  int clusters = 0;
  const auto key = std::make_tuple(d.device, (int)sizeof(T), K, (int)smem);
  {
    std::lock_guard<std::mutex> g(g_occ_mutex);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) clusters = it->second;
  }
  if (clusters == 0) {
    cudaError_t e;
    if (K > 1) {
      cfg.gridDim = dim3(K);
      e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    } else {
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
      clusters = per_sm * d.sms;
    }
    if (e != cudaSuccess) return e;
    if (clusters < 1) clusters = 1;
    std::lock_guard<std::mutex> g(g_occ_mutex);
    g_occ[key] = clusters;
  }
  const int64_t max_rows = a.N * a.C;  // upper bound on the valid tokens
  const int64_t nq = clusters < max_rows ? clusters : max_rows;
  cfg.gridDim = dim3((unsigned)(nq * K));
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename T>
cudaError_t launch_t(const FwdArgs& a, const DeviceInfo& d, cudaStream_t st) {
  switch (row_split(a.V * (int64_t)sizeof(T), "GRPO_LSE_CLUSTER")) {
    case 8:
      return launch_k<T, 8>(a, d, st);
    case 4:
      return launch_k<T, 4>(a, d, st);
    case 2:
      return launch_k<T, 2>(a, d, st);
    default:
      return launch_k<T, 1>(a, d, st);
  }
}

}  // namespace

cudaError_t launch_lse_gather(const FwdArgs& a, const DeviceInfo& d, cudaStream_t st) {
  if (a.N == 0 || a.C == 0) return cudaSuccess;
  return a.dtype == 0 ? launch_t<float>(a, d, st) : launch_t<uint16_t>(a, d, st);
}

}  // namespace grpo

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
// block cluster (split-V; K from lse_split: 1, whole rows per CTA, unless the
// batch has too few rows to occupy the GPU).  CTA k streams its 1/K of the
// row with 16-byte loads, reduces its (max, sum) over its 256 threads, and
// sends the partial to CTA 0 of the cluster through distributed shared
// memory; CTA 0 merges the K partials in rank order (deterministic) and
// writes logp and lse.
// The grid is persistent: as many clusters as fit on the GPU at once, each
// looping over valid rows r = cluster, cluster + #clusters, ... The row of
// valid token r is found by binary search in the prefix sums of the lengths
// that prep_kernel writes.
#include <stdlib.h>

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "host_ctx.cuh"

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
  pdl_wait();
  pdl_trigger();
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
  return launch_pdl(prep_kernel, dim3(1), dim3(1024), 0, st, 1, a.len, a.N, a.C,
                    reinterpret_cast<WsHeader*>(ws), reinterpret_cast<int32_t*>(ws + l.offsets),
                    reinterpret_cast<int32_t*>(ws + l.lens));
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
  // the log-probs-only call: this kernel also writes 0 to logp and lse past
  // each length (the loss forward's surrogate kernel does that otherwise)
  bool zero_past;
  // launched right after prep with the offsets table in shared memory: the
  // table is computed here from the raw lengths before waiting on prep
  bool early;
  const int32_t* len;  // raw lengths
};

// Ring of shared-memory stages filled by bulk copies (TMA).
constexpr int kStages = 3;
constexpr int kStageBytes = 16384;
constexpr int kConsumers = kThreads;          // 8 consumer warps
constexpr int kLseThreads = kConsumers + 32;  // + 1 producer warp
constexpr int kVecPerStage = kStageBytes / 16;
constexpr int kVecPerThread = kVecPerStage / kConsumers;
static_assert(kVecPerStage % kConsumers == 0, "stage must split evenly over consumers");

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

// Completion holding valid token r: the i with off[i] <= r < off[i+1].
__device__ __forceinline__ int locate(const int32_t* off, int64_t N, int64_t r) {
  int lo = 0, hi = (int)N;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= r)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

// Geometry of one CTA's share of one row: the slice [v0, v1) of the row,
// its 16-byte aligned interior [a, a + 8*nvec/..) moved by bulk copies, and
// the ragged head [v0, a) / tail [b, v1) read with scalar loads.
template <typename T>
struct Slice {
  const T* row;
  int64_t a, b, nvec;
  uint32_t bytes;  // interior bytes (multiple of 16)
  int nchunks;
};

template <typename T>
__device__ __forceinline__ Slice<T> slice_of(const T* row, int64_t v0, int64_t v1) {
  constexpr int EPV = Elt<T>::kPerVec;
  Slice<T> sl;
  sl.row = row;
  if (v0 >= v1) {
    sl.a = sl.b = v0;
    sl.nvec = 0;
  } else {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row + v0);
    const int64_t skip = (int64_t)(((16u - (unsigned)(addr & 15u)) & 15u) / sizeof(T));
    sl.a = min(v0 + skip, v1);
    sl.nvec = (v1 - sl.a) / EPV;
    sl.b = sl.a + sl.nvec * EPV;
  }
  sl.bytes = (uint32_t)(sl.nvec * 16);
  sl.nchunks = (int)((sl.bytes + kStageBytes - 1) / kStageBytes);
  return sl;
}

// CTA 0 of the cluster: merge the K partials of a row in rank order and
// write logp and lse of token (i, t).
template <int K, typename P>
__device__ __forceinline__ void finalize_row(const P& p, const float4* part, int64_t i,
                                             int64_t t) {
  float4 pk = part[0];
  float cm = pk.x, cs = pk.y, z = pk.z;
  bool has = pk.w != 0.f;
#pragma unroll
  for (int k = 1; k < K; ++k) {
    pk = part[k];
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
    pdl_wait();  // prep has reset the header
    atomicOr(&p.hdr->flags, kFlagTokenRange);
  }
}

// Persistent cluster kernel.  Warps 0..7 consume, warp 8 produces: its lane 0
// walks the same rows as the consumers and issues one bulk copy per stage of
// each row's interior, running ahead across rows as far as the ring allows.
// At the end of a row each CTA sends its (max, sum, target logit) partial to
// CTA 0 through distributed shared memory and arrives on the cluster
// barrier; the matching wait comes one row later, so no CTA stalls at the
// barrier, and CTA 0 merges row r's partials then.  Partials rotate over
// three slots: slot r%3 is rewritten for row r+3 only after every thread has
// passed the wait of row r+1, which CTA 0 reaches after merging row r.
template <typename T, int K>
__global__ void __launch_bounds__(kLseThreads, 3) lse_gather_kernel(const LseParams<T> p) {
  using E = Elt<T>;
  constexpr int EPV = E::kPerVec;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t s_full[kStages];
  __shared__ __align__(8) uint64_t s_empty[kStages];
  __shared__ float4 s_part[3][K];     // CTA 0: partial (m, s, z_y, has z_y) of each rank
  __shared__ float2 s_red[2][kWarps];  // per consumer warp (m, s)
  __shared__ float s_zy[3];
  __shared__ int64_t s_found[3];       // row whose target logit this CTA picked up
  __shared__ int s_abort;              // a bounded wait gave up
  __shared__ int32_t s_warp[kLseThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool producer = warp == kWarps;
  const uint32_t rank = K > 1 ? cluster_ctarank() : 0u;
  const int64_t q = K > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
  const int64_t nq = K > 1 ? (int64_t)nclusters_x() : (int64_t)gridDim.x;
  const uint32_t ring = smem_u32(smem);

  if (tid < 3) s_found[tid] = -1;
  if (tid == 0) {
    s_abort = 0;
    for (int k = 0; k < kStages; ++k) {
      mbar_init(smem_u32(&s_full[k]), 1);
      mbar_init(smem_u32(&s_empty[k]), kWarps);
    }
    mbar_init_fence();
  }
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes);
  const int32_t* off = p.offsets;
  if (p.early) {
    // every kernel before prep has completed (prep waits before it lets this
    // kernel launch): lengths, ids and logits can be read now; the header
    // prep resets is touched only after pdl_wait()
    pdl_trigger();
    block_clamped_offsets(p.len, p.N, p.C, s_off, s_warp);
    off = s_off;
  } else {
    pdl_wait();  // the previous kernel's writes (offsets, ids) are visible from here
    pdl_trigger();
    if (p.N + 1 <= kSmemOffsets) {
      for (int64_t k = tid; k <= p.N; k += kLseThreads) s_off[k] = p.offsets[k];
      off = s_off;
    }
  }
  // every CTA of the cluster is running and initialised before any
  // distributed-shared-memory store or bulk copy
  if (K > 1)
    cluster_sync();
  else
    __syncthreads();

  const int64_t tv = off[p.N];  // number of valid tokens
  const int64_t v0 = (int64_t)rank * p.chunk;
  const int64_t v1 = min(p.V, v0 + p.chunk);
  int stage = 0;
  uint32_t phase = 0;
  int64_t prev_i = 0, prev_t = 0;
  int64_t it = 0;
  uint32_t issued = 0;  // producer: bulk copies issued

  // the next row's (i, t, y) are fetched one row ahead, so the id load's
  // latency hides behind the current row
  int64_t i_nx = 0, t_nx = 0, y_nx = 0;
  if (q < tv) {
    i_nx = locate(off, p.N, q);
    t_nx = q - off[i_nx];
    if (!producer) y_nx = __ldg(p.ids + i_nx * p.T_len + p.P + t_nx);
  }
  for (int64_t r = q; r < tv; r += nq, ++it) {
    const int slot = (int)(it % 3);
    const int64_t i = i_nx, t = t_nx, y = y_nx;
    if (r + nq < tv) {
      i_nx = locate(off, p.N, r + nq);
      t_nx = r + nq - off[i_nx];
      if (!producer) y_nx = __ldg(p.ids + i_nx * p.T_len + p.P + t_nx);
    }
    const T* row = p.logits + (i * p.T_len + (p.P - 1 + t)) * p.V;
    const Slice<T> sl = slice_of(row, v0, v1);

    if (producer) {
      if (lane == 0) {
        const char* src = reinterpret_cast<const char*>(row + sl.a);
        for (int c = 0; c < sl.nchunks; ++c) {
          if (*(volatile int*)&s_abort) break;
          if (!mbar_wait(smem_u32(&s_empty[stage]), phase ^ 1u)) {
            pdl_wait();
            atomicOr(&p.hdr->flags, kFlagTimeout);
            *(volatile int*)&s_abort = 1;
            break;
          }
          const uint32_t nb = min((uint32_t)kStageBytes, sl.bytes - (uint32_t)c * kStageBytes);
          const uint32_t full = smem_u32(&s_full[stage]);
          mbar_arrive_expect_tx(full, nb);
          bulk_g2s(ring + stage * kStageBytes, src + (size_t)c * kStageBytes, nb, full);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      __syncwarp();
    } else {
      float m = -INFINITY, s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      const uint64_t L2 = f2_pack(kLog2e, kLog2e);
      uint64_t acc01 = f2_pack(0.f, 0.f), acc23 = f2_pack(0.f, 0.f);
      float zy = 0.f;
      bool found = false;
      // ragged head and tail (fewer than EPV elements each)
      int64_t e = -1;
      if (tid < sl.a - v0)
        e = v0 + tid;
      else if (tid >= 32 && tid - 32 < v1 - sl.b)
        e = sl.b + (tid - 32);
      if (e >= 0) {
        const float xv = E::load1(row + e);
        if (e == y) {
          zy = xv;
          found = true;
        }
        online1(xv, m, s0, s1, s2, s3);
      }
      // the target's vector: chunk cy, consumer thread ty, register slot uy
      const int64_t ky = (y >= sl.a && y < sl.b) ? (y - sl.a) / EPV : -1;
      const int ey = ky >= 0 ? (int)((y - sl.a) % EPV) : 0;
      const int cy = ky >= 0 ? (int)(ky / kVecPerStage) : -1;
      const int kl = ky >= 0 ? (int)(ky % kVecPerStage) : 0;
      const int ty = kl % kConsumers, uy = kl / kConsumers;
      for (int c = 0; c < sl.nchunks; ++c) {
        bool ok = !*(volatile int*)&s_abort;
        if (ok && !mbar_wait(smem_u32(&s_full[stage]), phase)) {
          pdl_wait();
          atomicOr(&p.hdr->flags, kFlagTimeout);
          *(volatile int*)&s_abort = 1;
          ok = false;
        }
        if (ok) {
          const int64_t vbase = (int64_t)c * kVecPerStage;
          (void)vbase;
          const int nv = (int)min((int64_t)kVecPerStage, sl.nvec - vbase);
          const uint32_t sbase = ring + stage * kStageBytes;
          uint4 d[kVecPerThread];
#pragma unroll
          for (int u = 0; u < kVecPerThread; ++u) {
            const int k = tid + u * kConsumers;
            d[u] = k < nv ? ld_shared_v4(sbase + 16u * k)
                          : make_uint4(E::kNegInf, E::kNegInf, E::kNegInf, E::kNegInf);
          }
          if (c == cy && tid == ty) {
#pragma unroll
            for (int u = 0; u < kVecPerThread; ++u)
              if (u == uy) zy = E::extract(d[u], ey);
            found = true;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&s_empty[stage]));  // stage may be refilled
          float x[kVecPerThread * EPV];
#pragma unroll
          for (int u = 0; u < kVecPerThread; ++u) E::unpack(d[u], x + u * EPV);
          const float bm = E::template batch_max<kVecPerThread>(d);
          if (bm > m) {
            const float sc = ex2((m - bm) * kLog2e);
            const uint64_t sc2 = f2_pack(sc, sc);
            acc01 = f2_mul(acc01, sc2);
            acc23 = f2_mul(acc23, sc2);
            s0 *= sc;  // holds the ragged elements, if any
            m = bm;
          }
          if (m != -INFINITY) {
            const float mL = m * kLog2e;
            const uint64_t nmL2 = f2_pack(-mL, -mL);
            // pairs: one packed FMA for two arguments, one packed add for
            // two sums; the fixed pairing keeps the summation order fixed
#pragma unroll
            for (int k = 0; k < kVecPerThread * EPV; k += 4) {
              acc01 = f2_add(acc01, f2_ex2(f2_fma(f2_pack(x[k + 0], x[k + 1]), L2, nmL2)));
              acc23 = f2_add(acc23, f2_ex2(f2_fma(f2_pack(x[k + 2], x[k + 3]), L2, nmL2)));
            }
          }
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      {
        // the ragged elements went into s0 (relative to the same running max)
        float a0, a1, a2, a3;
        f2_unpack(acc01, a0, a1);
        f2_unpack(acc23, a2, a3);
        s0 += a0;
        s1 += a1;
        s2 += a2;
        s3 += a3;
      }
      float s = (s0 + s1) + (s2 + s3);
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2b = __shfl_xor_sync(0xffffffffu, s, o);
        lse_merge(m, s, m2, s2b);
      }
      const int rb = (int)(it & 1);
      if (lane == 0) s_red[rb][warp] = make_float2(m, s);
      if (found) {
        s_zy[slot] = zy;
        s_found[slot] = r;
      }
      bar_sync_named(kConsumers);
      if (tid == 0) {
        float cm = s_red[rb][0].x, cs = s_red[rb][0].y;
#pragma unroll
        for (int k = 1; k < kWarps; ++k) lse_merge(cm, cs, s_red[rb][k].x, s_red[rb][k].y);
        const bool has = s_found[slot] == r;
        const float4 part = make_float4(cm, cs, has ? s_zy[slot] : 0.f, has ? 1.f : 0.f);
        if (K > 1) {
          st_cluster_f32x4(map_to_rank(smem_u32(&s_part[slot][rank]), 0), part);
          fence_cluster();  // the only store another CTA reads; see cluster_arrive_relaxed
        } else {
          s_part[slot][0] = part;
        }
      }
    }
    __syncwarp();  // the cluster barrier instructions are warp-aligned
    if (K > 1) {
      if (it > 0) {
        cluster_wait();  // row it-1: every CTA's partial has landed in CTA 0
        if (rank == 0 && tid == 0) finalize_row<K>(p, s_part[(it - 1) % 3], prev_i, prev_t);
      }
      cluster_arrive_relaxed();
    } else if (tid == 0) {
      finalize_row<K>(p, s_part[slot], i, t);
    }
    prev_i = i;
    prev_t = t;
  }
  __syncwarp();
  if (K > 1 && it > 0) {
    cluster_wait();
    if (rank == 0 && tid == 0) finalize_row<K>(p, s_part[(it - 1) % 3], prev_i, prev_t);
  }
  // after the rows, where little state is live (keeps the row loop's
  // register count)
  if (p.zero_past) {  // positions past each length: 0
    const int64_t nct = (int64_t)gridDim.x * kLseThreads;
    for (int64_t k = (int64_t)blockIdx.x * kLseThreads + tid; k < p.N * p.C; k += nct) {
      const int64_t i = k / p.C;
      if (k - i * p.C >= off[i + 1] - off[i]) {
        p.logp[k] = 0.f;
        p.lse[k] = 0.f;
      }
    }
  }
  // copies this CTA issued that no consumer waited for (only after a timeout)
  if (producer && lane == 0 && *(volatile int*)&s_abort) {
    for (uint32_t k = 0; k < kStages && k < issued; ++k) {
      const uint32_t n = issued - 1 - k;  // copy number n used stage n % kStages
      mbar_wait(smem_u32(&s_full[n % kStages]), (n / kStages) & 1u);
    }
  }
  // the grid completes only after prep has (the kernels after this one read
  // prep's table through this kernel's completion)
  if (tid == 0) pdl_wait();
}

// ---------------------------------------------------------------------------
// launch
// ---------------------------------------------------------------------------

namespace {

std::mutex g_occ_mutex;
std::map<std::tuple<int, int, int, int>, int> g_occ;  // (device, dtype, K, smem) -> clusters

template <typename T, int K>
cudaError_t launch_k(const FwdArgs& a, const DeviceInfo& d, cudaStream_t st, bool after_prep) {
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
  // no gradient weights requested: the log-probs-only call
  p.zero_past = a.w == nullptr;
  p.early = after_prep && a.N + 1 <= kSmemOffsets;
  p.len = a.len;

  const size_t smem = (size_t)kStages * kStageBytes +
                      (a.N + 1 <= kSmemOffsets ? sizeof(int32_t) * (size_t)(a.N + 1) : 0);
  auto kern = lse_gather_kernel<T, K>;
  {
    const int max_smem = kStages * kStageBytes + (int)sizeof(int32_t) * kSmemOffsets;
    cudaError_t e = ensure_dynamic_smem((const void*)kern, max_smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = K;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kLseThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = K > 1 ? 1 : 0;  // the occupancy query takes the cluster only

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
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kLseThreads, smem);
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
  if (K > 1) {
    cfg.numAttrs = 2;
  } else {
    attr[0] = attr[1];
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename T>
cudaError_t launch_t(const FwdArgs& a, const DeviceInfo& d, cudaStream_t st, bool after_prep) {
  switch (lse_split(a.V * (int64_t)sizeof(T), a.N * a.C, d.sms, "GRPO_LSE_CLUSTER")) {
    case 8:
      return launch_k<T, 8>(a, d, st, after_prep);
    case 4:
      return launch_k<T, 4>(a, d, st, after_prep);
    case 2:
      return launch_k<T, 2>(a, d, st, after_prep);
    default:
      return launch_k<T, 1>(a, d, st, after_prep);
  }
}

}  // namespace

cudaError_t launch_lse_gather(const FwdArgs& a, const DeviceInfo& d, cudaStream_t st,
                              bool after_prep) {
  if (a.N == 0 || a.C == 0) return cudaSuccess;
  return a.dtype == 0 ? launch_t<float>(a, d, st, after_prep)
                      : launch_t<uint16_t>(a, d, st, after_prep);
}

}  // namespace grpo

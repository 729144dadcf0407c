// Fused forward + backward over the scored rows: one HBM read of each scored
// row instead of two (the unfused forward reads it for the log-sum-exp and the
// backward reads it again for the softmax).
//
// The loss depends on a scored row only through its token's log-prob, and the
// row's gradient g*w_t*(onehot - softmax) needs only that token's (lse_t, w_t),
// which are known as soon as the row's log-sum-exp is: so a row can be read,
// reduced, and written back as gradient before moving on ("compute_logprobs",
// "The loss" and "loss.backward()" of "Making Dr GRPO go brrr",
// salahadawi.com, composed for one row at a time).
//
// Work layout: the forward's persistent grid, rows split over clusters of K
// CTAs as lse_split decides for the forward (K = 1, whole rows per CTA, unless
// the batch is small), and its bulk-copy ring.  For each row a CTA streams its
// row (slice) twice through the ring: pass 1 from HBM (normal L2 priority)
// for (max, sum, target logit); with K > 1 the partials are
// exchanged all-to-all through distributed shared memory and a cluster
// barrier, so every CTA merges them in rank order into the same lse and w;
// pass 2 writes the gradient, reading the row's first chunks from the
// shared-memory slots pass 1 loaded them into, and the rest from L2 where it
// is still there (whole rows keep ~90 MB live over the grid, so part of it
// comes from HBM again), last chunk first (the most recently loaded lines are
// the likeliest to be in L2).  Rows that score nothing are written with
// zeros by a separate store-only kernel launched after this one, which does
// not wait on it: its CTAs take the SM slots this persistent grid's CTAs free
// as they finish (with the head slots two CTAs fill an SM's shared memory;
// the host-memory variant holds none, and there they also run beside it).
// Per element the arithmetic is that of lse_gather_kernel and dlogits_kernel,
// and the per-token terms are token_terms(), so logp, lse, w and dlogits have
// the same bits as the unfused path; only the loss's summation order differs
// (per cluster, then clusters in order).
#include <stdlib.h>

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "host_ctx.cuh"
#include "host_rows.cuh"

namespace grpo {
namespace {

// A 4-stage ring and 3 head slots (7 x 16 KiB, two CTAs per SM): measured
// against 3 + 4, 2 + 5, 5 + 2 and 6 + 1 at the long-completion workload
// (10.28 ms against 10.31, 10.76, 10.39 and 10.57) and at 6,043 scored rows
// (0.857 ms against 0.863, 0.889, 0.866 and 0.874).
constexpr int kStages = 4;
constexpr int kStageBytes = 16384;
constexpr int kConsumers = kThreads;
constexpr int kFusedThreads = kConsumers + 32;
constexpr int kVecPerStage = kStageBytes / 16;
constexpr int kVecPerThread = kVecPerStage / kConsumers;
constexpr int kSmemOffsets = 4096;
// Chunks at the head of each row (slice) that pass 1 loads into slots of
// their own and pass 2 reads from there, not from L2: with whole rows per CTA
// the head of a row is the part likeliest to have left L2 by pass 2.  As many
// slots as leave two CTAs per SM beside the ring and the offsets table
// (keep_slots): three up to 191 completions, two above that, three again
// from 4,096 (the offsets table then stays in global memory).
constexpr int kKeepMax = 3;

template <typename T>
struct FusedParams {
  const T* logits;   // kHost: the device mapping of page-locked host logits
  T* staging;        // kHost: device buffer of the logits' shape (scored rows written)
  T* dlogits;
  int64_t T_len, P, C, V, N;
  const int64_t* ids;
  const int32_t* offsets;  // [N+1] prefix sums of the clamped lengths
  const float* adv;
  const float* old_logp;
  const float* ref_logp;
  const float* grad;       // device scalar or nullptr (1)
  float eps, beta;
  int agg;
  double norm;
  float* logp;
  float* lse;
  float* w;
  float* loss;
  WsHeader* hdr;
  double* partials;        // one per cluster
  int64_t chunk;
  int nkeep;               // head chunks held in shared memory (0 .. kKeepMax; 0 with kHost)
};

__device__ __forceinline__ int locate_row(const int32_t* off, int64_t N, int64_t r) {
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

// Pass 1's copies take normal L2 priority: measured against evict-last at the
// long-completion workload, evict-last lines that pass 2 has already read
// stay behind and crowd out newer ones (pass 2 re-read 5.6 GB from DRAM per
// launch with evict-last, 4.5 GB with normal priority; the call 10.35 ->
// 10.32 ms, and 0.1-0.4% faster on the smaller workloads).
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s_hint(uint32_t smem_dst, const void* gsrc, uint32_t bytes,
                                              uint32_t mbar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_dst),
      "l"(gsrc), "r"(bytes), "r"(mbar), "l"(pol)
      : "memory");
}

// kHost: the logits are in page-locked host memory.  Pass 1 then reads each
// scored row through the device mapping with plain 16-byte loads (consumers
// keep a stage's kVecPerThread loads in flight; the many CTAs fill the host
// link) and writes what it read to the same row of `staging`; pass 2 reads
// those vectors back, each thread the ones it wrote.  Element order, per-
// thread batching and arithmetic are those of the ring path, so every result
// has the same bits as with the logits in device memory; the producer warp
// only takes part in the cluster barriers.
template <typename T, int K, bool kHost>
__global__ void __launch_bounds__(kFusedThreads, 2) lse_grad_kernel(const FusedParams<T> p) {
  using E = Elt<T>;
  constexpr int EPV = E::kPerVec;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t s_full[kStages];
  __shared__ __align__(8) uint64_t s_empty[kStages];
  __shared__ __align__(8) uint64_t s_kfull[kKeepMax];   // head slot loaded
  __shared__ __align__(8) uint64_t s_kempty[kKeepMax];  // head slot read by pass 2
  __shared__ float4 s_part[2][K];  // every CTA: the K partials of a row
  __shared__ float2 s_red[kWarps];
  __shared__ float s_zy;
  __shared__ int64_t s_found;
  __shared__ float s_row[3];  // lse, -g*w/norm, has target (broadcast to consumers)
  __shared__ int s_abort;
  __shared__ bool s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool producer = warp == kWarps;
  const uint32_t rank = K > 1 ? cluster_ctarank() : 0u;
  const int64_t q = K > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
  const int64_t nq = K > 1 ? (int64_t)nclusters_x() : (int64_t)gridDim.x;
  const uint32_t ring = smem_u32(smem);

  if (tid == 0) {
    s_abort = 0;
    s_found = -1;
    for (int k = 0; k < kStages; ++k) {
      mbar_init(smem_u32(&s_full[k]), 1);
      mbar_init(smem_u32(&s_empty[k]), kWarps);
    }
    for (int k = 0; k < kKeepMax; ++k) {
      mbar_init(smem_u32(&s_kfull[k]), 1);
      mbar_init(smem_u32(&s_kempty[k]), kWarps);
    }
    mbar_init_fence();
  }
  pdl_wait();
  pdl_trigger();
  const uint32_t keep = ring + kStages * kStageBytes;  // head slots
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + (kStages + p.nkeep) * kStageBytes);
  const int32_t* off = p.offsets;
  if (p.N + 1 <= kSmemOffsets) {
    for (int64_t k = tid; k <= p.N; k += kFusedThreads) s_off[k] = p.offsets[k];
    off = s_off;
  }
  if (K > 1)
    cluster_sync();
  else
    __syncthreads();

  const float g = p.grad != nullptr ? __ldg(p.grad) : 1.f;
  const int64_t tv = off[p.N];
  const int64_t v0 = (int64_t)rank * p.chunk;
  const int64_t v1 = min(p.V, v0 + p.chunk);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0;
  // bit k: parity of head slot k's current use (flipped once per row that uses it)
  uint32_t kph = 0, kused = 0;
  double loss_acc = 0.0;  // rank 0, thread 0: sum of this cluster's ell
  const uint64_t pol_keep = l2_policy_evict_normal();
  const uint64_t pol_drop = l2_policy_evict_first();

  int64_t i_nx = 0, t_nx = 0, y_nx = 0;
  if (q < tv) {
    i_nx = locate_row(off, p.N, q);
    t_nx = q - off[i_nx];
    if (!producer) y_nx = __ldg(p.ids + i_nx * p.T_len + p.P + t_nx);
  }
  int64_t it = 0;
  for (int64_t r = q; r < tv; r += nq, ++it) {
    const int slot = (int)(it & 1);
    const int64_t i = i_nx, t = t_nx, y = y_nx;
    if (r + nq < tv) {
      i_nx = locate_row(off, p.N, r + nq);
      t_nx = r + nq - off[i_nx];
      if (!producer) y_nx = __ldg(p.ids + i_nx * p.T_len + p.P + t_nx);
    }
    const int64_t row_index = i * p.T_len + (p.P - 1 + t);
    const T* row = p.logits + row_index * p.V;
    T* orow = p.dlogits + row_index * p.V;
    T* srow = kHost ? p.staging + row_index * p.V : nullptr;
    int64_t a, b, nvec;
    if (v0 >= v1) {
      a = b = v0;
      nvec = 0;
    } else {
      const uintptr_t addr = reinterpret_cast<uintptr_t>(row + v0);
      const int64_t skip = (int64_t)(((16u - (unsigned)(addr & 15u)) & 15u) / sizeof(T));
      a = min(v0 + skip, v1);
      nvec = (v1 - a) / EPV;
      b = a + nvec * EPV;
    }
    const uint32_t bytes = (uint32_t)(nvec * 16);
    const int nchunks = (int)((bytes + kStageBytes - 1) / kStageBytes);
    const int nk = min(p.nkeep, nchunks);  // head chunks: slots, not the ring
    const uint32_t kmask = (1u << nk) - 1u;

    if (producer && kHost) {  // one arrival per row, as the consumers'
      if (K > 1) {
        cluster_arrive_relaxed();
        cluster_wait();
      }
      continue;
    }
    if (producer) {
      const char* src = reinterpret_cast<const char*>(row + a);
      for (int pass = 0; pass < 2; ++pass) {
        if (lane == 0) {
          for (int c = 0; c < nchunks; ++c) {
            if (*(volatile int*)&s_abort) break;
            if (c < nk) {  // a head chunk: its own slot in pass 1, nothing in pass 2
              if (pass == 1) continue;
              if (!mbar_wait(smem_u32(&s_kempty[c]), ((kph >> c) & 1u) ^ 1u)) {
                atomicOr(&p.hdr->flags, kFlagTimeout);
                *(volatile int*)&s_abort = 1;
                break;
              }
              const uint32_t nb = min((uint32_t)kStageBytes, bytes - (uint32_t)c * kStageBytes);
              const uint32_t full = smem_u32(&s_kfull[c]);
              mbar_arrive_expect_tx(full, nb);
              bulk_g2s_hint(keep + c * kStageBytes, src + (size_t)c * kStageBytes, nb, full,
                            pol_drop);
              kph ^= 1u << c;
              kused |= 1u << c;
              continue;
            }
            if (!mbar_wait(smem_u32(&s_empty[stage]), phase ^ 1u)) {
              atomicOr(&p.hdr->flags, kFlagTimeout);
              *(volatile int*)&s_abort = 1;
              break;
            }
            const int cc = pass == 0 ? c : nchunks - 1 - (c - nk);
            const uint32_t nb = min((uint32_t)kStageBytes, bytes - (uint32_t)cc * kStageBytes);
            const uint32_t full = smem_u32(&s_full[stage]);
            mbar_arrive_expect_tx(full, nb);
            bulk_g2s_hint(ring + stage * kStageBytes, src + (size_t)cc * kStageBytes, nb, full,
                          pass == 0 ? pol_keep : pol_drop);
            ++issued;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        __syncwarp();
        // arrive after pass 1 (the consumers need every CTA's arrival to
        // start pass 2, and pass 2's copies may wait on them); wait after
        // pass 2, before the next row's arrive
        if (K > 1) {
          if (pass == 0)
            cluster_arrive_relaxed();
          else
            cluster_wait();
        }
      }
      continue;
    }

    // ---------------- consumers: pass 1 (max, sum, target logit) --------
    float m = -INFINITY, s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    const uint64_t L2 = f2_pack(kLog2e, kLog2e);
    uint64_t acc01 = f2_pack(0.f, 0.f), acc23 = f2_pack(0.f, 0.f);
    float zy = 0.f;
    bool found = false;
    int64_t e = -1;  // this thread's ragged element (head or tail), if any
    if (tid < a - v0)
      e = v0 + tid;
    else if (tid >= 32 && tid - 32 < v1 - b)
      e = b + (tid - 32);
    float xe = 0.f;
    if (e >= 0) {
      xe = E::load1(row + e);
      if (kHost) E::store1(srow + e, xe);
      if (e == y) {
        zy = xe;
        found = true;
      }
      if (xe > m) m = xe;  // first value of this thread: no rescale needed
      if (m != -INFINITY) s0 += ex2(fmaf(xe, kLog2e, -m * kLog2e));
    }
    const int64_t ky = (y >= a && y < b) ? (y - a) / EPV : -1;
    const int ey = ky >= 0 ? (int)((y - a) % EPV) : 0;
    const int cy = ky >= 0 ? (int)(ky / kVecPerStage) : -1;
    const int kl = ky >= 0 ? (int)(ky % kVecPerStage) : 0;
    const int ty = kl % kConsumers, uy = kl / kConsumers;
    const uint4* hv = reinterpret_cast<const uint4*>(row + a);  // kHost: the host row
    uint4* sv = kHost ? reinterpret_cast<uint4*>(srow + a) : nullptr;
    for (int c = 0; c < nchunks; ++c) {
      const bool head = c < nk;
      bool ok = !*(volatile int*)&s_abort;
      if (!kHost && ok &&
          !mbar_wait(head ? smem_u32(&s_kfull[c]) : smem_u32(&s_full[stage]),
                     head ? (kph >> c) & 1u : phase)) {
        atomicOr(&p.hdr->flags, kFlagTimeout);
        *(volatile int*)&s_abort = 1;
        ok = false;
      }
      if (ok) {
        const int nv = (int)min((int64_t)kVecPerStage, nvec - (int64_t)c * kVecPerStage);
        const uint32_t sbase = head ? keep + c * kStageBytes : ring + stage * kStageBytes;
        uint4 d[kVecPerThread];
        if constexpr (kHost) {
          const int64_t base = (int64_t)c * kVecPerStage;
#pragma unroll
          for (int u = 0; u < kVecPerThread; ++u) {
            const int k = tid + u * kConsumers;
            d[u] = k < nv ? ld_stream(hv + base + k)
                          : make_uint4(E::kNegInf, E::kNegInf, E::kNegInf, E::kNegInf);
          }
#pragma unroll
          for (int u = 0; u < kVecPerThread; ++u) {
            const int k = tid + u * kConsumers;
            if (k < nv) sv[base + k] = d[u];  // stays in L2 for pass 2
          }
        } else {
#pragma unroll
          for (int u = 0; u < kVecPerThread; ++u) {
            const int k = tid + u * kConsumers;
            d[u] = k < nv ? ld_shared_v4(sbase + 16u * k)
                          : make_uint4(E::kNegInf, E::kNegInf, E::kNegInf, E::kNegInf);
          }
        }
        if (c == cy && tid == ty) {
#pragma unroll
          for (int u = 0; u < kVecPerThread; ++u)
            if (u == uy) zy = E::extract(d[u], ey);
          found = true;
        }
        if (!kHost && !head) {  // head slots stay until pass 2
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&s_empty[stage]));
        }
        float x[kVecPerThread * EPV];
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) E::unpack(d[u], x + u * EPV);
        const float bm = E::template batch_max<kVecPerThread>(d);
        if (bm > m) {
          const float sc = ex2((m - bm) * kLog2e);
          const uint64_t sc2 = f2_pack(sc, sc);
          acc01 = f2_mul(acc01, sc2);
          acc23 = f2_mul(acc23, sc2);
          s0 *= sc;
          m = bm;
        }
        if (m != -INFINITY) {
          const float mL = m * kLog2e;
          const uint64_t nmL2 = f2_pack(-mL, -mL);
#pragma unroll
          for (int k = 0; k < kVecPerThread * EPV; k += 4) {
            acc01 = f2_add(acc01, f2_ex2(f2_fma(f2_pack(x[k + 0], x[k + 1]), L2, nmL2)));
            acc23 = f2_add(acc23, f2_ex2(f2_fma(f2_pack(x[k + 2], x[k + 3]), L2, nmL2)));
          }
        }
      }
      if (!head && ++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    {
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
    if (lane == 0) s_red[warp] = make_float2(m, s);
    if (found) {
      s_zy = zy;
      s_found = r;
    }
    bar_sync_named(kConsumers);
    if (tid == 0) {
      float cm = s_red[0].x, cs = s_red[0].y;
#pragma unroll
      for (int k = 1; k < kWarps; ++k) lse_merge(cm, cs, s_red[k].x, s_red[k].y);
      const bool has = s_found == r;
      const float4 part = make_float4(cm, cs, has ? s_zy : 0.f, has ? 1.f : 0.f);
      if (K > 1) {
        for (uint32_t k = 0; k < (uint32_t)K; ++k)  // every CTA gets every partial
          st_cluster_f32x4(map_to_rank(smem_u32(&s_part[slot][rank]), k), part);
        fence_cluster();
      } else {
        s_part[slot][0] = part;
      }
    }
    __syncwarp();
    if (K > 1) {
      cluster_arrive_relaxed();
      cluster_wait();
    }
    // ---------------- the row's lse, logp and per-token terms -----------
    if (tid == 0) {
      float4 pk = s_part[slot][0];
      float cm = pk.x, cs = pk.y, z = pk.z;
      bool has = pk.w != 0.f;
#pragma unroll
      for (int k = 1; k < K; ++k) {
        pk = s_part[slot][k];
        lse_merge(cm, cs, pk.x, pk.y);
        if (pk.w != 0.f) {
          z = pk.z;
          has = true;
        }
      }
      const float l = cm + logf(cs);
      const int64_t o = i * p.C + t;
      float lp, wv;
      if (has) {
        lp = z - l;
        const TokenTerms tt =
            token_terms(lp, p.adv[i], p.old_logp != nullptr,
                        p.old_logp != nullptr ? p.old_logp[o] : 0.f, p.beta,
                        p.beta != 0.f ? p.ref_logp[o] : 0.f, p.eps);
        const double len_i = (double)(off[i + 1] - off[i]);
        const double denom = p.agg == 0 ? p.norm : p.norm * len_i;
        wv = (float)((double)tt.w / denom);
        if (rank == 0) loss_acc += p.agg == 0 ? (double)tt.ell : (double)tt.ell / len_i;
      } else {  // y outside [0, V)
        lp = __int_as_float(0x7fc00000);
        wv = lp;
        if (rank == 0) {
          loss_acc += (double)lp;
          atomicOr(&p.hdr->flags, kFlagTokenRange);
        }
      }
      if (rank == 0) {
        p.logp[o] = lp;
        p.lse[o] = has ? l : lp;
        p.w[o] = wv;
      }
      s_row[0] = l;
      s_row[1] = -(g * wv);
    }
    bar_sync_named(kConsumers);
    const float lse_t = s_row[0];
    const float ngw = s_row[1];
    const float lseL = lse_t * kLog2e;

    // ---------------- consumers: pass 2 (the gradient) ------------------
    uint4* ovp = reinterpret_cast<uint4*>(orow + a);
    // the head chunks from their slots first (frees them for the next row's
    // copies), then the others from L2, most recently read in pass 1 first
    for (int c2 = 0; c2 < nchunks; ++c2) {
      const bool head = c2 < nk;
      const int c = head ? c2 : nchunks - 1 - (c2 - nk);
      bool ok = !*(volatile int*)&s_abort;
      if (!kHost && !head && ok && !mbar_wait(smem_u32(&s_full[stage]), phase)) {
        atomicOr(&p.hdr->flags, kFlagTimeout);
        *(volatile int*)&s_abort = 1;
        ok = false;
      }
      if (ok) {
        const int nv = (int)min((int64_t)kVecPerStage, nvec - (int64_t)c * kVecPerStage);
        const uint32_t sbase = head ? keep + c * kStageBytes : ring + stage * kStageBytes;
        uint4 d[kVecPerThread];
        if constexpr (kHost) {  // the vectors this thread wrote in pass 1
          const int64_t base = (int64_t)c * kVecPerStage;
#pragma unroll
          for (int u = 0; u < kVecPerThread; ++u) {
            const int k = tid + u * kConsumers;
            if (k < nv) d[u] = __ldcg(sv + base + k);
          }
        } else {
#pragma unroll
          for (int u = 0; u < kVecPerThread; ++u) {
            const int k = tid + u * kConsumers;
            if (k < nv) d[u] = ld_shared_v4(sbase + 16u * k);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(head ? smem_u32(&s_kempty[c]) : smem_u32(&s_empty[stage]));
        }
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
          const int k = tid + u * kConsumers;
          if (k >= nv) break;
          float xv[EPV], ov[EPV];
          E::unpack(d[u], xv);
#pragma unroll
          for (int q2 = 0; q2 < EPV; ++q2) ov[q2] = ngw * ex2(fmaf(xv[q2], kLog2e, -lseL));
          if (c == cy && tid == ty && u == uy) {
            // 1 - p_y without cancellation
#pragma unroll
            for (int q2 = 0; q2 < EPV; ++q2)
              if (q2 == ey) ov[q2] = ngw * expm1f(xv[q2] - lse_t);
          }
          st_stream(ovp + (int64_t)c * kVecPerStage + k, E::pack(ov));
        }
      }
      if (!head && ++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    kph ^= kmask;
    if (e >= 0) {
      const float ov = e == y ? ngw * expm1f(xe - lse_t) : ngw * ex2(fmaf(xe, kLog2e, -lseL));
      E::store1(orow + e, ov);
    }
  }

  // copies this CTA issued that no consumer waited for (only after a timeout)
  if (producer && lane == 0 && *(volatile int*)&s_abort) {
    for (uint32_t k = 0; k < kStages && k < issued; ++k) {
      const uint32_t n = issued - 1 - k;
      mbar_wait(smem_u32(&s_full[n % kStages]), (n / kStages) & 1u);
    }
    for (int k = 0; k < kKeepMax; ++k)  // the last copy into each head slot used
      if ((kused >> k) & 1u) mbar_wait(smem_u32(&s_kfull[k]), ((kph >> k) & 1u) ^ 1u);
  }
  // the loss: each cluster's sum, then the last cluster adds them in order
  if (rank == 0 && tid == 0) {
    p.partials[q] = loss_acc;
    __threadfence();
    const unsigned ticket = atomicAdd(&p.hdr->ticket, 1u);
    s_last = ticket == (unsigned)nq - 1;
  }
  __syncthreads();
  if (rank == 0 && s_last && tid == 0) {
    __threadfence();
    double tot = 0.0;
    for (int64_t k = 0; k < nq; ++k) tot += reinterpret_cast<volatile double*>(p.partials)[k];
    *p.loss = (float)(tot / p.norm);
    p.hdr->ticket = 0;
  }
}

std::mutex g_occ_mutex;
std::map<std::tuple<int, int, int, int>, int> g_occ;

// Head slots per CTA: as many as fit beside the ring and the offsets table
// (offs bytes) with two CTAs per SM (half the SM's shared memory, less the
// per-block reservation and the kernel's static arrays), at most kKeepMax,
// and at most GRPO_FUSED_KEEP when that is set.
template <typename T, int K>
cudaError_t keep_slots(int device, size_t offs, int* n) {
  static std::map<int, long> avail;  // per device: dynamic bytes per CTA at two CTAs per SM
  static const int cap = [] {
    const char* v = getenv("GRPO_FUSED_KEEP");
    if (v == nullptr || *v == 0) return kKeepMax;
    const int k = atoi(v);
    return k < 0 ? 0 : (k > kKeepMax ? kKeepMax : k);
  }();
  long bytes = -1;
  {
    std::lock_guard<std::mutex> lk(g_occ_mutex);
    auto it = avail.find(device);
    if (it != avail.end()) bytes = it->second;
  }
  if (bytes < 0) {
    int per_sm = 0, reserved = 0;
    cudaError_t e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                           device);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, device);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, lse_grad_kernel<T, K, false>);
    if (e != cudaSuccess) return e;
    bytes = (long)per_sm / 2 - reserved - (long)fa.sharedSizeBytes;
    std::lock_guard<std::mutex> lk(g_occ_mutex);
    avail[device] = bytes;
  }
  long k = (bytes - (long)kStages * kStageBytes - (long)offs) / kStageBytes;
  if (k < 0) k = 0;
  if (k > cap) k = cap;
  *n = (int)k;
  return cudaSuccess;
}

// staging != nullptr: a.logits is the device mapping of host logits (kHost).
template <typename T, int K>
cudaError_t launch_k(const FwdArgs& a, const BwdArgs& bw, const DeviceInfo& d, cudaStream_t st,
                     void* staging) {
  constexpr int EPV = Elt<T>::kPerVec;
  const WsLayout l = ws_layout(a.N);
  char* ws = static_cast<char*>(a.ws);
  FusedParams<T> p;
  p.logits = static_cast<const T*>(a.logits);
  p.staging = static_cast<T*>(staging);
  p.dlogits = static_cast<T*>(bw.dlogits);
  p.T_len = a.P + a.C;
  p.P = a.P;
  p.C = a.C;
  p.V = a.V;
  p.N = a.N;
  p.ids = a.ids;
  p.offsets = reinterpret_cast<const int32_t*>(ws + l.offsets);
  p.adv = a.adv;
  p.old_logp = a.old_logp;
  p.ref_logp = a.ref_logp;
  p.grad = bw.grad;
  p.eps = a.eps;
  p.beta = a.beta;
  p.agg = a.agg;
  p.norm = default_norm(a);
  p.logp = a.logp;
  p.lse = a.lse;
  p.w = a.w;
  p.loss = a.loss;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.partials = reinterpret_cast<double*>(ws + l.partials);
  p.chunk = ((a.V + K - 1) / K + EPV - 1) / EPV * EPV;
  const size_t offs = a.N + 1 <= kSmemOffsets ? sizeof(int32_t) * (size_t)(a.N + 1) : 0;
  int nkeep = 0;
  if (cudaError_t e = keep_slots<T, K>(d.device, offs, &nkeep); e != cudaSuccess) return e;
  p.nkeep = staging != nullptr ? 0 : nkeep;

  const size_t smem_dev = (size_t)(kStages + nkeep) * kStageBytes + offs;
  const size_t smem = (size_t)(kStages + p.nkeep) * kStageBytes + offs;
  // the grid (and so the loss's summation order) is that of the device-memory
  // kernel in both modes
  auto kern = lse_grad_kernel<T, K, false>;
  auto kern_launch = staging != nullptr ? lse_grad_kernel<T, K, true> : kern;
  {
    const int max_smem =
        (kStages + kKeepMax) * kStageBytes + (int)sizeof(int32_t) * kSmemOffsets;
    cudaError_t e = ensure_dynamic_smem((const void*)kern, max_smem);
    if (e == cudaSuccess) e = ensure_dynamic_smem((const void*)kern_launch, max_smem);
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
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = smem_dev;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = K > 1 ? 1 : 0;
  int clusters = 0;
  const auto key = std::make_tuple(d.device, (int)sizeof(T), K, (int)smem_dev);
  {
    std::lock_guard<std::mutex> lk(g_occ_mutex);
    auto itc = g_occ.find(key);
    if (itc != g_occ.end()) clusters = itc->second;
  }
  if (clusters == 0) {
    cudaError_t e;
    if (K > 1) {
      cfg.gridDim = dim3(K);
      e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    } else {
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFusedThreads, smem_dev);
      clusters = per_sm * d.sms;
    }
    if (e != cudaSuccess) return e;
    if (clusters < 1) clusters = 1;
    if (clusters > kMaxLossBlocks) clusters = kMaxLossBlocks;  // one loss partial each
    std::lock_guard<std::mutex> lk(g_occ_mutex);
    g_occ[key] = clusters;
  }
  const int64_t max_rows = a.N * a.C;
  const int64_t nq = clusters < max_rows ? clusters : max_rows;
  cfg.gridDim = dim3((unsigned)(nq * K));
  cfg.dynamicSmemBytes = smem;
  if (K > 1) {
    cfg.numAttrs = 2;
  } else {
    attr[0] = attr[1];
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern_launch, p);
}

template <typename T>
cudaError_t launch_t(const FwdArgs& a, const BwdArgs& b, const DeviceInfo& d, cudaStream_t st,
                     void* staging) {
  switch (lse_split(a.V * (int64_t)sizeof(T), a.N * a.C, d.sms, "GRPO_FUSED_CLUSTER")) {
    case 8:
      return launch_k<T, 8>(a, b, d, st, staging);
    case 4:
      return launch_k<T, 4>(a, b, d, st, staging);
    case 2:
      return launch_k<T, 2>(a, b, d, st, staging);
    default:
      return launch_k<T, 1>(a, b, d, st, staging);
  }
}

}  // namespace

cudaError_t launch_lse_grad(const FwdArgs& a, const BwdArgs& b, const DeviceInfo& d,
                            cudaStream_t st) {
  if (a.N == 0 || a.C == 0) return cudaSuccess;
  return a.dtype == 0 ? launch_t<float>(a, b, d, st, nullptr)
                      : launch_t<uint16_t>(a, b, d, st, nullptr);
}

cudaError_t launch_lse_grad_host(const FwdArgs& a, const BwdArgs& b, void* staging,
                                 const DeviceInfo& d, cudaStream_t st) {
  if (a.N == 0 || a.C == 0) return cudaSuccess;
  return a.dtype == 0 ? launch_t<float>(a, b, d, st, staging)
                      : launch_t<uint16_t>(a, b, d, st, staging);
}

}  // namespace grpo

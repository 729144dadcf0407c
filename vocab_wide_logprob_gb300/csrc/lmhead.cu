// Log-probs of the sampled tokens straight from the policy's last hidden
// states: the LM-head projection logits = H * W^T ("model(...).logits" of
// "compute_logprobs" in "Making Dr GRPO go brrr", salahadawi.com) fused with
// the shifted log-softmax and gather, so the [rows, V] logits never reach
// HBM.  This is a dense contraction, so it runs on the 5th-generation tensor
// cores: tcgen05.mma with operands staged in shared memory by TMA and the
// fp32 accumulator in tensor memory (TMEM).
//
// Pipeline (one CTA per SM, persistent):
//   gather_rows_kernel   copies the hidden state of every scored row into a
//                        dense [rows, d] buffer (row r = valid token r)
//   lmhead_lse_kernel    work items (block of 128 rows, range of vocabulary
//                        tiles of 256).  Warp 0 issues TMA loads of a 128x64
//                        slab of H and a 256x64 slab of W per k-step into a
//                        4-stage ring (128-byte swizzle); warp 1 issues
//                        tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32) into
//                        one of two TMEM accumulators; warps 2-5 read the
//                        finished 128x256 tile from TMEM (one row per thread)
//                        and fold it into a running (max, sum of exp) and the
//                        target logit, while the MMAs fill the other buffer.
//                        Each item writes one partial per row.
//   lmhead_merge_kernel  merges a row's partials in order (deterministic) into
//                        lse and logp = z_y - lse, and zeroes positions past
//                        each length.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace grpo {
namespace {

constexpr int kBM = 128;          // rows per tile (TMEM lanes)
constexpr int kBN = 256;          // vocabulary columns per tile
constexpr int kBK = 64;           // k per stage: one 128-byte swizzle atom of bf16
constexpr int kLmStages = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KiB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KiB
constexpr int kStageBytesLm = kABytes + kBBytes;
constexpr int kLmThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kMaxSplits = 256;  // = kThreads: one candidate per thread

struct LmParams {
  int64_t N, P, C, V, d;
  const int32_t* offsets;  // prefix sums of the clamped lengths ([N+1])
  int4* geometry;          // (row blocks, splits, tiles per split): written by the gather
  float4* partials;        // [items][kBM] (max, sum, target logit, has target)
  WsHeader* hdr;
  int sms;                 // CTAs in the grid: the split count is chosen from it
};

// Row blocks and vocabulary splits for t_valid rows, computed once by the
// first CTA of gather_rows_kernel and read by the later kernels.  Candidate
// split counts s = 1 .. 256 (one per thread) are scored by how well their work
// items (row block, 1/s of the vocabulary tiles) fill the grid's rounds,
// counting both the items per round and the uneven last split of tiles; the
// smallest s within 0.01 of the best score wins (less merging, and every split
// re-reads its row block).  items = mb * s never exceeds 4 * sms + 2 * mb, the
// size of the partials buffer.
__device__ float lm_split_score(int32_t mb, int32_t sp, int32_t ntiles, int sms) {
  const int32_t items = mb * sp;
  if (sp > ntiles || items > 4 * sms + 2 * mb) return -1.f;
  const int32_t rounds = (items + sms - 1) / sms;
  const int32_t tps = (ntiles + sp - 1) / sp;
  return (float)items / (float)(rounds * sms) * (float)ntiles / (float)(tps * sp);
}

// Called by all kThreads (= kMaxSplits) threads of one CTA.
__device__ int4 lm_geometry_block(int64_t t_valid, int64_t V, int sms) {
  __shared__ float s_best[kWarps];
  __shared__ int s_pick[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t ntiles = (int32_t)((V + kBN - 1) / kBN);
  const int32_t mb = (int32_t)((t_valid + kBM - 1) / kBM);
  const int32_t sp = tid + 1;
  const float score = mb > 0 ? lm_split_score(mb, sp, ntiles, sms) : (sp == 1 ? 1.f : -1.f);
  float best = score;
  for (int o = 16; o > 0; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
  if (lane == 0) s_best[warp] = best;
  __syncthreads();
  best = s_best[0];
  for (int k = 1; k < kWarps; ++k) best = fmaxf(best, s_best[k]);
  int pick = (score >= 0.f && score >= best - 0.01f) ? sp : 1 << 30;
  for (int o = 16; o > 0; o >>= 1) pick = min(pick, __shfl_xor_sync(0xffffffffu, pick, o));
  if (lane == 0) s_pick[warp] = pick;
  __syncthreads();
  pick = s_pick[0];
  for (int k = 1; k < kWarps; ++k) pick = min(pick, s_pick[k]);
  if (pick > kMaxSplits) pick = 1;
  return make_int4(mb, pick, (ntiles + pick - 1) / pick, 0);
}

// ---- tensor memory and tcgen05 helpers ----------------------------------------

__device__ __forceinline__ uint64_t umma_sdesc(uint32_t saddr) {
  uint64_t dsc = 0;
  dsc |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
  dsc |= (uint64_t)1 << 16;                   // leading byte offset (unused: 128-byte swizzle)
  dsc |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 bytes
  dsc |= (uint64_t)1 << 46;                   // descriptor version
  dsc |= (uint64_t)2 << 61;                   // layout: 128-byte swizzle, K-major
  return dsc;
}

// D (f32) += A (bf16, K-major) * B (bf16, K-major)^T, M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t ad, uint64_t bd, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(ad), "l"(bd), "r"(kIdesc), "r"(acc)
      : "memory");
}
// Arrive on the mbarrier once every tcgen05 operation issued so far is done.
__device__ __forceinline__ void umma_commit(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
      : "memory");
}
__device__ __forceinline__ void tmem_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,"
      "%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tma_load_2d(uint32_t sdst, const CUtensorMap* map, int x, int y,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(sdst),
      "l"(map), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}

// ---- gather: dense [rows, d] copy of the scored rows' hidden states ----------

__global__ void __launch_bounds__(kThreads) gather_rows_kernel(const uint16_t* __restrict__ hidden,
                                                               uint16_t* __restrict__ dense,
                                                               const int32_t* __restrict__ off,
                                                               int64_t N, int64_t T, int64_t P,
                                                               int64_t d, int64_t V, int sms,
                                                               int4* __restrict__ geometry) {
  pdl_wait();
  pdl_trigger();
  const int64_t tv = off[N];
  if (blockIdx.x == 0) {
    const int4 g = lm_geometry_block(tv, V, sms);
    if (threadIdx.x == 0) *geometry = g;
  }
  const int64_t vec_per_row = d / 8;  // 16-byte vectors
  for (int64_t k = (int64_t)blockIdx.x * kThreads + threadIdx.x; k < tv * vec_per_row;
       k += (int64_t)gridDim.x * kThreads) {
    const int64_t r = k / vec_per_row, c = k - r * vec_per_row;
    int lo = 0, hi = (int)N;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (off[mid] <= r)
        lo = mid;
      else
        hi = mid;
    }
    const int64_t t = r - off[lo];
    const uint4* src = reinterpret_cast<const uint4*>(hidden + ((int64_t)lo * T + P - 1 + t) * d);
    reinterpret_cast<uint4*>(dense + r * d)[c] = ld_stream(src + c);
  }
}

// ---- the tensor-core kernel -----------------------------------------------------

__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_lse_kernel(const __grid_constant__ CUtensorMap map_h,
                      const __grid_constant__ CUtensorMap map_w, const int64_t* __restrict__ ids,
                      const LmParams p) {
  extern __shared__ __align__(1024) unsigned char lm_smem[];
  __shared__ __align__(8) uint64_t s_full[kLmStages];
  __shared__ __align__(8) uint64_t s_empty[kLmStages];
  __shared__ __align__(8) uint64_t s_acc_full[2];
  __shared__ __align__(8) uint64_t s_acc_empty[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* ring = lm_smem + ((1024 - (smem_u32(lm_smem) & 1023)) & 1023);
  const uint32_t ring_u32 = smem_u32(ring);

  if (tid == 0) {
    s_abort = 0;
    for (int k = 0; k < kLmStages; ++k) {
      mbar_init(smem_u32(&s_full[k]), 1);
      mbar_init(smem_u32(&s_empty[k]), 1);  // one tcgen05.commit per use
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&s_acc_full[k]), 1);   // tcgen05.commit after a tile's MMAs
      mbar_init(smem_u32(&s_acc_empty[k]), 4);  // one arrive per epilogue warp
    }
    mbar_init_fence();
  }
  if (warp == 1) {  // two 256-column fp32 accumulators: all 512 TMEM columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&s_tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait();
  pdl_trigger();

  const int64_t tv = p.offsets[p.N];
  const int4 geo = *p.geometry;
  const int64_t mb = geo.x, splits = geo.y, tps = geo.z;
  const int64_t ntiles = (p.V + kBN - 1) / kBN;
  const int64_t items = mb * splits;
  const int kblocks = (int)(p.d / kBK);

  if (warp == 0) {
    // ---------------- TMA producer -----------------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int64_t it = blockIdx.x; it < items && !*(volatile int*)&s_abort; it += gridDim.x) {
        const int64_t rb = it / splits, sp = it - rb * splits;
        const int64_t n0 = sp * tps, n1 = min(ntiles, n0 + tps);
        for (int64_t n = n0; n < n1; ++n) {
          for (int kb = 0; kb < kblocks; ++kb) {
            if (!mbar_wait(smem_u32(&s_empty[stage]), phase ^ 1u)) {
              atomicOr(&p.hdr->flags, kFlagTimeout);
              *(volatile int*)&s_abort = 1;
              break;
            }
            const uint32_t full = smem_u32(&s_full[stage]);
            const uint32_t sa = ring_u32 + stage * kStageBytesLm;
            mbar_arrive_expect_tx(full, kStageBytesLm);
            tma_load_2d(sa, &map_h, kb * kBK, (int)(rb * kBM), full);
            tma_load_2d(sa + kABytes, &map_w, kb * kBK, (int)(n * kBN), full);
            if (++stage == kLmStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (*(volatile int*)&s_abort) break;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ---------------------------------------------
    if (lane == 0) {
      int stage = 0, buf = 0;
      uint32_t phase = 0, aphase = 0;
      for (int64_t it = blockIdx.x; it < items && !*(volatile int*)&s_abort; it += gridDim.x) {
        const int64_t rb = it / splits, sp = it - rb * splits;
        const int64_t n0 = sp * tps, n1 = min(ntiles, n0 + tps);
        (void)rb;
        for (int64_t n = n0; n < n1; ++n) {
          // the epilogue has drained this accumulator
          if (!mbar_wait(smem_u32(&s_acc_empty[buf]), aphase ^ 1u)) {
            atomicOr(&p.hdr->flags, kFlagTimeout);
            *(volatile int*)&s_abort = 1;
            break;
          }
          tmem_fence_after();
          const uint32_t dacc = tmem + (uint32_t)(buf * kBN);
          bool ok = true;
          for (int kb = 0; kb < kblocks; ++kb) {
            if (!mbar_wait(smem_u32(&s_full[stage]), phase)) {
              atomicOr(&p.hdr->flags, kFlagTimeout);
              *(volatile int*)&s_abort = 1;
              ok = false;
              break;
            }
            tmem_fence_after();
            const uint32_t sa = ring_u32 + stage * kStageBytesLm;
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j)
              umma(dacc, umma_sdesc(sa + j * 32), umma_sdesc(sa + kABytes + j * 32),
                   (kb | j) ? 1u : 0u);
            umma_commit(smem_u32(&s_empty[stage]));  // the stage is free once these finish
            if (++stage == kLmStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit(smem_u32(&s_acc_full[buf]));  // the tile is complete in TMEM
          if (++buf == 2) {
            buf = 0;
            aphase ^= 1u;
          }
        }
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5, one accumulator row per thread ----
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 of this warp
    const int row_in_block = quarter * 32 + lane;
    int buf = 0;
    uint32_t aphase = 0;
    const uint64_t L2 = f2_pack(kLog2e, kLog2e);
    for (int64_t it = blockIdx.x; it < items && !*(volatile int*)&s_abort; it += gridDim.x) {
      const int64_t rb = it / splits, sp = it - rb * splits;
      const int64_t n0 = sp * tps, n1 = min(ntiles, n0 + tps);
      const int64_t r = rb * kBM + row_in_block;  // valid token of this thread
      int64_t y = -1;
      if (r < tv) {
        int lo = 0, hi = (int)p.N;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (p.offsets[mid] <= r)
            lo = mid;
          else
            hi = mid;
        }
        y = __ldg(ids + (int64_t)lo * (p.P + p.C) + p.P + (r - p.offsets[lo]));
      }
      float m = -INFINITY, s_extra = 0.f, zy = 0.f;
      uint64_t acc01 = f2_pack(0.f, 0.f), acc23 = f2_pack(0.f, 0.f);
      bool has = false;
      bool ok = true;
      for (int64_t n = n0; n < n1; ++n) {
        if (!mbar_wait(smem_u32(&s_acc_full[buf]), aphase)) {
          atomicOr(&p.hdr->flags, kFlagTimeout);
          *(volatile int*)&s_abort = 1;
          ok = false;
          break;
        }
        tmem_fence_after();
        const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * kBN);
        const int64_t vbase = n * kBN;
#pragma unroll 1
        for (int c = 0; c < kBN; c += 32) {
          float v[32];
          tmem_ld32(tbase + (uint32_t)c, v);
          const int64_t v0 = vbase + c;
          if (v0 + 32 > p.V) {  // the vocabulary's last tile: columns past V do not exist
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (v0 + j >= p.V) v[j] = -INFINITY;
          }
          if (y >= v0 && y < v0 + 32) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (v0 + j == y) zy = v[j];
            has = true;
          }
          float bm = v[0];
#pragma unroll
          for (int j = 1; j < 32; ++j) bm = fmaxf(bm, v[j]);
          if (bm > m) {
            const float sc = ex2((m - bm) * kLog2e);
            const uint64_t sc2 = f2_pack(sc, sc);
            acc01 = f2_mul(acc01, sc2);
            acc23 = f2_mul(acc23, sc2);
            s_extra *= sc;
            m = bm;
          }
          if (m != -INFINITY) {
            const float mL = m * kLog2e;
            const uint64_t nmL2 = f2_pack(-mL, -mL);
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              acc01 = f2_add(acc01, f2_ex2(f2_fma(f2_pack(v[j], v[j + 1]), L2, nmL2)));
              acc23 = f2_add(acc23, f2_ex2(f2_fma(f2_pack(v[j + 2], v[j + 3]), L2, nmL2)));
            }
          }
        }
        tmem_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s_acc_empty[buf]));  // accumulator may be reused
        if (++buf == 2) {
          buf = 0;
          aphase ^= 1u;
        }
      }
      if (!ok) break;
      float a0, a1, a2, a3;
      f2_unpack(acc01, a0, a1);
      f2_unpack(acc23, a2, a3);
      const float s = ((a0 + a1) + (a2 + a3)) + s_extra;
      if (r < tv) p.partials[it * kBM + row_in_block] = make_float4(m, s, zy, has ? 1.f : 0.f);
    }
  }

  // release tensor memory: every MMA this CTA issued has completed once the
  // epilogue consumed its tile (or, after a timeout, once the last commit lands)
  tmem_fence_before();
  __syncthreads();
  if (warp == 1) {
    tmem_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

// ---- merge: partials of a row in split order -> lse, logp ----------------------

__global__ void __launch_bounds__(kThreads) lmhead_merge_kernel(const LmParams p,
                                                                const int64_t* __restrict__ ids,
                                                                float* __restrict__ logp,
                                                                float* __restrict__ lse,
                                                                const int32_t* __restrict__ lens) {
  pdl_wait();
  pdl_trigger();
  const int64_t splits = p.geometry->y;
  const int64_t NC = p.N * p.C;
  for (int64_t k = (int64_t)blockIdx.x * kThreads + threadIdx.x; k < NC;
       k += (int64_t)gridDim.x * kThreads) {
    const int64_t i = k / p.C, t = k - i * p.C;
    if (t >= lens[i]) {
      logp[k] = 0.f;
      lse[k] = 0.f;
      continue;
    }
    const int64_t r = p.offsets[i] + t;
    const int64_t rb = r / kBM, rr = r - rb * kBM;
    float4 pk = p.partials[(rb * splits) * kBM + rr];
    float cm = pk.x, cs = pk.y, z = pk.z;
    bool has = pk.w != 0.f;
    for (int64_t sp = 1; sp < splits; ++sp) {
      pk = p.partials[(rb * splits + sp) * kBM + rr];
      lse_merge(cm, cs, pk.x, pk.y);
      if (pk.w != 0.f) {
        z = pk.z;
        has = true;
      }
    }
    const float l = cm + logf(cs);
    if (has) {
      logp[k] = z - l;
      lse[k] = l;
    } else {  // the sampled id is outside [0, V)
      logp[k] = __int_as_float(0x7fc00000);
      lse[k] = __int_as_float(0x7fc00000);
      atomicOr(&p.hdr->flags, kFlagTokenRange);
    }
  }
}

// ---- host side --------------------------------------------------------------------

std::mutex g_enc_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::lock_guard<std::mutex> lk(g_enc_mutex);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return cudaSuccess;
}

// 2-D bf16 tensor map over a row-major [rows, d] matrix, box 64 x box_rows,
// 128-byte swizzle (rows past `rows` read as zeros).
cudaError_t encode_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t d, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encoder(&enc);
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

LmLayout lm_layout(int64_t N, int64_t C, int64_t d, int sms) {
  LmLayout l;
  const WsLayout base = ws_layout(N);
  const int64_t rows = N * C;
  l.geometry = base.total;  // 16 bytes
  l.dense = align_up(base.total + 16, 1024);
  l.partials = align_up(l.dense + (size_t)rows * (size_t)d * 2, 256);
  const int64_t mb_max = (rows + kBM - 1) / kBM;
  const int64_t items_max = 4 * (int64_t)sms + 2 * mb_max;  // mb * splits bound
  l.total = align_up(l.partials + (size_t)items_max * kBM * sizeof(float4), 256);
  return l;
}

cudaError_t launch_lmhead(const void* hidden, const void* weight, const FwdArgs& a, int64_t d,
                          const DeviceInfo& dev, cudaStream_t st) {
  const WsLayout wl = ws_layout(a.N);
  const LmLayout ll = lm_layout(a.N, a.C, d, dev.sms);
  char* ws = static_cast<char*>(a.ws);
  const int32_t* off = reinterpret_cast<const int32_t*>(ws + wl.offsets);
  uint16_t* dense = reinterpret_cast<uint16_t*>(ws + ll.dense);
  const int64_t rows = a.N * a.C;

  int4* geometry = reinterpret_cast<int4*>(ws + ll.geometry);
  cudaError_t e = launch_pdl(gather_rows_kernel, dim3((unsigned)(dev.sms * 8)), dim3(kThreads), 0,
                             st, 1, static_cast<const uint16_t*>(hidden), dense, off, a.N,
                             a.P + a.C, a.P, d, a.V, dev.sms, geometry);
  if (e != cudaSuccess) return e;

  CUtensorMap map_h, map_w;
  if ((e = encode_2d(&map_h, dense, rows, d, kBM)) != cudaSuccess) return e;
  if ((e = encode_2d(&map_w, weight, a.V, d, kBN)) != cudaSuccess) return e;

  LmParams p;
  p.N = a.N;
  p.P = a.P;
  p.C = a.C;
  p.V = a.V;
  p.d = d;
  p.offsets = off;
  p.geometry = geometry;
  p.partials = reinterpret_cast<float4*>(ws + ll.partials);
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.sms = dev.sms;

  const int smem = kLmStages * kStageBytesLm + 1024;
  static bool attr_done = false;
  if (!attr_done) {
    if ((e = cudaFuncSetAttribute(lmhead_lse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  smem)) != cudaSuccess)
      return e;
    attr_done = true;
  }
  e = launch_pdl(lmhead_lse_kernel, dim3((unsigned)dev.sms), dim3(kLmThreads), (size_t)smem, st, 1,
                 map_h, map_w, a.ids, p);
  if (e != cudaSuccess) return e;
  int64_t blocks = (rows + kThreads - 1) / kThreads;
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  return launch_pdl(lmhead_merge_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, st, 1, p,
                    a.ids, a.logp, a.lse, reinterpret_cast<const int32_t*>(ws + wl.lens));
}

}  // namespace grpo

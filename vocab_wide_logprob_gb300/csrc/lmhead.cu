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
//                        dense [rows, d] buffer (row r = valid token r) and
//                        zeroes the rows up to the next multiple of 128
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
//
// The backward ("loss.backward()" through the projection) recomputes the
// logits with the same pipeline: lmhead_dz_kernel's epilogue turns each tile
// into the logits gradient g * w_t * (onehot(y_t) - exp(z - lse_t)), rounded
// to bf16, and stores it for the two gradient contractions (lmhead_bwd.cu).
#include <mutex>

#include "tc.cuh"

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
constexpr uint32_t kIdescLm = umma_idesc(kBM, kBN, false, false);

struct LmParams {
  int64_t N, P, C, V, d;
  const int32_t* offsets;  // prefix sums of the clamped lengths ([N+1])
  int4* geometry;          // [0] (row blocks, splits, tiles per split): written by the gather
  float4* partials;        // forward: [items][kBM] (max, sum, target logit, has target)
  WsHeader* hdr;
  int sms;                 // CTAs in the grid: the split count is chosen from it
  // logits-gradient pass only
  const float* lse;        // [N, C] from the forward
  const float* w;          // [N, C] d loss / d logp from the forward
  const float* grad;       // upstream scalar gradient (nullable: 1)
  uint16_t* dz;            // bf16 [rows, ldz]
  int64_t ldz;
};

// Split `ksteps` steps of work for each of `units` independent tiles into
// `splits` ranges so that the items (unit, range) fill the grid's rounds,
// counting both the items per round and the uneven last range; every range
// is non-empty and items <= max_items.  Candidate split counts 1 .. 256, one
// per thread of the calling CTA (kThreads threads); the smallest within 0.01
// of the best score wins (fewer partials to merge, and every range re-reads
// its unit's operand).  Returns (splits, steps per split).
__device__ float split_score(int32_t units, int32_t sp, int32_t ksteps, int sms,
                             int32_t max_items) {
  const int32_t items = units * sp;
  if (sp > ksteps || items > max_items) return -1.f;
  const int32_t sps = (ksteps + sp - 1) / sp;
  if ((int64_t)sps * (sp - 1) >= ksteps) return -1.f;  // the last range would be empty
  const int32_t rounds = (items + sms - 1) / sms;
  return (float)items / (float)(rounds * sms) * (float)ksteps / (float)(sps * sp);
}

__device__ int2 choose_split_block(int32_t units, int32_t ksteps, int sms, int32_t max_items) {
  __shared__ float s_best[kWarps];
  __shared__ int s_pick[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t sp = tid + 1;
  const float score =
      units > 0 ? split_score(units, sp, ksteps, sms, max_items) : (sp == 1 ? 1.f : -1.f);
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
  return make_int2(pick, (ksteps + pick - 1) / pick);
}

// ---- gather: dense [rows, d] copy of the scored rows' hidden states ----------

// geometry[0]: the projection pass (row blocks, vocabulary splits, tiles per
// split, 0).  With `grad_gemm`, geometry[1]: the hidden-state gradient
// contraction (row blocks, 256-wide d tiles, vocabulary splits, 64-wide
// k-steps per split).
__global__ void __launch_bounds__(kThreads) gather_rows_kernel(const uint16_t* __restrict__ hidden,
                                                               uint16_t* __restrict__ dense,
                                                               const int32_t* __restrict__ off,
                                                               int64_t N, int64_t T, int64_t P,
                                                               int64_t d, int64_t V, int sms,
                                                               int4* __restrict__ geometry,
                                                               int grad_gemm) {
  pdl_wait();
  pdl_trigger();
  const int64_t tv = off[N];
  const int32_t mb = (int32_t)((tv + kBM - 1) / kBM);
  if (blockIdx.x == 0) {
    const int32_t ntiles = (int32_t)((V + kBN - 1) / kBN);
    const int2 s = choose_split_block(mb, ntiles, sms, 4 * sms + 2 * mb);
    if (threadIdx.x == 0) geometry[0] = make_int4(mb, s.x, s.y, 0);
  }
  if (grad_gemm && blockIdx.x == (gridDim.x > 1 ? 1u : 0u)) {
    const int32_t nb = (int32_t)((d + 255) / 256);
    const int32_t ksteps = (int32_t)((V + kBN - 1) / kBN) * (kBN / kBK);
    const int2 s = choose_split_block(mb * nb, ksteps, sms, 2 * sms + mb * nb);
    if (threadIdx.x == 0) geometry[1] = make_int4(mb, nb, s.x, s.y);
  }
  const int64_t vec_per_row = d / 8;  // 16-byte vectors
  const int64_t rows_pad = (int64_t)mb * kBM;
  for (int64_t k = (int64_t)blockIdx.x * kThreads + threadIdx.x; k < rows_pad * vec_per_row;
       k += (int64_t)gridDim.x * kThreads) {
    const int64_t r = k / vec_per_row, c = k - r * vec_per_row;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);  // rows past the last scored one read as zeros
    if (r < tv) {
      int lo = 0, hi = (int)N;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= r)
          lo = mid;
        else
          hi = mid;
      }
      const int64_t t = r - off[lo];
      const uint4* src =
          reinterpret_cast<const uint4*>(hidden + ((int64_t)lo * T + P - 1 + t) * d);
      v = ld_stream(src + c);
    }
    reinterpret_cast<uint4*>(dense + r * d)[c] = v;
  }
}

// ---- the tensor-core pipeline ----------------------------------------------------

// Completion of the valid token r (binary search over the offsets).
__device__ __forceinline__ int completion_of(const int32_t* off, int64_t N, int64_t r) {
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

// kMode 0: log-sum-exp partials per row; kMode 1: the bf16 logits gradient.
template <int kMode>
__device__ __forceinline__ void lm_tile_pipeline(const CUtensorMap* map_h, const CUtensorMap* map_w,
                                                 const int64_t* __restrict__ ids,
                                                 const LmParams& p) {
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
  if (warp == 1) tmem_alloc(&s_tmem, 512);  // two 256-column fp32 accumulators
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait();
  pdl_trigger();

  const int64_t tv = p.offsets[p.N];
  const int4 geo = p.geometry[0];
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
            tma_load_2d(sa, map_h, kb * kBK, (int)(rb * kBM), full);
            tma_load_2d(sa + kABytes, map_w, kb * kBK, (int)(n * kBN), full);
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
              umma_bf16(dacc, umma_desc_k(sa + j * 32), umma_desc_k(sa + kABytes + j * 32),
                        kIdescLm, (kb | j) ? 1u : 0u);
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
    const float g = (kMode == 1 && p.grad != nullptr) ? __ldg(p.grad) : 1.f;
    for (int64_t it = blockIdx.x; it < items && !*(volatile int*)&s_abort; it += gridDim.x) {
      const int64_t rb = it / splits, sp = it - rb * splits;
      const int64_t n0 = sp * tps, n1 = min(ntiles, n0 + tps);
      const int64_t r = rb * kBM + row_in_block;  // valid token of this thread
      int64_t y = -1;
      float lse_r = 0.f, coef = 0.f;
      if (r < tv) {
        const int i = completion_of(p.offsets, p.N, r);
        const int64_t t = r - p.offsets[i];
        y = __ldg(ids + (int64_t)i * (p.P + p.C) + p.P + t);
        if (kMode == 1) {
          lse_r = __ldg(p.lse + (int64_t)i * p.C + t);
          coef = g * __ldg(p.w + (int64_t)i * p.C + t);
        }
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
          if constexpr (kMode == 0) {
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
          } else {
            // dz = coef * (onehot(y) - 2^(z log2 e - lse log2 e)), bf16 (round to nearest even)
            const float lL = lse_r * kLog2e;
            const uint64_t nlL2 = f2_pack(-lL, -lL);
            const uint64_t nc2 = f2_pack(-coef, -coef);
            uint32_t pk[16];
            if (y >= v0 && y < v0 + 32) {
              // the target column: coef * (1 - p_y) without cancellation, -expm1(z_y - lse)
              float zy_ = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (v0 + j == y) zy_ = v[j];
              const float dy = coef * -expm1f(zy_ - lse_r);
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                float a, b;
                f2_unpack(f2_mul(f2_ex2(f2_fma(f2_pack(v[j], v[j + 1]), L2, nlL2)), nc2), a, b);
                a = (v0 + j == y) ? dy : a;
                b = (v0 + j + 1 == y) ? dy : b;
                pk[j / 2] = pack_bf16x2(a, b);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                float a, b;
                f2_unpack(f2_mul(f2_ex2(f2_fma(f2_pack(v[j], v[j + 1]), L2, nlL2)), nc2), a, b);
                pk[j / 2] = pack_bf16x2(a, b);
              }
            }
            if (r >= tv) {  // padding rows of the last block: zeros
#pragma unroll
              for (int j = 0; j < 16; ++j) pk[j] = 0u;
            } else if (v0 + 32 > p.V) {  // columns past V: zeros
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (v0 + j >= p.V) pk[j >> 1] &= (j & 1) ? 0x0000ffffu : 0xffff0000u;
            }
            uint4* dst = reinterpret_cast<uint4*>(p.dz + r * p.ldz + v0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
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
      if constexpr (kMode == 0) {
        float a0, a1, a2, a3;
        f2_unpack(acc01, a0, a1);
        f2_unpack(acc23, a2, a3);
        const float s = ((a0 + a1) + (a2 + a3)) + s_extra;
        if (r < tv) p.partials[it * kBM + row_in_block] = make_float4(m, s, zy, has ? 1.f : 0.f);
      }
    }
  }

  // release tensor memory: every MMA this CTA issued has completed once the
  // epilogue consumed its tile (or, after a timeout, once the last commit lands)
  tmem_fence_before();
  __syncthreads();
  if (warp == 1) {
    tmem_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_lse_kernel(const __grid_constant__ CUtensorMap map_h,
                      const __grid_constant__ CUtensorMap map_w, const int64_t* __restrict__ ids,
                      const LmParams p) {
  lm_tile_pipeline<0>(&map_h, &map_w, ids, p);
}

__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_dz_kernel(const __grid_constant__ CUtensorMap map_h,
                     const __grid_constant__ CUtensorMap map_w, const int64_t* __restrict__ ids,
                     const LmParams p) {
  lm_tile_pipeline<1>(&map_h, &map_w, ids, p);
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

LmParams lm_params(const int32_t* off, int4* geometry, WsHeader* hdr, int64_t N, int64_t P,
                   int64_t C, int64_t V, int64_t d, int sms) {
  LmParams p = {};
  p.N = N;
  p.P = P;
  p.C = C;
  p.V = V;
  p.d = d;
  p.offsets = off;
  p.geometry = geometry;
  p.hdr = hdr;
  p.sms = sms;
  return p;
}

template <typename K>
cudaError_t launch_tiles(K kern, const void* dense, const void* weight, int64_t rows, int64_t d,
                         int64_t V, const int64_t* ids, const LmParams& p, const DeviceInfo& dev,
                         cudaStream_t st, bool* attr_done) {
  CUtensorMap map_h, map_w;
  cudaError_t e;
  if ((e = encode_bf16_2d(&map_h, dense, d, rows, d, kBM)) != cudaSuccess) return e;
  if ((e = encode_bf16_2d(&map_w, weight, d, V, d, kBN)) != cudaSuccess) return e;
  const int smem = kLmStages * kStageBytesLm + 1024;
  if (!*attr_done) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
      return e;
    *attr_done = true;
  }
  return launch_pdl(kern, dim3((unsigned)dev.sms), dim3(kLmThreads), (size_t)smem, st, 1, map_h,
                    map_w, ids, p);
}

}  // namespace

cudaError_t encode_bf16_2d(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                           int64_t pitch, int box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encoder(&enc);
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)pitch * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

LmLayout lm_layout(int64_t N, int64_t C, int64_t d, int sms) {
  LmLayout l;
  const WsLayout base = ws_layout(N);
  const int64_t rows = N * C;
  const int64_t mb_max = (rows + kBM - 1) / kBM;
  l.geometry = base.total;  // 2 x int4
  l.dense = align_up(base.total + 32, 1024);
  l.partials = align_up(l.dense + (size_t)(mb_max * kBM) * (size_t)d * 2, 256);
  const int64_t items_max = 4 * (int64_t)sms + 2 * mb_max;  // mb * splits bound
  l.total = align_up(l.partials + (size_t)items_max * kBM * sizeof(float4), 256);
  return l;
}

LmBwdLayout lm_bwd_layout(int64_t N, int64_t C, int64_t V, int64_t d, int sms) {
  LmBwdLayout l;
  const WsLayout base = ws_layout(N);
  const int64_t mb_max = (N * C + kBM - 1) / kBM;
  l.rows_cap = mb_max * kBM;
  l.ldz = (V + kBN - 1) / kBN * kBN;
  const int64_t nb = (d + 255) / 256;
  l.items_max = 2 * (int64_t)sms + mb_max * nb;
  l.geometry = base.total;
  l.dense = align_up(base.total + 32, 1024);
  l.dz = align_up(l.dense + (size_t)l.rows_cap * (size_t)d * 2, 1024);
  l.dh_partials = align_up(l.dz + (size_t)l.rows_cap * (size_t)l.ldz * 2, 1024);
  l.total = align_up(l.dh_partials + (size_t)l.items_max * kBM * 256 * sizeof(float), 256);
  return l;
}

cudaError_t launch_lmhead(const void* hidden, const void* weight, const FwdArgs& a, int64_t d,
                          const DeviceInfo& dev, cudaStream_t st) {
  const WsLayout wl = ws_layout(a.N);
  const LmLayout ll = lm_layout(a.N, a.C, d, dev.sms);
  char* ws = static_cast<char*>(a.ws);
  const int32_t* off = reinterpret_cast<const int32_t*>(ws + wl.offsets);
  uint16_t* dense = reinterpret_cast<uint16_t*>(ws + ll.dense);
  const int64_t rows = (a.N * a.C + kBM - 1) / kBM * kBM;

  int4* geometry = reinterpret_cast<int4*>(ws + ll.geometry);
  cudaError_t e = launch_pdl(gather_rows_kernel, dim3((unsigned)(dev.sms * 8)), dim3(kThreads), 0,
                             st, 1, static_cast<const uint16_t*>(hidden), dense, off, a.N,
                             a.P + a.C, a.P, d, a.V, dev.sms, geometry, 0);
  if (e != cudaSuccess) return e;

  LmParams p = lm_params(off, geometry, reinterpret_cast<WsHeader*>(ws), a.N, a.P, a.C, a.V, d,
                         dev.sms);
  p.partials = reinterpret_cast<float4*>(ws + ll.partials);
  static bool attr_done = false;
  if ((e = launch_tiles(lmhead_lse_kernel, dense, weight, rows, d, a.V, a.ids, p, dev, st,
                        &attr_done)) != cudaSuccess)
    return e;
  int64_t blocks = (a.N * a.C + kThreads - 1) / kThreads;
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  return launch_pdl(lmhead_merge_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, st, 1, p,
                    a.ids, a.logp, a.lse, reinterpret_cast<const int32_t*>(ws + wl.lens));
}

cudaError_t launch_lmhead_dz(const LmBwdArgs& a, const DeviceInfo& dev, cudaStream_t st) {
  const WsLayout wl = ws_layout(a.N);
  const LmBwdLayout bl = lm_bwd_layout(a.N, a.C, a.V, a.d, dev.sms);
  char* ws = static_cast<char*>(a.ws);
  const int32_t* off = reinterpret_cast<const int32_t*>(ws + wl.offsets);
  uint16_t* dense = reinterpret_cast<uint16_t*>(ws + bl.dense);
  int4* geometry = reinterpret_cast<int4*>(ws + bl.geometry);
  cudaError_t e = launch_pdl(gather_rows_kernel, dim3((unsigned)(dev.sms * 8)), dim3(kThreads), 0,
                             st, 1, static_cast<const uint16_t*>(a.hidden), dense, off, a.N,
                             a.P + a.C, a.P, a.d, a.V, dev.sms, geometry, 1);
  if (e != cudaSuccess) return e;
  LmParams p = lm_params(off, geometry, reinterpret_cast<WsHeader*>(ws), a.N, a.P, a.C, a.V, a.d,
                         dev.sms);
  p.lse = a.lse;
  p.w = a.w;
  p.grad = a.grad;
  p.dz = reinterpret_cast<uint16_t*>(ws + bl.dz);
  p.ldz = bl.ldz;
  static bool attr_done = false;
  return launch_tiles(lmhead_dz_kernel, dense, a.weight, bl.rows_cap, a.d, a.V, a.ids, p, dev,
                      st, &attr_done);
}

}  // namespace grpo

// Persistent, warp-specialised tcgen05 pipeline over CTA pairs (2-SM MMA),
// shared by the LM-head kernels.  Internal header.
//
// The grid is a whole number of clusters of two CTAs on two SMs.  A pair
// processes work items; an item is a sequence of accumulator tiles of
// M = 256 rows (128 per CTA) by N <= 256 columns, each reduced over a range of
// 64-wide k-steps.  Per CTA:
//   warp 0 (one lane)  TMA producer: loads this CTA's 128 rows of A and its half
//                      of B's N rows for each k-step into a ring of
//                      Op::kStages stages; the loads of both CTAs
//                      complete on the leader's `full` barrier.
//   warp 1 (one lane)  on the leader only: issues tcgen05.mma.cta_group::2
//                      (M = 256, K = 16) into one of two 256-column TMEM
//                      accumulators (or one of up to 512 columns); commits
//                      free the stage (`empty`) and publish the tile
//                      (`acc_full`) in both CTAs at once.
//   warps 2 ..         epilogue (Op::kEpiWarps = 4 or 8): each reads this CTA's
//                      TMEM lanes 32 (w % 4) .. + 31 of the finished tile (with
//                      8 warps, half of its columns each) and hands the
//                      accumulator back (`acc_empty` on the leader, one
//                      arrival per epilogue warp of both CTAs).
// Per CTA, A and B stage operands sit at the same shared-memory offsets, which
// is how the leader's descriptors address both CTAs' halves.  Every wait is
// bounded (one second); a timeout sets kFlagTimeout in the workspace header
// and makes the CTA stop issuing work, so the kernel always finishes.
//
// The Op class supplies the item geometry, the loads, the descriptors and
// the epilogue (see the LM-head kernels for the four uses).
#pragma once

#include "tc.cuh"

namespace grpo {

constexpr int kPairThreads = 192;  // with 4 epilogue warps
constexpr int kPairStages = 6;          // the default ring: 6 stages of 32 KiB
constexpr int kPairStageBytes = 32768;  // A 16 KiB + B half <= 16 KiB per CTA
constexpr int kPairBOffset = 16384;     // B half inside a stage
constexpr int kPairRingBytes = kPairStages * kPairStageBytes;

// Op:
//   static constexpr int kStages, kStageBytes   the ring (kStages * kStageBytes <= the
//                                               dynamic shared memory before `ring` + ...)
//   static constexpr int kEpiWarps              4 or 8 epilogue warps (kernel threads:
//                                               64 + 32 * kEpiWarps)
//   static constexpr int kAccCols               256: two accumulators, the epilogue of one
//                                               tile overlaps the MMAs of the next; 512:
//                                               one accumulator of up to 512 columns
//   int64_t items() const;  int tiles(int64_t it) const;
//   void krange(int64_t it, int t, int64_t* k0, int64_t* k1) const;
//   uint32_t bytes(int64_t it, int t) const;            this CTA's bytes per k-step
//   void load(uint32_t sa, int64_t it, int t, int64_t ks, uint32_t rank,
//             uint32_t mbar_cluster) const;             this CTA's TMA loads
//   void mma(uint32_t dacc, uint32_t sa, int64_t it, int t, bool first) const;  4 MMAs
//   void epi_begin(int64_t it); void epi_tile(int64_t it, int t, uint32_t tmem_lane_base,
//                  bool empty, int slice); void epi_end(int64_t it); void epi_finish();
template <class Op>
__device__ __forceinline__ void pair_pipeline(Op& op, uint32_t ring, WsHeader* hdr) {
  constexpr int kStages = Op::kStages;
  constexpr uint32_t kStageBytes = Op::kStageBytes;
  constexpr int kBufs = Op::kAccCols == 512 ? 1 : 2;
  constexpr uint32_t kAccCols = Op::kAccCols;
  constexpr int kEpi = Op::kEpiWarps;  // 4 or 8: one or two warps per TMEM lane quarter
  __shared__ __align__(8) uint64_t s_full[kStages];
  __shared__ __align__(8) uint64_t s_empty[kStages];
  __shared__ __align__(8) uint64_t s_acc_full[2];
  __shared__ __align__(8) uint64_t s_acc_empty[2];
  __shared__ __align__(8) uint64_t s_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (tid == 0) {
    s_abort = 0;
    for (int k = 0; k < kStages; ++k) {
      mbar_init(smem_u32(&s_full[k]), 1);   // leader: its producer's arrive (+ both CTAs' bytes)
      mbar_init(smem_u32(&s_empty[k]), 1);  // the leader's multicast commit
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&s_acc_full[k]), 1);   // the leader's multicast commit
      mbar_init(smem_u32(&s_acc_empty[k]), 2 * kEpi);  // leader: the epilogue warps of 2 CTAs
    }
    mbar_init(smem_u32(&s_drain), 1);  // the leader's last commit
    mbar_init_fence();
  }
  if (warp == 1) tmem_alloc_pair(&s_tmem, 512);  // all 512 columns: kBufs accumulators
  tmem_fence_before();
  pair_sync();  // barriers and TMEM exist in both CTAs before any cross-CTA use
  tmem_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_wait();
  pdl_trigger();
  op.setup();
  const int64_t items = op.items();
  auto timeout = [&]() {
    atomicOr(&hdr->flags, kFlagTimeout);
    *(volatile int*)&s_abort = 1;
  };
  auto aborted = [&]() { return *(volatile int*)&s_abort != 0; };

  if (warp == 0) {
    if (lane == 0) {  // ---------------- TMA producer (both CTAs) ----------------
      int stage = 0;
      uint32_t phase = 0;
      for (int64_t it = pair; it < items && !aborted(); it += npairs) {
        const int nt = op.tiles(it);
        for (int t = 0; t < nt && !aborted(); ++t) {
          int64_t k0, k1;
          op.krange(it, t, &k0, &k1);
          const uint32_t bytes = op.bytes(it, t);
          for (int64_t ks = k0; ks < k1; ++ks) {
            if (!mbar_wait(smem_u32(&s_empty[stage]), phase ^ 1u)) {
              timeout();
              break;
            }
            const uint32_t full = smem_u32(&s_full[stage]);
            if (rank == 0) mbar_arrive_expect_tx(full, 2u * bytes);
            op.load(ring + (uint32_t)stage * kStageBytes, it, t, ks, rank, map_to_rank(full, 0));
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {  // ---------------- MMA issuer (leader) ------------
      int stage = 0, buf = 0;
      uint32_t phase = 0, aphase = 0;
      for (int64_t it = pair; it < items && !aborted(); it += npairs) {
        const int nt = op.tiles(it);
        for (int t = 0; t < nt && !aborted(); ++t) {
          if (!mbar_wait(smem_u32(&s_acc_empty[buf]), aphase ^ 1u)) {
            timeout();
            break;
          }
          tmem_fence_after();
          const uint32_t dacc = tmem + (uint32_t)buf * kAccCols;
          int64_t k0, k1;
          op.krange(it, t, &k0, &k1);
          bool ok = true;
          for (int64_t ks = k0; ks < k1; ++ks) {
            if (!mbar_wait(smem_u32(&s_full[stage]), phase)) {
              timeout();
              ok = false;
              break;
            }
            tmem_fence_after();
            op.mma(dacc, ring + (uint32_t)stage * kStageBytes, it, t, ks == k0);
            umma_commit_pair(smem_u32(&s_empty[stage]));  // the stage is free in both CTAs
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit_pair(smem_u32(&s_acc_full[buf]));  // (an empty range: arrives at once)
          if (++buf == kBufs) {
            buf = 0;
            aphase ^= 1u;
          }
        }
      }
    }
  } else {  // ---------------- epilogue: warps 2 .. 2 + kEpi - 1 of both CTAs -----
    const int quarter = warp & 3;  // TMEM lanes 32 * quarter .. + 31
    const int slice = (warp - 2) >> 2;  // with 8 warps: which half of the columns
    int buf = 0;
    uint32_t aphase = 0;
    const uint32_t acc_empty_leader0 = map_to_rank(smem_u32(&s_acc_empty[0]), 0);
    const uint32_t acc_empty_leader1 = map_to_rank(smem_u32(&s_acc_empty[1]), 0);
    for (int64_t it = pair; it < items && !aborted(); it += npairs) {
      op.epi_begin(it);
      const int nt = op.tiles(it);
      bool ok = true;
      for (int t = 0; t < nt; ++t) {
        if (!mbar_wait(smem_u32(&s_acc_full[buf]), aphase)) {
          timeout();
          ok = false;
          break;
        }
        tmem_fence_after();
        int64_t k0, k1;
        op.krange(it, t, &k0, &k1);
        op.epi_tile(it, t, tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)buf * kAccCols,
                    k1 <= k0, slice);
        tmem_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(buf ? acc_empty_leader1 : acc_empty_leader0);
        if (++buf == kBufs) {
          buf = 0;
          aphase ^= 1u;
        }
      }
      if (!ok) break;
      op.epi_end(it);
    }
    op.epi_finish();
  }

  // Teardown: a last commit from the leader lands in both CTAs once every MMA
  // it issued has completed (at once when the epilogues consumed every tile;
  // after a timeout, it keeps TMEM allocated until the MMAs in flight finish);
  // then both CTAs free the pair's TMEM together.
  if (warp == 1 && lane == 0 && rank == 0) umma_commit_pair(smem_u32(&s_drain));
  if (tid == 0 && !mbar_wait(smem_u32(&s_drain), 0)) atomicOr(&hdr->flags, kFlagTimeout);
  tmem_fence_before();
  pair_sync();
  if (warp == 1) {
    tmem_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace grpo

// Tensor-core (tcgen05 + TMEM) and tensor-TMA helpers of the LM-head kernels,
// as inline PTX for sm_103a.  Internal header.
//
// Shared-memory operand layouts (bf16, 128-byte swizzle, 1024-byte aligned):
//   K-major  : rows of 64 K-elements (128 B); 8 rows form a 1024-byte atom;
//              atoms along M/N at 1024 B (the stride byte offset).  One TMA box
//              {64 K, rows} writes it.  A 16-wide K step advances the start
//              address by 32 B inside the atom.
//   MN-major : rows of 64 M/N-elements (128 B), one row per K index; 8 K rows
//              form an atom; K groups of 8 at 1024 B (the stride byte offset),
//              64-wide M/N blocks at `lbo` bytes (the leading byte offset).
//              One TMA box {64 M/N, k rows} per 64 M/N elements writes it.  A
//              16-wide K step advances the start address by 2 atoms (2048 B).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace grpo {

__device__ __forceinline__ uint64_t umma_desc_k(uint32_t saddr) {
  uint64_t dsc = 0;
  dsc |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
  dsc |= (uint64_t)1 << 16;                   // leading byte offset (unused: K-major, swizzled)
  dsc |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 bytes
  dsc |= (uint64_t)1 << 46;                   // descriptor version
  dsc |= (uint64_t)2 << 61;                   // layout: 128-byte swizzle
  return dsc;
}

__device__ __forceinline__ uint64_t umma_desc_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t dsc = 0;
  dsc |= (uint64_t)((saddr >> 4) & 0x3FFFu);        // start address
  dsc |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;    // leading byte offset: next 64 M/N elements
  dsc |= (uint64_t)(1024 >> 4) << 32;               // stride byte offset: next 8 K rows
  dsc |= (uint64_t)1 << 46;
  dsc |= (uint64_t)2 << 61;
  return dsc;
}

// Instruction descriptor of tcgen05.mma kind::f16: D f32, A and B bf16,
// transpose bits for MN-major operands, N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (tmem, f32) (+)= A * B^T, one elected thread.
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t ad, uint64_t bd,
                                          uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
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
// Whole warp: allocate / free `cols` TMEM columns (a power of two >= 32).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t tmem, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols)
               : "memory");
}
// Whole warp: 32 lanes x 32 consecutive fp32 columns; thread t gets lane t.
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
// The same 32-column load, issued without waiting: the registers are filled
// asynchronously and must not be read before tmem_ld_wait(r).
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
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
}
// Waits for this thread's TMEM loads.  The registers are operands of the
// wait, so no use of them can be placed before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
// 2-D tiled TMA load into this CTA's shared memory; x is the inner coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t sdst, const CUtensorMap* map, int x, int y,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(sdst),
      "l"(map), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}

// 3-D variant (coordinates x inner, y, z outer).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t sdst, const CUtensorMap* map, int x, int y,
                                                 int z, uint32_t mbar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sdst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(mbar_cluster)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t ssrc, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(map),
      "r"(x), "r"(y), "r"(z), "r"(ssrc)
      : "memory");
}

// 2-D TMA store of a shared-memory box to global memory (bulk async group of
// this thread); x is the inner coordinate.  Parts outside the tensor are not
// written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t ssrc, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   map),
               "r"(x), "r"(y), "r"(ssrc)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// At most N of this thread's bulk groups still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// At most N of this thread's bulk groups not yet complete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Generic-proxy writes to shared memory become visible to the TMA (async proxy).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// ---- CTA pairs (2-SM MMA, .cta_group::2) ----------------------------------------
// A cluster of two CTAs on two SMs computes one M = 256 tile: CTA r holds rows
// [128 r, 128 r + 128) of A and half of B's N rows in its own shared memory;
// one thread of the even CTA (the leader) issues the MMAs, which read both
// CTAs' operands and write each CTA's 128 rows of D into its own TMEM.

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// (map_to_rank: the shared::cluster address of a shared::cta offset in CTA
// `rank`; cluster_sync: a barrier over both CTAs; both in common.cuh.)
__device__ __forceinline__ void pair_sync() { cluster_sync(); }
// Whole warp in each CTA of the pair: allocate / free the same TMEM columns in both.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t tmem, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols)
               : "memory");
}
// Leader only: D (both CTAs' TMEM, M = 256) (+)= A * B^T.
__device__ __forceinline__ void umma_bf16_pair(uint32_t tmem_d, uint64_t ad, uint64_t bd,
                                               uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
      : "memory");
}
// Leader only: once the MMAs issued so far are done, arrive on the mbarrier at
// this shared::cta offset in both CTAs of the pair.
__device__ __forceinline__ void umma_commit_pair(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(mbar),
      "h"((uint16_t)3)
      : "memory");
}
// TMA load into this CTA's shared memory completing on an mbarrier of either
// CTA of the pair (`mbar_cluster` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t sdst, const CUtensorMap* map, int x, int y,
                                                 uint32_t mbar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(sdst),
      "l"(map), "r"(x), "r"(y), "r"(mbar_cluster)
      : "memory");
}
// Arrive on an mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t mbar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(mbar_cluster)
               : "memory");
}

// 2-D bf16 tensor map over a row-major [outer, inner] matrix with row pitch
// `pitch` elements, box {64, box_outer}, 128-byte swizzle; reads outside the
// extents return zeros.
cudaError_t encode_bf16_2d(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                           int64_t pitch, int box_outer);
// The logits gradient dz of the scored rows is kept in vocabulary slabs:
// [ldz / 64][rows][64] bf16, so that a TMA box of 64 vocabulary columns by
// 64 or 128 rows is one contiguous 8 or 16 KiB block.  Tensor map of that
// layout with box {64, box_rows, 1} (128-byte swizzle, loads) or, with
// `store`, box {32, 32, 1} (64-byte swizzle, the epilogue's stores).
cudaError_t encode_dz_slabs(CUtensorMap* map, void* base, int64_t rows, int64_t ldz, int box_rows,
                            bool store);
// Tensor map of a row-major [outer, inner] matrix for the epilogues' 32 x 32
// TMA stores: bf16 (64-byte rows, 64-byte swizzle) or fp32 (128-byte rows,
// 128-byte swizzle); pitch in elements.
cudaError_t encode_store_32x32(CUtensorMap* map, void* base, bool fp32, int64_t inner,
                               int64_t outer, int64_t pitch);

}  // namespace grpo

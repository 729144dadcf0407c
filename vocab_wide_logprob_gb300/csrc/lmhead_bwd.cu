// Gradients of the Dr. GRPO loss through the LM-head projection z = h W^T
// ("loss.backward()" over "model(...).logits" in "Making Dr GRPO go brrr",
// salahadawi.com; the page prints no gradient, this is the chain rule).  With
// dz the bf16 logits gradient of the scored rows (lmhead_dz_kernel):
//
//   dhidden[row] = dz[row] W        (rows x V) (V x d): K = vocabulary
//   dweight      = dz^T H_scored    (V x rows) (rows x d): K = scored rows
//
// Both are dense contractions on the tcgen05 tensor cores (CTA pairs, 2-SM
// MMA with M = 256, pair_pipeline.cuh) with the fp32 accumulator in TMEM.  The
// operands are read where they lie: W [V, d] and the dense scored hidden rows
// [rows, d] (row-major), and dz in 64-column vocabulary slabs
// [ldz / 64][rows][64]; each enters as an MN-major (transposed) shared-memory
// operand where the contraction runs over its row index, so nothing is
// transposed in memory.
//
// lmhead_grad_gemm_kernel<DhOp>   dhidden partials: items (range of
//     vocabulary k-steps, 256 rows, up to 512 columns of d), fp32 tiles in the
//     workspace
// lmhead_grad_gemm_kernel<DwOp>   dweight: items (256 vocabulary rows, 512
//     columns of d), K = every row of the pass, fp32 straight to dweight
//     [V, d]: stored by the first pass, added by TMA reductions in the others
// lmhead_dh_reduce_kernel         sums a row's partials in split order
//     (deterministic) into dhidden [N, P+C, d]; rows that score nothing get 0;
//     runs beside the dweight kernel
//
// The backward rows run in passes (lmhead.cuh, LmBwdLayout): each pass runs
// the logits-gradient kernel and these three over its rows, in stream order,
// so one pass's dz buffer serves them all.
//
// The epilogue warps drain TMEM into 32 x 32 shared-memory boxes (128-byte
// swizzle, one or two per warp) that TMA stores write out while the next box
// fills.
// d must be a multiple of 128: each CTA of a pair holds half of every MMA's
// N columns (256 or 128) as whole 64-column MN-major atoms.
#include "host_ctx.cuh"
#include "pair_pipeline.cuh"
#include "lmhead.cuh"

namespace grpo {
namespace {

constexpr int kRows = 256;                 // output rows per pair tile (128 per CTA)
constexpr int kGK = 64;                    // k per stage
constexpr int kGABytes = 128 * kGK * 2;    // this CTA's A: 16 KiB
constexpr uint32_t kMnAtomStride = 8192;   // 64 M/N elements x 64 K rows x 2 bytes (one TMA box)
constexpr int kEpiBoxBytes = 32 * 32 * 4;  // one 32 x 32 fp32 TMA-store box
constexpr int kDhN = 512;                  // dhidden: d columns per item (two MMAs of <= 256)
constexpr int64_t kDhTileFloats = (int64_t)kRows * kDhN;

struct GradParams {
  int64_t N, V, d;
  const int4* geometry;    // [geo_dh]: (row blocks, d tiles of 512, splits, k-steps per split);
                           // [2].x: the backward's rows
  int geo_dh;              // this pass's hidden-gradient geometry
  int64_t row0, rows_pass;  // this pass's first backward row, rows per pass
  int pass;
  int64_t ksteps_v;        // vocabulary k-steps of the hidden-state gradient (ldz / 64)
  WsHeader* hdr;
};

__device__ __forceinline__ int64_t rows_of_pass(const GradParams& p) {
  const int64_t rows = p.geometry[2].x;
  return rows <= p.row0 ? 0 : (rows - p.row0 < p.rows_pass ? rows - p.row0 : p.rows_pass);
}

// 2-D TMA reduction of a shared-memory box into global memory: each element
// of the box is added to the one it lands on (bulk async group of the
// calling thread).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t ssrc, int x,
                                                  int y) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], "
      "[%3];" ::"l"(map),
      "r"(x), "r"(y), "r"(ssrc)
      : "memory");
}

// Drains accumulator columns [c0, c1) of this warp's 32 TMEM lanes through
// kBoxes 32 x 32 fp32 boxes (128-byte swizzle) into TMA stores at (x0 + c, y),
// or with `add` TMA reductions that add the box to what is there.
template <int kBoxes>
__device__ __forceinline__ void drain_fp32(const CUtensorMap* map_out, uint32_t stg,
                                           uint32_t& chunk, uint32_t tbase, int c0, int c1,
                                           bool empty, int x0, int y, bool add = false) {
  const int lane = threadIdx.x & 31;
  // The next 32 columns' TMEM load is issued as soon as this chunk's values
  // sit in shared memory, so it runs while the TMA reads the box.
  uint32_t v[32];
  if (!empty && c0 < c1) tmem_ld32_issue(tbase + (uint32_t)c0, v);
  for (int c = c0; c < c1; c += 32) {
    if (!empty) {
      tmem_ld_wait(v);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0u;
    }
    // row `lane` of the box; 16-byte chunk q sits at q ^ (lane & 7)
    const uint32_t box = stg + (chunk % kBoxes) * (uint32_t)kEpiBoxBytes;
    if (lane == 0) bulk_wait_read<kBoxes - 1>();  // the store that last used this box has read it
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 8; ++q)
      st_shared_v4(box + (uint32_t)lane * 128u + ((uint32_t)(q ^ (lane & 7)) << 4), v[4 * q],
                   v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    fence_async_smem();
    __syncwarp();
    if (!empty && c + 32 < c1) tmem_ld32_issue(tbase + (uint32_t)(c + 32), v);
    if (lane == 0) {
      if (add)
        tma_reduce_add_2d(map_out, box, x0 + c, y);
      else
        tma_store_2d(map_out, box, x0 + c, y);
      bulk_commit();
    }
    ++chunk;
  }
}

// The d tile item `it` of the persistent loop works on.  Items come in
// aligned groups of nb (one unit: the same operand rows, its nb d tiles, the
// last one narrower when d is not a multiple of 512), and a pair takes every
// npairs-th item: with the tile fixed by `it % nb` the same pairs would always
// get the narrow tile (npairs even, nb = 2: even pairs 512 columns per item,
// odd pairs 384).  Rotating the tiles of each group by the round, it / npairs,
// gives every pair the tiles in turn; a group still runs in one round on
// neighbouring pairs (npairs a multiple of nb), sharing its operand in L2.
__device__ __forceinline__ int64_t rotated_tile(int64_t it, int64_t nb) {
  const int64_t npairs = gridDim.x >> 1;
  if (nb <= 1 || npairs % nb != 0) return it % nb;
  return (it % nb + it / npairs) % nb;
}

// An item's unit (it / nb), d tile and width, decoded once per item by each
// role's thread: the producer and the MMA issuer consult them at every
// k-step, where 64-bit divisions on every call would hold up the issue.
struct ItemTile {
  int64_t it = -1, unit = 0, n = 0;
  int w = 0;
};

// dhidden = dz W.  Items (vocabulary split, 256-row block, d tile of up to
// 512): A = dz (K-major, one {64 vocabulary, 128 rows} slab box per CTA), B =
// W (MN-major): the d tile is two MMAs of N0 <= 256 and N1 = width - N0
// columns sharing A, each split over the pair (N / 2 columns per CTA, whole
// 64-column atoms), accumulating into TMEM columns [0, N0) and [256, 256 + N1).
// Fewer operand bytes per FLOP than 256-column tiles: the kernel is bound by
// how fast operands arrive from L2, and its epilogue runs once per long item.
struct DhOp {
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kGABytes + 2 * 16384;  // A + up to 256 B columns
  static constexpr int kAccCols = 512;
  static constexpr int kEpiWarps = 4;  // the epilogue runs once per long item
  static constexpr int kBoxes = 2;
  const GradParams& p;
  const CUtensorMap* map_a;
  const CUtensorMap* map_b;
  const CUtensorMap* map_out;
  uint32_t rank, stg;
  int64_t nb, mb, sps, ksteps, n_items;
  uint32_t chunk;

  __device__ void setup() {
    nb = (p.d + kDhN - 1) / kDhN;
    const int4 g = p.geometry[p.geo_dh];
    mb = g.x;
    sps = g.w;
    ksteps = p.ksteps_v;
    n_items = (int64_t)g.x * g.y * g.z;
    chunk = 0;
  }
  // it / nb = split * mb + row block, its d tile rotated by the round
  // (rotated_tile): the items running at the same time share their vocabulary
  // range in L2.
  mutable ItemTile cur;
  __device__ const ItemTile& tile_of(int64_t it) const {
    if (it != cur.it) {
      cur.it = it;
      cur.unit = it / nb;
      cur.n = rotated_tile(it, nb);
      cur.w = (int)min((int64_t)kDhN, p.d - cur.n * kDhN);
    }
    return cur;
  }
  __device__ int64_t m_tile(int64_t it) const { return tile_of(it).unit % mb; }
  __device__ int64_t n_tile(int64_t it) const { return tile_of(it).n; }
  __device__ int width(int64_t it) const { return tile_of(it).w; }
  __device__ int64_t items() const { return n_items; }
  __device__ int tiles(int64_t) const { return 1; }
  __device__ void krange(int64_t it, int, int64_t* k0, int64_t* k1) const {
    *k0 = (tile_of(it).unit / mb) * sps;
    *k1 = min(ksteps, *k0 + sps);
  }
  __device__ uint32_t bytes(int64_t it, int) const {
    return (uint32_t)(kGABytes + (width(it) / 2) * kGK * 2);
  }
  __device__ void load(uint32_t sa, int64_t it, int, int64_t ks, uint32_t rk,
                       uint32_t mbar) const {
    const int64_t d0 = n_tile(it) * kDhN;
    const int w = width(it), n0 = min(w, 256), n1 = w - n0;
    tma_load_3d_pair(sa, map_a, 0, (int)(m_tile(it) * kRows + rk * 128), (int)ks, mbar);
    const uint32_t sb = sa + kGABytes;
    for (int j = 0; j < n0 / 128; ++j)  // first MMA: this CTA's n0 / 2 columns
      tma_load_2d_pair(sb + j * kMnAtomStride, map_b, (int)(d0 + rk * (n0 / 2) + 64 * j),
                       (int)(ks * kGK), mbar);
    for (int j = 0; j < n1 / 128; ++j)  // second MMA: this CTA's n1 / 2 columns
      tma_load_2d_pair(sb + 16384 + j * kMnAtomStride, map_b,
                       (int)(d0 + 256 + rk * (n1 / 2) + 64 * j), (int)(ks * kGK), mbar);
  }
  __device__ void mma(uint32_t dacc, uint32_t sa, int64_t it, int, bool first) const {
    const int w = width(it), n0 = min(w, 256), n1 = w - n0;
    const uint32_t id0 = umma_idesc(256, n0, false, true);
    const uint32_t id1 = umma_idesc(256, n1 > 0 ? n1 : 16, false, true);
    const uint32_t sb = sa + kGABytes;
#pragma unroll
    for (int j = 0; j < kGK / 16; ++j) {
      const uint64_t ad = umma_desc_k(sa + j * 32);
      const uint32_t acc = (first && j == 0) ? 0u : 1u;
      umma_bf16_pair(dacc, ad, umma_desc_mn(sb + j * 2048, kMnAtomStride), id0, acc);
      if (n1 > 0)
        umma_bf16_pair(dacc + 256, ad, umma_desc_mn(sb + 16384 + j * 2048, kMnAtomStride), id1,
                       acc);
    }
  }
  __device__ void epi_begin(int64_t) {}
  __device__ void epi_tile(int64_t it, int, uint32_t tbase, bool empty, int) {
    // partial tile (split * mb + row block) * nb + d tile: rows .. * 256 of an
    // [items * 256, 512] matrix
    const int quarter = (threadIdx.x >> 5) & 3;
    const int64_t tile = tile_of(it).unit * nb + n_tile(it);
    drain_fp32<kBoxes>(map_out, stg, chunk, tbase, 0, width(it), empty, 0,
                       (int)(tile * kRows + rank * 128 + quarter * 32));
  }
  __device__ void epi_end(int64_t) {}
  __device__ void epi_finish() {
    if ((threadIdx.x & 31) == 0) bulk_wait<0>();  // every store has completed
  }
};

// dweight = dz^T H.  Items (256-vocabulary block, d tile of kN), K = every
// scored row: A = dz^T (MN-major, two {64 vocabulary, 64 rows} slab boxes per
// CTA), B = H (MN-major, each CTA holding half of every MMA's N columns).
// kN = 256: two accumulators, so the epilogue of one item (128 KiB of fp32 per
// CTA) overlaps the next item's MMAs.  kN = 512: two MMAs share A (fewer
// operand bytes per FLOP), one accumulator.
template <int kN>
struct DwOp {
  static constexpr int kStages = kN == 512 ? 4 : kPairStages;
  static constexpr int kStageBytes = kGABytes + (kN / 2) * kGK * 2;
  static constexpr int kAccCols = kN;
  // the epilogue (kN fp32 columns per row per item) is as long as a good part
  // of the item's MMAs: two warps per TMEM lane quarter drain half each
  static constexpr int kEpiWarps = 8;
  static constexpr int kBoxes = 1;
  const GradParams& p;
  const CUtensorMap* map_a;
  const CUtensorMap* map_b;
  const CUtensorMap* map_out;
  uint32_t rank, stg;
  int64_t nb, ksteps, n_items;
  uint32_t chunk;

  __device__ void setup() {
    nb = (p.d + kN - 1) / kN;
    const int64_t rows = rows_of_pass(p);
    ksteps = (rows + kGK - 1) / kGK;  // rows past the pass's last one are zero
    // the first pass stores dweight (zeros when there is no row at all); the
    // others add to it, and one without rows has nothing to add
    n_items = (p.pass > 0 && rows == 0) ? 0 : (p.V + kRows - 1) / kRows * nb;
    chunk = 0;
  }
  mutable ItemTile cur;
  __device__ const ItemTile& tile_of(int64_t it) const {
    if (it != cur.it) {
      cur.it = it;
      cur.unit = it / nb;
      cur.n = rotated_tile(it, nb);
      cur.w = (int)min((int64_t)kN, p.d - cur.n * kN);
    }
    return cur;
  }
  __device__ int64_t m_tile(int64_t it) const { return tile_of(it).unit; }
  __device__ int64_t n_tile(int64_t it) const { return tile_of(it).n; }
  __device__ int width(int64_t it) const { return tile_of(it).w; }
  __device__ int64_t items() const { return n_items; }
  __device__ int tiles(int64_t) const { return 1; }
  __device__ void krange(int64_t, int, int64_t* k0, int64_t* k1) const {
    *k0 = 0;
    *k1 = ksteps;
  }
  __device__ uint32_t bytes(int64_t it, int) const {
    return (uint32_t)(kGABytes + (width(it) / 2) * kGK * 2);
  }
  __device__ void load(uint32_t sa, int64_t it, int, int64_t ks, uint32_t rk,
                       uint32_t mbar) const {
    const int64_t mt = m_tile(it), d0 = n_tile(it) * kN;
    const int w = width(it), n0 = min(w, 256), n1 = w - n0;
    for (int j = 0; j < 2; ++j)
      tma_load_3d_pair(sa + j * kMnAtomStride, map_a, 0, (int)(ks * kGK),
                       (int)(mt * (kRows / 64) + rk * 2 + j), mbar);
    const uint32_t sb = sa + kGABytes;
    const int hrow = (int)(p.row0 + ks * kGK);  // the pass's rows of the dense hidden states
    for (int j = 0; j < n0 / 128; ++j)
      tma_load_2d_pair(sb + j * kMnAtomStride, map_b, (int)(d0 + rk * (n0 / 2) + 64 * j), hrow,
                       mbar);
    for (int j = 0; j < n1 / 128; ++j)
      tma_load_2d_pair(sb + 16384 + j * kMnAtomStride, map_b,
                       (int)(d0 + 256 + rk * (n1 / 2) + 64 * j), hrow, mbar);
  }
  __device__ void mma(uint32_t dacc, uint32_t sa, int64_t it, int, bool first) const {
    const int w = width(it), n0 = min(w, 256), n1 = w - n0;
    const uint32_t id0 = umma_idesc(256, n0, true, true);
    const uint32_t id1 = umma_idesc(256, n1 > 0 ? n1 : 16, true, true);
    const uint32_t sb = sa + kGABytes;
#pragma unroll
    for (int j = 0; j < kGK / 16; ++j) {
      const uint64_t ad = umma_desc_mn(sa + j * 2048, kMnAtomStride);
      const uint32_t acc = (first && j == 0) ? 0u : 1u;
      umma_bf16_pair(dacc, ad, umma_desc_mn(sb + j * 2048, kMnAtomStride), id0, acc);
      if (n1 > 0)
        umma_bf16_pair(dacc + 256, ad, umma_desc_mn(sb + 16384 + j * 2048, kMnAtomStride), id1,
                       acc);
    }
  }
  __device__ void epi_begin(int64_t) {}
  __device__ void epi_tile(int64_t it, int, uint32_t tbase, bool empty, int slice) {
    // dweight [V, d] at (vocabulary row, d column); rows past V are not stored
    const int quarter = (threadIdx.x >> 5) & 3;
    const int half = width(it) / 2;
    drain_fp32<kBoxes>(map_out, stg, chunk, tbase, slice * half, (slice + 1) * half, empty,
                       (int)(n_tile(it) * kN), (int)(m_tile(it) * kRows + rank * 128 + quarter * 32),
                       p.pass > 0);
  }
  __device__ void epi_end(int64_t) {}
  __device__ void epi_finish() {
    if ((threadIdx.x & 31) == 0) bulk_wait<0>();  // every store has completed
  }
};

constexpr int kDwN = 512;  // dweight: d columns per item (measured faster than 256)

template <class Op>
__global__ void __launch_bounds__(64 + 32 * Op::kEpiWarps, 1)
    lmhead_grad_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                            const __grid_constant__ CUtensorMap map_b,
                            const __grid_constant__ CUtensorMap map_out, const GradParams p) {
  extern __shared__ __align__(1024) unsigned char g_smem[];
  const uint32_t ring = smem_u32(g_smem + ((1024 - (smem_u32(g_smem) & 1023)) & 1023));
  Op op{p, &map_a, &map_b, &map_out};
  op.rank = cluster_rank();
  op.stg = ring + Op::kStages * Op::kStageBytes +  // this epilogue warp's boxes
           (uint32_t)((threadIdx.x >> 5) - 2) * Op::kBoxes * kEpiBoxBytes;
  pair_pipeline(op, ring, p.hdr);
}

// dhidden [N, P+C, d]: row (i, P-1+t) is backward row r = tokrow[i*C + t]
// (-1: the token is not scored, or its weight is 0 and was skipped; then the
// row is 0).  The pass that holds backward row r writes that row: the sum of
// its split partials in split order; the first pass also writes every row of
// no backward row (zeros).  A CTA per output row (index arithmetic once per
// row), 16-byte accesses.
// Launched after the dweight kernel (programmatic dependent launch), it runs
// beside it: it starts once every dweight CTA has begun, which is after the
// dhidden kernel it reads from has completed, and it waits for the dweight
// kernel only before it exits, so the kernels after it still see both done.
constexpr int kReduceThreads = 128;

__global__ void __launch_bounds__(kReduceThreads)
    lmhead_dh_reduce_kernel(const float* __restrict__ partials, const int4* __restrict__ geometry,
                            int geo_dh, const int32_t* __restrict__ rowmap,
                            const int32_t* __restrict__ tokrow, int64_t N, int64_t P, int64_t C,
                            int64_t d, int64_t row0, int64_t rows_pass, int pass,
                            float* __restrict__ dh) {
  pdl_trigger();
  const int4 g = geometry[geo_dh];
  const int64_t mb = g.x, nb = g.y;
  const int splits = g.z;
  const int64_t T = P + C;
  const int d4 = (int)(d / 4);
  const int64_t split_stride = mb * nb * kDhTileFloats;
  const int64_t all = geometry[2].x;
  const int64_t rows = all <= row0 ? 0 : (all - row0 < rows_pass ? all - row0 : rows_pass);
  // this pass's backward rows
  for (int64_t rr = blockIdx.x; rr < rows; rr += gridDim.x) {
    const int64_t tok = rowmap[row0 + rr], i = tok / C, t = tok - i * C;
    float4* dst = reinterpret_cast<float4*>(dh + (i * T + P - 1 + t) * d);
    const int64_t rb = rr / kRows, rl = rr - rb * kRows;
    for (int k4 = threadIdx.x; k4 < d4; k4 += kReduceThreads) {
      const int k = 4 * k4, nt = k / kDhN, kk = k - nt * kDhN;
      // partial tile of split s: item (s * mb + rb) * nb + nt
      const float* src = partials + (rb * nb + nt) * kDhTileFloats + rl * kDhN + kk;
      // L2 loads (not L1): the partials were written by a kernel this one does not wait for
      float4 acc = __ldcg(reinterpret_cast<const float4*>(src));
#pragma unroll 4
      for (int s = 1; s < splits; ++s) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(src + s * split_stride));
        acc.x += x.x;
        acc.y += x.y;
        acc.z += x.z;
        acc.w += x.w;
      }
      dst[k4] = acc;
    }
  }
  // the rows of no backward row: prompt rows, the last row, rows past each
  // length and skipped tokens
  if (pass == 0) {
    for (int64_t row = blockIdx.x; row < N * T; row += gridDim.x) {
      const int64_t i = row / T, t = row - i * T - (P - 1);
      if (t >= 0 && t < C && tokrow[i * C + t] >= 0) continue;
      float4* dst = reinterpret_cast<float4*>(dh + row * d);
      for (int k4 = threadIdx.x; k4 < d4; k4 += kReduceThreads)
        dst[k4] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  pdl_wait();  // the dweight kernel launched before this one has completed
}

template <class Op>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out,
                        const GradParams& p, const DeviceInfo& dev, cudaStream_t st) {
  constexpr int smem = Op::kStages * Op::kStageBytes + Op::kEpiWarps * Op::kBoxes * kEpiBoxBytes +
                       1024;
  cudaError_t e = ensure_dynamic_smem((const void*)lmhead_grad_gemm_kernel<Op>, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(lmhead_grad_gemm_kernel<Op>, dim3((unsigned)(2 * lm_pairs(dev))),
                    dim3(64 + 32 * Op::kEpiWarps), (size_t)smem, st, 2, a, b, out, p);
}

}  // namespace

cudaError_t launch_lmhead_grads(const LmBwdArgs& a, int64_t pass, const DeviceInfo& dev,
                                cudaStream_t st) {
  const LmBwdLayout bl = lm_bwd_layout(a.N, a.C, a.V, a.d, dev.sms, a.rows_pass);
  char* ws = static_cast<char*>(a.ws);
  const int32_t* rowmap = reinterpret_cast<const int32_t*>(ws + bl.rowmap);
  const int32_t* tokrow = reinterpret_cast<const int32_t*>(ws + bl.tokrow);
  const uint16_t* dz = reinterpret_cast<const uint16_t*>(ws + bl.dz);
  const uint16_t* dense = reinterpret_cast<const uint16_t*>(ws + bl.dense);
  const int4* geometry = reinterpret_cast<const int4*>(ws + bl.geometry);
  float* partials = reinterpret_cast<float*>(ws + bl.dh_partials);

  GradParams p;
  p.N = a.N;
  p.V = a.V;
  p.d = a.d;
  p.geometry = geometry;
  p.geo_dh = lm_geo_dh(pass);
  p.row0 = pass * bl.rows_pass;
  p.rows_pass = bl.rows_pass;
  p.pass = (int)pass;
  p.ksteps_v = bl.ldz / kGK;
  p.hdr = reinterpret_cast<WsHeader*>(ws);

  // dhidden = dz W: A = dz (K-major, K = vocabulary), B = W (MN-major)
  CUtensorMap a_dh, b_dh, o_dh, a_dw, b_dw, o_dw;
  cudaError_t e;
  if ((e = encode_dz_slabs(&a_dh, const_cast<uint16_t*>(dz), bl.rows_pass, bl.ldz, 128,
                           false)) != cudaSuccess)
    return e;
  if ((e = encode_bf16_2d(&b_dh, a.weight, a.d, a.V, a.d, kGK)) != cudaSuccess) return e;
  if ((e = encode_store_32x32(&o_dh, partials, true, kDhN, bl.items_max * kRows, kDhN)) !=
      cudaSuccess)
    return e;
  if ((e = launch_gemm<DhOp>(a_dh, b_dh, o_dh, p, dev, st)) != cudaSuccess) return e;

  // dweight (+)= dz^T H: A = dz (MN-major, K = the pass's rows), B = H (MN-major)
  if ((e = encode_dz_slabs(&a_dw, const_cast<uint16_t*>(dz), bl.rows_pass, bl.ldz, 64,
                           false)) != cudaSuccess)
    return e;
  if ((e = encode_bf16_2d(&b_dw, dense, a.d, bl.rows_cap, a.d, kGK)) != cudaSuccess) return e;
  if ((e = encode_store_32x32(&o_dw, a.dweight, true, a.d, a.V, a.d)) != cudaSuccess) return e;
  if ((e = launch_gemm<DwOp<kDwN>>(a_dw, b_dw, o_dw, p, dev, st)) != cudaSuccess) return e;

  // the dhidden partials, summed beside the dweight kernel
  int64_t blocks = a.N * (a.P + a.C);  // a CTA per row
  if (blocks > 16 * (int64_t)dev.sms) blocks = 16 * (int64_t)dev.sms;
  if (blocks < 1) blocks = 1;
  return launch_pdl(lmhead_dh_reduce_kernel, dim3((unsigned)blocks), dim3(kReduceThreads), 0, st,
                    1, (const float*)partials, geometry, lm_geo_dh(pass), rowmap, tokrow, a.N, a.P,
                    a.C, a.d, p.row0, bl.rows_pass, (int)pass, a.dhidden);
}

}  // namespace grpo

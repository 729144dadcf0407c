// Log-probs of the sampled tokens straight from the policy's last hidden
// states: the LM-head projection logits = H * W^T ("model(...).logits" of
// "compute_logprobs" in "Making Dr GRPO go brrr", salahadawi.com) fused with
// the shifted log-softmax and gather, so the [rows, V] logits never reach
// HBM.  This is a dense contraction, so it runs on the 5th-generation tensor
// cores: tcgen05.mma on CTA pairs (2-SM MMA, M = 256) with operands staged in
// shared memory by TMA and the fp32 accumulator in tensor memory (TMEM).
//
//   gather_rows_kernel   copies the hidden state of every scored row into a
//                        dense [rows, d] buffer (row r = valid token r) and
//                        zeroes the rows up to the next multiple of 256
//                        (and zeroes logp and lse past each length)
//   lmhead_lse_kernel    work items (block of 256 rows, range of vocabulary
//                        tiles of 256) on the pair pipeline (pair_pipeline.cuh):
//                        each CTA loads 128 rows of H and 128 vocabulary rows
//                        of W per 64-wide k-step; the epilogue folds each
//                        finished 256-column tile of its 128 rows into a
//                        running (max, sum of exp) and the target logit.  Each
//                        item writes one partial per row and counts it; the
//                        thread that writes a row's last partial merges the
//                        row's partials in split order (deterministic) into lse
//                        and logp = z_y - lse.
//
// The backward ("loss.backward()" through the projection) recomputes the
// logits with the same pipeline: lmhead_dz_kernel's epilogue turns each tile
// into the logits gradient g * w_t * (onehot(y_t) - exp(z - lse_t)), rounded
// to bf16, and stores it by TMA, in 64-column vocabulary slabs, for the two
// gradient contractions (lmhead_bwd.cu).
#include <mutex>

#include "host_ctx.cuh"
#include "pair_pipeline.cuh"
#include "lmhead.cuh"

namespace grpo {
namespace {

constexpr int kRows = 256;        // rows per pair tile (128 per CTA)
constexpr int kVTile = 256;       // vocabulary columns per tile
constexpr int kK = 64;            // k per stage: one 128-byte swizzle atom of bf16
constexpr int kMaxSplits = 256;   // = kThreads: one candidate per thread
constexpr uint32_t kIdescLm = umma_idesc(256, kVTile, false, false);
constexpr int kLmSmem = kPairRingBytes + 1024;
constexpr int kDzSmem = kLmSmem + 8 * 4096;  // + two 2 KiB TMA-store boxes per epilogue warp

struct LmParams {
  int64_t N, P, C, V, d;
  const int32_t* offsets;  // prefix sums of the clamped lengths ([N+1])
  int4* geometry;          // [geo_index] (row blocks, splits, tiles per split): by the gather
  int geo_index;           // forward: 0; backward pass p: 3 + 2p
  int64_t row0;            // backward: the pass's first row (forward: 0)
  int64_t rows_pass;       // backward: rows per pass
  float4* partials;        // forward: [items][256] (max, sum, target logit, has target)
  uint32_t* counters;      // forward: partials written per row (zeroed by the gather)
  float* logp_out;         // forward: [N, C]
  float* lse_out;          // forward: [N, C]
  WsHeader* hdr;
  // logits-gradient pass only
  const float* lse;        // [N, C] from the forward
  const float* w;          // [N, C] d loss / d logp from the forward
  const float* grad;       // upstream scalar gradient (nullable: 1)
  const int32_t* rowmap;   // the token i*C + t of each backward row (geometry[2].x rows)
};

// Backward rows of pass `pass` out of `rows` in passes of `rows_pass`.
__device__ __forceinline__ int64_t pass_rows(int64_t rows, int64_t row0, int64_t rows_pass) {
  return rows <= row0 ? 0 : (rows - row0 < rows_pass ? rows - row0 : rows_pass);
}

// Split `ksteps` steps of work for each of `units` independent tiles into
// `splits` ranges so that the items (unit, range) fill the grid's rounds,
// counting both the items per round and the uneven last range; every range
// is non-empty and items <= max_items.  Candidate split counts 1 .. 256, one
// per thread of the calling CTA (kThreads threads); the smallest within 0.01
// of the best score wins (fewer partials to merge, and every range re-reads
// its unit's operand).  Returns (splits, steps per split).
__device__ float split_score(int32_t units, int32_t sp, int32_t ksteps, int slots,
                             int32_t max_items) {
  const int32_t items = units * sp;
  if (sp > ksteps || items > max_items) return -1.f;
  const int32_t sps = (ksteps + sp - 1) / sp;
  if ((int64_t)sps * (sp - 1) >= ksteps) return -1.f;  // the last range would be empty
  const int32_t rounds = (items + slots - 1) / slots;
  return (float)items / (float)(rounds * slots) * (float)ksteps / (float)(sps * sp);
}

__device__ int2 choose_split_block(int32_t units, int32_t ksteps, int slots, int32_t max_items) {
  __shared__ float s_best[kWarps];
  __shared__ int s_pick[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t sp = tid + 1;
  const float score =
      units > 0 ? split_score(units, sp, ksteps, slots, max_items) : (sp == 1 ? 1.f : -1.f);
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

// geometry[0]: the projection pass (256-row blocks, vocabulary splits, tiles
// per split, 0).  `pairs`: CTA pairs of the tensor-core kernels.
__global__ void __launch_bounds__(kThreads) gather_rows_kernel(const uint16_t* __restrict__ hidden,
                                                               uint16_t* __restrict__ dense,
                                                               const int32_t* __restrict__ off,
                                                               int64_t N, int64_t T, int64_t P,
                                                               int64_t d, int64_t V, int pairs,
                                                               int4* __restrict__ geometry,
                                                               uint32_t* __restrict__ counters,
                                                               float* __restrict__ logp,
                                                               float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  const int64_t tv = off[N];
  const int32_t mb = (int32_t)((tv + kRows - 1) / kRows);
  if (blockIdx.x == 0) {
    const int32_t ntiles = (int32_t)((V + kVTile - 1) / kVTile);
    const int2 s = choose_split_block(mb, ntiles, pairs, 4 * pairs + 2 * mb);
    if (threadIdx.x == 0) geometry[0] = make_int4(mb, s.x, s.y, 0);
  }
  const int64_t vec_per_row = d / 8;  // 16-byte vectors
  const int64_t rows_pad = (int64_t)mb * kRows;
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
  // the log-sum-exp kernel counts each row's partials from 0; positions past
  // each length are 0 in logp and lse
  const int64_t C = T - P;
  for (int64_t k = (int64_t)blockIdx.x * kThreads + threadIdx.x; k < N * C;
       k += (int64_t)gridDim.x * kThreads) {
    if (k < rows_pad) counters[k] = 0u;
    const int64_t i = k / C;
    if (k - i * C >= off[i + 1] - off[i]) {
      logp[k] = 0.f;
      lse[k] = 0.f;
    }
  }
  for (int64_t k = N * C + (int64_t)blockIdx.x * kThreads + threadIdx.x; k < rows_pad;
       k += (int64_t)gridDim.x * kThreads)
    counters[k] = 0u;
}

// ---- backward rows ------------------------------------------------------------------

// The backward's rows: the scored tokens (t < len_i) in token order, or with
// `skip` only those whose g * w is not exactly 0 (they contribute nothing to
// either gradient).  One CTA: each thread takes a contiguous run of tokens,
// counts its rows, and a block-wide exclusive scan of the counts places them:
// rowmap[row] = i * C + t, tokrow[i * C + t] = row or -1; geometry[2].x = rows.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
    active_rows_kernel(const int32_t* __restrict__ lens, const float* __restrict__ w,
                       const float* __restrict__ grad, int64_t N, int64_t C, int skip,
                       int32_t* __restrict__ rowmap, int32_t* __restrict__ tokrow,
                       int4* __restrict__ geometry) {
  __shared__ int32_t s_warp[kScanThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t NC = N * C;
  const float g = grad != nullptr ? __ldg(grad) : 1.f;
  const int64_t per = (NC + kScanThreads - 1) / kScanThreads;
  const int64_t k0 = min(NC, (int64_t)tid * per), k1 = min(NC, k0 + per);
  auto active = [&](int64_t k) {
    const int64_t i = k / C, t = k - i * C;
    return t < lens[i] && (!skip || g * w[k] != 0.f);
  };
  int32_t cnt = 0;
  for (int64_t k = k0; k < k1; ++k) cnt += active(k) ? 1 : 0;
  // block-wide exclusive scan of cnt
  int32_t x = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t v = s_warp[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    s_warp[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  int32_t row = x - cnt + (warp > 0 ? s_warp[warp - 1] : 0);
  for (int64_t k = k0; k < k1; ++k) {
    if (active(k)) {
      rowmap[row] = (int32_t)k;
      tokrow[k] = row++;
    } else {
      tokrow[k] = -1;
    }
  }
  if (tid == kScanThreads - 1) geometry[2] = make_int4(row, 0, 0, 0);
}

// Dense copy of the backward rows' hidden states (zero rows up to the next
// multiple of 256) and, for every pass of rows_pass rows, the geometries of
// the projection pass (geometry[3 + 2p]: 256-row blocks, vocabulary splits,
// tiles per split) and of the hidden-state gradient contraction
// (geometry[4 + 2p]: 256-row blocks, 512-wide d tiles, vocabulary splits,
// 64-wide k-steps per split).
__global__ void __launch_bounds__(kThreads)
    gather_active_rows_kernel(const uint16_t* __restrict__ hidden, uint16_t* __restrict__ dense,
                              const int32_t* __restrict__ rowmap, int64_t C, int64_t T, int64_t P,
                              int64_t d, int64_t V, int pairs, int64_t rows_pass, int64_t npass,
                              int4* __restrict__ geometry) {
  pdl_wait();
  pdl_trigger();
  const int64_t rows = geometry[2].x;
  const int32_t mb = (int32_t)((rows + kRows - 1) / kRows);
  for (int64_t pass = blockIdx.x; pass < npass; pass += gridDim.x) {  // uniform per CTA
    const int64_t rp = pass_rows(rows, pass * rows_pass, rows_pass);
    const int32_t mbp = (int32_t)((rp + kRows - 1) / kRows);
    const int32_t ntiles = (int32_t)((V + kVTile - 1) / kVTile);
    const int2 s0 = choose_split_block(mbp, ntiles, pairs, 4 * pairs + 2 * mbp);
    const int32_t nb = (int32_t)((d + 511) / 512);
    const int32_t ksteps = ntiles * (kVTile / kK);
    const int2 s1 = choose_split_block(mbp * nb, ksteps, pairs, 2 * pairs + mbp * nb);
    if (threadIdx.x == 0) {
      geometry[3 + 2 * pass] = make_int4(mbp, s0.x, s0.y, 0);
      geometry[4 + 2 * pass] = make_int4(mbp, nb, s1.x, s1.y);
    }
  }
  const int64_t vec_per_row = d / 8;  // 16-byte vectors
  const int64_t rows_pad = (int64_t)mb * kRows;
  for (int64_t k = (int64_t)blockIdx.x * kThreads + threadIdx.x; k < rows_pad * vec_per_row;
       k += (int64_t)gridDim.x * kThreads) {
    const int64_t r = k / vec_per_row, c = k - r * vec_per_row;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) {
      const int64_t tok = rowmap[r], i = tok / C, t = tok - i * C;
      const uint4* src =
          reinterpret_cast<const uint4*>(hidden + (i * T + P - 1 + t) * d);
      v = ld_stream(src + c);
    }
    reinterpret_cast<uint4*>(dense + r * d)[c] = v;
  }
}

// ---- the projection on the pair pipeline -------------------------------------------

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

// Items (256-row block, range of vocabulary tiles); a tile is 256 rows x 256
// vocabulary columns reduced over d.  kMode 0: log-sum-exp partials per row;
// kMode 1: the bf16 logits gradient, stored by TMA.
template <int kMode>
struct LmOp {
  static constexpr int kStages = kPairStages;
  static constexpr int kStageBytes = kPairStageBytes;
  static constexpr int kAccCols = 256;
  // the gradient epilogue (exp, scale, round, store per element) is the heavier
  // one: two warps per TMEM lane quarter, 128 columns each
  static constexpr int kEpiWarps = kMode == 1 ? 8 : 4;
  const LmParams& p;
  const CUtensorMap* map_h;
  const CUtensorMap* map_w;
  const CUtensorMap* map_dz;
  const int64_t* ids;
  uint32_t rank, stg;
  int64_t tv, mb, splits, tps, ntiles;
  int kblocks;
  // epilogue state of this thread's row
  int64_t r, y;
  float lse_r, coef, g, m, s_extra, zy;
  uint64_t acc01, acc23;
  int64_t tok;  // forward: the token i*C + t of this thread's row (-1: a padding row)
  bool has;
  uint32_t chunk;

  __device__ void setup() {
    tv = kMode == 1 ? pass_rows(p.geometry[2].x, p.row0, p.rows_pass)  // rows of the pass
                    : (int64_t)p.offsets[p.N];
    const int4 geo = p.geometry[p.geo_index];
    mb = geo.x;
    splits = geo.y;
    tps = geo.z;
    ntiles = (p.V + kVTile - 1) / kVTile;
    kblocks = (int)(p.d / kK);
    g = (kMode == 1 && p.grad != nullptr) ? __ldg(p.grad) : 1.f;
    chunk = 0;
  }
  // item it = (row block, vocabulary split), decoded once per item by each
  // role's thread (the producer asks at every k-step, where 64-bit divisions
  // on every call would hold up the issue)
  mutable int64_t c_it = -1, c_rb = 0, c_n0 = 0;
  __device__ void decode(int64_t it) const {
    if (it != c_it) {
      c_it = it;
      c_rb = it / splits;
      c_n0 = (it - c_rb * splits) * tps;
    }
  }
  __device__ int64_t items() const { return mb * splits; }
  __device__ int64_t first_tile(int64_t it) const {
    decode(it);
    return c_n0;
  }
  __device__ int tiles(int64_t it) const {
    const int64_t n0 = first_tile(it);
    return (int)(min(ntiles, n0 + tps) - n0);
  }
  __device__ void krange(int64_t, int, int64_t* k0, int64_t* k1) const {
    *k0 = 0;
    *k1 = kblocks;
  }
  __device__ uint32_t bytes(int64_t, int) const { return kPairStageBytes; }
  __device__ void load(uint32_t sa, int64_t it, int t, int64_t ks, uint32_t rk,
                       uint32_t mbar) const {
    decode(it);
    const int64_t rb = c_rb, n = c_n0 + t;
    tma_load_2d_pair(sa, map_h, (int)(ks * kK), (int)(p.row0 + rb * kRows + rk * 128), mbar);
    tma_load_2d_pair(sa + kPairBOffset, map_w, (int)(ks * kK), (int)(n * kVTile + rk * 128),
                     mbar);
  }
  __device__ void mma(uint32_t dacc, uint32_t sa, int64_t, int, bool first) const {
#pragma unroll
    for (int j = 0; j < kK / 16; ++j)
      umma_bf16_pair(dacc, umma_desc_k(sa + j * 32), umma_desc_k(sa + kPairBOffset + j * 32),
                     kIdescLm, (first && j == 0) ? 0u : 1u);
  }

  __device__ void epi_begin(int64_t it) {
    const int lane = threadIdx.x & 31, quarter = (threadIdx.x >> 5) & 3;
    r = (it / splits) * kRows + rank * 128 + quarter * 32 + lane;
    y = -1;
    tok = -1;
    lse_r = 0.f;
    coef = 0.f;
    if (r < tv) {
      int64_t i, t;
      if (kMode == 1) {  // the backward's rows: the row map
        const int64_t tok = p.rowmap[p.row0 + r];
        i = tok / p.C;
        t = tok - i * p.C;
      } else {           // every scored token, in order
        i = completion_of(p.offsets, p.N, r);
        t = r - p.offsets[i];
      }
      y = __ldg(ids + i * (p.P + p.C) + p.P + t);
      tok = i * p.C + t;
      if (kMode == 1) {
        lse_r = __ldg(p.lse + i * p.C + t);
        coef = g * __ldg(p.w + i * p.C + t);
      }
    }
    m = -INFINITY;
    s_extra = 0.f;
    zy = 0.f;
    acc01 = f2_pack(0.f, 0.f);
    acc23 = f2_pack(0.f, 0.f);
    has = false;
  }

  __device__ void epi_tile(int64_t it, int t, uint32_t tbase, bool, int slice) {
    const int lane = threadIdx.x & 31, quarter = (threadIdx.x >> 5) & 3;
    const uint64_t L2 = f2_pack(kLog2e, kLog2e);
    const int64_t vbase = (first_tile(it) + t) * kVTile;
    constexpr int kCols = kVTile * 4 / kEpiWarps;  // this warp's columns of the tile
#pragma unroll 1
    for (int c = slice * kCols; c < (slice + 1) * kCols; c += 32) {
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
        // row `lane` of this warp's 32 x 32 box; 16-byte chunk q sits at q ^ ((lane >> 1) & 3)
        const uint32_t box = stg + (chunk & 1u) * 2048u;
        if (lane == 0) bulk_wait_read<1>();  // the store that last used this box has read it
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared_v4(box + (uint32_t)lane * 64u + ((uint32_t)(q ^ ((lane >> 1) & 3)) << 4),
                       pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(map_dz, box, (int)(v0 & 63),
                       (int)((it / splits) * kRows + rank * 128 + quarter * 32), (int)(v0 >> 6));
          bulk_commit();
        }
        ++chunk;
      }
    }
  }

  __device__ void epi_end(int64_t it) {
    if constexpr (kMode == 0) {
      const int lane = threadIdx.x & 31, quarter = (threadIdx.x >> 5) & 3;
      float a0, a1, a2, a3;
      f2_unpack(acc01, a0, a1);
      f2_unpack(acc23, a2, a3);
      const float s = ((a0 + a1) + (a2 + a3)) + s_extra;
      if (r < tv) {
        const int64_t rr = rank * 128 + quarter * 32 + lane;  // the row within its block
        p.partials[it * kRows + rr] = make_float4(m, s, zy, has ? 1.f : 0.f);
        // The thread that writes a row's last partial merges the row: every
        // writer makes its partial visible before counting it, the last one
        // sees every count and so every partial.
        __threadfence();
        if (atomicAdd(p.counters + r, 1u) == (uint32_t)(splits - 1)) {
          __threadfence();
          merge_row(it / splits, rr);
        }
      }
    }
  }
  // Partials of row (block rb, row rr) in split order -> lse, logp.
  __device__ void merge_row(int64_t rb, int64_t rr) const {
    float4 pk = __ldcg(p.partials + (rb * splits) * kRows + rr);
    float cm = pk.x, cs = pk.y, z = pk.z;
    bool found = pk.w != 0.f;
    for (int64_t sp = 1; sp < splits; ++sp) {
      pk = __ldcg(p.partials + (rb * splits + sp) * kRows + rr);
      lse_merge(cm, cs, pk.x, pk.y);
      if (pk.w != 0.f) {
        z = pk.z;
        found = true;
      }
    }
    const float l = cm + logf(cs);
    if (found) {
      p.logp_out[tok] = z - l;
      p.lse_out[tok] = l;
    } else {  // the sampled id is outside [0, V)
      p.logp_out[tok] = __int_as_float(0x7fc00000);
      p.lse_out[tok] = __int_as_float(0x7fc00000);
      atomicOr(&p.hdr->flags, kFlagTokenRange);
    }
  }
  __device__ void epi_finish() {
    if (kMode == 1 && (threadIdx.x & 31) == 0) bulk_wait<0>();  // the gradient stores are done
  }
};

template <int kMode>
__device__ __forceinline__ void lm_kernel_body(const CUtensorMap* map_h, const CUtensorMap* map_w,
                                               const CUtensorMap* map_dz, const int64_t* ids,
                                               const LmParams& p) {
  extern __shared__ __align__(1024) unsigned char lm_smem[];
  const uint32_t ring = smem_u32(lm_smem + ((1024 - (smem_u32(lm_smem) & 1023)) & 1023));
  LmOp<kMode> op{p, map_h, map_w, map_dz, ids};
  op.rank = cluster_rank();
  op.stg = ring + kPairRingBytes + (uint32_t)((threadIdx.x >> 5) - 2) * 4096u;  // epilogue warps
  pair_pipeline(op, ring, p.hdr);
}

__global__ void __launch_bounds__(kPairThreads, 1)
    lmhead_lse_kernel(const __grid_constant__ CUtensorMap map_h,
                      const __grid_constant__ CUtensorMap map_w, const int64_t* __restrict__ ids,
                      const LmParams p) {
  lm_kernel_body<0>(&map_h, &map_w, nullptr, ids, p);
}

__global__ void __launch_bounds__(64 + 32 * LmOp<1>::kEpiWarps, 1)
    lmhead_dz_kernel(const __grid_constant__ CUtensorMap map_h,
                     const __grid_constant__ CUtensorMap map_w,
                     const __grid_constant__ CUtensorMap map_dz, const int64_t* __restrict__ ids,
                     const LmParams p) {
  lm_kernel_body<1>(&map_h, &map_w, &map_dz, ids, p);
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
                   int64_t C, int64_t V, int64_t d) {
  LmParams p = {};
  p.N = N;
  p.P = P;
  p.C = C;
  p.V = V;
  p.d = d;
  p.offsets = off;
  p.geometry = geometry;
  p.geo_index = 0;
  p.row0 = 0;
  p.rows_pass = INT64_MAX;
  p.hdr = hdr;
  return p;
}

}  // namespace

int lm_pairs(const DeviceInfo& dev) { return dev.sms / 2 > 0 ? dev.sms / 2 : 1; }

cudaError_t encode_bf16_2d(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                           int64_t pitch, int box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encoder(&enc);
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)pitch * 2};
  cuuint32_t box[2] = {(cuuint32_t)kK, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_store_32x32(CUtensorMap* map, void* base, bool fp32, int64_t inner,
                               int64_t outer, int64_t pitch) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encoder(&enc);
  if (e != cudaSuccess) return e;
  const int64_t es = fp32 ? 4 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)(pitch * es)};
  cuuint32_t box[2] = {32u, 32u};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   fp32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_dz_slabs(CUtensorMap* map, void* base, int64_t rows, int64_t ldz, int box_rows,
                            bool store) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encoder(&enc);
  if (e != cudaSuccess) return e;
  cuuint64_t dims[3] = {64u, (cuuint64_t)rows, (cuuint64_t)(ldz / 64)};
  cuuint64_t strides[2] = {128u, (cuuint64_t)rows * 128u};
  cuuint32_t box[3] = {store ? 32u : 64u, store ? 32u : (cuuint32_t)box_rows, 1u};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   store ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                   store ? CU_TENSOR_MAP_L2_PROMOTION_NONE : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

LmLayout lm_layout(int64_t N, int64_t C, int64_t d, int sms) {
  LmLayout l;
  const WsLayout base = ws_layout(N);
  const int64_t mb_max = (N * C + kRows - 1) / kRows;
  const int64_t pairs = sms / 2 > 0 ? sms / 2 : 1;
  l.geometry = base.total;  // 2 x int4
  l.dense = align_up(base.total + 32, 1024);
  l.partials = align_up(l.dense + (size_t)(mb_max * kRows) * (size_t)d * 2, 256);
  const int64_t items_max = 4 * pairs + 2 * mb_max;  // mb * splits bound
  l.counters = align_up(l.partials + (size_t)items_max * kRows * sizeof(float4), 256);
  l.total = align_up(l.counters + (size_t)(mb_max * kRows) * sizeof(uint32_t), 256);
  return l;
}

LmBwdLayout lm_bwd_layout(int64_t N, int64_t C, int64_t V, int64_t d, int sms,
                          int64_t rows_pass) {
  LmBwdLayout l;
  const WsLayout base = ws_layout(N);
  const int64_t mb_max = (N * C + kRows - 1) / kRows;
  const int64_t pairs = sms / 2 > 0 ? sms / 2 : 1;
  l.rows_cap = mb_max * kRows;
  l.rows_pass = rows_pass <= 0 ? l.rows_cap : (rows_pass + kRows - 1) / kRows * kRows;
  if (l.rows_pass > l.rows_cap) l.rows_pass = l.rows_cap;
  l.npass = l.rows_pass > 0 ? (l.rows_cap + l.rows_pass - 1) / l.rows_pass : 1;
  if (l.npass < 1) l.npass = 1;
  l.ldz = (V + kVTile - 1) / kVTile * kVTile;
  const int64_t nb = (d + 511) / 512;  // d tiles of the hidden-state gradient
  l.items_max = 2 * pairs + (l.rows_pass / kRows) * nb;
  l.geometry = base.total;
  l.rowmap = align_up(base.total + sizeof(int4) * (size_t)(3 + 2 * l.npass), 256);
  l.tokrow = align_up(l.rowmap + sizeof(int32_t) * (size_t)(N * C), 256);
  l.dense = align_up(l.tokrow + sizeof(int32_t) * (size_t)(N * C), 1024);
  l.dz = align_up(l.dense + (size_t)l.rows_cap * (size_t)d * 2, 1024);
  l.dh_partials = align_up(l.dz + (size_t)l.rows_pass * (size_t)l.ldz * 2, 1024);
  l.total = align_up(l.dh_partials + (size_t)l.items_max * kRows * 512 * sizeof(float), 256);
  return l;
}

cudaError_t launch_lmhead(const void* hidden, const void* weight, const FwdArgs& a, int64_t d,
                          const DeviceInfo& dev, cudaStream_t st) {
  const WsLayout wl = ws_layout(a.N);
  const LmLayout ll = lm_layout(a.N, a.C, d, dev.sms);
  char* ws = static_cast<char*>(a.ws);
  const int32_t* off = reinterpret_cast<const int32_t*>(ws + wl.offsets);
  uint16_t* dense = reinterpret_cast<uint16_t*>(ws + ll.dense);
  const int64_t rows = (a.N * a.C + kRows - 1) / kRows * kRows;
  const int pairs = lm_pairs(dev);

  int4* geometry = reinterpret_cast<int4*>(ws + ll.geometry);
  uint32_t* counters = reinterpret_cast<uint32_t*>(ws + ll.counters);
  cudaError_t e = launch_pdl(gather_rows_kernel, dim3((unsigned)(dev.sms * 8)), dim3(kThreads), 0,
                             st, 1, static_cast<const uint16_t*>(hidden), dense, off, a.N,
                             a.P + a.C, a.P, d, a.V, pairs, geometry, counters, a.logp, a.lse);
  if (e != cudaSuccess) return e;

  LmParams p = lm_params(off, geometry, reinterpret_cast<WsHeader*>(ws), a.N, a.P, a.C, a.V, d);
  p.partials = reinterpret_cast<float4*>(ws + ll.partials);
  p.counters = counters;
  p.logp_out = a.logp;
  p.lse_out = a.lse;
  CUtensorMap map_h, map_w;
  if ((e = encode_bf16_2d(&map_h, dense, d, rows, d, 128)) != cudaSuccess) return e;
  if ((e = encode_bf16_2d(&map_w, weight, d, a.V, d, 128)) != cudaSuccess) return e;
  if ((e = ensure_dynamic_smem((const void*)lmhead_lse_kernel, kLmSmem)) != cudaSuccess) return e;
  return launch_pdl(lmhead_lse_kernel, dim3((unsigned)(2 * pairs)), dim3(kPairThreads),
                    (size_t)kLmSmem, st, 2, map_h, map_w, a.ids, p);
}

cudaError_t launch_lmhead_bwd_rows(const LmBwdArgs& a, const DeviceInfo& dev, cudaStream_t st) {
  const WsLayout wl = ws_layout(a.N);
  const LmBwdLayout bl = lm_bwd_layout(a.N, a.C, a.V, a.d, dev.sms, a.rows_pass);
  char* ws = static_cast<char*>(a.ws);
  const int32_t* lens = reinterpret_cast<const int32_t*>(ws + wl.lens);
  int32_t* rowmap = reinterpret_cast<int32_t*>(ws + bl.rowmap);
  int32_t* tokrow = reinterpret_cast<int32_t*>(ws + bl.tokrow);
  uint16_t* dense = reinterpret_cast<uint16_t*>(ws + bl.dense);
  int4* geometry = reinterpret_cast<int4*>(ws + bl.geometry);
  const int pairs = lm_pairs(dev);
  cudaError_t e = launch_pdl(active_rows_kernel, dim3(1), dim3(kScanThreads), 0, st, 1, lens, a.w,
                             a.grad, a.N, a.C, a.skip_zero_weight ? 1 : 0, rowmap, tokrow,
                             geometry);
  if (e != cudaSuccess) return e;
  return launch_pdl(gather_active_rows_kernel, dim3((unsigned)(dev.sms * 8)), dim3(kThreads), 0,
                    st, 1, static_cast<const uint16_t*>(a.hidden), dense, (const int32_t*)rowmap,
                    a.C, a.P + a.C, a.P, a.d, a.V, pairs, bl.rows_pass, bl.npass, geometry);
}

cudaError_t launch_lmhead_dz(const LmBwdArgs& a, int64_t pass, const DeviceInfo& dev,
                             cudaStream_t st) {
  const WsLayout wl = ws_layout(a.N);
  const LmBwdLayout bl = lm_bwd_layout(a.N, a.C, a.V, a.d, dev.sms, a.rows_pass);
  char* ws = static_cast<char*>(a.ws);
  const int32_t* off = reinterpret_cast<const int32_t*>(ws + wl.offsets);
  const int32_t* rowmap = reinterpret_cast<const int32_t*>(ws + bl.rowmap);
  uint16_t* dense = reinterpret_cast<uint16_t*>(ws + bl.dense);
  int4* geometry = reinterpret_cast<int4*>(ws + bl.geometry);
  const int pairs = lm_pairs(dev);
  LmParams p = lm_params(off, geometry, reinterpret_cast<WsHeader*>(ws), a.N, a.P, a.C, a.V, a.d);
  p.geo_index = lm_geo_proj(pass);
  p.row0 = pass * bl.rows_pass;
  p.rows_pass = bl.rows_pass;
  p.lse = a.lse;
  p.w = a.w;
  p.grad = a.grad;
  p.rowmap = rowmap;
  uint16_t* dz = reinterpret_cast<uint16_t*>(ws + bl.dz);
  CUtensorMap map_h, map_w, map_dz;
  cudaError_t e;
  if ((e = encode_bf16_2d(&map_h, dense, a.d, bl.rows_cap, a.d, 128)) != cudaSuccess) return e;
  if ((e = encode_bf16_2d(&map_w, a.weight, a.d, a.V, a.d, 128)) != cudaSuccess) return e;
  if ((e = encode_dz_slabs(&map_dz, dz, bl.rows_pass, bl.ldz, 32, true)) != cudaSuccess) return e;
  if ((e = ensure_dynamic_smem((const void*)lmhead_dz_kernel, kDzSmem)) != cudaSuccess) return e;
  return launch_pdl(lmhead_dz_kernel, dim3((unsigned)(2 * pairs)),
                    dim3(64 + 32 * LmOp<1>::kEpiWarps), (size_t)kDzSmem, st, 2, map_h, map_w,
                    map_dz, a.ids, p);
}

}  // namespace grpo

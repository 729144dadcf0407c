// Gradients of the Dr. GRPO loss through the LM-head projection z = h W^T
// ("loss.backward()" over "model(...).logits" in "Making Dr GRPO go brrr",
// salahadawi.com; the page prints no gradient, this is the chain rule).  With
// dz the bf16 logits gradient of the scored rows (lmhead_dz_kernel):
//
//   dhidden[row] = dz[row] W        (rows x V) (V x d): K = vocabulary
//   dweight      = dz^T H_scored    (V x rows) (rows x d): K = scored rows
//
// Both are dense contractions on the tcgen05 tensor cores with the fp32
// accumulator in TMEM.  The operands are read in their natural row-major
// layouts: W [V, d], the dense scored hidden rows [rows, d] and dz
// [rows, ldz] enter as MN-major (transposed) shared-memory operands where the
// contraction runs over their row index, so nothing is transposed in memory.
//
// lmhead_grad_gemm_kernel<false>  dhidden partials: items (128 rows, 256
//     columns of d, range of vocabulary k-steps), fp32 tiles in the workspace
// lmhead_dh_reduce_kernel         sums a row's partials in split order
//     (deterministic) into dhidden [N, P+C, d]; rows that score nothing get 0
// lmhead_grad_gemm_kernel<true>   dweight: items (128 vocabulary rows, 256
//     columns of d), K = every scored row, fp32 straight to dweight [V, d]
//
// Warp roles as in the projection kernel: warp 0 TMA, warp 1 MMA, warps 2-5
// drain TMEM through a shared-memory transpose into coalesced 16-byte stores.
#include "tc.cuh"

namespace grpo {
namespace {

constexpr int kGM = 128;                  // output rows per tile (TMEM lanes)
constexpr int kGN = 256;                  // output columns per tile (the last d tile may be narrower)
constexpr int kGK = 64;                   // k per stage
constexpr int kGStages = 4;
constexpr int kGABytes = kGM * kGK * 2;   // 16 KiB
constexpr int kGBBytes = kGN * kGK * 2;   // 32 KiB (at the full tile width)
constexpr int kGStageBytes = kGABytes + kGBBytes;
constexpr int kGThreads = 192;
constexpr uint32_t kMnAtomStride = 8192;  // 64 M/N elements x 64 K rows x 2 bytes (one TMA box)
constexpr int kStagePitch = 36;           // floats per staged row: 16-byte aligned, no bank conflicts
constexpr int kEpiFloats = 4 * 32 * kStagePitch;
constexpr int kGSmem = kGStages * kGStageBytes + kEpiFloats * 4 + 1024;
constexpr int kTileFloats = kGM * kGN;

struct GradParams {
  int64_t N, V, d;
  const int32_t* offsets;  // [N+1]: offsets[N] = scored rows
  const int4* geometry;    // [1]: (row blocks, d tiles, splits, k-steps per split)
  int64_t ksteps_v;        // vocabulary k-steps of the hidden-state gradient (ldz / 64)
  float* out;              // <false>: partial tiles [items][128][256]; <true>: dweight [V, d]
  WsHeader* hdr;
};

struct GradItem {
  int64_t m_tile, n_tile, k0, k1;
};

template <bool kDW>
__device__ __forceinline__ GradItem grad_item(int64_t it, int64_t nb, int64_t splits, int64_t sps,
                                              int64_t ksteps) {
  GradItem g;
  if (kDW) {
    g.m_tile = it / nb;
    g.n_tile = it - g.m_tile * nb;
    g.k0 = 0;
    g.k1 = ksteps;
  } else {
    const int64_t s = it % splits, t = it / splits;
    g.n_tile = t % nb;
    g.m_tile = t / nb;
    g.k0 = s * sps;
    g.k1 = min(ksteps, g.k0 + sps);
  }
  return g;
}

template <bool kDW>
__global__ void __launch_bounds__(kGThreads, 1)
    lmhead_grad_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                            const __grid_constant__ CUtensorMap map_b, const GradParams p) {
  extern __shared__ __align__(1024) unsigned char g_smem[];
  __shared__ __align__(8) uint64_t s_full[kGStages];
  __shared__ __align__(8) uint64_t s_empty[kGStages];
  __shared__ __align__(8) uint64_t s_acc_full[2];
  __shared__ __align__(8) uint64_t s_acc_empty[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* ring = g_smem + ((1024 - (smem_u32(g_smem) & 1023)) & 1023);
  const uint32_t ring_u32 = smem_u32(ring);
  float* staging = reinterpret_cast<float*>(ring + kGStages * kGStageBytes);

  if (tid == 0) {
    s_abort = 0;
    for (int k = 0; k < kGStages; ++k) {
      mbar_init(smem_u32(&s_full[k]), 1);
      mbar_init(smem_u32(&s_empty[k]), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&s_acc_full[k]), 1);
      mbar_init(smem_u32(&s_acc_empty[k]), 4);
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
  const int64_t nb = (p.d + kGN - 1) / kGN;
  int64_t items, splits = 1, sps, ksteps;
  if (kDW) {
    ksteps = (tv + kGK - 1) / kGK;  // rows past tv are zero in both operands
    sps = ksteps;
    items = (p.V + kGM - 1) / kGM * nb;
  } else {
    const int4 g = p.geometry[1];
    splits = g.z;
    sps = g.w;
    ksteps = p.ksteps_v;
    items = (int64_t)g.x * g.y * splits;
  }

  if (warp == 0) {
    // ---------------- TMA producer -----------------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int64_t it = blockIdx.x; it < items && !*(volatile int*)&s_abort; it += gridDim.x) {
        const GradItem gi = grad_item<kDW>(it, nb, splits, sps, ksteps);
        const int nw = (int)min((int64_t)kGN, p.d - gi.n_tile * kGN);
        const uint32_t bytes = (uint32_t)(kGABytes + nw * kGK * 2);
        for (int64_t ks = gi.k0; ks < gi.k1; ++ks) {
          if (!mbar_wait(smem_u32(&s_empty[stage]), phase ^ 1u)) {
            atomicOr(&p.hdr->flags, kFlagTimeout);
            *(volatile int*)&s_abort = 1;
            break;
          }
          const uint32_t full = smem_u32(&s_full[stage]);
          const uint32_t sa = ring_u32 + stage * kGStageBytes;
          mbar_arrive_expect_tx(full, bytes);
          if (kDW) {  // dz^T: two {64 vocabulary, 64 rows} boxes (MN-major A)
            tma_load_2d(sa, &map_a, (int)(gi.m_tile * kGM), (int)(ks * kGK), full);
            tma_load_2d(sa + kMnAtomStride, &map_a, (int)(gi.m_tile * kGM + 64), (int)(ks * kGK),
                        full);
          } else {    // dz: one {64 vocabulary, 128 rows} box (K-major A)
            tma_load_2d(sa, &map_a, (int)(ks * kGK), (int)(gi.m_tile * kGM), full);
          }
          for (int j = 0; j < nw / 64; ++j)  // B: {64 of d, 64 k rows} boxes (MN-major)
            tma_load_2d(sa + kGABytes + j * kMnAtomStride, &map_b, (int)(gi.n_tile * kGN + 64 * j),
                        (int)(ks * kGK), full);
          if (++stage == kGStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ---------------------------------------------
    if (lane == 0) {
      int stage = 0, buf = 0;
      uint32_t phase = 0, aphase = 0;
      for (int64_t it = blockIdx.x; it < items && !*(volatile int*)&s_abort; it += gridDim.x) {
        const GradItem gi = grad_item<kDW>(it, nb, splits, sps, ksteps);
        const int nw = (int)min((int64_t)kGN, p.d - gi.n_tile * kGN);
        const uint32_t idesc = umma_idesc(kGM, nw, kDW, true);
        if (!mbar_wait(smem_u32(&s_acc_empty[buf]), aphase ^ 1u)) {
          atomicOr(&p.hdr->flags, kFlagTimeout);
          *(volatile int*)&s_abort = 1;
          break;
        }
        tmem_fence_after();
        const uint32_t dacc = tmem + (uint32_t)(buf * kGN);
        bool ok = true;
        for (int64_t ks = gi.k0; ks < gi.k1; ++ks) {
          if (!mbar_wait(smem_u32(&s_full[stage]), phase)) {
            atomicOr(&p.hdr->flags, kFlagTimeout);
            *(volatile int*)&s_abort = 1;
            ok = false;
            break;
          }
          tmem_fence_after();
          const uint32_t sa = ring_u32 + stage * kGStageBytes;
#pragma unroll
          for (int j = 0; j < kGK / 16; ++j) {
            const uint64_t ad = kDW ? umma_desc_mn(sa + j * 2048, kMnAtomStride)
                                    : umma_desc_k(sa + j * 32);
            const uint64_t bd = umma_desc_mn(sa + kGABytes + j * 2048, kMnAtomStride);
            umma_bf16(dacc, ad, bd, idesc, (ks > gi.k0 || j > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&s_empty[stage]));
          if (++stage == kGStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&s_acc_full[buf]));  // (no MMAs for an empty range: arrives at once)
        if (++buf == 2) {
          buf = 0;
          aphase ^= 1u;
        }
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5 ------------------------------------
    const int quarter = warp & 3;  // TMEM lanes (tile rows) 32*quarter .. +31
    float* stg = staging + quarter * 32 * kStagePitch;
    const int sub = lane >> 3, c4 = (lane & 7) * 4;
    int buf = 0;
    uint32_t aphase = 0;
    for (int64_t it = blockIdx.x; it < items && !*(volatile int*)&s_abort; it += gridDim.x) {
      const GradItem gi = grad_item<kDW>(it, nb, splits, sps, ksteps);
      const int nw = (int)min((int64_t)kGN, p.d - gi.n_tile * kGN);
      if (!mbar_wait(smem_u32(&s_acc_full[buf]), aphase)) {
        atomicOr(&p.hdr->flags, kFlagTimeout);
        *(volatile int*)&s_abort = 1;
        break;
      }
      tmem_fence_after();
      const bool empty = gi.k1 <= gi.k0;  // nothing accumulated: the tile is zero
      const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * kGN);
      for (int c = 0; c < nw; c += 32) {
        float v[32];
        if (!empty) {
          tmem_ld32(tbase + (uint32_t)c, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        // transpose through shared memory: thread = row -> 8 threads per row segment
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(stg + lane * kStagePitch + 4 * q) =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int row = 4 * k + sub;  // row of this warp's 32
          const float4 x = *reinterpret_cast<const float4*>(stg + row * kStagePitch + c4);
          const int64_t tr = quarter * 32 + row;  // row inside the 128-row tile
          if (kDW) {
            const int64_t v = gi.m_tile * kGM + tr;
            if (v < p.V)
              *reinterpret_cast<float4*>(p.out + v * p.d + gi.n_tile * kGN + c + c4) = x;
          } else {
            *reinterpret_cast<float4*>(p.out + it * kTileFloats + tr * kGN + c + c4) = x;
          }
        }
        __syncwarp();
      }
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_acc_empty[buf]));
      if (++buf == 2) {
        buf = 0;
        aphase ^= 1u;
      }
    }
  }

  tmem_fence_before();
  __syncthreads();
  if (warp == 1) {
    tmem_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dhidden [N, P+C, d]: the scored row (i, P-1+t), t < len_i, is valid token
// r = offsets[i] + t; its value is the sum of its split partials in order.
__global__ void __launch_bounds__(kThreads)
    lmhead_dh_reduce_kernel(const float* __restrict__ partials, const int4* __restrict__ geometry,
                            const int32_t* __restrict__ off, const int32_t* __restrict__ lens,
                            int64_t N, int64_t P, int64_t C, int64_t d, float* __restrict__ dh) {
  pdl_wait();
  pdl_trigger();
  const int4 g = geometry[1];
  const int64_t nb = g.y, splits = g.z;
  const int64_t T = P + C;
  const int64_t total4 = N * T * d / 4;
  for (int64_t e4 = (int64_t)blockIdx.x * kThreads + threadIdx.x; e4 < total4;
       e4 += (int64_t)gridDim.x * kThreads) {
    const int64_t e = e4 * 4;
    const int64_t row_all = e / d, k = e - row_all * d;
    const int64_t i = row_all / T, t = row_all - i * T - (P - 1);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t >= 0 && t < lens[i]) {
      const int64_t r = off[i] + t;
      const int64_t rb = r / kGM, rr = r - rb * kGM;
      const int64_t nt = k / kGN, kk = k - nt * kGN;
      const float* src = partials + ((rb * nb + nt) * splits) * kTileFloats + rr * kGN + kk;
      for (int64_t s = 0; s < splits; ++s) {
        const float4 x = *reinterpret_cast<const float4*>(src + s * kTileFloats);
        acc.x += x.x;
        acc.y += x.y;
        acc.z += x.z;
        acc.w += x.w;
      }
    }
    reinterpret_cast<float4*>(dh)[e4] = acc;
  }
}

template <bool kDW>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const GradParams& p,
                        const DeviceInfo& dev, cudaStream_t st) {
  static bool attr_done = false;
  cudaError_t e;
  if (!attr_done) {
    if ((e = cudaFuncSetAttribute(lmhead_grad_gemm_kernel<kDW>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem)) !=
        cudaSuccess)
      return e;
    attr_done = true;
  }
  return launch_pdl(lmhead_grad_gemm_kernel<kDW>, dim3((unsigned)dev.sms), dim3(kGThreads),
                    (size_t)kGSmem, st, 1, a, b, p);
}

}  // namespace

cudaError_t launch_lmhead_grads(const LmBwdArgs& a, const DeviceInfo& dev, cudaStream_t st) {
  const WsLayout wl = ws_layout(a.N);
  const LmBwdLayout bl = lm_bwd_layout(a.N, a.C, a.V, a.d, dev.sms);
  char* ws = static_cast<char*>(a.ws);
  const int32_t* off = reinterpret_cast<const int32_t*>(ws + wl.offsets);
  const int32_t* lens = reinterpret_cast<const int32_t*>(ws + wl.lens);
  const uint16_t* dz = reinterpret_cast<const uint16_t*>(ws + bl.dz);
  const uint16_t* dense = reinterpret_cast<const uint16_t*>(ws + bl.dense);
  const int4* geometry = reinterpret_cast<const int4*>(ws + bl.geometry);
  float* partials = reinterpret_cast<float*>(ws + bl.dh_partials);

  GradParams p;
  p.N = a.N;
  p.V = a.V;
  p.d = a.d;
  p.offsets = off;
  p.geometry = geometry;
  p.ksteps_v = bl.ldz / kGK;
  p.hdr = reinterpret_cast<WsHeader*>(ws);

  // dhidden = dz W: A = dz (K-major, K = vocabulary), B = W (MN-major)
  CUtensorMap a_dh, b_dh, a_dw, b_dw;
  cudaError_t e;
  if ((e = encode_bf16_2d(&a_dh, dz, bl.ldz, bl.rows_cap, bl.ldz, kGM)) != cudaSuccess) return e;
  if ((e = encode_bf16_2d(&b_dh, a.weight, a.d, a.V, a.d, kGK)) != cudaSuccess) return e;
  p.out = partials;
  if ((e = launch_gemm<false>(a_dh, b_dh, p, dev, st)) != cudaSuccess) return e;
  int64_t blocks = (a.N * (a.P + a.C) * a.d / 4 + kThreads - 1) / kThreads;
  if (blocks > 4 * (int64_t)dev.sms) blocks = 4 * (int64_t)dev.sms;
  if (blocks < 1) blocks = 1;
  if ((e = launch_pdl(lmhead_dh_reduce_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, st, 1,
                      (const float*)partials, geometry, off, lens, a.N, a.P, a.C, a.d,
                      a.dhidden)) != cudaSuccess)
    return e;

  // dweight = dz^T H: A = dz (MN-major, K = scored rows), B = H (MN-major)
  if ((e = encode_bf16_2d(&a_dw, dz, bl.ldz, bl.rows_cap, bl.ldz, kGK)) != cudaSuccess) return e;
  if ((e = encode_bf16_2d(&b_dw, dense, a.d, bl.rows_cap, a.d, kGK)) != cudaSuccess) return e;
  p.out = a.dweight;
  return launch_gemm<true>(a_dw, b_dw, p, dev, st);
}

}  // namespace grpo

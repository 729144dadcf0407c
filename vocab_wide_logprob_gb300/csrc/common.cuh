// Internal header of the GB300 (sm_103a) Dr. GRPO loss library: device
// helpers written as inline PTX, the workspace layout, and the launchers that
// api.cu calls.  Not part of the public ABI (include/grpo.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace grpo {

constexpr int kThreads = 256;  // threads per CTA of the streaming kernels
constexpr int kWarps = kThreads / 32;

// log2(e): exp(x) = 2^(x * log2(e)); the streaming kernels work in base 2 so
// that one FFMA feeds one ex2.approx.
constexpr float kLog2e = 1.4426950408889634f;

// Flag bits the kernels set in the workspace header (read by grpo_check_error).
constexpr uint32_t kFlagTokenRange = 1u;
constexpr uint32_t kFlagLengthRange = 2u;
constexpr uint32_t kFlagTimeout = 4u;

// Workspace: a 256-byte header, then the exclusive prefix sums of the
// clamped lengths (offsets[i] = sum of len[0..i), offsets[N] = number of
// valid tokens), the clamped lengths, and the per-block partial sums of the
// loss reduction.
struct WsHeader {
  uint32_t flags;   // kFlag* bits of the most recent forward call
  uint32_t ticket;  // arrival counter of the loss reduction's last-block step
  uint32_t pad[2];
};
constexpr int kMaxLossBlocks = 1024;

struct WsLayout {
  size_t offsets;   // int32[N + 1]
  size_t lens;      // int32[N]
  size_t partials;  // double[kMaxLossBlocks]
  size_t total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout ws_layout(int64_t N) {
  WsLayout l;
  l.offsets = 256;
  l.lens = align_up(l.offsets + sizeof(int32_t) * (size_t)(N + 1), 256);
  l.partials = align_up(l.lens + sizeof(int32_t) * (size_t)N, 256);
  l.total = align_up(l.partials + sizeof(double) * kMaxLossBlocks, 256);
  return l;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

// 2^x on the SFU (MUFU.EX2); flushes subnormal results to zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte load through the read-only path, not allocated in L1: every logits
// byte is read once per kernel.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// 16-byte streaming store (evict-first): dlogits is written once, not re-read.
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// bfloat16 -> float: the 16 stored bits are the high half of a binary32.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf16_bits_to_float(uint16_t u) {
  return __uint_as_float((uint32_t)u << 16);
}

// Two floats -> packed bfloat16x2 (round to nearest even), `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t u) {
  __nv_bfloat162 h;
  memcpy(&h, &u, sizeof h);
  return h;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// All threads of all CTAs of the cluster; release/acquire orders the
// shared::cluster stores before it with the loads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32x4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// Arrive without ordering this thread's memory operations: threads that
// stored nothing the other CTAs read skip the cluster-scope fence.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
// Release fence at cluster scope: orders this thread's earlier stores (to
// another CTA's shared memory) before its later relaxed arrive.
__device__ __forceinline__ void fence_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Named barrier 1 over the first `n` threads of the CTA (a subset of warps).
__device__ __forceinline__ void bar_sync_named(int n) {
  asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- programmatic dependent launch ----------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialisation and calls pdl_wait() before its first global-memory access:
// that waits for the previous kernel in the stream to complete and its
// writes to be visible, so no ordering is lost, while the launch and the
// shared-memory prologue overlap the previous kernel's tail.  pdl_trigger()
// lets the next kernel start launching; it is issued once this kernel's
// CTAs are all resident, so it cannot take their slots.  Two exceptions:
// the backward, launched right after the loss forward on the same stream,
// writes the rows that score nothing before its wait (dlogits.cu); and the
// loss forward's log-sum-exp kernel, launched right after prep (which waits
// before it triggers, so every kernel before prep has completed when it
// starts), reads the raw lengths and the logits before its wait, and waits
// only before it touches what prep writes (the workspace header).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// off[0..N]: exclusive prefix sums of the lengths clamped to [0, C] (what
// prep writes to the workspace), computed by every thread of one block into
// shared memory (N below 2^31); s_warp holds one int per warp.
static __device__ __noinline__ void block_clamped_offsets(const int32_t* __restrict__ len, int64_t N,
                                                         int64_t C, int32_t* off, int32_t* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = (int)N, c = (int)min(C, (int64_t)INT32_MAX);
  const int per = (n + (int)blockDim.x - 1) / (int)blockDim.x;
  const int k0 = min(tid * per, n), k1 = min(k0 + per, n);
  int32_t own = 0;
  for (int k = k0; k < k1; ++k) own += min(max(__ldg(len + k), 0), c);
  int32_t x = own;  // inclusive scan within the warp
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int32_t run = x - own;
  for (int k = 0; k < warp; ++k) run += s_warp[k];
  if (tid == 0) off[0] = 0;
  for (int k = k0; k < k1; ++k) {
    run += min(max(__ldg(len + k), 0), c);
    off[k + 1] = run;
  }
  __syncthreads();
}

// ---- packed float pairs (Blackwell f32x2 FMA/ADD/MUL: two lanes per
// instruction, each rounded exactly as the scalar instruction) ------------

__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// 2^x of both lanes on the SFU.
__device__ __forceinline__ uint64_t f2_ex2(uint64_t a) {
  float x, y;
  f2_unpack(a, x, y);
  return f2_pack(ex2(x), ex2(y));
}

// ---- mbarrier and bulk-copy (TMA) helpers ----------------------------------

__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}
// Makes barrier initialisation visible to the async proxy and the cluster.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(addr), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t addr) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(addr) : "memory");
}
// Tests phase `parity` of the barrier; while it is incomplete the thread is
// suspended in hardware (up to about 0.1 ms) instead of spinning, so waiting
// warps do not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity), "r"(100000u)
      : "memory");
  return ok != 0;
}
// Upper bound of any wait on an mbarrier: one second.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// Waits for phase `parity` of the barrier to complete; false after the limit.
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity) {
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(addr, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}
// One-dimensional bulk copy global -> this CTA's shared memory, completing
// `bytes` of transaction count on the mbarrier.  Both addresses 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t smem_dst, const void* gsrc, uint32_t bytes,
                                         uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_dst),
      "l"(gsrc), "r"(bytes), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Merge of two partial (max m, sum of exp(x - m)) pairs; the sums are kept
// relative to their own maximum, so merging rescales the smaller side.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) {  // both empty (or all -inf logits)
    m = M;
    s = 0.f;
    return;
  }
  s = s * ex2((m - M) * kLog2e) + s2 * ex2((m2 - M) * kLog2e);
  m = M;
}

// ---------------------------------------------------------------------------
// per-token loss terms ("The loss" / grpo_loss; the k3 KL term)
// ---------------------------------------------------------------------------

// For one valid token with log-prob lp: the per-token loss ell and
// w = d loss / d logp (before dividing by the normaliser).
//   r   = exp(lp - old)                      (1 when there is no old log-prob)
//   s   = min(r*A, clamp(r, 1-eps, 1+eps)*A)  -- clip the ratio, then * A
//   k3  = exp(d) - d - 1, d = ref - lp        (written expm1(d) - d)
//   ell = -s + beta*k3
//   w   = -(A*r if min() takes r*A, else 0) + beta*(1 - exp(d))
// NaN inputs give NaN results (the comparisons keep NaN).  Shared by the
// unfused and the fused forward so both give the same bits.
struct TokenTerms {
  float ell, w;
};
__device__ __forceinline__ TokenTerms token_terms(float lp, float A, bool has_old, float old,
                                                  float beta, float ref, float eps) {
  const float lo = 1.f - eps, hi = 1.f + eps;
  const float r = has_old ? expf(lp - old) : 1.f;
  const float unclipped = r * A;
  const float rc = r < lo ? lo : (r > hi ? hi : r);
  const float clipped = rc * A;
  const float s = unclipped < clipped ? unclipped : clipped;
  const float ds = unclipped <= clipped ? A * r : 0.f;
  float k3 = 0.f, dk3 = 0.f;
  if (beta != 0.f) {
    const float d = ref - lp;
    const float em1 = expm1f(d);
    k3 = em1 - d;
    dk3 = -em1;
  }
  TokenTerms tt;
  tt.ell = -s + beta * k3;
  tt.w = -ds + beta * dk3;
  return tt;
}

// ---------------------------------------------------------------------------
// element types: 16-byte vectors of float32 (4) or bfloat16 bit patterns (8)
// ---------------------------------------------------------------------------

template <typename T>
struct Elt;

template <>
struct Elt<float> {
  static constexpr int kPerVec = 4;
  static constexpr int kUnroll = 8;  // vectors in flight per thread
  static constexpr uint32_t kNegInf = 0xff800000u;
  __device__ static void unpack(const uint4& d, float* x) {
    x[0] = __uint_as_float(d.x);
    x[1] = __uint_as_float(d.y);
    x[2] = __uint_as_float(d.z);
    x[3] = __uint_as_float(d.w);
  }
  __device__ static float extract(const uint4& d, int e) {
    const uint32_t w = e == 0 ? d.x : (e == 1 ? d.y : (e == 2 ? d.z : d.w));
    return __uint_as_float(w);
  }
  __device__ static float load1(const float* p) { return __ldg(p); }
  template <int U>
  __device__ static float batch_max(const uint4* d) {
    float m = __uint_as_float(d[0].x);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      m = fmaxf(m, __uint_as_float(d[u].x));
      m = fmaxf(m, __uint_as_float(d[u].y));
      m = fmaxf(m, __uint_as_float(d[u].z));
      m = fmaxf(m, __uint_as_float(d[u].w));
    }
    return m;
  }
  __device__ static uint4 pack(const float* o) {
    return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                      __float_as_uint(o[3]));
  }
  __device__ static void store1(float* p, float v) { *p = v; }
};

template <>
struct Elt<uint16_t> {  // bfloat16 bit patterns
  static constexpr int kPerVec = 8;
  static constexpr int kUnroll = 4;
  static constexpr uint32_t kNegInf = 0xff80ff80u;
  __device__ static void unpack(const uint4& d, float* x) {
    x[0] = bf16_lo(d.x);
    x[1] = bf16_hi(d.x);
    x[2] = bf16_lo(d.y);
    x[3] = bf16_hi(d.y);
    x[4] = bf16_lo(d.z);
    x[5] = bf16_hi(d.z);
    x[6] = bf16_lo(d.w);
    x[7] = bf16_hi(d.w);
  }
  __device__ static float extract(const uint4& d, int e) {
    const int k = e >> 1;
    const uint32_t w = k == 0 ? d.x : (k == 1 ? d.y : (k == 2 ? d.z : d.w));
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
  }
  __device__ static float load1(const uint16_t* p) { return bf16_bits_to_float(__ldg(p)); }
  // Maximum of U vectors with packed bfloat16x2 max (exact; ignores NaN like
  // fmaxf), then one widening of the last pair.
  template <int U>
  __device__ static float batch_max(const uint4* d) {
    __nv_bfloat162 m = as_bf162(d[0].x);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      m = __hmax2(m, as_bf162(d[u].x));
      m = __hmax2(m, as_bf162(d[u].y));
      m = __hmax2(m, as_bf162(d[u].z));
      m = __hmax2(m, as_bf162(d[u].w));
    }
    return fmaxf(__low2float(m), __high2float(m));
  }
  __device__ static uint4 pack(const float* o) {
    return make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                      pack_bf16x2(o[6], o[7]));
  }
  __device__ static void store1(uint16_t* p, float v) {
    *p = (uint16_t)(pack_bf16x2(v, 0.f) & 0xffffu);
  }
};

// Number of CTAs a row of `row_bytes` is split over: the largest power of two
// <= max_split that keeps at least 32 KiB of the row per CTA.  `env` names an
// environment variable that may force 1, 2, 4 or 8.
int row_split(int64_t row_bytes, const char* env, int max_split);

// CTAs per scored row (a thread block cluster splitting the row over the
// vocabulary) of the log-sum-exp kernels: 1 when the batch's N*C rows (an
// upper bound of the scored rows) can occupy the GPU on their own, else the
// smallest of 2, 4, 8 with rows * K >= 4 * SMs, as row_split allows.  Whole
// rows per CTA measured faster on GB300 whenever there are enough of them
// (no cluster barrier per row); the split keeps small batches from idling
// most SMs.  Both kernels use this rule, so they split a row the same way
// and their results have the same bits.
int lse_split(int64_t row_bytes, int64_t rows_max, int sms, const char* env);

// CTAs per SM of an oversubscribed streaming grid: `def`, or the positive
// integer in environment variable `env`.
int grid_mult(const char* env, int def);

// ---------------------------------------------------------------------------
// launchers (defined in the kernel files, called by api.cu)
// ---------------------------------------------------------------------------

// Launch with programmatic stream serialisation (and an optional cluster).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = cluster_x;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = cluster_x > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

struct DeviceInfo {
  int device;
  int sms;
};

cudaError_t launch_mask(const int64_t* ids, int64_t N, int64_t P, int64_t C, int64_t eos,
                        uint8_t* mask, int32_t* len, cudaStream_t st);
cudaError_t launch_advantage(const float* R, int64_t B, int64_t G, int mode, float std_eps,
                             float* adv, int32_t* n_contrast, cudaStream_t st,
                             bool after_mask);

struct FwdArgs {
  const void* logits;
  int dtype;  // 0 f32, 1 bf16
  int64_t N, P, C, V;
  const int64_t* ids;
  const int32_t* len;
  const float* adv;
  const float* old_logp;
  const float* ref_logp;
  float eps, beta, norm;
  int agg;  // 0: token sum / norm (Dr. GRPO); 1: per-response mean / norm
  float* logp;
  float* lse;
  float* w;
  float* loss;
  void* ws;
};
// The constant the token sum is divided by when norm <= 0.
inline double default_norm(const FwdArgs& a) {
  return a.norm > 0.f ? (double)a.norm : (a.agg == 0 ? (double)a.N * (double)a.C : (double)a.N);
}
cudaError_t launch_prep(const FwdArgs& a, cudaStream_t st);
// after_prep: launched directly after launch_prep on the same stream (the
// kernel then reads the lengths and logits before its wait)
cudaError_t launch_lse_gather(const FwdArgs& a, const DeviceInfo& d, cudaStream_t st,
                              bool after_prep);
cudaError_t launch_surrogate(const FwdArgs& a, cudaStream_t st);

struct BwdArgs {
  const void* logits;
  int dtype;
  int64_t N, P, C, V;
  const int64_t* ids;
  const int32_t* len;
  const float* lse;
  const float* w;
  const float* grad;
  void* dlogits;
  bool skip_zero_weight;  // rows with g*w == 0: zeros, logits not read
  // the launch directly follows the loss forward on its stream: rows that
  // score nothing may be written before waiting on it
  bool after_fwd;
};
cudaError_t launch_dlogits(const BwdArgs& a, const DeviceInfo& d, cudaStream_t st);
// Store-only pass of the fused path: zero dlogits rows and masked logp/lse/w.
cudaError_t launch_zero_rows(const BwdArgs& a, const DeviceInfo& d, cudaStream_t st, float* logp,
                             float* lse, float* w);
// Fused forward + backward over the scored rows (after prep and zero rows).
cudaError_t launch_lse_grad(const FwdArgs& a, const BwdArgs& b, const DeviceInfo& d,
                            cudaStream_t st);

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, const DeviceInfo& d,
                        cudaStream_t st);

}  // namespace grpo

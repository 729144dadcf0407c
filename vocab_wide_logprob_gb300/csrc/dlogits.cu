// Gradient of the loss with respect to the logits ("loss.backward()" of
// "Making Dr GRPO go brrr", salahadawi.com; the page relies on autograd and
// prints no formula, so it is derived here).  The loss depends on a logits
// row only through logp_t = z_y - logsumexp(z) of the one token the row
// scores, so by the chain rule
//     d loss / d z_v = w_t * ([v == y] - softmax(z)_v),   w_t = d loss / d logp_t,
// and every row that scores no valid token (prompt rows 0..P-2, the last row
// P+C-1, rows past the first EOS) has gradient 0.
//
// One streaming pass writes the whole [N, P+C, V] buffer: a scored row reads
// its logits once (16-byte loads) and writes g*w_t*(onehot - exp(z - lse_t));
// any other row is written with zeros and not read.  The target column uses
// 1 - p_y = -expm1(z_y - lse) to keep its precision when p_y is close to 1.
// Work items are (row, 1/K of the row), walked by a grid-stride loop.
//
// Item order.  By default the items go in memory order and every CTA waits
// for the preceding kernel first.  A row that scores nothing depends only on
// the lengths, though, and the loss forward's kernels write neither the
// lengths nor dlogits; so when the host knows this launch directly follows
// the loss forward on its stream (`zero_first`), the items are ordered with
// every such row first: those rows are written without waiting, while the
// forward's last kernels still run, and a CTA waits only before its first
// scored row (which needs lse and w).  Each CTA then computes the prefix sums
// of the lengths itself (batches of up to kZeroFirstMaxN completions).
#include "common.cuh"

namespace grpo {

constexpr int kZeroFirstMaxN = 1024;
constexpr int kPrefixPerThread = kZeroFirstMaxN / kThreads;

template <typename T>
struct DlParams {
  const T* logits;
  T* dlogits;
  int64_t N, P, C, V, T_len;
  const int64_t* ids;
  const int32_t* len;
  const float* lse;
  const float* w;
  const float* grad;  // device scalar or nullptr (1)
  int64_t chunk;      // elements per work item (multiple of kPerVec)
  int64_t split;      // work items per row
  // store-only mode (the fused forward+backward writes the scored rows):
  // also zero logp, lse and w [N, C] past each length
  float* logp_out;
  float* lse_out;
  float* w_out;
  int skip_zero_weight;  // a scored row with g*w == 0 is written with zeros, not read
  int zero_first;        // rows that score nothing first, written before the wait (N <= 1024)
};

// s_pre[i] = sum of min(max(len[k], 0), C) over k < i, for i = 0..N (N <=
// kZeroFirstMaxN), computed by the whole CTA.  Reads the lengths through L2:
// they are not written by any kernel still running.
__device__ __forceinline__ void length_prefix(const int32_t* __restrict__ len, int64_t N,
                                              int64_t C, int32_t* s_pre, int32_t* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (int)((N + kThreads - 1) / kThreads);
  const int k0 = tid * per;
  int32_t v[kPrefixPerThread];
  int32_t own = 0;
#pragma unroll
  for (int u = 0; u < kPrefixPerThread; ++u) {
    int32_t L = 0;
    if (u < per && k0 + u < N) {
      L = __ldcg(len + k0 + u);
      L = L < 0 ? 0 : (L > C ? (int32_t)C : L);
    }
    v[u] = L;
    own += L;
  }
  int32_t x = own;  // inclusive scan within the warp
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  int32_t run = x - own;
  for (int k = 0; k < warp; ++k) run += s_warp[k];
  if (tid == 0) s_pre[0] = 0;
#pragma unroll
  for (int u = 0; u < kPrefixPerThread; ++u)
    if (u < per && k0 + u < N) {
      run += v[u];
      s_pre[k0 + u + 1] = run;
    }
  __syncthreads();
}

// kZeroOnly: write only the rows that score nothing (and the masked
// per-token outputs); scored rows are left to lse_grad_kernel, which is
// launched just before this kernel and writes disjoint rows and positions,
// so no CTA waits on it before writing (the lengths were written before
// either started): the zeros stream out while lse_grad_kernel runs.
// Resident CTAs per SM the register budget is held to: 5 for bf16 (the
// oversubscribed grid streams faster with more of them), 4 for fp32 (whose
// wider unroll would spill at 5).
template <typename T>
constexpr int dl_min_blocks() {
  return sizeof(T) == 2 ? 5 : 4;
}

template <typename T, bool kZeroOnly>
__global__ void __launch_bounds__(kThreads, dl_min_blocks<T>()) dlogits_kernel(const DlParams<T> p) {
  using E = Elt<T>;
  constexpr int EPV = E::kPerVec;
  constexpr int U = E::kUnroll;
  const int tid = threadIdx.x;
  __shared__ int32_t s_pre[kZeroFirstMaxN + 1];
  __shared__ int32_t s_warp[kThreads / 32];
  const bool zero_first = !kZeroOnly && p.zero_first;
  bool waited = false;  // the preceding kernel's outputs (lse, w) are visible once set
  if (zero_first) {
    length_prefix(p.len, p.N, p.C, s_pre, s_warp);
  } else if (!kZeroOnly) {
    pdl_wait();
    waited = true;
  }
  pdl_trigger();
  const int64_t items = p.N * p.T_len * p.split;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  if (kZeroOnly) {
    for (int64_t k = (int64_t)blockIdx.x * kThreads + tid; k < p.N * p.C;
         k += (int64_t)gridDim.x * kThreads) {
      const int64_t i = k / p.C;
      int64_t L = __ldg(p.len + i);
      L = L < 0 ? 0 : (L > p.C ? p.C : L);
      if (k - i * p.C >= L) {
        p.logp_out[k] = 0.f;
        p.lse_out[k] = 0.f;
        p.w_out[k] = 0.f;
      }
    }
  }
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int64_t r = item / p.split;
    const int64_t j = item - r * p.split;
    int64_t row, i, L;
    if (!zero_first) {
      row = r;
      i = row / p.T_len;
      L = __ldg(p.len + i);
      L = L < 0 ? 0 : (L > p.C ? p.C : L);
    } else if (r < p.N * p.T_len - s_pre[p.N]) {  // rows that score nothing come first
      // zero row r: completion i has i*T_len - s_pre[i] zero rows before it
      // (every completion has at least one, its last row), its own being the
      // prompt rows 0..P-2 and then the rows past its length
      int lo = 0, hi = (int)p.N;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)mid * p.T_len - s_pre[mid] <= r)
          lo = mid;
        else
          hi = mid;
      }
      i = lo;
      L = s_pre[lo + 1] - s_pre[lo];
      const int64_t q = r - (i * p.T_len - s_pre[lo]);
      row = i * p.T_len + (q < p.P - 1 ? q : q + L);
    } else {  // then the scored rows, last first: the forward read those most
              // recently, so they are the likeliest to be still in L2
      const int64_t sr = (int64_t)s_pre[p.N] - 1 - (r - (p.N * p.T_len - s_pre[p.N]));
      int lo = 0, hi = (int)p.N;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pre[mid] <= sr)
          lo = mid;
        else
          hi = mid;
      }
      i = lo;
      L = s_pre[lo + 1] - s_pre[lo];
      row = i * p.T_len + p.P - 1 + (sr - s_pre[lo]);
    }
    const int64_t t = row - i * p.T_len - (p.P - 1);  // completion token this row scores
    const int64_t v0 = j * p.chunk;
    const int64_t v1 = min(p.V, v0 + p.chunk);
    if (v0 >= v1) continue;
    T* orow = p.dlogits + row * p.V;
    const T* zrow = p.logits + row * p.V;
    // 16-byte aligned interior [a, b) of the output slice
    const uintptr_t oaddr = reinterpret_cast<uintptr_t>(orow + v0);
    const int64_t skip = (int64_t)(((16u - (unsigned)(oaddr & 15u)) & 15u) / sizeof(T));
    const int64_t a = min(v0 + skip, v1);
    const int64_t nvec = (v1 - a) / EPV;
    const int64_t b = a + nvec * EPV;
    uint4* ovp = reinterpret_cast<uint4*>(orow + a);

    bool zero_row = t < 0 || t >= L;  // the row scores nothing
    float gw = 0.f;
    if (!zero_row && !kZeroOnly) {
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      gw = (p.grad != nullptr ? __ldg(p.grad) : 1.f) * __ldg(p.w + i * p.C + t);
      if (p.skip_zero_weight && gw == 0.f) zero_row = true;  // its gradient is 0
    }
    if (zero_row) {  // zeros, logits not read
      for (int64_t k = tid; k < nvec; k += kThreads) st_stream(ovp + k, zero);
      if (tid < a - v0) E::store1(orow + v0 + tid, 0.f);
      if (tid >= 32 && tid - 32 < v1 - b) E::store1(orow + b + (tid - 32), 0.f);
      continue;
    }
    if (kZeroOnly) continue;
    const int64_t k_tok = i * p.C + t;
    const float ngw = -gw;
    const float lse_t = __ldg(p.lse + k_tok);
    const float lseL = lse_t * kLog2e;
    const int64_t y = __ldg(p.ids + i * p.T_len + p.P + t);
    // vector path only when logits and dlogits share the 16-byte phase
    const bool same_phase =
        ((reinterpret_cast<uintptr_t>(zrow + a) ^ reinterpret_cast<uintptr_t>(orow + a)) & 15u) == 0;
    if (same_phase) {
      const uint4* zvp = reinterpret_cast<const uint4*>(zrow + a);
      const int64_t ky = (y >= a && y < b) ? (y - a) / EPV : -1;
      const int ey = ky >= 0 ? (int)((y - a) % EPV) : 0;
      for (int64_t k0 = tid; k0 < nvec; k0 += (int64_t)kThreads * U) {
        uint4 d[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t k = k0 + (int64_t)u * kThreads;
          if (k < nvec) d[u] = ld_stream(zvp + k);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t k = k0 + (int64_t)u * kThreads;
          if (k >= nvec) break;
          float x[EPV], o[EPV];
          E::unpack(d[u], x);
#pragma unroll
          for (int e = 0; e < EPV; ++e) o[e] = ngw * ex2(fmaf(x[e], kLog2e, -lseL));
          if (k == ky) {
            // 1 - p_y without cancellation
            const float zy = E::extract(d[u], ey);
#pragma unroll
            for (int e = 0; e < EPV; ++e)
              if (e == ey) o[e] = ngw * expm1f(zy - lse_t);
          }
          st_stream(ovp + k, E::pack(o));
        }
      }
    } else {
      for (int64_t v = a + tid; v < b; v += kThreads) {
        const float x = E::load1(zrow + v);
        const float o = v == y ? ngw * expm1f(x - lse_t) : ngw * ex2(fmaf(x, kLog2e, -lseL));
        E::store1(orow + v, o);
      }
    }
    int64_t e = -1;
    if (tid < a - v0)
      e = v0 + tid;
    else if (tid >= 32 && tid - 32 < v1 - b)
      e = b + (tid - 32);
    if (e >= 0) {
      const float x = E::load1(zrow + e);
      const float o = e == y ? ngw * expm1f(x - lse_t) : ngw * ex2(fmaf(x, kLog2e, -lseL));
      E::store1(orow + e, o);
    }
  }
  // The kernel must not complete before the preceding one (the next launch
  // on the stream relies on it): when no CTA has waited (the store-only mode,
  // or no scored row in the batch), CTA 0 does.
  if (!waited && blockIdx.x == 0) pdl_wait();
}

namespace {

template <typename T, bool kZeroOnly>
cudaError_t launch_t(const BwdArgs& a, const DeviceInfo& d, cudaStream_t st, float* logp,
                     float* lse, float* w_out) {
  constexpr int EPV = Elt<T>::kPerVec;
  DlParams<T> p;
  p.logits = static_cast<const T*>(a.logits);
  p.dlogits = static_cast<T*>(a.dlogits);
  p.N = a.N;
  p.P = a.P;
  p.C = a.C;
  p.V = a.V;
  p.T_len = a.P + a.C;
  p.ids = a.ids;
  p.len = a.len;
  p.lse = a.lse;
  p.w = a.w;
  p.grad = a.grad;
  p.logp_out = logp;
  p.lse_out = lse;
  p.w_out = w_out;
  p.skip_zero_weight = a.skip_zero_weight ? 1 : 0;
  p.zero_first = !kZeroOnly && a.after_fwd && a.N <= kZeroFirstMaxN ? 1 : 0;
  p.split = row_split(a.V * (int64_t)sizeof(T), "GRPO_BWD_SPLIT", 8);
  p.chunk = ((a.V + p.split - 1) / p.split + EPV - 1) / EPV * EPV;
  // An oversubscribed grid (many more CTAs than fit at once, grid-stride over
  // the items) streams stores faster than a persistent one: measured 7.3 vs
  // 6.5 TB/s for a pure write stream on GB300.
  const int64_t items = a.N * (a.P + a.C) * p.split;
  int64_t grid = (int64_t)grid_mult("GRPO_BWD_GRID", 256) * d.sms;
  if (grid > items) grid = items;
  return launch_pdl(dlogits_kernel<T, kZeroOnly>, dim3((unsigned)grid), dim3(kThreads), 0, st,
                    1, p);
}

}  // namespace

cudaError_t launch_dlogits(const BwdArgs& a, const DeviceInfo& d, cudaStream_t st) {
  if (a.N == 0) return cudaSuccess;
  return a.dtype == 0 ? launch_t<float, false>(a, d, st, nullptr, nullptr, nullptr)
                      : launch_t<uint16_t, false>(a, d, st, nullptr, nullptr, nullptr);
}

cudaError_t launch_zero_rows(const BwdArgs& a, const DeviceInfo& d, cudaStream_t st, float* logp,
                             float* lse, float* w) {
  if (a.N == 0) return cudaSuccess;
  return a.dtype == 0 ? launch_t<float, true>(a, d, st, logp, lse, w)
                      : launch_t<uint16_t, true>(a, d, st, logp, lse, w);
}

}  // namespace grpo

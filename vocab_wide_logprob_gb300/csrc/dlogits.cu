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
// Work items are (row, 1/K of the row); a persistent grid walks them in
// memory order.
#include "common.cuh"

namespace grpo {

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
};

// kZeroOnly: write only the rows that score nothing (and the masked
// per-token outputs); scored rows are left to lse_grad_kernel.
template <typename T, bool kZeroOnly>
__global__ void __launch_bounds__(kThreads) dlogits_kernel(const DlParams<T> p) {
  using E = Elt<T>;
  constexpr int EPV = E::kPerVec;
  constexpr int U = E::kUnroll;
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const float g = p.grad != nullptr ? __ldg(p.grad) : 1.f;
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
    const int64_t row = item / p.split;
    const int64_t j = item - row * p.split;
    const int64_t i = row / p.T_len;
    const int64_t t = row - i * p.T_len - (p.P - 1);  // completion token this row scores
    const int64_t v0 = j * p.chunk;
    const int64_t v1 = min(p.V, v0 + p.chunk);
    if (v0 >= v1) continue;
    int64_t L = __ldg(p.len + i);
    L = L < 0 ? 0 : (L > p.C ? p.C : L);
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
      gw = g * __ldg(p.w + i * p.C + t);
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

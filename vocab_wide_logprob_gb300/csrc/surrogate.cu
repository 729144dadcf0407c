// Clipped surrogate, k3 KL term, per-token gradient weight and the scalar
// loss ("The loss" / grpo_loss and section "Dr. GRPO" of "Making Dr GRPO go
// brrr", salahadawi.com).  Per valid token:
//     r   = exp(logp - old)                (exactly 1 without old log-probs)
//     s   = min(r*A, clamp(r, 1-eps, 1+eps)*A)   -- clip the ratio, then * A
//     k3  = exp(ref - logp) - (ref - logp) - 1   (written expm1(d) - d)
//     ell = -s + beta*k3
//     w   = d loss / d logp = (-(A*r if min() takes r*A, else 0)
//                              + beta*(1 - exp(ref - logp))) / norm
// and loss = (sum of ell over valid tokens) / norm: token-sum aggregation over
// a constant, not a per-response mean.  The mask multiplies the per-token
// loss (masked positions contribute nothing and are never read), never the
// ratio.
//
// The sum is deterministic: each thread accumulates its positions in index
// order in float64, each CTA reduces in a fixed tree, and the last CTA to
// finish adds the per-CTA partials in CTA order.
#include "common.cuh"

namespace grpo {

struct SurParams {
  int64_t N, C;
  const int32_t* lens;  // clamped lengths (workspace)
  const float* adv;
  const float* old_logp;
  const float* ref_logp;
  float eps, beta;
  int agg;
  double norm;
  float* logp;
  float* lse;
  float* w;
  float* loss;
  WsHeader* hdr;
  double* partials;
};

__global__ void __launch_bounds__(kThreads) surrogate_kernel(const SurParams p) {
  __shared__ double s_red[kWarps];
  __shared__ bool s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Trigger first: the backward that follows can then launch while the
  // log-sum-exp kernel still runs and write its rows that score nothing (it
  // waits on this kernel before it reads lse or w).
  pdl_trigger();
  pdl_wait();
  const int64_t NC = p.N * p.C;
  double acc = 0.0;
  for (int64_t k = (int64_t)blockIdx.x * kThreads + tid; k < NC;
       k += (int64_t)gridDim.x * kThreads) {
    const int64_t i = k / p.C, t = k - i * p.C;
    if (t >= p.lens[i]) {  // past the first EOS: outputs 0, inputs unread
      p.logp[k] = 0.f;
      p.lse[k] = 0.f;
      p.w[k] = 0.f;
      continue;
    }
    const float lp = p.logp[k];
    const TokenTerms tt =
        token_terms(lp, p.adv[i], p.old_logp != nullptr,
                    p.old_logp != nullptr ? p.old_logp[k] : 0.f, p.beta,
                    p.beta != 0.f ? p.ref_logp[k] : 0.f, p.eps);
    // the constant this token is divided by; the per-response mean also
    // divides by the completion's length
    const double denom = p.agg == 0 ? p.norm : p.norm * (double)p.lens[i];
    p.w[k] = (float)((double)tt.w / denom);
    acc += p.agg == 0 ? (double)tt.ell : (double)tt.ell / (double)p.lens[i];
  }
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) s_red[warp] = acc;
  __syncthreads();
  if (tid == 0) {
    double b = s_red[0];
#pragma unroll
    for (int k = 1; k < kWarps; ++k) b += s_red[k];
    p.partials[blockIdx.x] = b;
    __threadfence();
    const unsigned ticket = atomicAdd(&p.hdr->ticket, 1u);
    s_last = ticket == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  // last CTA: every other CTA's partial is visible (fence before its ticket)
  __threadfence();
  double v = 0.0;
  for (int64_t b = tid; b < gridDim.x; b += kThreads)
    v += reinterpret_cast<volatile double*>(p.partials)[b];
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  if (tid == 0) {
    double tot = s_red[0];
#pragma unroll
    for (int k = 1; k < kWarps; ++k) tot += s_red[k];
    *p.loss = (float)(tot / p.norm);
    p.hdr->ticket = 0;
  }
}

cudaError_t launch_surrogate(const FwdArgs& a, cudaStream_t st) {
  const WsLayout l = ws_layout(a.N);
  char* ws = static_cast<char*>(a.ws);
  SurParams p;
  p.N = a.N;
  p.C = a.C;
  p.lens = reinterpret_cast<const int32_t*>(ws + l.lens);
  p.adv = a.adv;
  p.old_logp = a.old_logp;
  p.ref_logp = a.ref_logp;
  p.eps = a.eps;
  p.beta = a.beta;
  p.agg = a.agg;
  p.norm = default_norm(a);
  p.logp = a.logp;
  p.lse = a.lse;
  p.w = a.w;
  p.loss = a.loss;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.partials = reinterpret_cast<double*>(ws + l.partials);
  const int64_t NC = a.N * a.C;
  int64_t blocks = (NC + kThreads - 1) / kThreads;
  if (blocks > kMaxLossBlocks) blocks = kMaxLossBlocks;
  if (blocks < 1) blocks = 1;
  return launch_pdl(surrogate_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, st, 1, p);
}

}  // namespace grpo

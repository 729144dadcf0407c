// C ABI of the library (declared in include/grpo.h): argument validation on
// the host, then the launches on the caller's stream.  Nothing here allocates
// device memory or synchronises, except grpo_check_error.
#include <math.h>
#include <stdlib.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "host_ctx.cuh"
#include "lmhead.cuh"
#include "host_rows.cuh"
#include "selftest.cuh"
#include "grpo.h"

namespace grpo {

int row_split(int64_t row_bytes, const char* env, int max_split) {
  if (env != nullptr) {
    if (const char* s = getenv(env)) {
      const int k = atoi(s);
      if (k == 1 || k == 2 || k == 4 || k == 8) return k;
    }
  }
  int k = 1;
  while (k < max_split && row_bytes / (2 * k) >= 32768) k *= 2;
  return k;
}

int lse_split(int64_t row_bytes, int64_t rows_max, int sms, const char* env) {
  int k = 1;
  while (k < 8 && rows_max * k < 4 * (int64_t)sms) k *= 2;
  return row_split(row_bytes, env, k);
}

int grid_mult(const char* env, int def) {
  if (const char* s = getenv(env)) {
    const int k = atoi(s);
    if (k > 0 && k <= 4096) return k;
  }
  return def;
}

namespace {

// SM count per device ordinal (ordinals below 64; others are asked each time)
std::atomic<int> g_sms[64] = {};

cudaError_t current_device(DeviceInfo* d) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  d->device = dev;
  int n = dev >= 0 && dev < 64 ? g_sms[dev].load(std::memory_order_relaxed) : 0;
  if (n == 0) {
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_sms[dev].store(n, std::memory_order_relaxed);
  }
  d->sms = n;
  return cudaSuccess;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// What the library enqueued last on a stream, and which memory it touches.
// Two launches may touch memory before waiting on the kernel before them,
// when the host knows that kernel: the backward, right after the loss
// forward, writes the rows that score nothing (it reads only the lengths and
// writes only dlogits before its wait); the advantage, right after the mask,
// computes its groups (it reads the rewards and writes the advantages).  Each
// may do so only when its own buffers are disjoint from those of the call
// before it (what that call writes must not be read or written, what it
// reads must not be written); otherwise it waits first as every launch does.
// So every entry point that enqueues work calls stream_take_last() first, and
// a successful loss forward or mask call records itself and its buffers.
// Calls from several host threads on one stream are ordered as their launches
// are only if the caller orders them.
enum LastCall { kLastOther = 0, kLastLossFwd = 1, kLastMask = 2 };

struct Span {  // [lo, hi) in the process's (unified) address space
  uintptr_t lo = 0, hi = 0;
};
Span span(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return p == nullptr ? Span{} : Span{a, a + bytes};
}
struct CallRecord {
  int kind = kLastOther;
  Span writes[5];
  Span reads[6];
};
bool overlaps(const Span* set, int n, Span x) {
  if (x.lo == x.hi) return false;
  for (int k = 0; k < n; ++k)
    if (set[k].lo < x.hi && x.lo < set[k].hi) return true;
  return false;
}
// Whether a launch that writes `w` and reads `r` before its wait may follow
// the recorded call without waiting on it.
bool disjoint_from(const CallRecord& c, Span w, Span r) {
  return !overlaps(c.writes, 5, w) && !overlaps(c.reads, 6, w) && !overlaps(c.writes, 5, r);
}

std::mutex g_order_mutex;
std::map<std::pair<unsigned long long, cudaStream_t>, CallRecord> g_last_call;

// A stream handle names a stream of the current context (the legacy default
// stream 0 is a different stream in each), so records are kept per context.
std::pair<unsigned long long, cudaStream_t> order_key(cudaStream_t st) {
  unsigned long long ctx = 0;
  if (current_context_id(&ctx) != cudaSuccess) (void)cudaGetLastError();
  return {ctx, st};
}

// grpo_set_early_start(0) turns the two early starts off process-wide.
std::atomic<int> g_early_start{1};

// The library's last call on `st` (kind kLastOther if not recorded, or if
// early starts are off); forgets it.
CallRecord stream_take_last(cudaStream_t st) {
  const auto key = order_key(st);
  std::lock_guard<std::mutex> lk(g_order_mutex);
  const auto it = g_last_call.find(key);
  if (it == g_last_call.end()) return CallRecord{};
  const CallRecord last = it->second;
  g_last_call.erase(it);
  return g_early_start.load() ? last : CallRecord{};
}
void stream_take_after_fwd(cudaStream_t st) { (void)stream_take_last(st); }

void stream_mark_last(cudaStream_t st, const CallRecord& rec) {
  const auto key = order_key(st);
  std::lock_guard<std::mutex> lk(g_order_mutex);
  g_last_call[key] = rec;
}

// a*b*c without int64 overflow, or -1
int64_t mul3(int64_t a, int64_t b, int64_t c) {
  if (a < 0 || b < 0 || c < 0) return -1;
  if (a == 0 || b == 0 || c == 0) return 0;
  if (a > INT64_MAX / b) return -1;
  const int64_t ab = a * b;
  if (ab > INT64_MAX / c) return -1;
  return ab * c;
}

grpo_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GRPO_OK : GRPO_ERR_CUDA; }

// Shape checks shared by the loss calls.
grpo_status check_shapes(grpo_dtype dtype, int64_t N, int64_t P, int64_t C, int64_t V) {
  if (dtype != GRPO_F32 && dtype != GRPO_BF16) return GRPO_ERR_UNSUPPORTED;
  if (N < 0 || P < 1 || C < 0 || V < 1) return GRPO_ERR_INVALID_ARG;
  if (P > INT64_MAX - C) return GRPO_ERR_UNSUPPORTED;  // P + C is formed below
  if (N > 0 && C > 0 && N > (int64_t)INT32_MAX / C) return GRPO_ERR_UNSUPPORTED;  // N*C < 2^31
  const int64_t elems = mul3(N, P + C, V);
  if (elems < 0 || elems > INT64_MAX / 4) return GRPO_ERR_UNSUPPORTED;
  return GRPO_OK;
}

}  // namespace
}  // namespace grpo

using namespace grpo;

extern "C" {

const char* grpo_status_string(grpo_status s) {
  switch (s) {
    case GRPO_OK:
      return "ok";
    case GRPO_ERR_INVALID_ARG:
      return "invalid argument";
    case GRPO_ERR_UNSUPPORTED:
      return "unsupported dtype or size";
    case GRPO_ERR_WORKSPACE:
      return "workspace missing or too small";
    case GRPO_ERR_MISALIGNED:
      return "pointer misaligned";
    case GRPO_ERR_CUDA:
      return "CUDA runtime error";
    case GRPO_ERR_TOKEN_RANGE:
      return "a scored token id is outside [0, V)";
    case GRPO_ERR_LENGTH_RANGE:
      return "a completion length is outside [0, C]";
    case GRPO_ERR_TIMEOUT:
      return "a device-side wait timed out";
  }
  return "unknown status";
}

grpo_status grpo_mask(const int64_t* input_ids, int64_t N, int64_t P, int64_t C, int64_t eos_id,
                      uint8_t* mask, int32_t* len, grpo_stream_t stream) {
  if (N < 0 || P < 0 || C < 0) return GRPO_ERR_INVALID_ARG;
  if (N == 0) return GRPO_OK;
  if (len == nullptr || (C > 0 && input_ids == nullptr)) return GRPO_ERR_INVALID_ARG;
  if (P > INT64_MAX - C || mul3(N, P + C, 8) < 0 || C > INT32_MAX) return GRPO_ERR_UNSUPPORTED;
  if (!aligned(input_ids, 8) || !aligned(len, 4)) return GRPO_ERR_MISALIGNED;
  stream_take_last(stream);
  const cudaError_t e = launch_mask(input_ids, N, P, C, eos_id, mask, len, (cudaStream_t)stream);
  if (e == cudaSuccess) {
    CallRecord rec;
    rec.kind = kLastMask;
    rec.writes[0] = span(mask, (size_t)(N * C));
    rec.writes[1] = span(len, sizeof(int32_t) * (size_t)N);
    rec.reads[0] = span(input_ids, sizeof(int64_t) * (size_t)(N * (P + C)));
    stream_mark_last(stream, rec);
  }
  return from_cuda(e);
}

grpo_status grpo_advantage(const float* rewards, int64_t B, int64_t G, float* adv,
                           grpo_stream_t stream) {
  if (B < 0 || G < 1) return GRPO_ERR_INVALID_ARG;
  if (B == 0) return GRPO_OK;
  if (rewards == nullptr || adv == nullptr) return GRPO_ERR_INVALID_ARG;
  if (mul3(B, G, 4) < 0 || B > INT32_MAX) return GRPO_ERR_UNSUPPORTED;
  if (!aligned(rewards, 4) || !aligned(adv, 4)) return GRPO_ERR_MISALIGNED;
  const CallRecord last = stream_take_last(stream);
  const bool after_mask =
      last.kind == kLastMask && disjoint_from(last, span(adv, sizeof(float) * (size_t)(B * G)),
                                              span(rewards, sizeof(float) * (size_t)(B * G)));
  return from_cuda(
      launch_advantage(rewards, B, G, 0, 0.f, adv, nullptr, (cudaStream_t)stream, after_mask));
}

grpo_status grpo_advantage_ex(const float* rewards, int64_t B, int64_t G, grpo_adv_mode mode,
                              float std_eps, float* adv, int32_t* n_contrast,
                              grpo_stream_t stream) {
  if (B < 0 || G < 1) return GRPO_ERR_INVALID_ARG;
  if (mode != GRPO_ADV_DR && mode != GRPO_ADV_STD) return GRPO_ERR_UNSUPPORTED;
  if (!(std_eps >= 0.f) || isinf(std_eps)) return GRPO_ERR_INVALID_ARG;
  if (B > 0 && (rewards == nullptr || adv == nullptr)) return GRPO_ERR_INVALID_ARG;
  if (mul3(B, G, 4) < 0 || B > INT32_MAX) return GRPO_ERR_UNSUPPORTED;
  if (!aligned(rewards, 4) || !aligned(adv, 4) || !aligned(n_contrast, 4))
    return GRPO_ERR_MISALIGNED;
  const CallRecord last = stream_take_last(stream);
  const bool after_mask =
      last.kind == kLastMask && disjoint_from(last, span(adv, sizeof(float) * (size_t)(B * G)),
                                              span(rewards, sizeof(float) * (size_t)(B * G)));
  return from_cuda(launch_advantage(rewards, B, G, (int)mode, std_eps, adv, n_contrast,
                                    (cudaStream_t)stream, after_mask));
}

grpo_status grpo_workspace_size(int64_t N, int64_t C, int64_t V, size_t* bytes) {
  if (bytes == nullptr || N < 0 || C < 0 || V < 1) return GRPO_ERR_INVALID_ARG;
  if (N > 0 && C > 0 && N > (int64_t)INT32_MAX / C) return GRPO_ERR_UNSUPPORTED;
  *bytes = ws_layout(N).total;
  return GRPO_OK;
}

}  // extern "C"

namespace {

// mode 0: full forward; 1: log-probs only (no loss, w or adv needed).
grpo_status loss_fwd_impl(const void* logits, grpo_dtype dtype, int64_t N, int64_t P, int64_t C,
                          int64_t V, const int64_t* input_ids, const int32_t* len,
                          const float* adv, const float* old_logp, const float* ref_logp,
                          float eps, float beta, float norm, int agg, float* logp, float* lse,
                          float* w, float* loss, void* workspace, size_t workspace_bytes,
                          grpo_stream_t stream, int mode) {
  grpo_status s = check_shapes(dtype, N, P, C, V);
  if (s != GRPO_OK) return s;
  if (!(eps >= 0.f && eps < 1.f) || !(beta >= 0.f) || isinf(beta) || isnan(norm) || isinf(norm))
    return GRPO_ERR_INVALID_ARG;
  if (agg != 0 && agg != 1) return GRPO_ERR_UNSUPPORTED;
  if ((mode == 0 && loss == nullptr) || workspace == nullptr) return GRPO_ERR_INVALID_ARG;
  if (N > 0 && (len == nullptr || (mode == 0 && adv == nullptr))) return GRPO_ERR_INVALID_ARG;
  if (N > 0 && C > 0 &&
      (logits == nullptr || input_ids == nullptr || logp == nullptr || lse == nullptr ||
       (mode == 0 && w == nullptr)))
    return GRPO_ERR_INVALID_ARG;
  if (mode == 0 && beta != 0.f && ref_logp == nullptr && N > 0 && C > 0)
    return GRPO_ERR_INVALID_ARG;
  const size_t esize = dtype == GRPO_F32 ? 4 : 2;
  if (!aligned(logits, esize) || !aligned(input_ids, 8) || !aligned(len, 4) ||
      !aligned(adv, 4) || !aligned(old_logp, 4) || !aligned(ref_logp, 4) || !aligned(logp, 4) ||
      !aligned(lse, 4) || !aligned(w, 4) || !aligned(loss, 4) || !aligned(workspace, 256))
    return GRPO_ERR_MISALIGNED;
  if (workspace_bytes < ws_layout(N).total) return GRPO_ERR_WORKSPACE;

  FwdArgs a;
  a.logits = logits;
  a.dtype = dtype == GRPO_F32 ? 0 : 1;
  a.N = N;
  a.P = P;
  a.C = C;
  a.V = V;
  a.ids = input_ids;
  a.len = len;
  a.adv = adv;
  a.old_logp = old_logp;
  a.ref_logp = beta != 0.f ? ref_logp : nullptr;
  a.eps = eps;
  a.beta = beta;
  a.norm = norm;
  a.agg = agg;
  a.logp = logp;
  a.lse = lse;
  a.w = w;
  a.loss = loss;
  a.ws = workspace;
  const cudaStream_t st = (cudaStream_t)stream;
  DeviceInfo d;
  cudaError_t e = current_device(&d);
  if (e != cudaSuccess) return GRPO_ERR_CUDA;
  stream_take_after_fwd(st);
  // the prep kernel also resets the error flags and the reduction ticket
  if ((e = launch_prep(a, st)) != cudaSuccess) return GRPO_ERR_CUDA;
  if (N == 0 || C == 0)
    return mode == 0 ? from_cuda(cudaMemsetAsync(loss, 0, sizeof(float), st)) : GRPO_OK;
  if ((e = launch_lse_gather(a, d, st, true)) != cudaSuccess) return GRPO_ERR_CUDA;
  if (mode == 1) return GRPO_OK;  // the log-sum-exp kernel zeroed the masked positions
  if ((e = launch_surrogate(a, st)) != cudaSuccess) return GRPO_ERR_CUDA;
  CallRecord rec;
  rec.kind = kLastLossFwd;
  const size_t nc4 = sizeof(float) * (size_t)(N * C);
  rec.writes[0] = span(logp, nc4);
  rec.writes[1] = span(lse, nc4);
  rec.writes[2] = span(w, nc4);
  rec.writes[3] = span(loss, sizeof(float));
  rec.writes[4] = span(workspace, workspace_bytes);
  rec.reads[0] = span(logits, (size_t)mul3(N, P + C, V) * (dtype == GRPO_F32 ? 4 : 2));
  rec.reads[1] = span(input_ids, sizeof(int64_t) * (size_t)(N * (P + C)));
  rec.reads[2] = span(len, sizeof(int32_t) * (size_t)N);
  rec.reads[3] = span(adv, sizeof(float) * (size_t)N);
  rec.reads[4] = span(old_logp, nc4);
  rec.reads[5] = span(a.ref_logp, nc4);
  stream_mark_last(st, rec);
  return GRPO_OK;
}

}  // namespace

extern "C" {

grpo_status grpo_loss_fwd(const void* logits, grpo_dtype dtype, int64_t N, int64_t P, int64_t C,
                          int64_t V, const int64_t* input_ids, const int32_t* len,
                          const float* adv, const float* old_logp, const float* ref_logp,
                          float eps, float beta, float norm, float* logp, float* lse, float* w,
                          float* loss, void* workspace, size_t workspace_bytes,
                          grpo_stream_t stream) {
  return loss_fwd_impl(logits, dtype, N, P, C, V, input_ids, len, adv, old_logp, ref_logp, eps,
                       beta, norm, 0, logp, lse, w, loss, workspace, workspace_bytes, stream, 0);
}

grpo_status grpo_loss_fwd_ex(const void* logits, grpo_dtype dtype, int64_t N, int64_t P,
                             int64_t C, int64_t V, const int64_t* input_ids, const int32_t* len,
                             const float* adv, const float* old_logp, const float* ref_logp,
                             float eps, float beta, float norm, grpo_aggregation agg,
                             float* logp, float* lse, float* w, float* loss, void* workspace,
                             size_t workspace_bytes, grpo_stream_t stream) {
  return loss_fwd_impl(logits, dtype, N, P, C, V, input_ids, len, adv, old_logp, ref_logp, eps,
                       beta, norm, (int)agg, logp, lse, w, loss, workspace, workspace_bytes,
                       stream, 0);
}

grpo_status grpo_logprobs(const void* logits, grpo_dtype dtype, int64_t N, int64_t P, int64_t C,
                          int64_t V, const int64_t* input_ids, const int32_t* len, float* logp,
                          float* lse, void* workspace, size_t workspace_bytes,
                          grpo_stream_t stream) {
  return loss_fwd_impl(logits, dtype, N, P, C, V, input_ids, len, nullptr, nullptr, nullptr, 0.f,
                       0.f, 0.f, 0, logp, lse, nullptr, nullptr, workspace, workspace_bytes,
                       stream, 1);
}

grpo_status grpo_loss_bwd_ex(const void* logits, grpo_dtype dtype, int64_t N, int64_t P,
                             int64_t C, int64_t V, const int64_t* input_ids, const int32_t* len,
                             const float* lse, const float* w, const float* grad_loss,
                             void* dlogits, uint32_t flags, grpo_stream_t stream) {
  if (flags & ~(uint32_t)GRPO_BWD_SKIP_ZERO_WEIGHT) return GRPO_ERR_UNSUPPORTED;
  grpo_status s = check_shapes(dtype, N, P, C, V);
  if (s != GRPO_OK) return s;
  if (N == 0) return GRPO_OK;
  if (dlogits == nullptr || len == nullptr) return GRPO_ERR_INVALID_ARG;
  if (C > 0 && (logits == nullptr || input_ids == nullptr || lse == nullptr || w == nullptr))
    return GRPO_ERR_INVALID_ARG;
  const size_t esize = dtype == GRPO_F32 ? 4 : 2;
  if (!aligned(logits, esize) || !aligned(dlogits, esize) || !aligned(input_ids, 8) ||
      !aligned(len, 4) || !aligned(lse, 4) || !aligned(w, 4) || !aligned(grad_loss, 4))
    return GRPO_ERR_MISALIGNED;
  const size_t bytes = (size_t)mul3(N, P + C, V) * esize;
  const char* lo = static_cast<const char*>(logits);
  const char* dl = static_cast<const char*>(dlogits);
  if (logits != nullptr && dl < lo + bytes && lo < dl + bytes) return GRPO_ERR_INVALID_ARG;

  BwdArgs a;
  a.logits = logits;
  a.dtype = dtype == GRPO_F32 ? 0 : 1;
  a.N = N;
  a.P = P;
  a.C = C;
  a.V = V;
  a.ids = input_ids;
  a.len = len;
  a.lse = lse;
  a.w = w;
  a.grad = grad_loss;
  a.dlogits = dlogits;
  a.skip_zero_weight = (flags & GRPO_BWD_SKIP_ZERO_WEIGHT) != 0;
  DeviceInfo d;
  if (current_device(&d) != cudaSuccess) return GRPO_ERR_CUDA;
  {
    // before its wait the backward writes dlogits (zero rows) and reads len
    const CallRecord last = stream_take_last(stream);
    a.after_fwd = last.kind == kLastLossFwd &&
                  disjoint_from(last, span(dlogits, bytes), span(len, sizeof(int32_t) * (size_t)N));
  }
  return from_cuda(launch_dlogits(a, d, (cudaStream_t)stream));
}

grpo_status grpo_loss_bwd(const void* logits, grpo_dtype dtype, int64_t N, int64_t P, int64_t C,
                          int64_t V, const int64_t* input_ids, const int32_t* len,
                          const float* lse, const float* w, const float* grad_loss,
                          void* dlogits, grpo_stream_t stream) {
  return grpo_loss_bwd_ex(logits, dtype, N, P, C, V, input_ids, len, lse, w, grad_loss, dlogits, 0u,
                          stream);
}

}  // extern "C"

namespace {

// Launches prep and the gather of the scored rows from host memory (through
// the buffer's device mapping `host_src`) into the same rows of `staging`.
grpo_status launch_host_gather(const void* host_src, void* staging, size_t esize, int64_t N,
                               int64_t P, int64_t C, int64_t V, const int32_t* len,
                               void* workspace, const DeviceInfo& d, cudaStream_t st) {
  FwdArgs a = {};
  a.N = N;
  a.P = P;
  a.C = C;
  a.V = V;
  a.len = len;
  a.ws = workspace;
  if (launch_prep(a, st) != cudaSuccess) return GRPO_ERR_CUDA;
  return from_cuda(launch_gather_host_rows(host_src, staging, esize, a, d, st));
}

// grpo_loss_fwd_bwd_ex; with host_src (the device mapping of page-locked
// host logits, validated by the caller) the scored rows are first gathered
// from it into `logits`, the staging buffer.
grpo_status fwd_bwd_impl(const void* logits, grpo_dtype dtype, int64_t N, int64_t P, int64_t C,
                         int64_t V, const int64_t* input_ids, const int32_t* len,
                         const float* adv, const float* old_logp, const float* ref_logp,
                         float eps, float beta, float norm, grpo_aggregation agg,
                         const float* grad_loss, float* logp, float* lse, float* w, float* loss,
                         void* dlogits, void* workspace, size_t workspace_bytes,
                         grpo_stream_t stream, const void* host_src) {
  if (agg != GRPO_AGG_TOKEN_SUM && agg != GRPO_AGG_SEQ_MEAN) return GRPO_ERR_UNSUPPORTED;
  grpo_status s = check_shapes(dtype, N, P, C, V);
  if (s != GRPO_OK) return s;
  const size_t esize = dtype == GRPO_F32 ? 4 : 2;
  if (N > 0 && dlogits == nullptr) return GRPO_ERR_INVALID_ARG;
  if (!aligned(dlogits, esize) || !aligned(grad_loss, 4)) return GRPO_ERR_MISALIGNED;
  if (N > 0 && logits != nullptr) {
    const size_t bytes = (size_t)mul3(N, P + C, V) * esize;
    const char* lo = static_cast<const char*>(logits);
    const char* dl = static_cast<const char*>(dlogits);
    if (dl < lo + bytes && lo < dl + bytes) return GRPO_ERR_INVALID_ARG;
  }
  const bool same_phase = ((reinterpret_cast<uintptr_t>(logits) ^
                            reinterpret_cast<uintptr_t>(dlogits)) & 15u) == 0;
  if (N > 0 && C > 0) {
    // the forward's validation (pointers, eps, beta, norm, workspace), before
    // anything is enqueued
    if (!(eps >= 0.f && eps < 1.f) || !(beta >= 0.f) || isinf(beta) || isnan(norm) ||
        isinf(norm))
      return GRPO_ERR_INVALID_ARG;
    if (loss == nullptr || workspace == nullptr || len == nullptr || adv == nullptr ||
        logits == nullptr || input_ids == nullptr || logp == nullptr || lse == nullptr ||
        w == nullptr)
      return GRPO_ERR_INVALID_ARG;
    if (beta != 0.f && ref_logp == nullptr) return GRPO_ERR_INVALID_ARG;
    if (!aligned(logits, esize) || !aligned(input_ids, 8) || !aligned(len, 4) ||
        !aligned(adv, 4) || !aligned(old_logp, 4) || !aligned(ref_logp, 4) ||
        !aligned(logp, 4) || !aligned(lse, 4) || !aligned(w, 4) || !aligned(loss, 4) ||
        !aligned(workspace, 256))
      return GRPO_ERR_MISALIGNED;
    if (workspace_bytes < ws_layout(N).total) return GRPO_ERR_WORKSPACE;
  }
  if (N == 0 || C == 0 || !same_phase) {  // nothing to fuse, or no common vector grid
    if (host_src != nullptr && N > 0 && C > 0) {
      DeviceInfo d;
      if (current_device(&d) != cudaSuccess) return GRPO_ERR_CUDA;
      stream_take_after_fwd((cudaStream_t)stream);
      s = launch_host_gather(host_src, const_cast<void*>(logits), esize, N, P, C, V, len,
                             workspace, d, (cudaStream_t)stream);
      if (s != GRPO_OK) return s;
    }
    s = grpo_loss_fwd_ex(logits, dtype, N, P, C, V, input_ids, len, adv, old_logp, ref_logp, eps,
                         beta, norm, agg, logp, lse, w, loss, workspace, workspace_bytes, stream);
    if (s != GRPO_OK) return s;
    return grpo_loss_bwd(logits, dtype, N, P, C, V, input_ids, len, lse, w, grad_loss, dlogits,
                         stream);
  }

  FwdArgs a;
  a.logits = logits;
  a.dtype = dtype == GRPO_F32 ? 0 : 1;
  a.N = N;
  a.P = P;
  a.C = C;
  a.V = V;
  a.ids = input_ids;
  a.len = len;
  a.adv = adv;
  a.old_logp = old_logp;
  a.ref_logp = beta != 0.f ? ref_logp : nullptr;
  a.eps = eps;
  a.beta = beta;
  a.norm = norm;
  a.agg = (int)agg;
  a.logp = logp;
  a.lse = lse;
  a.w = w;
  a.loss = loss;
  a.ws = workspace;
  BwdArgs b;
  b.logits = logits;
  b.dtype = a.dtype;
  b.N = N;
  b.P = P;
  b.C = C;
  b.V = V;
  b.ids = input_ids;
  b.len = len;
  b.lse = lse;
  b.w = w;
  b.grad = grad_loss;
  b.dlogits = dlogits;
  b.skip_zero_weight = false;
  b.after_fwd = false;
  const cudaStream_t st = (cudaStream_t)stream;
  DeviceInfo d;
  if (current_device(&d) != cudaSuccess) return GRPO_ERR_CUDA;
  stream_take_after_fwd(st);
  if (host_src != nullptr && ((reinterpret_cast<uintptr_t>(host_src) ^
                               reinterpret_cast<uintptr_t>(logits)) & 15u) == 0) {
    // The gradient kernel reads the scored rows from host memory itself
    // (writing them to the staging buffer for its second pass), so its
    // arithmetic runs while the rows cross the host link; the zero writer
    // runs beside it (this variant holds no head slots in shared memory).
    FwdArgs ah = a;
    ah.logits = host_src;
    if (launch_prep(ah, st) != cudaSuccess) return GRPO_ERR_CUDA;
    if (launch_lse_grad_host(ah, b, const_cast<void*>(logits), d, st) != cudaSuccess)
      return GRPO_ERR_CUDA;
    return from_cuda(launch_zero_rows(b, d, st, logp, lse, w));
  }
  if (host_src != nullptr) {
    // Host rows in another 16-byte phase than the staging buffer: gather them
    // first.  The zero writer goes between the gather and the gradient kernel:
    // it needs no logits, so it writes while the gather waits on the host link
    // (it does not wait on the gather; its CTA 0 waits before exiting, so the
    // gradient kernel, which waits on it, sees the gathered rows).
    grpo_status g = launch_host_gather(host_src, const_cast<void*>(logits), esize, N, P, C, V,
                                       len, workspace, d, st);
    if (g != GRPO_OK) return g;
    if (launch_zero_rows(b, d, st, logp, lse, w) != cudaSuccess) return GRPO_ERR_CUDA;
    return from_cuda(launch_lse_grad(a, b, d, st));
  }
  if (launch_prep(a, st) != cudaSuccess) return GRPO_ERR_CUDA;
  if (launch_lse_grad(a, b, d, st) != cudaSuccess) return GRPO_ERR_CUDA;
  return from_cuda(launch_zero_rows(b, d, st, logp, lse, w));
}

}  // namespace

extern "C" {

grpo_status grpo_loss_fwd_bwd_ex(const void* logits, grpo_dtype dtype, int64_t N, int64_t P,
                                 int64_t C, int64_t V, const int64_t* input_ids,
                                 const int32_t* len, const float* adv, const float* old_logp,
                                 const float* ref_logp, float eps, float beta, float norm,
                                 grpo_aggregation agg, const float* grad_loss, float* logp,
                                 float* lse, float* w, float* loss, void* dlogits, void* workspace,
                                 size_t workspace_bytes, grpo_stream_t stream) {
  return fwd_bwd_impl(logits, dtype, N, P, C, V, input_ids, len, adv, old_logp, ref_logp, eps,
                      beta, norm, agg, grad_loss, logp, lse, w, loss, dlogits, workspace,
                      workspace_bytes, stream, nullptr);
}

// [p, p + bytes) must be page-locked host memory the device can address:
// its first and its last byte both registered host memory, mapped by the
// device `bytes - 1` apart (a buffer pinned or registered shorter than the
// array fails the second test).  *dev_ptr receives the device address of p.
static grpo_status host_range(const void* p, size_t bytes, void** dev_ptr) {
  cudaPointerAttributes first, last;
  if (cudaPointerGetAttributes(&first, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return GRPO_ERR_INVALID_ARG;
  }
  if (first.type != cudaMemoryTypeHost || first.devicePointer == nullptr)
    return GRPO_ERR_INVALID_ARG;
  const char* end = static_cast<const char*>(p) + (bytes - 1);
  if (cudaPointerGetAttributes(&last, end) != cudaSuccess) {
    (void)cudaGetLastError();
    return GRPO_ERR_INVALID_ARG;
  }
  if (last.type != cudaMemoryTypeHost ||
      static_cast<const char*>(last.devicePointer) !=
          static_cast<const char*>(first.devicePointer) + (bytes - 1))
    return GRPO_ERR_INVALID_ARG;
  *dev_ptr = first.devicePointer;
  return GRPO_OK;
}

grpo_status grpo_loss_fwd_bwd_host(const void* host_logits, grpo_dtype dtype, int64_t N,
                                   int64_t P, int64_t C, int64_t V, const int64_t* input_ids,
                                   const int32_t* len, const float* adv, const float* old_logp,
                                   const float* ref_logp, float eps, float beta, float norm,
                                   const float* grad_loss, float* logp, float* lse, float* w,
                                   float* loss, void* dlogits, void* staging, void* workspace,
                                   size_t workspace_bytes, grpo_stream_t stream) {
  grpo_status s = check_shapes(dtype, N, P, C, V);
  if (s != GRPO_OK) return s;
  const size_t esize = dtype == GRPO_F32 ? 4 : 2;
  const size_t bytes = (size_t)mul3(N, P + C, V) * esize;
  // dlogits: device memory, or page-locked host memory (all of it) that the
  // kernels write through its device mapping, across the host link
  void* dl_dev = dlogits;
  bool dl_host = false;
  if (dlogits != nullptr && bytes > 0) {
    cudaPointerAttributes da;
    if (cudaPointerGetAttributes(&da, dlogits) != cudaSuccess) {
      (void)cudaGetLastError();
      return GRPO_ERR_INVALID_ARG;
    }
    if (da.type == cudaMemoryTypeUnregistered) return GRPO_ERR_INVALID_ARG;  // pageable
    if (da.type == cudaMemoryTypeHost) {
      s = host_range(dlogits, bytes, &dl_dev);
      if (s != GRPO_OK) return s;
      dl_host = true;
    }
  }
  if (N == 0 || C == 0)
    return grpo_loss_fwd_bwd(staging, dtype, N, P, C, V, input_ids, len, adv, old_logp, ref_logp,
                             eps, beta, norm, grad_loss, logp, lse, w, loss, dl_dev, workspace,
                             workspace_bytes, stream);
  if (host_logits == nullptr || staging == nullptr || len == nullptr || workspace == nullptr)
    return GRPO_ERR_INVALID_ARG;
  if (!aligned(host_logits, esize) || !aligned(staging, esize) || !aligned(len, 4) ||
      !aligned(workspace, 256))
    return GRPO_ERR_MISALIGNED;
  if (workspace_bytes < ws_layout(N).total) return GRPO_ERR_WORKSPACE;
  // the logits must be page-locked host memory the device can address, all
  // of it: the kernels read any scored row, up to the last byte
  void* host_dev = nullptr;
  s = host_range(host_logits, bytes, &host_dev);
  if (s != GRPO_OK) return s;
  // dlogits overlaps neither the logits nor the staging buffer
  const char* dl = static_cast<const char*>(dlogits);
  const char* other = dl_host ? static_cast<const char*>(host_logits)
                              : static_cast<const char*>(staging);
  if (dlogits != nullptr && dl < other + bytes && other < dl + bytes) return GRPO_ERR_INVALID_ARG;
  return fwd_bwd_impl(staging, dtype, N, P, C, V, input_ids, len, adv, old_logp, ref_logp, eps,
                      beta, norm, GRPO_AGG_TOKEN_SUM, grad_loss, logp, lse, w, loss, dl_dev,
                      workspace, workspace_bytes, stream, host_dev);
}

grpo_status grpo_loss_fwd_bwd(const void* logits, grpo_dtype dtype, int64_t N, int64_t P,
                              int64_t C, int64_t V, const int64_t* input_ids, const int32_t* len,
                              const float* adv, const float* old_logp, const float* ref_logp,
                              float eps, float beta, float norm, const float* grad_loss,
                              float* logp, float* lse, float* w, float* loss, void* dlogits,
                              void* workspace, size_t workspace_bytes, grpo_stream_t stream) {
  return grpo_loss_fwd_bwd_ex(logits, dtype, N, P, C, V, input_ids, len, adv, old_logp, ref_logp,
                              eps, beta, norm, GRPO_AGG_TOKEN_SUM, grad_loss, logp, lse, w, loss,
                              dlogits, workspace, workspace_bytes, stream);
}

grpo_status grpo_lmhead_workspace_size(int64_t N, int64_t C, int64_t V, int64_t d,
                                       size_t* bytes) {
  if (bytes == nullptr || N < 0 || C < 0 || V < 1) return GRPO_ERR_INVALID_ARG;
  if (d < 128 || d % 128 != 0) return GRPO_ERR_UNSUPPORTED;
  if (N > 0 && C > 0 && N > (int64_t)INT32_MAX / C) return GRPO_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if (current_device(&dev) != cudaSuccess) return GRPO_ERR_CUDA;
  *bytes = lm_layout(N, C, d, dev.sms).total;
  return GRPO_OK;
}

}  // extern "C"

namespace {

// Checks shared by the LM-head calls (bf16 hidden [N, P+C, d], weight [V, d]).
grpo_status lmhead_check(const void* hidden, const void* weight, int64_t N, int64_t P, int64_t C,
                         int64_t V, int64_t d, const int64_t* input_ids, const int32_t* len,
                         const void* workspace) {
  grpo_status s = check_shapes(GRPO_BF16, N, P, C, V);
  if (s != GRPO_OK) return s;
  if (d < 128 || d % 128 != 0) return GRPO_ERR_UNSUPPORTED;
  if (V > (int64_t)INT32_MAX - 256 || mul3(N, P + C, d) < 0) return GRPO_ERR_UNSUPPORTED;
  if (workspace == nullptr || (N > 0 && len == nullptr)) return GRPO_ERR_INVALID_ARG;
  if (N > 0 && C > 0 && (hidden == nullptr || weight == nullptr || input_ids == nullptr))
    return GRPO_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(input_ids, 8) || !aligned(len, 4) ||
      !aligned(workspace, 256))
    return GRPO_ERR_MISALIGNED;
  return GRPO_OK;
}

// mode 0: log-probs only; 1: log-probs, then the loss.
grpo_status lmhead_fwd_impl(const void* hidden, const void* weight, int64_t N, int64_t P, int64_t C,
                            int64_t V, int64_t d, const int64_t* input_ids, const int32_t* len,
                            const float* adv, const float* old_logp, const float* ref_logp,
                            float eps, float beta, float norm, int agg, float* logp, float* lse,
                            float* w, float* loss, void* workspace, size_t workspace_bytes,
                            grpo_stream_t stream, int mode) {
  if (agg != GRPO_AGG_TOKEN_SUM && agg != GRPO_AGG_SEQ_MEAN) return GRPO_ERR_UNSUPPORTED;
  grpo_status s = lmhead_check(hidden, weight, N, P, C, V, d, input_ids, len, workspace);
  if (s != GRPO_OK) return s;
  if (N > 0 && C > 0 && (logp == nullptr || lse == nullptr)) return GRPO_ERR_INVALID_ARG;
  if (mode == 1) {
    if (!(eps >= 0.f && eps < 1.f) || !(beta >= 0.f) || isinf(beta) || isnan(norm) ||
        isinf(norm))
      return GRPO_ERR_INVALID_ARG;
    if (loss == nullptr || (N > 0 && adv == nullptr) || (N > 0 && C > 0 && w == nullptr))
      return GRPO_ERR_INVALID_ARG;
    if (beta != 0.f && ref_logp == nullptr && N > 0 && C > 0) return GRPO_ERR_INVALID_ARG;
  }
  if (!aligned(logp, 4) || !aligned(lse, 4) || !aligned(adv, 4) || !aligned(old_logp, 4) ||
      !aligned(ref_logp, 4) || !aligned(w, 4) || !aligned(loss, 4))
    return GRPO_ERR_MISALIGNED;
  DeviceInfo dev;
  if (current_device(&dev) != cudaSuccess) return GRPO_ERR_CUDA;
  if (workspace_bytes < lm_layout(N, C, d, dev.sms).total) return GRPO_ERR_WORKSPACE;
  stream_take_after_fwd(stream);
  FwdArgs a = {};
  a.dtype = 1;
  a.N = N;
  a.P = P;
  a.C = C;
  a.V = V;
  a.ids = input_ids;
  a.len = len;
  a.adv = adv;
  a.old_logp = old_logp;
  a.ref_logp = beta != 0.f ? ref_logp : nullptr;
  a.eps = eps;
  a.beta = beta;
  a.norm = norm;
  a.agg = agg;
  a.logp = logp;
  a.lse = lse;
  a.w = w;
  a.loss = loss;
  a.ws = workspace;
  const cudaStream_t st = (cudaStream_t)stream;
  if (launch_prep(a, st) != cudaSuccess) return GRPO_ERR_CUDA;
  if (N == 0 || C == 0)
    return mode == 1 ? from_cuda(cudaMemsetAsync(loss, 0, sizeof(float), st)) : GRPO_OK;
  cudaError_t e = launch_lmhead(hidden, weight, a, d, dev, st);
  if (e != cudaSuccess || mode == 0) return from_cuda(e);
  return from_cuda(launch_surrogate(a, st));
}

}  // namespace

extern "C" {

grpo_status grpo_lmhead_logprobs(const void* hidden, const void* weight, int64_t N, int64_t P,
                                 int64_t C, int64_t V, int64_t d, const int64_t* input_ids,
                                 const int32_t* len, float* logp, float* lse, void* workspace,
                                 size_t workspace_bytes, grpo_stream_t stream) {
  return lmhead_fwd_impl(hidden, weight, N, P, C, V, d, input_ids, len, nullptr, nullptr, nullptr,
                         0.f, 0.f, 0.f, GRPO_AGG_TOKEN_SUM, logp, lse, nullptr, nullptr, workspace,
                         workspace_bytes, stream, 0);
}

grpo_status grpo_lmhead_loss_fwd(const void* hidden, const void* weight, int64_t N, int64_t P,
                                 int64_t C, int64_t V, int64_t d, const int64_t* input_ids,
                                 const int32_t* len, const float* adv, const float* old_logp,
                                 const float* ref_logp, float eps, float beta, float norm,
                                 float* logp, float* lse, float* w, float* loss, void* workspace,
                                 size_t workspace_bytes, grpo_stream_t stream) {
  return lmhead_fwd_impl(hidden, weight, N, P, C, V, d, input_ids, len, adv, old_logp, ref_logp,
                         eps, beta, norm, GRPO_AGG_TOKEN_SUM, logp, lse, w, loss, workspace,
                         workspace_bytes, stream, 1);
}

grpo_status grpo_lmhead_loss_fwd_ex(const void* hidden, const void* weight, int64_t N, int64_t P,
                                    int64_t C, int64_t V, int64_t d, const int64_t* input_ids,
                                    const int32_t* len, const float* adv, const float* old_logp,
                                    const float* ref_logp, float eps, float beta, float norm,
                                    grpo_aggregation agg, float* logp, float* lse, float* w,
                                    float* loss, void* workspace, size_t workspace_bytes,
                                    grpo_stream_t stream) {
  return lmhead_fwd_impl(hidden, weight, N, P, C, V, d, input_ids, len, adv, old_logp, ref_logp,
                         eps, beta, norm, (int)agg, logp, lse, w, loss, workspace, workspace_bytes,
                         stream, 1);
}

grpo_status grpo_lmhead_bwd_workspace_size_rows(int64_t N, int64_t C, int64_t V, int64_t d,
                                                int64_t rows_per_pass, size_t* bytes) {
  if (bytes == nullptr || N < 0 || C < 0 || V < 1 || rows_per_pass < 0)
    return GRPO_ERR_INVALID_ARG;
  if (d < 128 || d % 128 != 0) return GRPO_ERR_UNSUPPORTED;
  if (N > 0 && C > 0 && N > (int64_t)INT32_MAX / C) return GRPO_ERR_UNSUPPORTED;
  if (V > (int64_t)INT32_MAX - 256) return GRPO_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if (current_device(&dev) != cudaSuccess) return GRPO_ERR_CUDA;
  *bytes = lm_bwd_layout(N, C, V, d, dev.sms, rows_per_pass).total;
  return GRPO_OK;
}

grpo_status grpo_lmhead_bwd_workspace_size(int64_t N, int64_t C, int64_t V, int64_t d,
                                           size_t* bytes) {
  return grpo_lmhead_bwd_workspace_size_rows(N, C, V, d, 0, bytes);
}

grpo_status grpo_lmhead_loss_bwd(const void* hidden, const void* weight, int64_t N, int64_t P,
                                 int64_t C, int64_t V, int64_t d, const int64_t* input_ids,
                                 const int32_t* len, const float* lse, const float* w,
                                 const float* grad_loss, float* dhidden, float* dweight,
                                 void* workspace, size_t workspace_bytes, grpo_stream_t stream) {
  return grpo_lmhead_loss_bwd_ex(hidden, weight, N, P, C, V, d, input_ids, len, lse, w, grad_loss,
                                 dhidden, dweight, 0u, workspace, workspace_bytes, stream);
}

grpo_status grpo_lmhead_loss_bwd_ex(const void* hidden, const void* weight, int64_t N, int64_t P,
                                    int64_t C, int64_t V, int64_t d, const int64_t* input_ids,
                                    const int32_t* len, const float* lse, const float* w,
                                    const float* grad_loss, float* dhidden, float* dweight,
                                    uint32_t flags, void* workspace, size_t workspace_bytes,
                                    grpo_stream_t stream) {
  if (flags & ~GRPO_BWD_SKIP_ZERO_WEIGHT) return GRPO_ERR_UNSUPPORTED;
  grpo_status s = lmhead_check(hidden, weight, N, P, C, V, d, input_ids, len, workspace);
  if (s != GRPO_OK) return s;
  if (dweight == nullptr || (N > 0 && dhidden == nullptr)) return GRPO_ERR_INVALID_ARG;
  if (N > 0 && C > 0 && (lse == nullptr || w == nullptr)) return GRPO_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !aligned(w, 4) || !aligned(grad_loss, 4) || !aligned(dhidden, 16) ||
      !aligned(dweight, 16))
    return GRPO_ERR_MISALIGNED;
  DeviceInfo dev;
  if (current_device(&dev) != cudaSuccess) return GRPO_ERR_CUDA;
  // rows per pass: as many as the workspace holds (every possible row when it
  // is grpo_lmhead_bwd_workspace_size bytes), at least one block of 256
  const int64_t blocks = (N * C + 255) / 256;
  int64_t lo = 1, hi = blocks > 0 ? blocks : 1;
  if (workspace_bytes < lm_bwd_layout(N, C, V, d, dev.sms, 256).total) return GRPO_ERR_WORKSPACE;
  while (lo < hi) {  // the layout grows with the rows per pass
    const int64_t mid = (lo + hi + 1) / 2;
    if (lm_bwd_layout(N, C, V, d, dev.sms, mid * 256).total <= workspace_bytes)
      lo = mid;
    else
      hi = mid - 1;
  }
  const LmBwdLayout bl = lm_bwd_layout(N, C, V, d, dev.sms, lo * 256);
  stream_take_after_fwd(stream);
  FwdArgs f = {};
  f.N = N;
  f.P = P;
  f.C = C;
  f.V = V;
  f.len = len;
  f.ws = workspace;
  const cudaStream_t st = (cudaStream_t)stream;
  if (launch_prep(f, st) != cudaSuccess) return GRPO_ERR_CUDA;
  if (N == 0 || C == 0) {  // nothing is scored: both gradients are zero
    if (cudaMemsetAsync(dweight, 0, (size_t)V * (size_t)d * 4, st) != cudaSuccess)
      return GRPO_ERR_CUDA;
    const int64_t nh = mul3(N, P + C, d);
    return nh == 0 ? GRPO_OK : from_cuda(cudaMemsetAsync(dhidden, 0, (size_t)nh * 4, st));
  }
  LmBwdArgs a;
  a.hidden = hidden;
  a.weight = weight;
  a.N = N;
  a.P = P;
  a.C = C;
  a.V = V;
  a.d = d;
  a.ids = input_ids;
  a.lse = lse;
  a.w = w;
  a.grad = grad_loss;
  a.dhidden = dhidden;
  a.dweight = dweight;
  a.ws = workspace;
  a.rows_pass = bl.rows_pass;
  a.skip_zero_weight = (flags & GRPO_BWD_SKIP_ZERO_WEIGHT) != 0;
  if (launch_lmhead_bwd_rows(a, dev, st) != cudaSuccess) return GRPO_ERR_CUDA;
  for (int64_t pass = 0; pass < bl.npass; ++pass) {
    if (launch_lmhead_dz(a, pass, dev, st) != cudaSuccess) return GRPO_ERR_CUDA;
    cudaError_t e = launch_lmhead_grads(a, pass, dev, st);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return GRPO_OK;
}

grpo_status grpo_check_error(const void* workspace, grpo_stream_t stream) {
  if (workspace == nullptr) return GRPO_ERR_INVALID_ARG;
  uint32_t flags = 0;
  const cudaStream_t st = (cudaStream_t)stream;
  stream_take_after_fwd(st);
  if (cudaMemcpyAsync(&flags, workspace, sizeof flags, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return GRPO_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GRPO_ERR_CUDA;
  if (flags & kFlagTokenRange) return GRPO_ERR_TOKEN_RANGE;
  if (flags & kFlagLengthRange) return GRPO_ERR_LENGTH_RANGE;
  if (flags & kFlagTimeout) return GRPO_ERR_TIMEOUT;
  return GRPO_OK;
}

void grpo_set_early_start(int enable) { g_early_start.store(enable != 0 ? 1 : 0); }

grpo_status grpo_selftest_timeout(void* workspace, grpo_stream_t stream) {
  if (workspace == nullptr) return GRPO_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return GRPO_ERR_MISALIGNED;
  stream_take_after_fwd(stream);
  return from_cuda(launch_selftest_timeout(workspace, (cudaStream_t)stream));
}

grpo_status grpo_copy(void* dst, const void* src, size_t bytes, grpo_stream_t stream) {
  if (bytes == 0) return GRPO_OK;
  if (dst == nullptr || src == nullptr) return GRPO_ERR_INVALID_ARG;
  if (!aligned(dst, 16) || !aligned(src, 16) || bytes % 16 != 0) return GRPO_ERR_MISALIGNED;
  const char* d8 = static_cast<const char*>(dst);
  const char* s8 = static_cast<const char*>(src);
  if (d8 < s8 + bytes && s8 < d8 + bytes) return GRPO_ERR_INVALID_ARG;
  DeviceInfo d;
  if (current_device(&d) != cudaSuccess) return GRPO_ERR_CUDA;
  stream_take_after_fwd(stream);
  return from_cuda(launch_copy(dst, src, bytes, d, (cudaStream_t)stream));
}

}  // extern "C"

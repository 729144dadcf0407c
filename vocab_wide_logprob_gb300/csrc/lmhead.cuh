// Internal header of the LM-head kernels (the projection logits = H W^T on
// the tensor cores, forward and backward): workspace layouts and launchers
// that api.cu calls.
#pragma once

#include "common.cuh"

namespace grpo {

// LM-head log-probs (tensor cores): workspace beyond the base layout holds a
// dense copy of the scored rows' hidden states and the per-item partials.
struct LmLayout {
  size_t geometry;  // int4: row blocks, vocabulary splits, tiles per split
  size_t dense;     // bf16 [N*C rounded up to 256, d]
  size_t partials;  // float4 [items][256]
  size_t counters;  // uint32 [N*C rounded up to 256]: partials written per row
  size_t total;
};
LmLayout lm_layout(int64_t N, int64_t C, int64_t d, int sms);
// After launch_prep: gather, then the tensor-core log-sum-exp (whose last
// partial of a row merges the row).
cudaError_t launch_lmhead(const void* hidden, const void* weight, const FwdArgs& a, int64_t d,
                          const DeviceInfo& dev, cudaStream_t st);

// Gradients through the LM head.  The backward rows (the scored tokens, or
// those whose g * w is not 0) run in passes of up to rows_pass rows each:
// every pass forms its rows' bf16 logits gradient and both contractions over
// it (dweight is stored by the first pass and added to by the others), so the
// logits-gradient buffer holds rows_pass rows, not every possible row.
// Workspace beyond the base layout: the geometries, the row maps, the dense
// scored hidden rows, one pass's bf16 logits gradient and the split partials
// of one pass's hidden-state gradient.
struct LmBwdLayout {
  size_t geometry;     // int4 [3 + 2 * npass]: [2].x = rows; per pass p: [3 + 2p] the
                       // projection pass, [4 + 2p] the hidden-gradient contraction
  size_t rowmap;       // int32 [N*C]: the token i*C + t of each backward row
  size_t tokrow;       // int32 [N*C]: the backward row of token i*C + t, or -1
  size_t dense;        // bf16 [rows_cap, d]
  size_t dz;           // bf16 [ldz / 64][rows_pass][64] (vocabulary slabs of one pass)
  size_t dh_partials;  // fp32 [items_max][256][512]
  size_t total;
  int64_t rows_cap;    // N*C rounded up to 256
  int64_t rows_pass;   // backward rows per pass: a multiple of 256, <= rows_cap
  int64_t npass;       // rows_cap / rows_pass, rounded up
  int64_t ldz;         // V rounded up to 256
  int64_t items_max;
};
// rows_pass <= 0 or >= N*C: one pass over every possible row.
LmBwdLayout lm_bwd_layout(int64_t N, int64_t C, int64_t V, int64_t d, int sms,
                          int64_t rows_pass = 0);
inline int lm_geo_proj(int64_t pass) { return 3 + 2 * (int)pass; }
inline int lm_geo_dh(int64_t pass) { return 4 + 2 * (int)pass; }
struct LmBwdArgs {
  const void* hidden;   // bf16 [N, P+C, d]
  const void* weight;   // bf16 [V, d]
  int64_t N, P, C, V, d;
  const int64_t* ids;
  const float* lse;     // [N, C]
  const float* w;       // [N, C]
  const float* grad;    // nullable: 1
  float* dhidden;       // fp32 [N, P+C, d]
  float* dweight;       // fp32 [V, d]
  void* ws;
  int64_t rows_pass;    // the layout's rows per pass
  bool skip_zero_weight;  // rows whose g * w is exactly 0 take no part (their dhidden is 0)
};
// CTA pairs of the tensor-core kernels on this device.
int lm_pairs(const DeviceInfo& dev);
// After launch_prep: the backward rows, the dense hidden rows and every pass's
// geometries.
cudaError_t launch_lmhead_bwd_rows(const LmBwdArgs& a, const DeviceInfo& dev, cudaStream_t st);
// Pass `pass`: the logits gradient of its rows.
cudaError_t launch_lmhead_dz(const LmBwdArgs& a, int64_t pass, const DeviceInfo& dev,
                             cudaStream_t st);
// After launch_lmhead_dz of the same pass: the hidden-state and weight
// gradient contractions over its rows.
cudaError_t launch_lmhead_grads(const LmBwdArgs& a, int64_t pass, const DeviceInfo& dev,
                                cudaStream_t st);

}  // namespace grpo

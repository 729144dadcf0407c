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

// Gradients through the LM head.  Workspace beyond the base layout: the two
// geometries, the dense scored hidden rows, the bf16 logits gradient of the
// scored rows, and the split partials of the hidden-state gradient.
struct LmBwdLayout {
  size_t geometry;     // int4[3]: projection pass; hidden-gradient contraction; (rows, ...)
  size_t rowmap;       // int32 [N*C]: the token i*C + t of each backward row
  size_t tokrow;       // int32 [N*C]: the backward row of token i*C + t, or -1
  size_t dense;        // bf16 [rows_cap, d]
  size_t dz;           // bf16 [ldz / 64][rows_cap][64] (vocabulary slabs)
  size_t dh_partials;  // fp32 [items_max][256][512]
  size_t total;
  int64_t rows_cap;    // N*C rounded up to 256
  int64_t ldz;         // V rounded up to 256
  int64_t items_max;
};
LmBwdLayout lm_bwd_layout(int64_t N, int64_t C, int64_t V, int64_t d, int sms);
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
  bool skip_zero_weight;  // rows whose g * w is exactly 0 take no part (their dhidden is 0)
};
// CTA pairs of the tensor-core kernels on this device.
int lm_pairs(const DeviceInfo& dev);
// After launch_prep: gather (+ both geometries) and the logits-gradient pass.
cudaError_t launch_lmhead_dz(const LmBwdArgs& a, const DeviceInfo& dev, cudaStream_t st);
// After launch_lmhead_dz: the hidden-state and weight gradient contractions.
cudaError_t launch_lmhead_grads(const LmBwdArgs& a, const DeviceInfo& dev, cudaStream_t st);

}  // namespace grpo

/*
 * grpo.h -- C ABI of the GB300 (sm_103a) Dr. GRPO loss library.
 *
 * The library computes the data-parallel hot path of one Dr. GRPO update
 * step over policy logits, forward and backward, as the page "Making Dr GRPO
 * go brrr" (salahadawi.com, "i-made-a-kernel-22x-faster-it-made-my-training-
 * loop-3x-slower") defines it:
 *
 *   grpo_mask       "The completion mask" (build_completion_mask)
 *   grpo_advantage  "Dr. GRPO": A_i = R_i - mean of the group, no sigma
 *   grpo_loss_fwd   "compute_logprobs" (shift, log_softmax, gather) and
 *                   "The loss" (grpo_loss): clipped surrogate, optional k3 KL
 *                   term, token-sum aggregation divided by a constant
 *   grpo_loss_bwd   "loss.backward()": d loss / d logits
 *
 * Shapes: N = B*G completions (completions b*G .. b*G+G-1 answer prompt b),
 * P prompt tokens, C completion tokens, T = P + C, vocabulary V.  Completion
 * token t of sequence i is input_ids[i, P+t]; it is scored by logits row
 * P-1+t of sequence i ("logits at position t predict the token at t+1").
 *
 * Conventions for every call:
 *  - All array pointers are DEVICE pointers to dense row-major arrays.  The
 *    caller owns all memory; the library never allocates, frees or keeps a
 *    pointer after a call returns.
 *  - Calls only enqueue work on `stream` and return without synchronising,
 *    except grpo_check_error.  Results are bitwise reproducible run to run
 *    for the same inputs and shapes on the same GPU model.
 *  - Arguments are validated on the host before anything is enqueued; a
 *    validation failure returns an error and enqueues nothing.  A failed
 *    launch returns GRPO_ERR_CUDA.  No C++ exception crosses this boundary.
 *  - Data-dependent problems (a scored token id outside [0, V), a length
 *    outside [0, C]) cannot be seen on the host without a synchronisation;
 *    the kernels record them in the workspace and grpo_check_error reports
 *    them.  The kernels never trap.
 *  - Within one call, the output arrays and the workspace must not overlap
 *    one another or that call's inputs (inputs may share memory).  Buffers
 *    of different calls may overlap; stream order then applies.
 *  - Inputs at positions the mask excludes (old_logp and ref_logp past the
 *    first EOS) are never read; outputs there are 0.
 *  - Index arithmetic is 64-bit; N*C must be below 2^31.
 */
#ifndef GRPO_H
#define GRPO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *grpo_stream_t;

typedef enum {
    GRPO_OK = 0,
    GRPO_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad eps/beta/G */
    GRPO_ERR_UNSUPPORTED = 2,  /* dtype or size outside what the kernels take */
    GRPO_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required  */
    GRPO_ERR_MISALIGNED = 4,   /* pointer not aligned as documented           */
    GRPO_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed */
    GRPO_ERR_TOKEN_RANGE = 6,  /* a scored token id was outside [0, V)        */
    GRPO_ERR_LENGTH_RANGE = 7, /* a completion length was outside [0, C]      */
    GRPO_ERR_TIMEOUT = 8       /* a bounded device-side wait gave up          */
} grpo_status;

typedef enum { GRPO_F32 = 0, GRPO_BF16 = 1 } grpo_dtype;

/* Group advantage ("GRPO" and "Dr. GRPO" sections). */
typedef enum {
    GRPO_ADV_DR = 0, /* A = R - mean (Dr. GRPO: no sigma)                        */
    GRPO_ADV_STD = 1 /* A = (R - mean) / (sigma + std_eps) (original GRPO)       */
} grpo_adv_mode;

/* Aggregation of the per-token loss ("Dr. GRPO" section). */
typedef enum {
    GRPO_AGG_TOKEN_SUM = 0, /* sum over valid tokens / norm (Dr. GRPO; norm <= 0: N*C)   */
    GRPO_AGG_SEQ_MEAN = 1   /* sum_i (sum_t / len_i) / norm (original GRPO 1/|o_i|;
                               norm <= 0: N)                                            */
} grpo_aggregation;

/* grpo_loss_bwd_ex flags. */
#define GRPO_BWD_SKIP_ZERO_WEIGHT 1u /* a row whose g*w_t is exactly 0 is written with +0 and
                                        not read (the reads it saves are left out of the
                                        byte count a caller reports)                       */

/* Static English description of a status code. */
const char *grpo_status_string(grpo_status status);

/*
 * grpo_mask -- completion mask ("The completion mask", build_completion_mask).
 *
 * input_ids [N, P+C] int64, 8-byte aligned; only columns P .. P+C-1 (the
 *           completion) are read.
 * mask      [N, C] uint8 out, may be NULL: 1 at positions up to and including
 *           the first id equal to eos_id, 0 after it; every position 1 when
 *           the completion holds no EOS (the torch.where fallback that keeps
 *           argmax's 0 on a row without EOS from masking the completion).
 * len       [N] int32 out: the number of 1s of each mask row, i.e. the first
 *           EOS index + 1, or C.  The loss calls take `len`: the mask is a
 *           prefix of each row.
 * N, P, C >= 0.  N == 0 enqueues nothing.
 */
grpo_status grpo_mask(const int64_t *input_ids, int64_t N, int64_t P, int64_t C,
                      int64_t eos_id, uint8_t *mask, int32_t *len, grpo_stream_t stream);

/*
 * grpo_advantage -- Dr. GRPO group advantage (section "Dr. GRPO": both
 * denominators removed, A_i = R_i - mu; code "rewards_grouped -
 * rewards_grouped.mean(dim=1, keepdim=True)").
 *
 * rewards [B*G] float32, grouped as [B, G]; adv [B*G] float32 out:
 * adv_i = R_i - (sum of the group's rewards) / G, in float32.  For binary
 * rewards and power-of-two G every step is exact.  B >= 0, G >= 1.
 *
 * Stream order: when the library's previous call on this stream (and device)
 * was grpo_mask and rewards and adv are disjoint from that call's mask and
 * len (adv also from its input_ids; the library checks the address ranges),
 * the advantages are computed while that call's kernel may still run;
 * otherwise the call waits for it as usual.  The same holds for
 * grpo_advantage_ex without n_contrast.
 */
grpo_status grpo_advantage(const float *rewards, int64_t B, int64_t G, float *adv,
                           grpo_stream_t stream);

/*
 * grpo_advantage_ex -- grpo_advantage with the original GRPO option and the
 * reward-contrast count.  mode GRPO_ADV_DR is grpo_advantage; GRPO_ADV_STD
 * divides by sigma + std_eps, sigma = sqrt(sum over the group (R - mean)^2 / G)
 * (section "GRPO": "Compute the advantage as A_i = (R_i - mu)/sigma inside the
 * group"); std_eps >= 0 keeps a uniform group at 0.  n_contrast, if not NULL,
 * is one int32 in device memory that receives the number of groups whose
 * rewards are not all equal (the analysis page's "useful groups": a uniform
 * group has no task-reward advantage).
 */
grpo_status grpo_advantage_ex(const float *rewards, int64_t B, int64_t G, grpo_adv_mode mode,
                              float std_eps, float *adv, int32_t *n_contrast,
                              grpo_stream_t stream);

/*
 * grpo_workspace_size -- bytes of device scratch grpo_loss_fwd needs for N
 * completions of C tokens (a few bytes per completion).  The workspace needs
 * no initialisation; grpo_loss_fwd resets what it uses.  It must be 256-byte
 * aligned and must not be shared by calls that may run concurrently.
 */
grpo_status grpo_workspace_size(int64_t N, int64_t C, int64_t V, size_t *bytes);

/*
 * grpo_loss_fwd -- per-token log-probs and the Dr. GRPO loss.
 *
 * logits    [N, P+C, V] of `dtype` (float32 or bfloat16), aligned to its
 *           element size, read-only.  Only the rows that score a valid token
 *           (rows P-1 .. P-2+len_i of sequence i) are read.
 * input_ids [N, P+C] int64; len [N] int32 (from grpo_mask); adv [N] float32.
 * old_logp  [N, C] float32 or NULL.  NULL means the old policy equals the
 *           current one (inner step 0): the ratio is exactly 1.
 * ref_logp  [N, C] float32; may be NULL only when beta == 0.
 * eps in [0, 1): clip range; beta >= 0: k3 KL weight.
 * norm      the constant the token sum is divided by; norm <= 0 selects N*C
 *           (the padded completion width times N).  P >= 1.
 *
 * Per valid token (t < len_i), with y = input_ids[i, P+t] and z the logits
 * row P-1+t of sequence i:
 *   lse   = log sum_v exp(z_v)                  (float32 accumulation)
 *   logp  = z_y - lse
 *   r     = exp(logp - old)                     (1 when old_logp == NULL)
 *   s     = min(r*A_i, clamp(r, 1-eps, 1+eps)*A_i)
 *   k3    = exp(ref - logp) - (ref - logp) - 1  (0 when beta == 0)
 *   ell   = -s + beta*k3
 *   w     = d loss / d logp = (-(r*A_i if min() selects r*A_i, else 0)
 *                              + beta*(1 - exp(ref - logp))) / norm
 *   loss  = (sum over valid tokens of ell) / norm   (float64 accumulation
 *                                                    in a fixed order)
 * Outputs: logp, lse, w [N, C] float32 (0 past each length); loss: one
 * float32 in device memory.
 * workspace: device scratch of at least grpo_workspace_size bytes.
 */
grpo_status grpo_loss_fwd(const void *logits, grpo_dtype dtype, int64_t N, int64_t P, int64_t C,
                          int64_t V, const int64_t *input_ids, const int32_t *len,
                          const float *adv, const float *old_logp, const float *ref_logp,
                          float eps, float beta, float norm, float *logp, float *lse, float *w,
                          float *loss, void *workspace, size_t workspace_bytes,
                          grpo_stream_t stream);

/*
 * grpo_loss_fwd_static -- grpo_loss_fwd without a workspace argument, for
 * callers that cannot allocate device memory.  The pages have no counterpart:
 * this is a convenience of this library.
 *
 * Who needs it: code that runs where cudaMalloc is off limits -- inside a
 * caching allocator or memory pool that must not be re-entered, in a plugin
 * host that only lends out the buffers it owns, or in a runtime that forbids
 * allocation once it has started.  Such callers still pass all inputs and
 * outputs exactly as for grpo_loss_fwd (same arguments, same results).
 *
 * Scratch: a 64 KiB array compiled into the library as a __device__ variable;
 * every GPU that loads the library holds it until the process exits.  It
 * covers N <= 4096 completions; a larger N returns GRPO_ERR_UNSUPPORTED and
 * enqueues nothing.  Nothing is allocated and no allocating routine is called.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  The address is kept per CUDA context (keyed on
 * the context's id), so after cudaDeviceReset, or in another context made
 * current on the same device, the next call looks it up again; that call too
 * should come before any capture.
 * All calls share the one array and it keeps the last call's contents; each
 * call resets what must start at zero before using it.  Calls whose work can
 * overlap on the GPU (different streams, or different host threads) race on
 * the array and must be serialised by the caller.  Data-dependent errors are
 * recorded in this shared array, so grpo_check_error cannot report them: a
 * scored token id outside [0, V) still shows as a NaN log-prob.
 */
grpo_status grpo_loss_fwd_static(const void *logits, grpo_dtype dtype, int64_t N, int64_t P,
                                 int64_t C, int64_t V, const int64_t *input_ids,
                                 const int32_t *len, const float *adv, const float *old_logp,
                                 const float *ref_logp, float eps, float beta, float norm,
                                 float *logp, float *lse, float *w, float *loss,
                                 grpo_stream_t stream);

/*
 * grpo_loss_fwd_ex -- grpo_loss_fwd with a choice of aggregation:
 * GRPO_AGG_TOKEN_SUM is grpo_loss_fwd; GRPO_AGG_SEQ_MEAN divides each
 * completion's token sum by its length, then the sum over completions by norm
 * (norm <= 0 selects N): the original GRPO's per-response 1/|o_i| mean that
 * Dr. GRPO replaces (section "Dr. GRPO").  w includes the same weights.
 */
grpo_status grpo_loss_fwd_ex(const void *logits, grpo_dtype dtype, int64_t N, int64_t P,
                             int64_t C, int64_t V, const int64_t *input_ids, const int32_t *len,
                             const float *adv, const float *old_logp, const float *ref_logp,
                             float eps, float beta, float norm, grpo_aggregation agg,
                             float *logp, float *lse, float *w, float *loss, void *workspace,
                             size_t workspace_bytes, grpo_stream_t stream);

/*
 * grpo_logprobs -- log-probs only, no loss: the no-grad passes of the update
 * loop ("old_logprobs = policy.logprobs(completions).detach()", the same for
 * the reference policy; section "Dr. GRPO" pseudo-code and "Putting it
 * together").  logp, lse [N, C] float32 as in grpo_loss_fwd (0 past each
 * length); workspace as for grpo_loss_fwd.  grpo_check_error reports token and
 * length errors.
 */
grpo_status grpo_logprobs(const void *logits, grpo_dtype dtype, int64_t N, int64_t P, int64_t C,
                          int64_t V, const int64_t *input_ids, const int32_t *len, float *logp,
                          float *lse, void *workspace, size_t workspace_bytes,
                          grpo_stream_t stream);

/*
 * grpo_loss_bwd -- gradient of (grad_loss * loss) with respect to the logits.
 *
 * Inputs as for grpo_loss_fwd, plus lse and w from it; grad_loss is one
 * float32 in device memory (the upstream gradient of the scalar loss) or NULL
 * for 1.
 * dlogits [N, P+C, V] of `dtype`, fully written:
 *   a row that scores valid token t:  g*w_t*([v == y] - exp(z_v - lse_t)),
 *   every other row (prompt rows 0..P-2, row P+C-1, rows past the first EOS):
 *   0, as autograd through the slice and the mask gives.
 * bfloat16 results are rounded to nearest even from float32.  dlogits must
 * not overlap logits.  Lengths are clamped to [0, C].
 *
 * Stream order: when the library's previous call on this stream (and
 * device) was grpo_loss_fwd or grpo_loss_fwd_ex, and dlogits overlaps none of
 * that call's buffers and len none of the buffers it writes (the library
 * keeps their address ranges and checks), the rows that score nothing are
 * written while that forward's last kernels may still run (they depend only
 * on len); otherwise, and after any other preceding work, the call waits for
 * it as usual.  Either way the results are those of stream order (see
 * grpo_set_early_start for kernels of other code in between).
 */
grpo_status grpo_loss_bwd(const void *logits, grpo_dtype dtype, int64_t N, int64_t P, int64_t C,
                          int64_t V, const int64_t *input_ids, const int32_t *len,
                          const float *lse, const float *w, const float *grad_loss,
                          void *dlogits, grpo_stream_t stream);

/*
 * grpo_loss_bwd_ex -- grpo_loss_bwd with flags (0 or GRPO_BWD_SKIP_ZERO_WEIGHT).
 * With GRPO_BWD_SKIP_ZERO_WEIGHT a scored row whose g*w_t is exactly 0 (a
 * group with no reward contrast and beta == 0, as the analysis page's
 * "no contrast" case) is written with +0 without reading its logits; its exact
 * gradient is (+/-)0 everywhere.
 */
grpo_status grpo_loss_bwd_ex(const void *logits, grpo_dtype dtype, int64_t N, int64_t P,
                             int64_t C, int64_t V, const int64_t *input_ids, const int32_t *len,
                             const float *lse, const float *w, const float *grad_loss,
                             void *dlogits, uint32_t flags, grpo_stream_t stream);

/*
 * grpo_loss_fwd_bwd -- grpo_loss_fwd and grpo_loss_bwd in one pass over each
 * scored row: the row is read from HBM once (its log-sum-exp, log-prob and
 * gradient weight are formed, then its gradient is written) instead of once by
 * each call.  Same method ("compute_logprobs", "The loss", "loss.backward()"),
 * composed per row; it needs the upstream gradient when the forward runs.
 *
 * Arguments: those of grpo_loss_fwd, then grad_loss (one float32 in device
 * memory, or NULL for 1) and dlogits [N, P+C, V] as in grpo_loss_bwd.
 * Results: logp, lse, w and dlogits have the same bits as grpo_loss_fwd
 * followed by grpo_loss_bwd; the loss is summed in another fixed order
 * (per cluster, then clusters in order), so it agrees to float rounding.
 * When logits and dlogits do not start at the same offset modulo 16 bytes the
 * call runs the two passes instead (same results).
 */
grpo_status grpo_loss_fwd_bwd(const void *logits, grpo_dtype dtype, int64_t N, int64_t P,
                              int64_t C, int64_t V, const int64_t *input_ids, const int32_t *len,
                              const float *adv, const float *old_logp, const float *ref_logp,
                              float eps, float beta, float norm, const float *grad_loss,
                              float *logp, float *lse, float *w, float *loss, void *dlogits,
                              void *workspace, size_t workspace_bytes, grpo_stream_t stream);

/*
 * grpo_loss_fwd_bwd_host -- grpo_loss_fwd_bwd for logits that sit in
 * page-locked host memory (cudaHostAlloc, or cudaHostRegister, mapped into the
 * device's address space).  The loss reads only the scored rows, row P-1+t of
 * sequence i for t < len_i ("compute_logprobs" and the completion mask), so
 * only those rows cross the host link, read through the buffer's device
 * mapping, and they are written to the same rows of `staging`, device memory
 * of the logits' shape [N, P+C, V] (its other rows are neither read nor
 * written).  When host_logits, staging and dlogits share their address modulo
 * 16 bytes, the gradient kernel reads the host rows itself and computes while
 * they arrive; otherwise a copy kernel fills `staging` first and
 * grpo_loss_fwd_bwd runs on it.  Results are bit-identical to
 * grpo_loss_fwd_bwd on the same logits in device memory either way.
 *
 * Arguments: those of grpo_loss_fwd_bwd with host_logits for logits, plus
 * staging (device, logits' size, element-aligned, not overlapping dlogits).
 * dlogits may be device memory or, like host_logits, page-locked host memory
 * mapped into the device's address space: the kernels then write every row
 * of the gradient (zero rows included) straight into it across the host link,
 * while the scored rows of the logits come the other way (the results are
 * the same bits; completion of the stream work means the host buffer holds
 * them).  The other pointers are device memory as for grpo_loss_fwd_bwd.
 * Returns GRPO_ERR_INVALID_ARG when host_logits (or a host dlogits) is not
 * page-locked host memory the device can address over its whole size
 * (N*(P+C)*V elements: the first and the last byte are checked), when
 * dlogits is pageable host memory, or when a host dlogits overlaps
 * host_logits.
 */
grpo_status grpo_loss_fwd_bwd_host(const void *host_logits, grpo_dtype dtype, int64_t N,
                                   int64_t P, int64_t C, int64_t V, const int64_t *input_ids,
                                   const int32_t *len, const float *adv, const float *old_logp,
                                   const float *ref_logp, float eps, float beta, float norm,
                                   const float *grad_loss, float *logp, float *lse, float *w,
                                   float *loss, void *dlogits, void *staging, void *workspace,
                                   size_t workspace_bytes, grpo_stream_t stream);

/* grpo_loss_fwd_bwd with the aggregation choice of grpo_loss_fwd_ex. */
grpo_status grpo_loss_fwd_bwd_ex(const void *logits, grpo_dtype dtype, int64_t N, int64_t P,
                                 int64_t C, int64_t V, const int64_t *input_ids,
                                 const int32_t *len, const float *adv, const float *old_logp,
                                 const float *ref_logp, float eps, float beta, float norm,
                                 grpo_aggregation agg, const float *grad_loss, float *logp,
                                 float *lse, float *w, float *loss, void *dlogits, void *workspace,
                                 size_t workspace_bytes, grpo_stream_t stream);

/*
 * grpo_lmhead_logprobs -- log-probs of the sampled tokens straight from the
 * policy's last hidden states, with the LM-head projection fused in: the
 * logits (hidden x W^T, "model(...).logits" in "compute_logprobs") are formed
 * tile by tile on the tensor cores and reduced on the fly, never written to
 * memory.  Same results as grpo_logprobs on logits = hidden x W^T computed in
 * float32 (up to the order of the float32 sums).
 *
 * hidden [N, P+C, d] bfloat16 (row P-1+t of sequence i scores token t);
 * weight [V, d] bfloat16 (the LM head, row v = the output embedding of token
 * v); both 16-byte aligned; d a multiple of 128.  input_ids, len, logp, lse as
 * for grpo_logprobs (0 past each length).  workspace: at least
 * grpo_lmhead_workspace_size bytes (it holds a dense copy of the scored rows'
 * hidden states, 2*d bytes per completion token, and a few KB of partials).
 */
grpo_status grpo_lmhead_workspace_size(int64_t N, int64_t C, int64_t V, int64_t d,
                                       size_t *bytes);
grpo_status grpo_lmhead_logprobs(const void *hidden, const void *weight, int64_t N, int64_t P,
                                 int64_t C, int64_t V, int64_t d, const int64_t *input_ids,
                                 const int32_t *len, float *logp, float *lse, void *workspace,
                                 size_t workspace_bytes, grpo_stream_t stream);

/*
 * grpo_lmhead_loss_fwd -- the Dr. GRPO loss forward from hidden states:
 * grpo_lmhead_logprobs followed by the surrogate, KL and token-sum reduction
 * of grpo_loss_fwd ("The loss", grpo_loss).  Arguments as for those two
 * calls; `workspace` at least grpo_lmhead_workspace_size bytes.  Outputs logp,
 * lse, w and the device scalar loss, with grpo_loss_fwd's meaning.
 */
grpo_status grpo_lmhead_loss_fwd(const void *hidden, const void *weight, int64_t N, int64_t P,
                                 int64_t C, int64_t V, int64_t d, const int64_t *input_ids,
                                 const int32_t *len, const float *adv, const float *old_logp,
                                 const float *ref_logp, float eps, float beta, float norm,
                                 float *logp, float *lse, float *w, float *loss, void *workspace,
                                 size_t workspace_bytes, grpo_stream_t stream);

/* grpo_lmhead_loss_fwd with the aggregation choice of grpo_loss_fwd_ex. */
grpo_status grpo_lmhead_loss_fwd_ex(const void *hidden, const void *weight, int64_t N, int64_t P,
                                    int64_t C, int64_t V, int64_t d, const int64_t *input_ids,
                                    const int32_t *len, const float *adv, const float *old_logp,
                                    const float *ref_logp, float eps, float beta, float norm,
                                    grpo_aggregation agg, float *logp, float *lse, float *w,
                                    float *loss, void *workspace, size_t workspace_bytes,
                                    grpo_stream_t stream);

/*
 * grpo_lmhead_loss_bwd -- gradients of g * loss with respect to the hidden
 * states and the LM head ("loss.backward()" through "model(...).logits" =
 * hidden x W^T; the chain rule, which the pages do not print).  Per scored
 * row (sequence i, row P-1+t, t < len_i) the logits gradient
 * dz = g * w[i, t] * (onehot(y) - softmax(z)) is recomputed from the logits
 * on the tensor cores (lse and w as grpo_lmhead_loss_fwd left them), rounded
 * to bfloat16 (the dtype of the logits), and contracted:
 *   dhidden[i, P-1+t, :] = dz W        dweight = sum over scored rows dz^T h
 * with float32 accumulation.  Rows that score nothing get dhidden = 0.
 *
 * hidden, weight, N, P, C, V, d, input_ids, len as for grpo_lmhead_logprobs;
 * lse, w [N, C] float32 from the forward; grad_loss: device scalar (NULL: 1).
 * dhidden [N, P+C, d] float32 and dweight [V, d] float32, 16-byte aligned,
 * fully written (accumulate into your own buffers yourself).
 *
 * Workspace and passes: the scored rows are processed in passes of up to R
 * rows (R a multiple of 256): each pass recomputes its rows' logits, forms
 * their bfloat16 gradient in the workspace (2 * R * V bytes, V rounded up to
 * 256) and runs both contractions over it; dweight is written by the first
 * pass and added to by the others (a tensor-memory-accelerator reduction, in
 * pass order).  The call takes R as large as `workspace_bytes` allows, so
 * grpo_lmhead_bwd_workspace_size (R covering all N*C possible rows: one pass)
 * and grpo_lmhead_bwd_workspace_size_rows(..., rows_per_pass) (R =
 * rows_per_pass rounded up to 256; 0 means all N*C) both give valid sizes;
 * the smallest accepted workspace is the one for R = 256.  A caller that
 * knows the number of scored tokens T (the sum of len) can pass
 * rows_per_pass = T for one pass over a workspace sized by the rows that are
 * actually scored; more scored rows than that only add passes.  Results are
 * deterministic for a given workspace size (fixed summation orders); a
 * different R changes the order of dweight's (and dhidden's) float sums, so
 * results agree to float rounding.
 */
grpo_status grpo_lmhead_bwd_workspace_size(int64_t N, int64_t C, int64_t V, int64_t d,
                                           size_t *bytes);
grpo_status grpo_lmhead_bwd_workspace_size_rows(int64_t N, int64_t C, int64_t V, int64_t d,
                                                int64_t rows_per_pass, size_t *bytes);
grpo_status grpo_lmhead_loss_bwd(const void *hidden, const void *weight, int64_t N, int64_t P,
                                 int64_t C, int64_t V, int64_t d, const int64_t *input_ids,
                                 const int32_t *len, const float *lse, const float *w,
                                 const float *grad_loss, float *dhidden, float *dweight,
                                 void *workspace, size_t workspace_bytes, grpo_stream_t stream);

/*
 * grpo_lmhead_loss_bwd with flags: GRPO_BWD_SKIP_ZERO_WEIGHT leaves out the
 * scored rows whose g * w is exactly 0 (no reward contrast in the group and
 * beta = 0: "Dr. GRPO", the analysis page's no-contrast groups), whose
 * gradient rows are 0: their logits are not recomputed and they take no part
 * in the two contractions; their dhidden rows are +0.  dweight is the same sum
 * over fewer (all-zero) terms, so it agrees to float rounding.
 */
grpo_status grpo_lmhead_loss_bwd_ex(const void *hidden, const void *weight, int64_t N, int64_t P,
                                    int64_t C, int64_t V, int64_t d, const int64_t *input_ids,
                                    const int32_t *len, const float *lse, const float *w,
                                    const float *grad_loss, float *dhidden, float *dweight,
                                    uint32_t flags, void *workspace, size_t workspace_bytes,
                                    grpo_stream_t stream);

/*
 * grpo_check_error -- synchronises `stream`, then reports what the kernels of
 * the most recent grpo_loss_fwd on `workspace` recorded: GRPO_OK,
 * GRPO_ERR_TOKEN_RANGE (a scored id outside [0, V); its logp and lse are NaN),
 * GRPO_ERR_LENGTH_RANGE (a length outside [0, C]; it was clamped), or
 * GRPO_ERR_TIMEOUT.  GRPO_ERR_CUDA if the synchronisation itself failed.
 */
grpo_status grpo_check_error(const void *workspace, grpo_stream_t stream);

/*
 * grpo_selftest_timeout -- diagnostic of the kernels' bounded waits.  Every
 * wait of the library's kernels on a shared-memory barrier gives up after
 * one second, records GRPO_ERR_TIMEOUT in the workspace and lets the kernel
 * finish instead of hanging.  This call launches one CTA that waits on a
 * barrier nothing completes: about one second later the kernel has recorded
 * the timeout in `workspace` (any workspace of grpo_workspace_size bytes,
 * 256-byte aligned; only its error flags are touched) and exited, so
 * grpo_check_error(workspace) returns GRPO_ERR_TIMEOUT and the stream and
 * context stay usable.  Reset the flags (any loss forward on the workspace
 * does) before reusing the workspace for error checks.
 */
grpo_status grpo_selftest_timeout(void *workspace, grpo_stream_t stream);

/*
 * grpo_set_early_start -- the two early starts (grpo_loss_bwd right after
 * grpo_loss_fwd, grpo_advantage right after grpo_mask; see those calls) are
 * on by default (enable != 0) and can be turned off process-wide (0).  The
 * library checks its own two calls' buffers, but it cannot see other code's
 * launches: a kernel enqueued between the two calls that itself lets its
 * successor start early (programmatic dependent launch) and reads dlogits or
 * writes len (or the advantage call's buffers) needs them off.  Kernels
 * launched the ordinary way are complete before either call touches memory.
 */
void grpo_set_early_start(int enable);

/*
 * grpo_copy -- dst[0 .. bytes) = src[0 .. bytes) with 16-byte vector loads and
 * streaming stores: the device-to-device copy ceiling the HBM roofline of the
 * other kernels is compared with.  Both pointers 16-byte aligned, bytes a
 * multiple of 16, no overlap.
 */
grpo_status grpo_copy(void *dst, const void *src, size_t bytes, grpo_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GRPO_H */

/*
 * Dr. GRPO loss over policy logits -- float64 CPU oracle.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  This is the plain, slow reference
 * the CUDA library is checked against.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no source,
 * header, table or constant with the CUDA path, and the CUDA path never loads
 * it.
 *
 * Every function restates one step of the method as the page "Making Dr GRPO
 * go brrr" (salahadawi.com, "i-made-a-kernel-22x-faster-it-made-my-training-
 * loop-3x-slower") defines it:
 *   - "The completion mask"  (build_completion_mask): 1 up to and including the
 *     first EOS, 0 after it; a completion with no EOS is entirely valid.
 *   - "compute_logprobs": logits at position t score token t+1, so completion
 *     token t is scored by logits row P-1+t; log_softmax over the vocabulary,
 *     then gather at the sampled id.
 *   - "Dr. GRPO": A_i = R_i - mean of the group, no division by sigma;
 *     token-sum aggregation divided by a constant, not a per-response mean.
 *   - "The loss" (grpo_loss): ratio r = exp(logp - logp_old); surrogate
 *     min(r*A, clamp(r, 1-eps, 1+eps)*A); the mask multiplies the per-token
 *     loss; clip the ratio first, then multiply by A.
 *   - the pseudo-code's "loss += beta * kl(logprobs, ref_logprobs)"; the page
 *     does not print the estimator, so this oracle uses the k3 estimator
 *     exp(ref - logp) - (ref - logp) - 1, aggregated like the surrogate.
 *   - "loss.backward()": the gradient with respect to the logits, derived by
 *     the chain rule (the page does not print it):
 *       d loss / d z_{row,v} = w_t * ([v == y] - softmax(z_row)_v),
 *       w_t = d loss / d logp_t.
 *
 * Arithmetic is IEEE double in the plain order of the definitions, with no
 * blocking or fusion; sums over tokens use a long double accumulator in index
 * order.  Rows are independent, so the row loops run on a few POSIX threads;
 * each row is computed by exactly one thread, which keeps every result
 * independent of the thread count.
 *
 * Logits arrive as IEEE binary32, as bfloat16 bit patterns (the upper 16 bits
 * of a binary32), or as binary64 (used for finite differences).  All convert
 * to double exactly.
 *
 * Return codes: 0 = ok, -1 = bad argument, -2 = a sampled token id outside
 * [0, V).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

static int dtype_ok(int dtype)
{
    return dtype == ORACLE_F32 || dtype == ORACLE_BF16 || dtype == ORACLE_F64;
}

/* ------------------------------------------------------------------------ */
/* element access                                                            */
/* ------------------------------------------------------------------------ */

/* Value of element v of a logits row, converted exactly to double. */
static double logit_at(const void *row, int dtype, int64_t v)
{
    if (dtype == ORACLE_F64)
        return ((const double *)row)[v];
    if (dtype == ORACLE_F32)
        return (double)((const float *)row)[v];
    /* bfloat16: the stored 16 bits are the high half of a binary32 */
    uint32_t bits = (uint32_t)((const uint16_t *)row)[v] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static size_t elem_size(int dtype)
{
    return dtype == ORACLE_F64 ? 8u : (dtype == ORACLE_F32 ? 4u : 2u);
}

static const void *row_ptr(const void *base, int dtype, int64_t row, int64_t V)
{
    return (const char *)base + (size_t)row * (size_t)V * elem_size(dtype);
}

/* ------------------------------------------------------------------------ */
/* a minimal parallel-for over independent items                            */
/* ------------------------------------------------------------------------ */

typedef void (*item_fn)(void *ctx, int64_t item);

struct pf_arg {
    item_fn fn;
    void *ctx;
    int64_t begin, end;
};

static void *pf_worker(void *p)
{
    struct pf_arg *a = (struct pf_arg *)p;
    for (int64_t k = a->begin; k < a->end; ++k)
        a->fn(a->ctx, k);
    return NULL;
}

static int g_threads = 0; /* 0: one per online core */

void oracle_set_threads(int n) { g_threads = n; }

int oracle_get_threads(void)
{
    if (g_threads > 0)
        return g_threads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    if (n < 1)
        n = 1;
    if (n > 256)
        n = 256;
    return (int)n;
}

/* Runs fn(ctx, k) for k in [0, n); contiguous static chunks, one per thread. */
static void parallel_for(int64_t n, item_fn fn, void *ctx)
{
    int nt = oracle_get_threads();
    if (n < 2 || nt < 2) {
        for (int64_t k = 0; k < n; ++k)
            fn(ctx, k);
        return;
    }
    if ((int64_t)nt > n)
        nt = (int)n;
    pthread_t tid[256];
    struct pf_arg arg[256];
    int started = 0;
    for (int t = 0; t < nt; ++t) {
        arg[t].fn = fn;
        arg[t].ctx = ctx;
        arg[t].begin = n * t / nt;
        arg[t].end = n * (t + 1) / nt;
        if (t == 0)
            continue;
        if (pthread_create(&tid[t], NULL, pf_worker, &arg[t]) != 0) {
            /* could not start a thread: do its share on this one */
            pf_worker(&arg[t]);
            arg[t].fn = NULL;
        } else {
            ++started;
        }
    }
    pf_worker(&arg[0]);
    for (int t = 1; t < nt; ++t)
        if (arg[t].fn != NULL)
            pthread_join(tid[t], NULL);
    (void)started;
}

/* ------------------------------------------------------------------------ */
/* completion mask  ("The completion mask", build_completion_mask)          */
/* ------------------------------------------------------------------------ */

/*
 * ids:  [N, T] row-major, T = P + C; the completion of row i is ids[i, P:P+C].
 * mask: [N, C] out, 1 for positions up to and including the first EOS of the
 *       completion, 0 after it; all 1 when the completion holds no EOS.
 * len:  [N] out, the number of 1s in the mask row.
 */
int oracle_mask(const int64_t *ids, int64_t N, int64_t P, int64_t C, int64_t eos,
                uint8_t *mask, int32_t *len)
{
    if (N < 0 || P < 0 || C < 0 || (N > 0 && (!ids || !len)))
        return -1;
    int64_t T = P + C;
    for (int64_t i = 0; i < N; ++i) {
        int64_t first_eos = -1;
        for (int64_t j = 0; j < C; ++j) {
            if (ids[i * T + P + j] == eos) {
                first_eos = j;
                break;
            }
        }
        int has_eos = first_eos >= 0;
        /* positions <= first EOS; no EOS: the whole completion is real */
        if (mask)
            for (int64_t j = 0; j < C; ++j)
                mask[i * C + j] = (uint8_t)(has_eos ? j <= first_eos : 1);
        len[i] = (int32_t)(has_eos ? first_eos + 1 : C);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* group advantage  ("Dr. GRPO": A_i = R_i - mu, no sigma)                  */
/* ------------------------------------------------------------------------ */

/* R, A: [B*G]; completions b*G .. b*G+G-1 form group b (prompts repeated G
 * times with repeat_interleave, rewards viewed as [B, G]). */
int oracle_advantage(const double *R, int64_t B, int64_t G, double *A)
{
    if (B < 0 || G < 1 || (B > 0 && (!R || !A)))
        return -1;
    for (int64_t b = 0; b < B; ++b) {
        double sum = 0.0;
        for (int64_t g = 0; g < G; ++g)
            sum += R[b * G + g];
        double mu = sum / (double)G;
        for (int64_t g = 0; g < G; ++g)
            A[b * G + g] = R[b * G + g] - mu;
    }
    return 0;
}

/*
 * Original GRPO advantage (section "GRPO": "Compute the advantage as
 * A_i = (R_i - mu)/sigma inside the group"; section "Dr. GRPO" removes the
 * sigma).  sigma is the standard deviation of the group's rewards,
 * sqrt(sum (R - mu)^2 / G); std_eps is added to it so a uniform group gives 0
 * instead of 0/0.
 */
int oracle_advantage_std(const double *R, int64_t B, int64_t G, double std_eps, double *A)
{
    if (B < 0 || G < 1 || !(std_eps >= 0.0) || (B > 0 && (!R || !A)))
        return -1;
    for (int64_t b = 0; b < B; ++b) {
        double sum = 0.0;
        for (int64_t g = 0; g < G; ++g)
            sum += R[b * G + g];
        double mu = sum / (double)G;
        double ss = 0.0;
        for (int64_t g = 0; g < G; ++g)
            ss += (R[b * G + g] - mu) * (R[b * G + g] - mu);
        double sigma = sqrt(ss / (double)G);
        for (int64_t g = 0; g < G; ++g)
            A[b * G + g] = (R[b * G + g] - mu) / (sigma + std_eps);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* reward contrast  ("The Quiet Library", "The sparse-reward bottleneck":   */
/* a group whose completions all get the same reward carries no contrast,   */
/* so its advantages are all zero; the useful groups are the others)        */
/* ------------------------------------------------------------------------ */

/* R: [B*G] grouped as [B, G].  *count = the number of groups b whose G
 * rewards are not all equal to one another. */
int oracle_contrast_count(const double *R, int64_t B, int64_t G, int64_t *count)
{
    if (B < 0 || G < 1 || !count || (B > 0 && !R))
        return -1;
    int64_t useful = 0;
    for (int64_t b = 0; b < B; ++b) {
        const double *grp = R + b * G;
        int all_equal = 1;
        for (int64_t k = 1; k < G && all_equal; ++k)
            if (grp[k] != grp[0])
                all_equal = 0;
        if (!all_equal)
            useful += 1;
    }
    *count = useful;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* log-probabilities  ("compute_logprobs": shift, log_softmax, gather)       */
/* ------------------------------------------------------------------------ */

/* log sum_v exp(z_v) of one row, by its plain definition with the maximum
 * factored out (two passes: maximum, then the sum). */
static double row_logsumexp(const void *row, int dtype, int64_t V)
{
    double mx = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double z = logit_at(row, dtype, v);
        if (z > mx || isnan(z))
            mx = z;
        if (isnan(mx))
            return NAN;
    }
    if (isinf(mx))
        return mx; /* all -inf: log 0 = -inf;  any +inf: +inf */
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v)
        s += exp(logit_at(row, dtype, v) - mx);
    return mx + log(s);
}

/*
 * Independent rows: logp[k] = z_k[y_k] - logsumexp(z_k) for each of n rows,
 * rows[k] = rows + k*V elements.  lse may be NULL.
 */
struct rows_ctx {
    const void *rows;
    int dtype;
    int64_t V;
    const int64_t *y;
    double *logp, *lse;
    int bad;
};

static void rows_item(void *p, int64_t k)
{
    struct rows_ctx *c = (struct rows_ctx *)p;
    const void *row = row_ptr(c->rows, c->dtype, k, c->V);
    int64_t y = c->y[k];
    if (y < 0 || y >= c->V) {
        __atomic_store_n(&c->bad, 1, __ATOMIC_RELAXED);
        c->logp[k] = NAN;
        if (c->lse)
            c->lse[k] = NAN;
        return;
    }
    double l = row_logsumexp(row, c->dtype, c->V);
    c->logp[k] = logit_at(row, c->dtype, y) - l;
    if (c->lse)
        c->lse[k] = l;
}

int oracle_logp_rows(const void *rows, int dtype, int64_t n, int64_t V, const int64_t *y,
                     double *logp, double *lse)
{
    if (n < 0 || V < 1 || !dtype_ok(dtype))
        return -1;
    if (n > 0 && (!rows || !y || !logp))
        return -1;
    struct rows_ctx c = {rows, dtype, V, y, logp, lse, 0};
    parallel_for(n, rows_item, &c);
    return c.bad ? -2 : 0;
}

/*
 * Whole batch: logits [N, T, V], ids [N, T], len [N] (from oracle_mask).
 * Completion token t of row i (t < len_i) is y = ids[i, P+t], scored by the
 * logits row P-1+t of sequence i.  logp, lse: [N, C]; 0 where t >= len_i.
 */
struct batch_ctx {
    const void *logits;
    int dtype;
    int64_t T, V, P, C;
    const int64_t *ids;
    const int32_t *len;
    double *logp, *lse;
    int bad;
};

static void batch_item(void *p, int64_t k)
{
    struct batch_ctx *c = (struct batch_ctx *)p;
    int64_t i = k / c->C, t = k % c->C;
    if (t >= c->len[i]) {
        c->logp[k] = 0.0;
        if (c->lse)
            c->lse[k] = 0.0;
        return;
    }
    int64_t y = c->ids[i * c->T + c->P + t];
    const void *row = row_ptr(c->logits, c->dtype, i * c->T + (c->P - 1 + t), c->V);
    if (y < 0 || y >= c->V) {
        __atomic_store_n(&c->bad, 1, __ATOMIC_RELAXED);
        c->logp[k] = NAN;
        if (c->lse)
            c->lse[k] = NAN;
        return;
    }
    double l = row_logsumexp(row, c->dtype, c->V);
    c->logp[k] = logit_at(row, c->dtype, y) - l;
    if (c->lse)
        c->lse[k] = l;
}

int oracle_logp(const void *logits, int dtype, int64_t N, int64_t P, int64_t C, int64_t V,
                const int64_t *ids, const int32_t *len, double *logp, double *lse)
{
    if (N < 0 || P < 1 || C < 0 || V < 1 || !dtype_ok(dtype))
        return -1;
    if (N > 0 && (!len || (C > 0 && (!logits || !ids || !logp))))
        return -1;
    for (int64_t i = 0; i < N; ++i)
        if (len[i] < 0 || len[i] > C)
            return -1;
    struct batch_ctx c = {logits, dtype, P + C, V, P, C, ids, len, logp, lse, 0};
    parallel_for(N * C, batch_item, &c);
    return c.bad ? -2 : 0;
}

/* ------------------------------------------------------------------------ */
/* loss  ("The loss", grpo_loss; "Dr. GRPO" aggregation; KL term)           */
/* ------------------------------------------------------------------------ */

static double clamp_d(double x, double lo, double hi)
{
    return x < lo ? lo : (x > hi ? hi : x);
}

/*
 * logp, old, ref, w, ell: [N, C]; A, len: [N].
 * old == NULL means "old log-probs equal the current ones" (inner step 0):
 * the ratio is exactly 1.  ref may be NULL only when beta == 0.
 * norm <= 0 selects the default constant N*C.
 *
 * Per valid token (t < len_i):
 *   r    = exp(logp - old)
 *   s    = min(r*A, clamp(r, 1-eps, 1+eps)*A)
 *   k3   = exp(ref - logp) - (ref - logp) - 1
 *   ell  = -s + beta*k3
 * loss = (sum of ell over valid tokens) / norm.
 * w = d loss / d logp per token:
 *   d s / d logp = A*r when the unclipped term is the one min() selects
 *   (r*A <= clamp(r)*A; both terms are equal inside the clip range), else 0;
 *   d k3 / d logp = 1 - exp(ref - logp);
 *   w = (-(d s / d logp) + beta*(d k3 / d logp)) / norm.
 * Masked positions (t >= len_i) give w = ell = 0 and are never read.
 */
/*
 * agg selects the aggregation (section "Dr. GRPO"):
 *   0  token sum divided by a constant: loss = sum_i sum_t ell / norm
 *      (norm <= 0 selects N*C) -- Dr. GRPO;
 *   1  per-response mean, then the mean over responses: loss =
 *      sum_i (sum_t ell) / len_i / norm (norm <= 0 selects N) -- original
 *      GRPO's 1/|o_i|; a completion with no valid token contributes 0.
 * w = d loss / d logp follows the same weights.
 */
int oracle_loss_agg(const double *logp, const double *old, const double *ref, const double *A,
                    const int32_t *len, int64_t N, int64_t C, double eps, double beta,
                    double norm, int agg, double *loss, double *w, double *ell);

int oracle_loss(const double *logp, const double *old, const double *ref, const double *A,
                const int32_t *len, int64_t N, int64_t C, double eps, double beta, double norm,
                double *loss, double *w, double *ell)
{
    return oracle_loss_agg(logp, old, ref, A, len, N, C, eps, beta, norm, 0, loss, w, ell);
}

int oracle_loss_agg(const double *logp, const double *old, const double *ref, const double *A,
                    const int32_t *len, int64_t N, int64_t C, double eps, double beta,
                    double norm, int agg, double *loss, double *w, double *ell)
{
    if (agg != 0 && agg != 1)
        return -1;
    if (N < 0 || C < 0 || !loss || !(eps >= 0.0 && eps < 1.0) || !(beta >= 0.0))
        return -1;
    if (beta != 0.0 && !ref)
        return -1;
    if (N > 0 && C > 0 && (!logp || !A || !len))
        return -1;
    if (!(norm > 0.0))
        norm = agg == 0 ? (double)N * (double)C : (double)N;
    long double total = 0.0L;
    for (int64_t i = 0; i < N; ++i) {
        double a = A[i];
        /* the constant every token of completion i is divided by */
        double denom = agg == 0 ? norm : norm * (double)(len[i] > 0 ? len[i] : 1);
        for (int64_t t = 0; t < C; ++t) {
            int64_t k = i * C + t;
            if (t >= len[i]) {
                if (w)
                    w[k] = 0.0;
                if (ell)
                    ell[k] = 0.0;
                continue;
            }
            double lp = logp[k];
            double r = old ? exp(lp - old[k]) : 1.0;
            double unclipped = r * a;
            double clipped = clamp_d(r, 1.0 - eps, 1.0 + eps) * a;
            double s = unclipped < clipped ? unclipped : clipped;
            double ds = unclipped <= clipped ? a * r : 0.0;
            double k3 = 0.0, dk3 = 0.0;
            if (beta != 0.0) {
                double d = ref[k] - lp;
                k3 = exp(d) - d - 1.0;
                dk3 = 1.0 - exp(d);
            }
            double l = -s + beta * k3;
            total += (long double)l * ((long double)norm / (long double)denom);
            if (w)
                w[k] = (-ds + beta * dk3) / denom;
            if (ell)
                ell[k] = l;
        }
    }
    *loss = (double)(total / (long double)norm);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* gradient with respect to the logits  ("loss.backward()")                  */
/* ------------------------------------------------------------------------ */

/* One scored row: out[v] = gw * ([v == y] - exp(z_v - lse)). */
int oracle_dlogits_row(const void *row, int dtype, int64_t V, int64_t y, double lse, double gw,
                       double *out)
{
    if (!row || !out || V < 1 || !dtype_ok(dtype))
        return -1;
    if (y < 0 || y >= V)
        return -2;
    for (int64_t v = 0; v < V; ++v) {
        double p = exp(logit_at(row, dtype, v) - lse);
        out[v] = gw * ((v == y ? 1.0 : 0.0) - p);
    }
    return 0;
}

/*
 * Whole batch: out [N, T, V] = d (g * loss) / d logits.  Rows that score no
 * valid completion token (prompt rows 0..P-2, the last row T-1, and rows past
 * the first EOS) do not enter the loss and get 0.  lse and w come from
 * oracle_logp and oracle_loss; g is the upstream scalar gradient.
 */
struct dl_ctx {
    const void *logits;
    int dtype;
    int64_t T, V, P, C;
    const int64_t *ids;
    const int32_t *len;
    const double *lse, *w;
    double g;
    double *out;
    int bad;
};

static void dl_item(void *p, int64_t row)
{
    struct dl_ctx *c = (struct dl_ctx *)p;
    int64_t i = row / c->T, pos = row % c->T;
    int64_t t = pos - (c->P - 1); /* completion token this row scores */
    double *o = c->out + (size_t)row * (size_t)c->V;
    if (t < 0 || t >= c->len[i]) {
        for (int64_t v = 0; v < c->V; ++v)
            o[v] = 0.0;
        return;
    }
    int64_t k = i * c->C + t;
    int64_t y = c->ids[i * c->T + c->P + t];
    if (oracle_dlogits_row(row_ptr(c->logits, c->dtype, row, c->V), c->dtype, c->V, y,
                           c->lse[k], c->g * c->w[k], o) != 0)
        __atomic_store_n(&c->bad, 1, __ATOMIC_RELAXED);
}

int oracle_dlogits(const void *logits, int dtype, int64_t N, int64_t P, int64_t C, int64_t V,
                   const int64_t *ids, const int32_t *len, const double *lse, const double *w,
                   double g, double *out)
{
    if (N < 0 || P < 1 || C < 0 || V < 1 || !dtype_ok(dtype))
        return -1;
    if (N > 0 && (!logits || !ids || !len || !lse || !w || !out))
        return -1;
    struct dl_ctx c = {logits, dtype, P + C, V, P, C, ids, len, lse, w, g, out, 0};
    parallel_for(N * (P + C), dl_item, &c);
    return c.bad ? -2 : 0;
}

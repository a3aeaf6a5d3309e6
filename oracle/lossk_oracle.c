/*
 * lossk_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the fused LM-head loss computes.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library; the product path never does.  It shares no code,
 * header, constant or table with the CUDA library: every constant below is
 * restated here from the pages.
 *
 * Sources (page title, section):
 *   [P1] "Loss functions and resident-context kernels", section "lossk: the
 *        loss is where the memory goes" (function table), section "Status
 *        codes", section "A worked example: uniform logits give exactly
 *        log(vocab)", section "The two budgets are genuinely different
 *        questions", section "Chunk invariance is checked to the last bit",
 *        section "The backward's gradient check is a cancellation identity".
 *   [P3] "Fuse distillation + z-loss in the triton monolithic path (#507)",
 *        section "What it does" (label-family gradient shape, z-loss folding,
 *        shared loss mask and divisor).
 *
 * Arithmetic rules:
 *   - Inputs arrive as float (every bf16 or fp32 value is exact in float);
 *     every operation after that is double.
 *   - Build with -ffp-contract=off so that a*b+c is never fused: the same
 *     source gives the same bits on x86-64 and aarch64.
 *   - Every logit is one dot product summed in ascending k; every sum over
 *     the vocabulary runs in ascending v; every sum over tokens runs in
 *     ascending t.  Threads (OpenMP) only split independent rows, so the
 *     result never depends on the thread count or on the chunk size.
 *
 * Parity: every function here is pinned by tests/test_oracle_pins.py
 * (closed forms, the pages' printed values, finite differences, library
 * routines in fp64, brute force).  The distillation functions at a
 * temperature other than 1 are pinned only by identities (T-scaling,
 * superposition, finite differences); the pages print no distillation value.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- status vocabulary, [P1] "Status codes" ---------------------------- */
enum {
    OR_OK = 580,
    OR_EMPTY_DIMENSION = 581,
    OR_LENGTH_MISMATCH = 582,
    OR_DIMENSION_TOO_LARGE = 583,
    OR_WORK_BUDGET_EXCEEDED = 584,
    OR_NON_FINITE_SCALAR = 585,
    OR_TARGET_OUT_OF_RANGE = 586,
    OR_CHUNK_EXCEEDS_BUDGET = 587,
    OR_UNKNOWN_OBJECTIVE = 588
};

/* LOSS_MAX_WORK_CELLS = 2^46 and LOSS_MAX_LOGIT_CELLS = 2^27 are printed on
 * [P1] (function table).  The per-dimension ceiling is not printed; this
 * oracle reads it as 2^24 for every dimension. */
static const int64_t OR_MAX_WORK_CELLS = (int64_t)1 << 46;
static const int64_t OR_MAX_LOGIT_CELLS = (int64_t)1 << 27;
static const int64_t OR_MAX_DIM = (int64_t)1 << 24;

const char *oracle_status_name(int code)
{
    switch (code) {
    case 580: return "ok";
    case 581: return "empty_dimension";
    case 582: return "length_mismatch";
    case 583: return "dimension_too_large";
    case 584: return "work_budget_exceeded";
    case 585: return "non_finite_scalar";
    case 586: return "target_id_out_of_range";
    case 587: return "chunk_exceeds_logit_budget";
    case 588: return "unknown_objective";
    default: return "unknown_status";
    }
}

/* loss_work_fits, [P1] function table: the three-factor product fits the
 * ceiling, decided by successive integer division so nothing overflows.
 * For positive integers n*d*V <= C  <=>  n <= floor(floor(C/d)/V). */
int oracle_work_fits(int64_t n, int64_t d, int64_t V, int64_t ceiling)
{
    if (n < 1 || d < 1 || V < 1 || ceiling < 0) return 0;
    int64_t q = ceiling / d;
    q = q / V;
    return n <= q;
}

/* loss_dims_check, [P1] function table. */
int oracle_dims_check(int64_t n, int64_t d, int64_t V)
{
    if (n < 1 || d < 1 || V < 1) return OR_EMPTY_DIMENSION;
    if (n > OR_MAX_DIM || d > OR_MAX_DIM || V > OR_MAX_DIM) return OR_DIMENSION_TOO_LARGE;
    if (!oracle_work_fits(n, d, V, OR_MAX_WORK_CELLS)) return OR_WORK_BUDGET_EXCEEDED;
    return OR_OK;
}

/* loss_chunk_check, [P1] function table: refuse (never clamp) a chunk whose
 * chunk*vocab would exceed 2^27; exactly 2^27 is allowed. */
int oracle_chunk_check(int64_t chunk, int64_t V)
{
    if (chunk < 1 || V < 1) return OR_EMPTY_DIMENSION;
    if (chunk > OR_MAX_LOGIT_CELLS / V) return OR_CHUNK_EXCEEDS_BUDGET;
    return OR_OK;
}

/* loss_logit_cells, [P1] function table: chunk*vocab as a double, negative
 * for a malformed request. */
double oracle_logit_cells(int64_t chunk, int64_t V)
{
    if (chunk < 1 || V < 1) return -1.0;
    return (double)chunk * (double)V;
}

/* loss_targets_in_range, [P1] function table: every one of the first n
 * targets lies in [0, V); a negative id is refused, not read as a mask. */
int oracle_targets_in_range(const int64_t *y, int64_t n, int64_t V)
{
    for (int64_t t = 0; t < n; ++t)
        if (y[t] < 0 || y[t] >= V) return 0;
    return 1;
}

/* ce_peak_logit_cells, [P1] opening example and function table.
 * out[0] chunked cells = min(chunk, n)*V, out[1] materialised cells = n*V,
 * out[2] ratio = materialised/chunked; *n_chunks = ceil(n/chunk).
 * Returns the status of the chunk argument (the numbers are still reported
 * when the chunk is over budget).  Malformed: cells -1, ratio 0, chunks 0. */
int oracle_peak_logit_cells(int64_t n, int64_t V, int64_t chunk, double *out, int64_t *n_chunks)
{
    if (n < 1 || V < 1 || chunk < 1) {
        out[0] = -1.0; out[1] = -1.0; out[2] = 0.0; *n_chunks = 0;
        return OR_EMPTY_DIMENSION;
    }
    int64_t held = chunk < n ? chunk : n;
    out[0] = (double)held * (double)V;
    out[1] = (double)n * (double)V;
    out[2] = out[1] / out[0];
    *n_chunks = (n + chunk - 1) / chunk;
    return oracle_chunk_check(chunk, V);
}

/* ---- arithmetic helpers ------------------------------------------------- */

/* One logit: sum_k h[k]*w[k], ascending k, in double. */
static double dot_asc(const float *h, const float *w, int64_t d)
{
    double acc = 0.0;
    for (int64_t k = 0; k < d; ++k) acc += (double)h[k] * (double)w[k];
    return acc;
}

/* Max-shifted log-sum-exp over x[0..V), ascending v: m + log(sum exp(x-m)).
 * This is the stable reduction the pages name (numerical_stability.logsumexp,
 * body not printed; the max-shifted form is the plain reading). */
static double lse_row(const double *x, int64_t V)
{
    double m = x[0];
    for (int64_t v = 1; v < V; ++v) if (x[v] > m) m = x[v];
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) s += exp(x[v] - m);
    return m + log(s);
}

/* A block of logit rows: buf[r][v] = H[t] . W[v] (dot_asc) for the R tokens
 * t = rows[r] (or t = t0 + r when rows is NULL) and every v < V.  Each
 * element is the one dot product above; the buffer is filled tile by tile
 * (64 tokens x 64 vocabulary rows, tiles spread over the threads) so that a
 * weight row is read from memory once per tile of tokens instead of once per
 * token.  The fill order changes no element. */
static void fill_logits(const float *H, const float *W, const int64_t *rows, int64_t t0, int64_t R,
                        int64_t d, int64_t V, double *buf)
{
    const int64_t TB = 64;
    #pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t rb = 0; rb < R; rb += TB)
        for (int64_t vb = 0; vb < V; vb += TB) {
            const int64_t r1 = rb + TB < R ? rb + TB : R, v1 = vb + TB < V ? vb + TB : V;
            for (int64_t r = rb; r < r1; ++r) {
                const float *h = H + (rows ? rows[r] : t0 + r) * d;
                for (int64_t v = vb; v < v1; ++v) buf[r * V + v] = dot_asc(h, W + v * d, d);
            }
        }
}

static int64_t count_valid(const uint8_t *mask, int64_t n)
{
    if (!mask) return n;
    int64_t c = 0;
    for (int64_t t = 0; t < n; ++t) c += mask[t] ? 1 : 0;
    return c;
}

static int scalar_ok(double x) { return isfinite(x); }

/* ---- cross-entropy from materialised logits, [P1] ce_from_logits_flat ---
 * Per token t (ascending): lse_t, ce_t = lse_t - x[t][y_t], z_t = lse_t^2
 * ([P3] z-loss: forward scalar log_sum_exp^2).  Masked tokens (mask 0) keep
 * lse_t but have ce_t = z_t = 0 and no gradient.
 * scal[0] = total = sum_t m_t(ce_t + wz z_t) / N_valid, scal[1] = ce mean,
 * scal[2] = z mean; sums sequential in t.  N_valid = 0 gives zeros.
 * grad (optional, [n][V]): G = alpha_t((1 + 2 wz lse_t) p_tv - [v == y_t]),
 * alpha_t = grad_scale m_t / N_valid ([P3] label-family gradient shape,
 * prob_coeff*softmax - label_coeff*onehot, with the z coefficient folded). */
int oracle_ce_from_logits(const float *logits, const int64_t *y, const uint8_t *mask,
                          int64_t n, int64_t V, double wz, double grad_scale,
                          double *lse_out, double *ce_out, double *scal, double *grad)
{
    if (n < 1 || V < 1) return OR_EMPTY_DIMENSION;
    if (n > OR_MAX_DIM || V > OR_MAX_DIM) return OR_DIMENSION_TOO_LARGE;
    if (!scalar_ok(wz) || wz < 0.0 || !scalar_ok(grad_scale)) return OR_NON_FINITE_SCALAR;
    if (!oracle_targets_in_range(y, n, V)) return OR_TARGET_OUT_OF_RANGE;
    int64_t nvalid = count_valid(mask, n);
    double *zt = (double *)malloc(sizeof(double) * (size_t)n);
    #pragma omp parallel
    {
        double *row = (double *)malloc(sizeof(double) * (size_t)V);
        #pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            const float *x = logits + t * V;
            for (int64_t v = 0; v < V; ++v) row[v] = (double)x[v];
            double lse = lse_row(row, V);
            int on = mask ? (mask[t] != 0) : 1;
            lse_out[t] = lse;
            ce_out[t] = on ? lse - row[y[t]] : 0.0;
            zt[t] = on ? lse * lse : 0.0;
            if (grad) {
                double alpha = nvalid > 0 && on ? grad_scale / (double)nvalid : 0.0;
                double c = alpha * (1.0 + 2.0 * wz * lse);
                for (int64_t v = 0; v < V; ++v) {
                    double g = c * exp(row[v] - lse);
                    if (v == y[t]) g -= alpha;
                    grad[t * V + v] = g;
                }
            }
        }
        free(row);
    }
    double sum_tok = 0.0, sum_ce = 0.0, sum_z = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        sum_tok += ce_out[t] + wz * zt[t];
        sum_ce += ce_out[t];
        sum_z += zt[t];
    }
    free(zt);
    if (nvalid > 0) {
        scal[0] = sum_tok / (double)nvalid;
        scal[1] = sum_ce / (double)nvalid;
        scal[2] = sum_z / (double)nvalid;
    } else {
        scal[0] = scal[1] = scal[2] = 0.0;
    }
    return OR_OK;
}

/* Shared argument checks of the fused calls, in the order: 581, 583, 584,
 * 587 (chunk, when given), 585 (scalars), 586 (targets, when given). */
static int fused_checks(int64_t n, int64_t d, int64_t V, int64_t chunk, const int64_t *y,
                        double wz, double grad_scale)
{
    int st = oracle_dims_check(n, d, V);
    if (st != OR_OK) return st;
    if (chunk != 0) {
        st = oracle_chunk_check(chunk, V);
        if (st != OR_OK) return st;
    }
    if (!scalar_ok(wz) || wz < 0.0 || !scalar_ok(grad_scale)) return OR_NON_FINITE_SCALAR;
    if (y && !oracle_targets_in_range(y, n, V)) return OR_TARGET_OUT_OF_RANGE;
    return OR_OK;
}

/* ---- fused projection + chunked cross-entropy, [P1] fused_linear_ce_flat --
 * H [n][d], W [V][d] row-major.  A [chunk][V] double buffer holds the logits
 * of one chunk of tokens at a time and is reused; per-token values and the
 * token-order sums are therefore the same bits for every chunk size
 * ([P1] "Chunk invariance is checked to the last bit").
 * Outputs as oracle_ce_from_logits (no gradient). */
int oracle_ce_fwd(const float *H, const float *W, const int64_t *y, const uint8_t *mask,
                  int64_t n, int64_t d, int64_t V, int64_t chunk, double wz,
                  double *lse_out, double *ce_out, double *scal)
{
    if (chunk < 1) return OR_EMPTY_DIMENSION;
    int st = fused_checks(n, d, V, chunk, y, wz, 1.0);
    if (st != OR_OK) return st;
    int64_t nvalid = count_valid(mask, n);
    int64_t rows_max = chunk < n ? chunk : n;
    double *buf = (double *)malloc(sizeof(double) * (size_t)(rows_max * V));
    double *zt = (double *)malloc(sizeof(double) * (size_t)n);
    for (int64_t t0 = 0; t0 < n; t0 += chunk) {
        int64_t rows = n - t0 < chunk ? n - t0 : chunk;
        /* project the chunk: buf[r][v] = H[t0+r] . W[v] */
        fill_logits(H, W, NULL, t0, rows, d, V, buf);
        /* reduce each row to (lse, target logit) and drop the chunk */
        #pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t t = t0 + r;
            double lse = lse_row(buf + r * V, V);
            int on = mask ? (mask[t] != 0) : 1;
            lse_out[t] = lse;
            ce_out[t] = on ? lse - buf[r * V + y[t]] : 0.0;
            zt[t] = on ? lse * lse : 0.0;
        }
    }
    double sum_tok = 0.0, sum_ce = 0.0, sum_z = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        sum_tok += ce_out[t] + wz * zt[t];
        sum_ce += ce_out[t];
        sum_z += zt[t];
    }
    free(zt);
    free(buf);
    if (nvalid > 0) {
        scal[0] = sum_tok / (double)nvalid;
        scal[1] = sum_ce / (double)nvalid;
        scal[2] = sum_z / (double)nvalid;
    } else {
        scal[0] = scal[1] = scal[2] = 0.0;
    }
    return OR_OK;
}

/* ---- analytic backward, [P1] fused_linear_ce_bwd_flat --------------------
 * Gradient of grad_scale * total with respect to H and W:
 *   G_tv  = alpha_t((1 + 2 wz lse_t) p_tv - [v == y_t]), p_tv = exp(s_tv - lse_t)
 *   dH_t  = sum_v G_tv W_v     (ascending v)
 *   dW_v  = sum_t G_tv H_t     (ascending t)
 * The pages do not chunk the backward; this oracle computes G a block of
 * tokens at a time only to bound memory, and adds each block into dW in
 * ascending t, so the block size changes no bit. */
int oracle_ce_bwd(const float *H, const float *W, const int64_t *y, const uint8_t *mask,
                  int64_t n, int64_t d, int64_t V, double wz, double grad_scale,
                  double *dH, double *dW)
{
    int st = fused_checks(n, d, V, 0, y, wz, grad_scale);
    if (st != OR_OK) return st;
    int64_t nvalid = count_valid(mask, n);
    memset(dH, 0, sizeof(double) * (size_t)(n * d));
    memset(dW, 0, sizeof(double) * (size_t)(V * d));
    if (nvalid == 0) return OR_OK;
    const int64_t B = 64;
    double *G = (double *)malloc(sizeof(double) * (size_t)(B * V));
    for (int64_t t0 = 0; t0 < n; t0 += B) {
        int64_t rows = n - t0 < B ? n - t0 : B;
        #pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t t = t0 + r;
            double *g = G + r * V;
            for (int64_t v = 0; v < V; ++v) g[v] = dot_asc(H + t * d, W + v * d, d);
            double lse = lse_row(g, V);
            int on = mask ? (mask[t] != 0) : 1;
            double alpha = on ? grad_scale / (double)nvalid : 0.0;
            double c = alpha * (1.0 + 2.0 * wz * lse);
            for (int64_t v = 0; v < V; ++v) {
                double gv = c * exp(g[v] - lse);
                if (v == y[t]) gv -= alpha;
                g[v] = gv;
            }
            double *dh = dH + t * d;
            for (int64_t v = 0; v < V; ++v) {
                const float *w = W + v * d;
                for (int64_t k = 0; k < d; ++k) dh[k] += g[v] * (double)w[k];
            }
        }
        #pragma omp parallel for schedule(static)
        for (int64_t v = 0; v < V; ++v) {
            double *dw = dW + v * d;
            for (int64_t r = 0; r < rows; ++r) {
                double gv = G[r * V + v];
                const float *h = H + (t0 + r) * d;
                for (int64_t k = 0; k < d; ++k) dw[k] += gv * (double)h[k];
            }
        }
    }
    free(G);
    return OR_OK;
}

/* ---- sampled rows, for checks at sizes where the whole oracle is too slow --
 * Per listed token: lse, target logit and (optionally) the dH row, each
 * computed exactly as above from that token's own logit row; and per listed
 * vocabulary row the dW row, given every token's lse (from oracle_ce_fwd). */
int oracle_ce_token_rows(const float *H, const float *W, const int64_t *y, const uint8_t *mask,
                         int64_t n, int64_t d, int64_t V, double wz, double grad_scale,
                         const int64_t *rows, int64_t n_rows,
                         double *lse_out, double *tgt_out, double *dH_rows)
{
    int st = fused_checks(n, d, V, 0, y, wz, grad_scale);
    if (st != OR_OK) return st;
    int64_t nvalid = count_valid(mask, n);
    /* the listed tokens' logit rows, a block of at most 256 at a time */
    const int64_t RB = 256;
    double *blk = (double *)malloc(sizeof(double) * (size_t)((n_rows < RB ? n_rows : RB) * V));
    for (int64_t i0 = 0; i0 < n_rows; i0 += RB) {
        const int64_t nb = n_rows - i0 < RB ? n_rows - i0 : RB;
        fill_logits(H, W, rows + i0, 0, nb, d, V, blk);
        #pragma omp parallel for schedule(dynamic, 1)
        for (int64_t ib = 0; ib < nb; ++ib) {
            const int64_t i = i0 + ib, t = rows[i];
            const double *s = blk + ib * V;
            double lse = lse_row(s, V);
            lse_out[i] = lse;
            tgt_out[i] = s[y[t]];
            if (dH_rows) {
                int on = mask ? (mask[t] != 0) : 1;
                double alpha = (on && nvalid > 0) ? grad_scale / (double)nvalid : 0.0;
                double c = alpha * (1.0 + 2.0 * wz * lse);
                double *dh = dH_rows + i * d;
                for (int64_t k = 0; k < d; ++k) dh[k] = 0.0;
                for (int64_t v = 0; v < V; ++v) {
                    double gv = c * exp(s[v] - lse);
                    if (v == y[t]) gv -= alpha;
                    const float *w = W + v * d;
                    for (int64_t k = 0; k < d; ++k) dh[k] += gv * (double)w[k];
                }
            }
        }
    }
    free(blk);
    return OR_OK;
}

int oracle_ce_dweight_rows(const float *H, const float *W, const int64_t *y, const uint8_t *mask,
                           int64_t n, int64_t d, int64_t V, double wz, double grad_scale,
                           const double *lse_all, const int64_t *vrows, int64_t n_vrows,
                           double *dW_rows)
{
    int st = fused_checks(n, d, V, 0, y, wz, grad_scale);
    if (st != OR_OK) return st;
    int64_t nvalid = count_valid(mask, n);
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_vrows; ++i) {
        int64_t v = vrows[i];
        double *dw = dW_rows + i * d;
        for (int64_t k = 0; k < d; ++k) dw[k] = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            int on = mask ? (mask[t] != 0) : 1;
            if (!on || nvalid == 0) continue;
            double alpha = grad_scale / (double)nvalid;
            double s = dot_asc(H + t * d, W + v * d, d);
            double gv = alpha * (1.0 + 2.0 * wz * lse_all[t]) * exp(s - lse_all[t]);
            if (v == y[t]) gv -= alpha;
            const float *h = H + t * d;
            for (int64_t k = 0; k < d; ++k) dw[k] += gv * (double)h[k];
        }
    }
    return OR_OK;
}

/* ---- distillation against a full teacher distribution -------------------
 * [P3] "What it does": the distribution-family loss compares the student
 * softmax with a full teacher distribution (cross-entropy, forward-KL,
 * reverse-KL), shares the loss mask and divisor, and folds z-loss over the
 * same student softmax: forward lse^2, gradient 2 g_z lse q_j.  The pages do
 * not print the formulas; this oracle takes the plain reading:
 *   a = s/T, b = teacher/T, q = softmax(a), p = softmax(b),
 *   log q = a - lse(a), log p = b - lse(b)
 *   CE  = -sum p log q;  fKL = sum p (log p - log q);  rKL = sum q (log q - log p)
 *   z   = lse(a)^2
 *   dL/ds_v: CE, fKL: (q_v - p_v)/T;  rKL: q_v (log q_v - log p_v - rKL)/T
 *   dz/ds_v = 2 lse(a) q_v / T
 * token_t = m_t (L_t + wz z_t); total = sum_t token_t / N_valid; gradient of
 * grad_scale*total.  direction: 0 CE, 1 forward-KL, 2 reverse-KL; other ->
 * 588 (the pages reserve it for an objective beyond cross-entropy).
 * teacher [n][V]; per_token[t] = L_t (0 when masked); scal = {total,
 * distill mean, z mean}; dH/dW may be NULL to skip the backward. */
static double distill_row(const double *s, const float *teach, int64_t V, int direction,
                          double T, double *a, double *b, double *lse_a_out, double *g_out)
{
    for (int64_t v = 0; v < V; ++v) { a[v] = s[v] / T; b[v] = (double)teach[v] / T; }
    double la = lse_row(a, V), lb = lse_row(b, V);
    double L = 0.0;
    /* An entry of probability 0 (a logit of -inf: a vocabulary entry masked
     * out of the row) adds nothing: the limit x log x -> 0 as x -> 0.  Where the
     * weighting probability is positive and the other one is 0, the term is
     * +inf, and so is the loss. */
    for (int64_t v = 0; v < V; ++v) {
        double lq = a[v] - la, lp = b[v] - lb;
        double q = exp(lq), p = exp(lp);
        if (direction == 0) L -= p > 0.0 ? p * lq : 0.0;
        else if (direction == 1) L += p > 0.0 ? p * (lp - lq) : 0.0;
        else L += q > 0.0 ? q * (lq - lp) : 0.0;
    }
    if (g_out) {
        for (int64_t v = 0; v < V; ++v) {
            double lq = a[v] - la, lp = b[v] - lb;
            double q = exp(lq), p = exp(lp);
            g_out[v] = direction == 2 ? (q > 0.0 ? q * (lq - lp - L) / T : 0.0) : (q - p) / T;
        }
    }
    *lse_a_out = la;
    return L;
}

int oracle_distill(const float *H, const float *W, const float *teacher, const uint8_t *mask,
                   int64_t n, int64_t d, int64_t V, int64_t chunk, int direction, double T,
                   double wz, double grad_scale, double *per_token, double *lse_out,
                   double *scal, double *dH, double *dW)
{
    if (chunk < 1) return OR_EMPTY_DIMENSION;
    int st = fused_checks(n, d, V, chunk, NULL, wz, grad_scale);
    if (st != OR_OK) return st;
    if (!scalar_ok(T) || T <= 0.0) return OR_NON_FINITE_SCALAR;
    if (direction < 0 || direction > 2) return OR_UNKNOWN_OBJECTIVE;
    int64_t nvalid = count_valid(mask, n);
    double *zt = (double *)malloc(sizeof(double) * (size_t)n);
    if (dH) memset(dH, 0, sizeof(double) * (size_t)(n * d));
    if (dW) memset(dW, 0, sizeof(double) * (size_t)(V * d));
    int64_t rows_max = chunk < n ? chunk : n;
    double *G = (double *)malloc(sizeof(double) * (size_t)(rows_max * V));
    for (int64_t t0 = 0; t0 < n; t0 += chunk) {
        int64_t rows = n - t0 < chunk ? n - t0 : chunk;
        #pragma omp parallel
        {
            double *s = (double *)malloc(sizeof(double) * (size_t)V);
            double *a = (double *)malloc(sizeof(double) * (size_t)V);
            double *b = (double *)malloc(sizeof(double) * (size_t)V);
            #pragma omp for schedule(static)
            for (int64_t r = 0; r < rows; ++r) {
                int64_t t = t0 + r;
                for (int64_t v = 0; v < V; ++v) s[v] = dot_asc(H + t * d, W + v * d, d);
                double la;
                double *g = G + r * V;
                double L = distill_row(s, teacher + t * V, V, direction, T, a, b, &la, g);
                int on = mask ? (mask[t] != 0) : 1;
                per_token[t] = on ? L : 0.0;
                zt[t] = on ? la * la : 0.0;
                if (lse_out) lse_out[t] = la;
                double alpha = (on && nvalid > 0) ? grad_scale / (double)nvalid : 0.0;
                for (int64_t v = 0; v < V; ++v) {
                    double q = exp(a[v] - la);
                    g[v] = alpha * (g[v] + 2.0 * wz * la * q / T);
                }
                if (dH) {
                    double *dh = dH + t * d;
                    for (int64_t v = 0; v < V; ++v) {
                        const float *w = W + v * d;
                        for (int64_t k = 0; k < d; ++k) dh[k] += g[v] * (double)w[k];
                    }
                }
            }
            free(s); free(a); free(b);
        }
        if (dW) {
            #pragma omp parallel for schedule(static)
            for (int64_t v = 0; v < V; ++v) {
                double *dw = dW + v * d;
                for (int64_t r = 0; r < rows; ++r) {
                    double gv = G[r * V + v];
                    const float *h = H + (t0 + r) * d;
                    for (int64_t k = 0; k < d; ++k) dw[k] += gv * (double)h[k];
                }
            }
        }
    }
    double sum_tok = 0.0, sum_l = 0.0, sum_z = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        sum_tok += per_token[t] + wz * zt[t];
        sum_l += per_token[t];
        sum_z += zt[t];
    }
    free(G);
    free(zt);
    if (nvalid > 0) {
        scal[0] = sum_tok / (double)nvalid;
        scal[1] = sum_l / (double)nvalid;
        scal[2] = sum_z / (double)nvalid;
    } else {
        scal[0] = scal[1] = scal[2] = 0.0;
    }
    return OR_OK;
}

/* ---- distillation from given student logits, [P3] "Changes" -------------
 * The from-distribution forward/backward on materialised student logits
 * (the (loss, z_loss, grad_logits) shape): per token the same L_t, lse(a)
 * and gradient as oracle_distill, with s = logits[t] instead of H W^T.
 * reduce_sum = 0: means over N_valid (as oracle_distill); 1: sums over the
 * counted tokens, alpha_t = grad_scale m_t (this oracle's reading of the
 * "sum" reduction the pages' parity suite lists beside masking and scaling).
 * grad [n][V] may be NULL. */
int oracle_distill_from_logits(const float *logits, const float *teacher, const uint8_t *mask,
                               int64_t n, int64_t V, int direction, double T, double wz,
                               double grad_scale, int reduce_sum, double *per_token,
                               double *lse_out, double *scal, double *grad)
{
    if (n < 1 || V < 1) return OR_EMPTY_DIMENSION;
    if (n > OR_MAX_DIM || V > OR_MAX_DIM) return OR_DIMENSION_TOO_LARGE;
    if (!scalar_ok(wz) || wz < 0.0 || !scalar_ok(grad_scale) || !scalar_ok(T) || T <= 0.0)
        return OR_NON_FINITE_SCALAR;
    if (direction < 0 || direction > 2) return OR_UNKNOWN_OBJECTIVE;
    int64_t nvalid = count_valid(mask, n);
    double *zt = (double *)malloc(sizeof(double) * (size_t)n);
    #pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)V);
        double *a = (double *)malloc(sizeof(double) * (size_t)V);
        double *b = (double *)malloc(sizeof(double) * (size_t)V);
        double *g = grad ? (double *)malloc(sizeof(double) * (size_t)V) : NULL;
        #pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            for (int64_t v = 0; v < V; ++v) s[v] = (double)logits[t * V + v];
            double la;
            double L = distill_row(s, teacher + t * V, V, direction, T, a, b, &la, g);
            int on = mask ? (mask[t] != 0) : 1;
            per_token[t] = on ? L : 0.0;
            zt[t] = on ? la * la : 0.0;
            lse_out[t] = la;
            if (grad) {
                double alpha = 0.0;
                if (on) alpha = reduce_sum ? grad_scale : (nvalid > 0 ? grad_scale / (double)nvalid : 0.0);
                for (int64_t v = 0; v < V; ++v) {
                    double q = exp(a[v] - la);
                    grad[t * V + v] = alpha * (g[v] + 2.0 * wz * la * q / T);
                }
            }
        }
        free(s); free(a); free(b); free(g);
    }
    double sum_tok = 0.0, sum_l = 0.0, sum_z = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        sum_tok += per_token[t] + wz * zt[t];
        sum_l += per_token[t];
        sum_z += zt[t];
    }
    free(zt);
    double div = reduce_sum ? 1.0 : (double)nvalid;
    if (!reduce_sum && nvalid == 0) {
        scal[0] = scal[1] = scal[2] = 0.0;
    } else {
        scal[0] = sum_tok / div;
        scal[1] = sum_l / div;
        scal[2] = sum_z / div;
    }
    return OR_OK;
}

/* Sampled distillation rows: per listed token, L_t, lse(a) and the dH row.
 * The listed tokens' logit rows are computed a block of at most 256 tokens
 * at a time (fill_logits), then each row is reduced on its own. */
int oracle_distill_token_rows(const float *H, const float *W, const float *teacher,
                              const uint8_t *mask, int64_t n, int64_t d, int64_t V,
                              int direction, double T, double wz, double grad_scale,
                              const int64_t *rows, int64_t n_rows,
                              double *loss_out, double *lse_out, double *dH_rows)
{
    int st = fused_checks(n, d, V, 0, NULL, wz, grad_scale);
    if (st != OR_OK) return st;
    if (!scalar_ok(T) || T <= 0.0) return OR_NON_FINITE_SCALAR;
    if (direction < 0 || direction > 2) return OR_UNKNOWN_OBJECTIVE;
    int64_t nvalid = count_valid(mask, n);
    const int64_t RB = 256;
    double *blk = (double *)malloc(sizeof(double) * (size_t)((n_rows < RB ? n_rows : RB) * V));
    for (int64_t i0 = 0; i0 < n_rows; i0 += RB) {
        const int64_t nb = n_rows - i0 < RB ? n_rows - i0 : RB;
        fill_logits(H, W, rows + i0, 0, nb, d, V, blk);
        #pragma omp parallel
        {
            double *a = (double *)malloc(sizeof(double) * (size_t)V);
            double *b = (double *)malloc(sizeof(double) * (size_t)V);
            double *g = (double *)malloc(sizeof(double) * (size_t)V);
            #pragma omp for schedule(dynamic, 1)
            for (int64_t ib = 0; ib < nb; ++ib) {
                const int64_t i = i0 + ib, t = rows[i];
                double la;
                double L = distill_row(blk + ib * V, teacher + t * V, V, direction, T, a, b, &la, g);
                int on = mask ? (mask[t] != 0) : 1;
                loss_out[i] = L;
                lse_out[i] = la;
                if (dH_rows) {
                    double alpha = (on && nvalid > 0) ? grad_scale / (double)nvalid : 0.0;
                    double *dh = dH_rows + i * d;
                    for (int64_t k = 0; k < d; ++k) dh[k] = 0.0;
                    for (int64_t v = 0; v < V; ++v) {
                        double q = exp(a[v] - la);
                        double gv = alpha * (g[v] + 2.0 * wz * la * q / T);
                        const float *w = W + v * d;
                        for (int64_t k = 0; k < d; ++k) dh[k] += gv * (double)w[k];
                    }
                }
            }
            free(a); free(b); free(g);
        }
    }
    free(blk);
    return OR_OK;
}

/* Sampled distillation d_weight rows, for checks at sizes where the whole
 * oracle is too slow.  Per listed vocabulary row v, dW_v = sum_t G_tv H_t in
 * ascending t, with G_tv exactly as in oracle_distill: the student's lse(a)
 * and L_t of every token are given (from oracle_distill_token_rows over all
 * tokens); the teacher's lse(b) is recomputed here from each teacher row. */
int oracle_distill_dweight_rows(const float *H, const float *W, const float *teacher,
                                const uint8_t *mask, int64_t n, int64_t d, int64_t V,
                                int direction, double T, double wz, double grad_scale,
                                const double *lse_all, const double *loss_all,
                                const int64_t *vrows, int64_t n_vrows, double *dW_rows)
{
    int st = fused_checks(n, d, V, 0, NULL, wz, grad_scale);
    if (st != OR_OK) return st;
    if (!scalar_ok(T) || T <= 0.0) return OR_NON_FINITE_SCALAR;
    if (direction < 0 || direction > 2) return OR_UNKNOWN_OBJECTIVE;
    int64_t nvalid = count_valid(mask, n);
    double *lb = (double *)malloc(sizeof(double) * (size_t)n);
    #pragma omp parallel
    {
        double *b = (double *)malloc(sizeof(double) * (size_t)V);
        #pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            const float *tr = teacher + t * V;
            for (int64_t v = 0; v < V; ++v) b[v] = (double)tr[v] / T;
            lb[t] = lse_row(b, V);
        }
        free(b);
    }
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_vrows; ++i) {
        int64_t v = vrows[i];
        double *dw = dW_rows + i * d;
        for (int64_t k = 0; k < d; ++k) dw[k] = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            int on = mask ? (mask[t] != 0) : 1;
            if (!on || nvalid == 0) continue;
            double alpha = grad_scale / (double)nvalid;
            double a = dot_asc(H + t * d, W + v * d, d) / T;
            double b = (double)teacher[t * V + v] / T;
            double lq = a - lse_all[t], lp = b - lb[t];
            double q = exp(lq), p = exp(lp);
            double g = direction == 2 ? (q > 0.0 ? q * (lq - lp - loss_all[t]) / T : 0.0) : (q - p) / T;
            double gv = alpha * (g + 2.0 * wz * lse_all[t] * q / T);
            const float *h = H + t * d;
            for (int64_t k = 0; k < d; ++k) dw[k] += gv * (double)h[k];
        }
    }
    free(lb);
    return OR_OK;
}

/* The token reduction of oracle_distill and oracle_ce_fwd on its own, for
 * per-token values computed row by row (oracle_distill_token_rows over every
 * token): loss[t] is L_t (or ce_t) of every token whether counted or not,
 * lse[t] the token's log-sum-exp; masked tokens add nothing.  Sums run in
 * ascending t; scal = {total, loss mean, z mean} ([P3] shared mask and
 * divisor), zeros when N_valid = 0. */
int oracle_reduce_tokens(const double *loss, const double *lse, const uint8_t *mask, int64_t n,
                         double wz, double *scal)
{
    if (n < 1) return OR_EMPTY_DIMENSION;
    if (!scalar_ok(wz) || wz < 0.0) return OR_NON_FINITE_SCALAR;
    int64_t nvalid = count_valid(mask, n);
    double sum_tok = 0.0, sum_l = 0.0, sum_z = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        int on = mask ? (mask[t] != 0) : 1;
        double l = on ? loss[t] : 0.0, z = on ? lse[t] * lse[t] : 0.0;
        sum_tok += l + wz * z;
        sum_l += l;
        sum_z += z;
    }
    if (nvalid > 0) {
        scal[0] = sum_tok / (double)nvalid;
        scal[1] = sum_l / (double)nvalid;
        scal[2] = sum_z / (double)nvalid;
    } else {
        scal[0] = scal[1] = scal[2] = 0.0;
    }
    return OR_OK;
}

/* ---- vocabulary-parallel cross-entropy -----------------------------------
 * [P3] "Changes" (its tests add a tensor-parallel distributed subtest) and
 * "Validation" (the world_size=2 tensor-parallel subtests): the weight's
 * vocabulary rows are split into contiguous shards, one per rank.  The pages
 * do not print the exchange; the plain reading, which this oracle states:
 *
 *   shard p holds rows [v0, v0 + Vs) of a vocabulary of V_total.  Per token
 *   its partials are  lse_p = log sum_{v in shard} exp(s_tv),  the target
 *   logit s_{t,y_t} when v0 <= y_t < v0 + Vs (else 0), and a flag 1/0 saying
 *   which.  The whole row's log-sum-exp is the max-shifted log of the sum of
 *   exp(lse_p) over the shards, the target logit comes from the one shard
 *   whose flag is set, and everything after that (ce, z, the token mean) is
 *   the unsharded loss's.  The backward of a shard is the unsharded
 *   backward restricted to the shard's vocabulary columns, with the whole
 *   row's lse: it gives the shard's d_weight rows and its share of d_hidden,
 *   whose sum over the shards is d_hidden.
 *
 * partials layout: [3][n] for one shard, [P][3][n] gathered in shard order. */
int oracle_ce_shard_fwd(const float *H, const float *Ws, const int64_t *y, int64_t n, int64_t d,
                        int64_t Vs, int64_t v0, int64_t V_total, double *partials)
{
    if (n < 1 || d < 1 || Vs < 1 || V_total < 1) return OR_EMPTY_DIMENSION;
    if (v0 < 0 || v0 > V_total - Vs) return OR_LENGTH_MISMATCH;
    if (!oracle_targets_in_range(y, n, V_total)) return OR_TARGET_OUT_OF_RANGE;
    #pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Vs);
        #pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            for (int64_t v = 0; v < Vs; ++v) s[v] = dot_asc(H + t * d, Ws + v * d, d);
            int64_t yl = y[t] - v0;
            int in = yl >= 0 && yl < Vs;
            partials[t] = lse_row(s, Vs);
            partials[n + t] = in ? s[yl] : 0.0;
            partials[2 * n + t] = in ? 1.0 : 0.0;
        }
        free(s);
    }
    return OR_OK;
}

int oracle_ce_shard_combine(const double *partials, int64_t P, int64_t n, const uint8_t *mask,
                            double wz, double *lse_out, double *ce_out, double *scal)
{
    if (n < 1 || P < 1) return OR_EMPTY_DIMENSION;
    if (!scalar_ok(wz) || wz < 0.0) return OR_NON_FINITE_SCALAR;
    for (int64_t t = 0; t < n; ++t) {
        double flags = 0.0;
        for (int64_t p = 0; p < P; ++p) flags += partials[(p * 3 + 2) * n + t];
        if (flags != 1.0) return OR_TARGET_OUT_OF_RANGE;   /* no shard, or two, hold the target */
    }
    int64_t nvalid = count_valid(mask, n);
    double sum_tok = 0.0, sum_ce = 0.0, sum_z = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        double m = partials[t];
        for (int64_t p = 1; p < P; ++p)
            if (partials[p * 3 * n + t] > m) m = partials[p * 3 * n + t];
        double acc = 0.0, tgt = 0.0;
        for (int64_t p = 0; p < P; ++p) {
            acc += exp(partials[p * 3 * n + t] - m);
            if (partials[(p * 3 + 2) * n + t] != 0.0) tgt = partials[(p * 3 + 1) * n + t];
        }
        double lse = m + log(acc);
        int on = mask ? (mask[t] != 0) : 1;
        lse_out[t] = lse;
        ce_out[t] = on ? lse - tgt : 0.0;
        double z = on ? lse * lse : 0.0;
        sum_tok += ce_out[t] + wz * z;
        sum_ce += ce_out[t];
        sum_z += z;
    }
    if (nvalid > 0) {
        scal[0] = sum_tok / (double)nvalid;
        scal[1] = sum_ce / (double)nvalid;
        scal[2] = sum_z / (double)nvalid;
    } else {
        scal[0] = scal[1] = scal[2] = 0.0;
    }
    return OR_OK;
}

int oracle_ce_shard_bwd(const float *H, const float *Ws, const int64_t *y, const uint8_t *mask,
                        int64_t n, int64_t d, int64_t Vs, int64_t v0, int64_t V_total, double wz,
                        double grad_scale, const double *lse_all, double *dH_part, double *dW_shard)
{
    if (n < 1 || d < 1 || Vs < 1 || V_total < 1) return OR_EMPTY_DIMENSION;
    if (v0 < 0 || v0 > V_total - Vs) return OR_LENGTH_MISMATCH;
    if (!scalar_ok(wz) || wz < 0.0 || !scalar_ok(grad_scale)) return OR_NON_FINITE_SCALAR;
    if (!oracle_targets_in_range(y, n, V_total)) return OR_TARGET_OUT_OF_RANGE;
    int64_t nvalid = count_valid(mask, n);
    double *G = (double *)malloc(sizeof(double) * (size_t)(n * Vs));
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        int on = mask ? (mask[t] != 0) : 1;
        double alpha = (on && nvalid > 0) ? grad_scale / (double)nvalid : 0.0;
        double c = alpha * (1.0 + 2.0 * wz * lse_all[t]);
        for (int64_t v = 0; v < Vs; ++v) {
            double g = c * exp(dot_asc(H + t * d, Ws + v * d, d) - lse_all[t]);
            if (v0 + v == y[t]) g -= alpha;
            G[t * Vs + v] = g;
        }
        if (dH_part) {
            double *dh = dH_part + t * d;
            for (int64_t k = 0; k < d; ++k) dh[k] = 0.0;
            for (int64_t v = 0; v < Vs; ++v) {
                const float *w = Ws + v * d;
                for (int64_t k = 0; k < d; ++k) dh[k] += G[t * Vs + v] * (double)w[k];
            }
        }
    }
    if (dW_shard) {
        #pragma omp parallel for schedule(static)
        for (int64_t v = 0; v < Vs; ++v) {
            double *dw = dW_shard + v * d;
            for (int64_t k = 0; k < d; ++k) dw[k] = 0.0;
            for (int64_t t = 0; t < n; ++t) {
                const float *h = H + t * d;
                for (int64_t k = 0; k < d; ++k) dw[k] += G[t * Vs + v] * (double)h[k];
            }
        }
    }
    free(G);
    return OR_OK;
}

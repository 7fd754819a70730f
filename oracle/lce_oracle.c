/*
 * lce_oracle.c -- float64 CPU oracle for the chunked language-model-head
 * cross-entropy ("chunked NLL loss").
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the timed
 * CPU baseline of the benchmark load this library. The product path
 * (chunked_lm_head_gemm_gb300) never links, imports or calls it, and it
 * shares no code, header, table or helper with the CUDA path.
 *
 * What it computes, stated from the source pages:
 *   - "Training Beyond 1M Tokens" (TRL guide), section "The loss is the
 *     first thing to break": the last decoder layer gives hidden states of
 *     shape L x H; multiplying by the LM-head weights gives logits of shape
 *     L x V; the loss is a cross entropy of those logits against the target
 *     labels.
 *   - Same guide, section "The massive logits matrix: chunk it": the loss is
 *     a sum over rows and the softmax runs along the vocabulary of one row,
 *     so rows may be processed in pieces and the pieces summed. The oracle
 *     does the plain whole-matrix computation; chunking is the CUDA path's
 *     business and must give the same numbers.
 *   - Reduction (the pages leave it open): labels equal to ignore_index, or
 *     outside [0, V), are ignored; the loss is the sum of per-row losses
 *     over the remaining rows divided by their count N. With N = 0 the loss
 *     and both gradients are 0.
 *
 * The plain definition, written out in float64, row by row:
 *   z[i][j]  = sum_k h[i][k] * W[j][k]                      (logits)
 *   lse[i]   = m_i + log( sum_j exp(z[i][j] - m_i) ),  m_i = max_j z[i][j]
 *   loss     = (1/N) * sum_{valid i} ( lse[i] - z[i][y_i] )
 *   G[i][j]  = dloss/N * ( exp(z[i][j] - lse[i]) - [j == y_i] )  (valid i)
 *            = 0                                                  (ignored i)
 *   dH       = G W        (L x H)
 *   dW       = G^T h      (V x H)
 * The max shift m_i is the textbook way to evaluate log-sum-exp without
 * overflow; it does not change the value.
 *
 * Two variants of the per-row loss, neither on the pages (they define only
 * the plain cross entropy above), selected by eps and zcoef (both 0 gives
 * the plain loss through the plain code):
 *   - label smoothing eps: the cross entropy against the smoothed target
 *     q_j = (1 - eps) [j == y_i] + eps / V instead of the one-hot,
 *       loss_i = sum_j q_j (lse[i] - z[i][j]);
 *   - z-loss zcoef: loss_i += zcoef * lse[i]^2.
 *   Then loss = (1/N) sum_{valid i} loss_i as before, and
 *   G[i][j] = dloss/N * ( (1 + 2 zcoef lse[i]) exp(z[i][j] - lse[i]) - q_j ).
 *
 * Inputs are widened to float64 exactly: dtype 0 = bfloat16 (raw 16-bit
 * patterns), 1 = float32, 2 = float64. All arithmetic is float64; the
 * exponential and logarithm are the C library's exp() and log().
 *
 * Parity is pinned in the tests (not here): against PyTorch's float64
 * cross_entropy + autograd, against central finite differences, against the
 * W = 0 closed form, and against invariants (gradient rows sum to zero,
 * shift invariance, row-permutation invariance).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_LABEL_RANGE 4
#define ORACLE_NO_MEMORY 7

/* ---- element access: widen one input element to float64 ---------------- */

static double widen(const void *base, int dtype, int64_t idx) {
    if (dtype == 0) {
        /* bfloat16 is the top half of an IEEE float32 */
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (dtype == 1) return (double)((const float *)base)[idx];
    return ((const double *)base)[idx];
}

/* Copy rows [r0, r0+n) of a row-major (rows x cols) input into float64. */
static void widen_rows(const void *base, int dtype, int64_t cols, int64_t r0,
                       int64_t n, double *out) {
    for (int64_t r = 0; r < n; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = widen(base, dtype, (r0 + r) * cols + c);
}

static int label_is_valid(int64_t y, int64_t V, int64_t ignore_index) {
    return y != ignore_index && y >= 0 && y < V;
}

/* N = number of rows whose label takes part in the loss. *bad is set when a
 * label is neither ignore_index nor inside [0, V). */
static int64_t count_valid(const int64_t *labels, int64_t L, int64_t V,
                           int64_t ignore_index, int *bad) {
    int64_t n = 0;
    *bad = 0;
    for (int64_t i = 0; i < L; ++i) {
        if (label_is_valid(labels[i], V, ignore_index))
            ++n;
        else if (labels[i] != ignore_index)
            *bad = 1;
    }
    return n;
}

/* ---- one row: logits, log-sum-exp --------------------------------------- */

/* Dot product of a float64 row with row j of W, W kept in its input type. */
static double dot_row(const double *x, const void *W, int dtype, int64_t j,
                      int64_t H) {
    double acc = 0.0;
    if (dtype == 0) {
        const uint16_t *w = (const uint16_t *)W + j * H;
        for (int64_t k = 0; k < H; ++k) {
            uint32_t bits = (uint32_t)w[k] << 16;
            float f;
            memcpy(&f, &bits, sizeof f);
            acc += x[k] * (double)f;
        }
    } else if (dtype == 1) {
        const float *w = (const float *)W + j * H;
        for (int64_t k = 0; k < H; ++k) acc += x[k] * (double)w[k];
    } else {
        const double *w = (const double *)W + j * H;
        for (int64_t k = 0; k < H; ++k) acc += x[k] * w[k];
    }
    return acc;
}

/* z[j] = sum_k h_row[k] * W[j][k] for every j < V. */
static void row_logits(const double *h_row, const void *W, int dtype,
                       int64_t H, int64_t V, double *z) {
    for (int64_t j = 0; j < V; ++j) z[j] = dot_row(h_row, W, dtype, j, H);
}

static double row_lse(const double *z, int64_t V) {
    double m = -INFINITY;
    for (int64_t j = 0; j < V; ++j)
        if (z[j] > m) m = z[j];
    double s = 0.0;
    for (int64_t j = 0; j < V; ++j) s += exp(z[j] - m);
    return m + log(s);
}

/* ---- threading ---------------------------------------------------------- */

typedef struct {
    /* problem */
    const void *h;
    int dtype;
    const void *W;    /* V x H, input type */
    const int64_t *labels;
    int64_t L, H, V, ignore_index;
    /* which rows: rows[r] for r in [r0, r1) if rows != NULL, else r itself */
    const int64_t *rows;
    int64_t r0, r1;
    /* outputs (any may be NULL) */
    double *lse, *zy;
    double *G;    /* nrows x V, only for the backward */
    double gscale; /* dloss / N, 0 when N == 0 */
    double eps, zcoef; /* loss variant (both 0: plain cross entropy) */
    double *term;  /* per-row loss of a variant (0 for ignored rows) */
    int status;
} row_job;

/* One row's loss under the variants: the cross entropy against the smoothed
 * target q_j = (1 - eps) [j == y] + eps / V, plus zcoef * lse^2. */
static double row_term(const double *z, int64_t V, int64_t y, double lse,
                       double eps, double zcoef) {
    double t = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        double q = (j == y ? 1.0 - eps : 0.0) + eps / (double)V;
        t += q * (lse - z[j]);
    }
    return t + zcoef * lse * lse;
}

static void *row_worker(void *arg) {
    row_job *jb = (row_job *)arg;
    double *hrow = (double *)malloc((size_t)jb->H * sizeof(double));
    double *z = (double *)malloc((size_t)jb->V * sizeof(double));
    if (!hrow || !z) {
        free(hrow);
        free(z);
        jb->status = ORACLE_NO_MEMORY;
        return NULL;
    }
    for (int64_t r = jb->r0; r < jb->r1; ++r) {
        int64_t i = jb->rows ? jb->rows[r] : r;
        widen_rows(jb->h, jb->dtype, jb->H, i, 1, hrow);
        row_logits(hrow, jb->W, jb->dtype, jb->H, jb->V, z);
        double lse = row_lse(z, jb->V);
        int64_t y = jb->labels[i];
        int valid = label_is_valid(y, jb->V, jb->ignore_index);
        if (jb->lse) jb->lse[r] = lse;
        if (jb->zy) jb->zy[r] = valid ? z[y] : NAN;
        if (jb->term)
            jb->term[r] = valid ? row_term(z, jb->V, y, lse, jb->eps,
                                           jb->zcoef)
                                : 0.0;
        if (jb->G) {
            double *g = jb->G + r * jb->V;
            if (!valid || jb->gscale == 0.0) {
                for (int64_t j = 0; j < jb->V; ++j) g[j] = 0.0;
            } else if (jb->eps == 0.0 && jb->zcoef == 0.0) {
                for (int64_t j = 0; j < jb->V; ++j)
                    g[j] = jb->gscale * exp(z[j] - lse);
                g[y] -= jb->gscale;
            } else {
                /* d loss_i / d z_j = (1 + 2 zcoef lse) p_j - q_j */
                const double zf = 1.0 + 2.0 * jb->zcoef * lse;
                const double qu = jb->eps / (double)jb->V;
                for (int64_t j = 0; j < jb->V; ++j)
                    g[j] = jb->gscale * (zf * exp(z[j] - lse) - qu);
                g[y] -= jb->gscale * (1.0 - jb->eps);
            }
        }
    }
    free(hrow);
    free(z);
    jb->status = ORACLE_OK;
    return NULL;
}

/* Run row_worker over [0, nrows) split into nthreads contiguous pieces. */
static int run_rows(row_job proto, int64_t nrows, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;
    row_job *jobs = (row_job *)calloc((size_t)nthreads, sizeof(row_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return ORACLE_NO_MEMORY;
    }
    int64_t per = (nrows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].r0 = t * per < nrows ? t * per : nrows;
        jobs[t].r1 = (t + 1) * per < nrows ? (t + 1) * per : nrows;
        pthread_create(&tid[t], NULL, row_worker, &jobs[t]);
    }
    int st = ORACLE_OK;
    for (int t = 0; t < nthreads; ++t) {
        pthread_join(tid[t], NULL);
        if (jobs[t].status != ORACLE_OK) st = jobs[t].status;
    }
    free(jobs);
    free(tid);
    return st;
}

static double *widen_all(const void *x, int dtype, int64_t rows, int64_t cols) {
    double *d = (double *)malloc((size_t)(rows * cols) * sizeof(double));
    if (d) widen_rows(x, dtype, cols, 0, rows, d);
    return d;
}

static int check_args(const void *h, const void *W, int dtype,
                      const int64_t *labels, int64_t L, int64_t H, int64_t V) {
    if (!h || !W || !labels) return ORACLE_BAD_ARG;
    if (dtype < 0 || dtype > 2) return ORACLE_BAD_ARG;
    if (L < 1 || H < 1 || V < 1) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

static int check_variant(double eps, double zcoef) {
    if (!(eps >= 0.0 && eps <= 1.0) || !(zcoef >= 0.0 && zcoef < INFINITY))
        return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

static int is_plain(double eps, double zcoef) {
    return eps == 0.0 && zcoef == 0.0;
}

/* ---- public entry points ------------------------------------------------ */

/*
 * Forward: lse[L], zy[L] (logit at the label, NaN for ignored rows),
 * loss = sum_valid(lse - zy) / N (0 when N == 0), n_valid = N; with a loss
 * variant (eps or zcoef not 0) the summed per-row loss is row_term's.
 * Returns ORACLE_LABEL_RANGE (results still written, those rows ignored)
 * when some label is neither ignore_index nor in [0, V).
 */
int lce_oracle_forward(const void *h, const void *W, int dtype,
                       const int64_t *labels, int64_t L, int64_t H, int64_t V,
                       int64_t ignore_index, double eps, double zcoef,
                       int nthreads, double *lse, double *zy, double *loss,
                       int64_t *n_valid) {
    int st = check_args(h, W, dtype, labels, L, H, V);
    if (st) return st;
    if ((st = check_variant(eps, zcoef))) return st;
    int bad = 0;
    int64_t n = count_valid(labels, L, V, ignore_index, &bad);
    const int plain = is_plain(eps, zcoef);
    double *lse_buf = lse ? lse : (double *)malloc((size_t)L * sizeof(double));
    double *zy_buf = zy ? zy : (double *)malloc((size_t)L * sizeof(double));
    double *term = plain ? NULL : (double *)malloc((size_t)L * sizeof(double));
    if (!lse_buf || !zy_buf || (!plain && !term)) {
        st = ORACLE_NO_MEMORY;
        goto out;
    }
    row_job proto = {0};
    proto.h = h;
    proto.dtype = dtype;
    proto.W = W;
    proto.labels = labels;
    proto.L = L;
    proto.H = H;
    proto.V = V;
    proto.ignore_index = ignore_index;
    proto.lse = lse_buf;
    proto.zy = zy_buf;
    proto.eps = eps;
    proto.zcoef = zcoef;
    proto.term = term;
    st = run_rows(proto, L, nthreads);
    if (st) goto out;
    {
        double total = 0.0;
        for (int64_t i = 0; i < L; ++i)
            if (label_is_valid(labels[i], V, ignore_index))
                total += plain ? lse_buf[i] - zy_buf[i] : term[i];
        if (loss) *loss = n > 0 ? total / (double)n : 0.0;
        if (n_valid) *n_valid = n;
    }
    st = bad ? ORACLE_LABEL_RANGE : ORACLE_OK;
out:
    if (!lse) free(lse_buf);
    if (!zy) free(zy_buf);
    free(term);
    return st;
}

/* out[:] += a * W[j][:], W kept in its input type. */
static void axpy_row(double a, const void *W, int dtype, int64_t j, int64_t H,
                     double *out) {
    if (dtype == 0) {
        const uint16_t *w = (const uint16_t *)W + j * H;
        for (int64_t k = 0; k < H; ++k) {
            uint32_t bits = (uint32_t)w[k] << 16;
            float f;
            memcpy(&f, &bits, sizeof f);
            out[k] += a * (double)f;
        }
    } else if (dtype == 1) {
        const float *w = (const float *)W + j * H;
        for (int64_t k = 0; k < H; ++k) out[k] += a * (double)w[k];
    } else {
        const double *w = (const double *)W + j * H;
        for (int64_t k = 0; k < H; ++k) out[k] += a * w[k];
    }
}

typedef struct {
    const double *G;  /* L x V */
    const void *W;    /* V x H, input type */
    int dtype;
    const double *hd; /* L x H */
    int64_t L, H, V;
    int64_t a0, a1;   /* row range (dH) or vocab range (dW) */
    double *dH, *dW;
    const int64_t *vrows; /* dW rows to compute: vrows[a] (NULL: a itself) */
} mm_job;

/* dH[i][:] = sum_j G[i][j] * W[j][:] for i in [a0, a1) */
static void *dH_worker(void *arg) {
    mm_job *jb = (mm_job *)arg;
    for (int64_t i = jb->a0; i < jb->a1; ++i) {
        double *out = jb->dH + i * jb->H;
        for (int64_t k = 0; k < jb->H; ++k) out[k] = 0.0;
        const double *g = jb->G + i * jb->V;
        for (int64_t j = 0; j < jb->V; ++j)
            if (g[j] != 0.0) axpy_row(g[j], jb->W, jb->dtype, j, jb->H, out);
    }
    return NULL;
}

/* dW[j][:] = sum_i G[i][j] * h[i][:] for the vocabulary ids j of [a0, a1)
 * (or of vrows[a0..a1) when a subset was asked for; out row a then). */
static void *dW_worker(void *arg) {
    mm_job *jb = (mm_job *)arg;
    for (int64_t a = jb->a0; a < jb->a1; ++a) {
        const int64_t j = jb->vrows ? jb->vrows[a] : a;
        double *out = jb->dW + a * jb->H;
        for (int64_t k = 0; k < jb->H; ++k) out[k] = 0.0;
        for (int64_t i = 0; i < jb->L; ++i) {
            double g = jb->G[i * jb->V + j];
            if (g == 0.0) continue;
            const double *hr = jb->hd + i * jb->H;
            for (int64_t k = 0; k < jb->H; ++k) out[k] += g * hr[k];
        }
    }
    return NULL;
}

static void run_mm(mm_job proto, int64_t n, int nthreads, void *(*fn)(void *)) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = (int)n;
    mm_job jobs[256];
    pthread_t tid[256];
    if (nthreads > 256) nthreads = 256;
    int64_t per = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].a0 = t * per < n ? t * per : n;
        jobs[t].a1 = (t + 1) * per < n ? (t + 1) * per : n;
        pthread_create(&tid[t], NULL, fn, &jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(tid[t], NULL);
}

/*
 * Backward for the whole problem: given the upstream gradient dloss of the
 * scalar loss, writes dH (L x H) and/or dW in float64 (either may be NULL).
 * dW is V x H, or, when vrows is not NULL, the nvrows x H rows dW[vrows[a]].
 * Holds G (L x V float64) in host memory, so it is for shapes whose L x V
 * fits.
 */
int lce_oracle_backward(const void *h, const void *W, int dtype,
                        const int64_t *labels, int64_t L, int64_t H, int64_t V,
                        int64_t ignore_index, double eps, double zcoef,
                        double dloss, int nthreads, double *dH, double *dW,
                        const int64_t *vrows, int64_t nvrows) {
    int st = check_args(h, W, dtype, labels, L, H, V);
    if (st) return st;
    if ((st = check_variant(eps, zcoef))) return st;
    if (vrows) {
        if (nvrows < 1) return ORACLE_BAD_ARG;
        for (int64_t a = 0; a < nvrows; ++a)
            if (vrows[a] < 0 || vrows[a] >= V) return ORACLE_BAD_ARG;
    }
    int bad = 0;
    int64_t n = count_valid(labels, L, V, ignore_index, &bad);
    double *hd = widen_all(h, dtype, L, H);
    double *G = (double *)malloc((size_t)(L * V) * sizeof(double));
    if (!hd || !G) {
        st = ORACLE_NO_MEMORY;
        goto out;
    }
    {
        row_job proto = {0};
        proto.h = h;
        proto.dtype = dtype;
        proto.W = W;
        proto.labels = labels;
        proto.L = L;
        proto.H = H;
        proto.V = V;
        proto.ignore_index = ignore_index;
        proto.G = G;
        proto.eps = eps;
        proto.zcoef = zcoef;
        proto.gscale = n > 0 ? dloss / (double)n : 0.0;
        st = run_rows(proto, L, nthreads);
        if (st) goto out;
    }
    {
        mm_job mp = {G, W, dtype, hd, L, H, V, 0, 0, dH, dW, vrows};
        if (dH) run_mm(mp, L, nthreads, dH_worker);
        if (dW) run_mm(mp, vrows ? nvrows : V, nthreads, dW_worker);
    }
    st = bad ? ORACLE_LABEL_RANGE : ORACLE_OK;
out:
    free(hd);
    free(G);
    return st;
}

/*
 * Selected rows of a problem of any size: for each rows[r], lse, the logit
 * at the label (NaN if ignored) and, if dH_rows is not NULL, that row of dH
 * (nrows x H). N is counted over all L labels, so the values are those of
 * the whole problem. Cost: nrows * H * V multiply-adds (twice with dH).
 */
int lce_oracle_rows(const void *h, const void *W, int dtype,
                    const int64_t *labels, int64_t L, int64_t H, int64_t V,
                    int64_t ignore_index, double eps, double zcoef,
                    double dloss, const int64_t *rows, int64_t nrows,
                    int nthreads, double *lse, double *zy, double *dH_rows) {
    int st = check_args(h, W, dtype, labels, L, H, V);
    if (st) return st;
    if ((st = check_variant(eps, zcoef))) return st;
    if (!rows || nrows < 1) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= L) return ORACLE_BAD_ARG;
    int bad = 0;
    int64_t n = count_valid(labels, L, V, ignore_index, &bad);
    double *G = dH_rows ? (double *)malloc((size_t)(nrows * V) * sizeof(double))
                        : NULL;
    if (dH_rows && !G) {
        st = ORACLE_NO_MEMORY;
        goto out;
    }
    {
        row_job proto = {0};
        proto.h = h;
        proto.dtype = dtype;
        proto.W = W;
        proto.labels = labels;
        proto.L = L;
        proto.H = H;
        proto.V = V;
        proto.ignore_index = ignore_index;
        proto.rows = rows;
        proto.lse = lse;
        proto.zy = zy;
        proto.G = G;
        proto.eps = eps;
        proto.zcoef = zcoef;
        proto.gscale = n > 0 ? dloss / (double)n : 0.0;
        st = run_rows(proto, nrows, nthreads);
        if (st) goto out;
    }
    if (dH_rows) {
        mm_job mp = {G, W, dtype, NULL, nrows, H, V, 0, 0, dH_rows, NULL, NULL};
        run_mm(mp, nrows, nthreads, dH_worker);
    }
    st = bad ? ORACLE_LABEL_RANGE : ORACLE_OK;
out:
    free(G);
    return st;
}

/*
 * Forward and backward of the whole problem from one pass over the logits:
 * what lce_oracle_forward and lce_oracle_backward return for the same
 * arguments (any output may be NULL), with each row's logits computed once
 * instead of twice. Holds G (L x V float64) like lce_oracle_backward.
 */
int lce_oracle_forward_backward(const void *h, const void *W, int dtype,
                                const int64_t *labels, int64_t L, int64_t H,
                                int64_t V, int64_t ignore_index, double eps,
                                double zcoef, double dloss, int nthreads,
                                double *lse, double *zy, double *loss,
                                int64_t *n_valid, double *dH, double *dW,
                                const int64_t *vrows, int64_t nvrows) {
    int st = check_args(h, W, dtype, labels, L, H, V);
    if (st) return st;
    if ((st = check_variant(eps, zcoef))) return st;
    if (vrows) {
        if (nvrows < 1) return ORACLE_BAD_ARG;
        for (int64_t a = 0; a < nvrows; ++a)
            if (vrows[a] < 0 || vrows[a] >= V) return ORACLE_BAD_ARG;
    }
    int bad = 0;
    int64_t n = count_valid(labels, L, V, ignore_index, &bad);
    const int plain = is_plain(eps, zcoef);
    double *lse_buf = lse ? lse : (double *)malloc((size_t)L * sizeof(double));
    double *zy_buf = zy ? zy : (double *)malloc((size_t)L * sizeof(double));
    double *term = plain ? NULL : (double *)malloc((size_t)L * sizeof(double));
    double *hd = widen_all(h, dtype, L, H);
    double *G = (double *)malloc((size_t)(L * V) * sizeof(double));
    if (!lse_buf || !zy_buf || (!plain && !term) || !hd || !G) {
        st = ORACLE_NO_MEMORY;
        goto out;
    }
    {
        row_job proto = {0};
        proto.h = h;
        proto.dtype = dtype;
        proto.W = W;
        proto.labels = labels;
        proto.L = L;
        proto.H = H;
        proto.V = V;
        proto.ignore_index = ignore_index;
        proto.lse = lse_buf;
        proto.zy = zy_buf;
        proto.term = term;
        proto.G = G;
        proto.eps = eps;
        proto.zcoef = zcoef;
        proto.gscale = n > 0 ? dloss / (double)n : 0.0;
        st = run_rows(proto, L, nthreads);
        if (st) goto out;
    }
    {
        double total = 0.0;
        for (int64_t i = 0; i < L; ++i)
            if (label_is_valid(labels[i], V, ignore_index))
                total += plain ? lse_buf[i] - zy_buf[i] : term[i];
        if (loss) *loss = n > 0 ? total / (double)n : 0.0;
        if (n_valid) *n_valid = n;
    }
    {
        mm_job mp = {G, W, dtype, hd, L, H, V, 0, 0, dH, dW, vrows};
        if (dH) run_mm(mp, L, nthreads, dH_worker);
        if (dW) run_mm(mp, vrows ? nvrows : V, nthreads, dW_worker);
    }
    st = bad ? ORACLE_LABEL_RANGE : ORACLE_OK;
out:
    if (!lse) free(lse_buf);
    if (!zy) free(zy_buf);
    free(term);
    free(hd);
    free(G);
    return st;
}

/* N over all rows; *bad_out = 1 if some label is out of range. */
int64_t lce_oracle_count_valid(const int64_t *labels, int64_t L, int64_t V,
                               int64_t ignore_index, int *bad_out) {
    int bad = 0;
    int64_t n = count_valid(labels, L, V, ignore_index, &bad);
    if (bad_out) *bad_out = bad;
    return n;
}

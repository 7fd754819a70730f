/*
 * mlp_oracle.c -- float64 CPU oracle for the gated MLP of a decoder layer,
 * the second workload of the row-chunking idea.
 *
 * TEST INFRASTRUCTURE, like lce_oracle.c: only the tests, the smoke check and
 * the benchmark's CPU baseline load it; it shares no code with the CUDA path.
 *
 * What it computes, from "Training Beyond 1M Tokens" (TRL guide), section
 * "One GPU is not enough: split the sequence across many": one MLP line of
 * the model is down_proj(act_fn(gate_proj(x)) * up_proj(x)), whose four
 * intermediate-width tensors are what fills the card at long sequence
 * length. With x [L][H], the three projections' weights in nn.Linear layout
 * Wg [I][H], Wu [I][H], Wd [H][I], and act_fn = SiLU (the activation of the
 * Qwen3 models the guide trains; the guide itself only says act_fn):
 *   g = x Wg^T,  u = x Wu^T                      [L][I]
 *   a = silu(g) * u,   silu(t) = t / (1 + exp(-t))
 *   y = a Wd^T                                   [L][H]
 * and, given the upstream gradient dy [L][H]:
 *   da  = dy Wd                                  [L][I]
 *   dWd = dy^T a                                 [H][I]
 *   du  = da * silu(g)
 *   dg  = da * u * silu'(g),  silu'(t) = s (1 + t (1 - s)),  s = 1/(1+exp(-t))
 *   dx  = dg Wg + du Wu                          [L][H]
 *   dWg = dg^T x,  dWu = du^T x                  [I][H]
 * Every row of x is independent in all of these except the weight
 * gradients, which are sums over rows -- why the rows can be tiled.
 *
 * All arithmetic is float64; inputs are widened exactly (dtype 0 = bf16 raw
 * bits, 1 = float32, 2 = float64).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MLP_OK 0
#define MLP_BAD_ARG 1
#define MLP_NO_MEMORY 7

static double mlp_widen(const void *base, int dtype, int64_t idx) {
    if (dtype == 0) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (dtype == 1) return (double)((const float *)base)[idx];
    return ((const double *)base)[idx];
}

static double *mlp_widen_all(const void *x, int dtype, int64_t n) {
    double *d = (double *)malloc((size_t)n * sizeof(double));
    if (d)
        for (int64_t i = 0; i < n; ++i) d[i] = mlp_widen(x, dtype, i);
    return d;
}

static double silu(double t) { return t / (1.0 + exp(-t)); }

static double silu_grad(double t) {
    double s = 1.0 / (1.0 + exp(-t));
    return s * (1.0 + t * (1.0 - s));
}

typedef struct {
    const double *x, *Wg, *Wu, *Wd, *dy;
    int64_t L, H, I;
    int64_t a0, a1; /* range of rows (or of weight rows for dW jobs) */
    double *g, *u, *a, *y, *dg, *du, *dx, *dWg, *dWu, *dWd;
} mlp_job;

/* g, u, a for rows [a0, a1); y too if requested. */
static void *fwd_worker(void *arg) {
    mlp_job *j = (mlp_job *)arg;
    for (int64_t r = j->a0; r < j->a1; ++r) {
        const double *xr = j->x + r * j->H;
        for (int64_t i = 0; i < j->I; ++i) {
            const double *wg = j->Wg + i * j->H, *wu = j->Wu + i * j->H;
            double sg = 0.0, su = 0.0;
            for (int64_t k = 0; k < j->H; ++k) {
                sg += xr[k] * wg[k];
                su += xr[k] * wu[k];
            }
            j->g[r * j->I + i] = sg;
            j->u[r * j->I + i] = su;
            j->a[r * j->I + i] = silu(sg) * su;
        }
        if (j->y) {
            const double *ar = j->a + r * j->I;
            for (int64_t h = 0; h < j->H; ++h) {
                const double *wd = j->Wd + h * j->I;
                double s = 0.0;
                for (int64_t i = 0; i < j->I; ++i) s += ar[i] * wd[i];
                j->y[r * j->H + h] = s;
            }
        }
    }
    return NULL;
}

/* da = dy Wd, then dg, du, dx for rows [a0, a1). */
static void *bwd_rows_worker(void *arg) {
    mlp_job *j = (mlp_job *)arg;
    for (int64_t r = j->a0; r < j->a1; ++r) {
        const double *dyr = j->dy + r * j->H;
        for (int64_t i = 0; i < j->I; ++i) {
            double da = 0.0;
            for (int64_t h = 0; h < j->H; ++h) da += dyr[h] * j->Wd[h * j->I + i];
            double g = j->g[r * j->I + i], u = j->u[r * j->I + i];
            j->du[r * j->I + i] = da * silu(g);
            j->dg[r * j->I + i] = da * u * silu_grad(g);
        }
        if (j->dx) {
            double *dxr = j->dx + r * j->H;
            for (int64_t k = 0; k < j->H; ++k) dxr[k] = 0.0;
            for (int64_t i = 0; i < j->I; ++i) {
                double cg = j->dg[r * j->I + i], cu = j->du[r * j->I + i];
                const double *wg = j->Wg + i * j->H, *wu = j->Wu + i * j->H;
                for (int64_t k = 0; k < j->H; ++k) dxr[k] += cg * wg[k] + cu * wu[k];
            }
        }
    }
    return NULL;
}

/* dWg, dWu rows i in [a0, a1): sum over rows r of dg[r][i] x[r][:]. */
static void *dWgu_worker(void *arg) {
    mlp_job *j = (mlp_job *)arg;
    for (int64_t i = j->a0; i < j->a1; ++i) {
        double *og = j->dWg ? j->dWg + i * j->H : NULL;
        double *ou = j->dWu ? j->dWu + i * j->H : NULL;
        for (int64_t k = 0; k < j->H; ++k) {
            if (og) og[k] = 0.0;
            if (ou) ou[k] = 0.0;
        }
        for (int64_t r = 0; r < j->L; ++r) {
            const double *xr = j->x + r * j->H;
            double cg = j->dg[r * j->I + i], cu = j->du[r * j->I + i];
            for (int64_t k = 0; k < j->H; ++k) {
                if (og) og[k] += cg * xr[k];
                if (ou) ou[k] += cu * xr[k];
            }
        }
    }
    return NULL;
}

/* dWd rows h in [a0, a1): sum over rows r of dy[r][h] a[r][:]. */
static void *dWd_worker(void *arg) {
    mlp_job *j = (mlp_job *)arg;
    for (int64_t h = j->a0; h < j->a1; ++h) {
        double *o = j->dWd + h * j->I;
        for (int64_t i = 0; i < j->I; ++i) o[i] = 0.0;
        for (int64_t r = 0; r < j->L; ++r) {
            double c = j->dy[r * j->H + h];
            const double *ar = j->a + r * j->I;
            for (int64_t i = 0; i < j->I; ++i) o[i] += c * ar[i];
        }
    }
    return NULL;
}

static void mlp_run(mlp_job proto, int64_t n, int nthreads,
                    void *(*fn)(void *)) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > n) nthreads = n > 0 ? (int)n : 1;
    mlp_job jobs[256];
    pthread_t tid[256];
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
 * Forward y = (silu(x Wg^T) * (x Wu^T)) Wd^T, and backward for the given dy
 * (dy may be NULL: forward only). Any output pointer may be NULL.
 */
int mlp_oracle(const void *x, const void *Wg, const void *Wu, const void *Wd,
               int dtype, int64_t L, int64_t H, int64_t I, const double *dy,
               int nthreads, double *y, double *dx, double *dWg, double *dWu,
               double *dWd) {
    if (!x || !Wg || !Wu || !Wd || dtype < 0 || dtype > 2 || L < 1 || H < 1 ||
        I < 1)
        return MLP_BAD_ARG;
    int st = MLP_OK;
    double *xd = mlp_widen_all(x, dtype, L * H);
    double *wg = mlp_widen_all(Wg, dtype, I * H);
    double *wu = mlp_widen_all(Wu, dtype, I * H);
    double *wd = mlp_widen_all(Wd, dtype, H * I);
    double *g = (double *)malloc((size_t)(L * I) * sizeof(double));
    double *u = (double *)malloc((size_t)(L * I) * sizeof(double));
    double *a = (double *)malloc((size_t)(L * I) * sizeof(double));
    double *dg = dy ? (double *)malloc((size_t)(L * I) * sizeof(double)) : NULL;
    double *du = dy ? (double *)malloc((size_t)(L * I) * sizeof(double)) : NULL;
    if (!xd || !wg || !wu || !wd || !g || !u || !a || (dy && (!dg || !du))) {
        st = MLP_NO_MEMORY;
        goto out;
    }
    {
        mlp_job p;
        memset(&p, 0, sizeof p);
        p.x = xd;
        p.Wg = wg;
        p.Wu = wu;
        p.Wd = wd;
        p.dy = dy;
        p.L = L;
        p.H = H;
        p.I = I;
        p.g = g;
        p.u = u;
        p.a = a;
        p.y = y;
        p.dg = dg;
        p.du = du;
        p.dx = dx;
        p.dWg = dWg;
        p.dWu = dWu;
        p.dWd = dWd;
        mlp_run(p, L, nthreads, fwd_worker);
        if (dy) {
            mlp_run(p, L, nthreads, bwd_rows_worker);
            if (dWg || dWu) mlp_run(p, I, nthreads, dWgu_worker);
            if (dWd) mlp_run(p, H, nthreads, dWd_worker);
        }
    }
out:
    free(xd);
    free(wg);
    free(wu);
    free(wd);
    free(g);
    free(u);
    free(a);
    free(dg);
    free(du);
    return st;
}

/*
 * The library's C ABI (include/lce.h) driven from a plain C program, with no
 * Python in between; test infrastructure, built and run by
 * tests/test_c_program.py.
 *
 * Without arguments it checks what needs no GPU: status strings, workspace
 * and chunk sizes, and argument errors returned before any device work.
 * With --gpu it runs a small ragged problem (300 rows, H 64, 1000 ids, 10%
 * of the labels ignored) on device buffers from the CUDA runtime through
 * lce_forward + lce_backward, lce_forward_backward + lce_scale_gradients and
 * the label-smoothing / z-loss calls, and compares every output with the
 * float64 oracle (oracle/liblce_oracle.so, linked as test infrastructure)
 * on the same bf16 inputs: loss relative error <= 1e-3, lse absolute error
 * <= 2e-3, dH and dW relative Frobenius error <= 1e-2; then the
 * sequence-tiled MLP (lce_mlp_forward, lce_mlp_backward) against the MLP
 * oracle, every output within a relative Frobenius error of 1e-2.
 *
 * Exit status 0 when every check passes, 1 otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "lce.h"

/* The oracle's single-pass entry point (oracle/lce_oracle.c); dtype 0 =
 * bf16 bit patterns. */
int lce_oracle_forward_backward(const void *h, const void *W, int dtype,
                                const int64_t *labels, int64_t L, int64_t H,
                                int64_t V, int64_t ignore_index, double eps,
                                double zcoef, double dloss, int nthreads,
                                double *lse, double *zy, double *loss,
                                int64_t *n_valid, double *dH, double *dW,
                                const int64_t *vrows, int64_t nvrows);

/* The MLP oracle (oracle/mlp_oracle.c): dy widened to float64. */
int mlp_oracle(const void *x, const void *Wg, const void *Wu, const void *Wd,
               int dtype, int64_t L, int64_t H, int64_t I, const double *dy,
               int nthreads, double *y, double *dx, double *dWg, double *dWu,
               double *dWd);

static int failures = 0;

static void check(int ok, const char *what) {
  printf("%s %s\n", ok ? "ok  " : "FAIL", what);
  if (!ok) ++failures;
}

/* ---- inputs: a 64-bit linear congruential generator, bf16 by rounding ---- */
static uint64_t lcg_state = 0x9E3779B97F4A7C15ull;
static double lcg_uniform(void) { /* [0, 1) */
  lcg_state = lcg_state * 6364136223846793005ull + 1442695040888963407ull;
  return (double)(lcg_state >> 11) * (1.0 / 9007199254740992.0);
}
static double lcg_normal(void) { /* Box-Muller */
  double u1 = lcg_uniform(), u2 = lcg_uniform();
  if (u1 < 1e-300) u1 = 1e-300;
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}
static uint16_t to_bf16(float f) { /* round to nearest even */
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double rel_fro(const double *got, const double *ref, size_t n) {
  double num = 0.0, den = 0.0;
  for (size_t i = 0; i < n; ++i) {
    num += (got[i] - ref[i]) * (got[i] - ref[i]);
    den += ref[i] * ref[i];
  }
  return den > 0.0 ? sqrt(num / den) : sqrt(num);
}

static int no_gpu_checks(void) {
  check(strcmp(lce_status_string(LCE_OK), "LCE_OK") == 0, "status string");
  check(strcmp(lce_status_string(LCE_ERR_WORKSPACE), "LCE_ERR_WORKSPACE") == 0,
        "status string of an error");
  check(lce_workspace_size(0, 64, 1000, LCE_BF16, 0) == 0,
        "workspace size of an empty problem is 0");
  check(lce_workspace_size(300, 12, 1000, LCE_BF16, 0) == 0,
        "workspace size with H not a multiple of 8 is 0");
  check(lce_workspace_size(300, 64, 1000, LCE_BF16, 128) > 0,
        "workspace size of a valid problem");
  check(lce_default_chunk_rows(131072, 4096, 151936) > 0,
        "default chunk of the 8B shard");
  float loss = 0.f, lse[4];
  check(lce_forward(NULL, NULL, LCE_BF16, NULL, 4, 8, 8, -100, &loss, lse,
                    NULL, 0, NULL) == LCE_ERR_INVALID_ARG,
        "null operands are refused before any device work");
  lce_loss_opts bad = {1.5f, 0.f};
  check(lce_forward_ex(NULL, NULL, LCE_BF16, NULL, 4, 8, 8, -100, &bad, &loss,
                       lse, NULL, 0, NULL) == LCE_ERR_INVALID_ARG,
        "label smoothing above 1 is refused");
  return failures;
}

#define CU(x)                                                           \
  do {                                                                  \
    cudaError_t e_ = (x);                                               \
    if (e_ != cudaSuccess) {                                            \
      printf("FAIL %s: %s\n", #x, cudaGetErrorString(e_));              \
      return 1;                                                         \
    }                                                                   \
  } while (0)

static int gpu_checks(void) {
  const int64_t L = 300, H = 64, V = 1000, chunk = 128;
  const int64_t ignore = -100;
  const float dloss = 0.5f;
  const size_t nh = (size_t)(L * H), nw = (size_t)(V * H);

  uint16_t *h = malloc(nh * 2), *W = malloc(nw * 2), *dH_b = malloc(nh * 2);
  int64_t *y = malloc((size_t)L * 8);
  float *lse = malloc((size_t)L * 4), *dW = malloc(nw * 4);
  double *r_lse = malloc((size_t)L * 8), *r_dH = malloc(nh * 8),
         *r_dW = malloc(nw * 8), *g_dH = malloc(nh * 8), *g_dW = malloc(nw * 8);
  if (!h || !W || !dH_b || !y || !lse || !dW || !r_lse || !r_dH || !r_dW ||
      !g_dH || !g_dW) {
    printf("FAIL host allocation\n");
    return 1;
  }
  for (size_t i = 0; i < nh; ++i) h[i] = to_bf16((float)lcg_normal());
  for (size_t i = 0; i < nw; ++i) W[i] = to_bf16((float)(0.05 * lcg_normal()));
  for (int64_t i = 0; i < L; ++i) {
    y[i] = (int64_t)(lcg_uniform() * (double)V);
    if (i % 10 == 3) y[i] = ignore;
  }

  void *d_h, *d_W, *d_dH, *d_ws;
  int64_t *d_y;
  float *d_loss, *d_lse, *d_dW, *d_dloss;
  const size_t ws_bytes = lce_workspace_size(L, H, V, LCE_BF16, chunk);
  CU(cudaMalloc(&d_h, nh * 2));
  CU(cudaMalloc(&d_W, nw * 2));
  CU(cudaMalloc(&d_dH, nh * 2));
  CU(cudaMalloc((void **)&d_y, (size_t)L * 8));
  CU(cudaMalloc((void **)&d_loss, 4));
  CU(cudaMalloc((void **)&d_lse, (size_t)L * 4));
  CU(cudaMalloc((void **)&d_dW, nw * 4));
  CU(cudaMalloc((void **)&d_dloss, 4));
  CU(cudaMalloc(&d_ws, ws_bytes));
  CU(cudaMemcpy(d_h, h, nh * 2, cudaMemcpyHostToDevice));
  CU(cudaMemcpy(d_W, W, nw * 2, cudaMemcpyHostToDevice));
  CU(cudaMemcpy(d_y, y, (size_t)L * 8, cudaMemcpyHostToDevice));
  CU(cudaMemcpy(d_dloss, &dloss, 4, cudaMemcpyHostToDevice));

  /* three ways through the library: recomputing, fused, and a variant */
  const lce_loss_opts opts[3] = {{0.f, 0.f}, {0.f, 0.f}, {0.1f, 1e-3f}};
  const char *names[3] = {"forward + backward", "forward_backward",
                          "forward_ex + backward_ex (eps 0.1, z 1e-3)"};
  for (int way = 0; way < 3; ++way) {
    lce_status st;
    if (way == 0) {
      st = lce_forward(d_h, d_W, LCE_BF16, d_y, L, H, V, ignore, d_loss, d_lse,
                       d_ws, ws_bytes, NULL);
      if (st == LCE_OK)
        st = lce_backward(d_h, d_W, LCE_BF16, d_y, d_lse, L, H, V, ignore,
                          d_dloss, chunk, d_dH, d_dW, d_ws, ws_bytes, NULL);
    } else if (way == 1) {
      st = lce_forward_backward(d_h, d_W, LCE_BF16, d_y, L, H, V, ignore,
                                chunk, d_loss, d_lse, d_dH, d_dW, d_ws,
                                ws_bytes, NULL);
      if (st == LCE_OK)
        st = lce_scale_gradients(d_dH, LCE_BF16, L, H, d_dW, V, d_dloss,
                                 NULL);
    } else {
      st = lce_forward_ex(d_h, d_W, LCE_BF16, d_y, L, H, V, ignore, &opts[2],
                          d_loss, d_lse, d_ws, ws_bytes, NULL);
      if (st == LCE_OK)
        st = lce_backward_ex(d_h, d_W, LCE_BF16, d_y, d_lse, L, H, V, ignore,
                             &opts[2], d_dloss, chunk, d_dH, d_dW, d_ws,
                             ws_bytes, NULL);
    }
    char what[160];
    snprintf(what, sizeof what, "%s: calls return LCE_OK", names[way]);
    check(st == LCE_OK, what);
    if (st != LCE_OK) {
      printf("     status %s\n", lce_status_string(st));
      continue;
    }
    snprintf(what, sizeof what, "%s: device error word clear", names[way]);
    check(lce_get_error(NULL) == LCE_OK, what);

    float loss = 0.f;
    CU(cudaMemcpy(&loss, d_loss, 4, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(lse, d_lse, (size_t)L * 4, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(dH_b, d_dH, nh * 2, cudaMemcpyDeviceToHost));
    CU(cudaMemcpy(dW, d_dW, nw * 4, cudaMemcpyDeviceToHost));

    double r_loss = 0.0;
    int64_t r_n = 0;
    const int ost = lce_oracle_forward_backward(
        h, W, 0, y, L, H, V, ignore, opts[way].label_smoothing,
        opts[way].z_loss, dloss, 4, r_lse, NULL, &r_loss, &r_n, r_dH, r_dW,
        NULL, 0);
    snprintf(what, sizeof what, "%s: oracle ran", names[way]);
    check(ost == 0, what);

    double lse_err = 0.0;
    for (int64_t i = 0; i < L; ++i) {
      const double d = fabs((double)lse[i] - r_lse[i]);
      if (d > lse_err) lse_err = d;
    }
    for (size_t i = 0; i < nh; ++i) g_dH[i] = from_bf16(dH_b[i]);
    for (size_t i = 0; i < nw; ++i) g_dW[i] = (double)dW[i];
    const double loss_err = fabs((double)loss - r_loss) / fabs(r_loss);
    const double eh = rel_fro(g_dH, r_dH, nh), ew = rel_fro(g_dW, r_dW, nw);
    printf("     loss %.6f (oracle %.6f), lse err %.2e, dH err %.2e, "
           "dW err %.2e\n", loss, r_loss, lse_err, eh, ew);
    snprintf(what, sizeof what, "%s: loss within 1e-3", names[way]);
    check(loss_err <= 1e-3, what);
    snprintf(what, sizeof what, "%s: lse within 2e-3", names[way]);
    check(lse_err <= 2e-3, what);
    snprintf(what, sizeof what, "%s: dH within 1e-2", names[way]);
    check(eh <= 1e-2, what);
    snprintf(what, sizeof what, "%s: dW within 1e-2", names[way]);
    check(ew <= 1e-2, what);
  }

  /* a workspace one byte short of what the backward needs is refused
   * before anything is queued (the forward alone needs less) */
  check(lce_backward(d_h, d_W, LCE_BF16, d_y, d_lse, L, H, V, ignore, d_dloss,
                     chunk, d_dH, d_dW, d_ws, ws_bytes - 1,
                     NULL) == LCE_ERR_WORKSPACE,
        "short workspace refused");

  cudaFree(d_h);
  cudaFree(d_W);
  cudaFree(d_dH);
  cudaFree(d_y);
  cudaFree(d_loss);
  cudaFree(d_lse);
  cudaFree(d_dW);
  cudaFree(d_dloss);
  cudaFree(d_ws);
  free(h);
  free(W);
  free(dH_b);
  free(y);
  free(lse);
  free(dW);
  free(r_lse);
  free(r_dH);
  free(r_dW);
  free(g_dH);
  free(g_dW);
  return failures;
}

/* The sequence-tiled gated MLP: 200 rows in chunks of 128 (a ragged
 * second chunk), H 64, I 192; y, dx, dWg, dWu, dWd against the oracle,
 * relative Frobenius error <= 1e-2 each. */
static int mlp_checks(void) {
  const int64_t L = 200, H = 64, I = 192, chunk = 128;
  const size_t nx = (size_t)(L * H), nw = (size_t)(I * H);
  uint16_t *x = malloc(nx * 2), *wg = malloc(nw * 2), *wu = malloc(nw * 2),
           *wd = malloc(nw * 2), *dy = malloc(nx * 2), *yb = malloc(nx * 2),
           *dxb = malloc(nx * 2);
  float *dwg = malloc(nw * 4), *dwu = malloc(nw * 4), *dwd = malloc(nw * 4);
  double *dy64 = malloc(nx * 8), *r[5], *g[5];
  for (int k = 0; k < 5; ++k) {
    r[k] = malloc((k < 2 ? nx : nw) * 8);
    g[k] = malloc((k < 2 ? nx : nw) * 8);
  }
  if (!x || !wg || !wu || !wd || !dy || !yb || !dxb || !dwg || !dwu || !dwd ||
      !dy64 || !r[4] || !g[4]) {
    printf("FAIL host allocation\n");
    return 1;
  }
  for (size_t i = 0; i < nx; ++i) x[i] = to_bf16((float)lcg_normal());
  for (size_t i = 0; i < nw; ++i) {
    wg[i] = to_bf16((float)(0.05 * lcg_normal()));
    wu[i] = to_bf16((float)(0.05 * lcg_normal()));
    wd[i] = to_bf16((float)(0.05 * lcg_normal()));
  }
  for (size_t i = 0; i < nx; ++i) {
    dy[i] = to_bf16((float)(0.1 * lcg_normal()));
    dy64[i] = from_bf16(dy[i]);
  }
  void *d_x, *d_wg, *d_wu, *d_wd, *d_dy, *d_y, *d_dx, *d_ws;
  float *d_dwg, *d_dwu, *d_dwd;
  const size_t ws_bytes = lce_mlp_workspace_size(L, H, I, chunk);
  check(ws_bytes > 0, "MLP workspace size");
  CU(cudaMalloc(&d_x, nx * 2));
  CU(cudaMalloc(&d_wg, nw * 2));
  CU(cudaMalloc(&d_wu, nw * 2));
  CU(cudaMalloc(&d_wd, nw * 2));
  CU(cudaMalloc(&d_dy, nx * 2));
  CU(cudaMalloc(&d_y, nx * 2));
  CU(cudaMalloc(&d_dx, nx * 2));
  CU(cudaMalloc((void **)&d_dwg, nw * 4));
  CU(cudaMalloc((void **)&d_dwu, nw * 4));
  CU(cudaMalloc((void **)&d_dwd, nw * 4));
  CU(cudaMalloc(&d_ws, ws_bytes));
  CU(cudaMemcpy(d_x, x, nx * 2, cudaMemcpyHostToDevice));
  CU(cudaMemcpy(d_wg, wg, nw * 2, cudaMemcpyHostToDevice));
  CU(cudaMemcpy(d_wu, wu, nw * 2, cudaMemcpyHostToDevice));
  CU(cudaMemcpy(d_wd, wd, nw * 2, cudaMemcpyHostToDevice));
  CU(cudaMemcpy(d_dy, dy, nx * 2, cudaMemcpyHostToDevice));
  lce_status st = lce_mlp_forward(d_x, d_wg, d_wu, d_wd, L, H, I, chunk, d_y,
                                  d_ws, ws_bytes, NULL);
  if (st == LCE_OK)
    st = lce_mlp_backward(d_x, d_wg, d_wu, d_wd, d_dy, L, H, I, chunk, d_dx,
                          d_dwg, d_dwu, d_dwd, d_ws, ws_bytes, NULL);
  check(st == LCE_OK, "MLP forward + backward return LCE_OK");
  if (st != LCE_OK) return failures;
  check(lce_get_error(NULL) == LCE_OK, "MLP: device error word clear");
  CU(cudaMemcpy(yb, d_y, nx * 2, cudaMemcpyDeviceToHost));
  CU(cudaMemcpy(dxb, d_dx, nx * 2, cudaMemcpyDeviceToHost));
  CU(cudaMemcpy(dwg, d_dwg, nw * 4, cudaMemcpyDeviceToHost));
  CU(cudaMemcpy(dwu, d_dwu, nw * 4, cudaMemcpyDeviceToHost));
  CU(cudaMemcpy(dwd, d_dwd, nw * 4, cudaMemcpyDeviceToHost));
  check(mlp_oracle(x, wg, wu, wd, 0, L, H, I, dy64, 4, r[0], r[1], r[2], r[3],
                   r[4]) == 0,
        "MLP oracle ran");
  for (size_t i = 0; i < nx; ++i) {
    g[0][i] = from_bf16(yb[i]);
    g[1][i] = from_bf16(dxb[i]);
  }
  for (size_t i = 0; i < nw; ++i) {
    g[2][i] = dwg[i];
    g[3][i] = dwu[i];
    g[4][i] = dwd[i];
  }
  const char *names[5] = {"MLP y", "MLP dx", "MLP dWg", "MLP dWu", "MLP dWd"};
  for (int k = 0; k < 5; ++k) {
    const double e = rel_fro(g[k], r[k], k < 2 ? nx : nw);
    char what[80];
    snprintf(what, sizeof what, "%s within 1e-2 (err %.2e)", names[k], e);
    check(e <= 1e-2, what);
  }
  cudaFree(d_x);
  cudaFree(d_wg);
  cudaFree(d_wu);
  cudaFree(d_wd);
  cudaFree(d_dy);
  cudaFree(d_y);
  cudaFree(d_dx);
  cudaFree(d_dwg);
  cudaFree(d_dwu);
  cudaFree(d_dwd);
  cudaFree(d_ws);
  free(x);
  free(wg);
  free(wu);
  free(wd);
  free(dy);
  free(yb);
  free(dxb);
  free(dwg);
  free(dwu);
  free(dwd);
  free(dy64);
  for (int k = 0; k < 5; ++k) {
    free(r[k]);
    free(g[k]);
  }
  return failures;
}

int main(int argc, char **argv) {
  no_gpu_checks();
  if (argc > 1 && strcmp(argv[1], "--gpu") == 0) {
    if (gpu_checks() != 0 && failures == 0) ++failures;
    if (mlp_checks() != 0 && failures == 0) ++failures;
  }
  printf("%d failure(s)\n", failures);
  return failures ? 1 : 0;
}

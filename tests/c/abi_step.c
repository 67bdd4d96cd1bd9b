/*
 * abi_step.c -- the C ABI used from plain C, with no Python and no PyTorch:
 * cudaMalloc'd buffers, a cudaStream_t, dpopt_reduce_adam for two steps on
 * one rank's shard, dpopt_stream_status, and the results checked against the
 * CPU oracle (oracle/oracle.c, linked as test infrastructure only).
 * Built and run by tests/test_gpu_c_abi.py; prints "ok" and exits 0 on
 * success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "dpopt.h"

/* the oracle's entry point (oracle/oracle.c) */
int orc_reduce_adam_shard(const void *const *grads, int dtype, int n, int64_t numel,
                          int shard_rank, float *master, float *m, float *v, uint16_t *out,
                          float lr, float beta1, float beta2, float eps, float weight_decay,
                          int64_t step, int nthreads);

#define N 4
#define S 10007 /* shard elements: ragged against the 8-element groups */
#define RANK 2

static uint64_t rng = 0x9E3779B97F4A7C15ull;
static double uniform(void) { /* xorshift64*, in [-1, 1) */
  rng ^= rng >> 12;
  rng ^= rng << 25;
  rng ^= rng >> 27;
  return (double)((rng * 0x2545F4914F6CDD1Dull) >> 11) / 4503599627370496.0 - 1.0;
}

static uint16_t bf16_trunc(float x) { /* any bf16 value serves as input */
  uint32_t u;
  memcpy(&u, &x, 4);
  return (uint16_t)(u >> 16);
}

static int check(cudaError_t e, const char *what) {
  if (e != cudaSuccess) {
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    exit(2);
  }
  return 0;
}

static int64_t bf16_order(uint16_t h) { return (h & 0x8000) ? -(int64_t)(h & 0x7FFF) : h; }

int main(void) {
  const int64_t numel = (int64_t)N * S;
  const float lr = 1e-3f, b1 = 0.9f, b2 = 0.999f, eps = 1e-8f;
  uint16_t *hg[N];
  void *dg[N];
  for (int r = 0; r < N; ++r) {
    hg[r] = malloc(numel * 2);
    for (int64_t i = 0; i < numel; ++i) hg[r][i] = bf16_trunc((float)(uniform() * 1e-3));
    check(cudaMalloc(&dg[r], numel * 2), "cudaMalloc");
    check(cudaMemcpy(dg[r], hg[r], numel * 2, cudaMemcpyHostToDevice), "cudaMemcpy");
  }
  float *th = malloc(S * 4), *m = calloc(S, 4), *v = calloc(S, 4);
  uint16_t *out = malloc(S * 2);
  for (int64_t i = 0; i < S; ++i) th[i] = (float)(uniform() * 0.02);
  float *dth, *dm, *dv;
  void *dout;
  check(cudaMalloc((void **)&dth, S * 4), "cudaMalloc");
  check(cudaMalloc((void **)&dm, S * 4), "cudaMalloc");
  check(cudaMalloc((void **)&dv, S * 4), "cudaMalloc");
  check(cudaMalloc(&dout, S * 2), "cudaMalloc");
  check(cudaMemcpy(dth, th, S * 4, cudaMemcpyHostToDevice), "cudaMemcpy");
  check(cudaMemset(dm, 0, S * 4), "cudaMemset");
  check(cudaMemset(dv, 0, S * 4), "cudaMemset");
  cudaStream_t st;
  check(cudaStreamCreate(&st), "cudaStreamCreate");

  /* an argument error is reported synchronously, with a message */
  if (dpopt_reduce_adam((const void *const *)dg, N, numel, RANK, 4096, dth, dm, dv, dout, lr, b1,
                        b2, eps, 0, st) != DPOPT_ERR_INVALID_ARG ||
      strlen(dpopt_last_error()) == 0) {
    fprintf(stderr, "step 0 was not rejected\n");
    return 1;
  }
  for (int64_t t = 1; t <= 2; ++t) {
    int rc = dpopt_reduce_adam((const void *const *)dg, N, numel, RANK, 4096, dth, dm, dv, dout,
                               lr, b1, b2, eps, t, st);
    if (rc == DPOPT_OK) rc = dpopt_stream_status(st);
    if (rc != DPOPT_OK) {
      fprintf(stderr, "step %lld: %s (%s)\n", (long long)t, dpopt_status_string(rc),
              dpopt_last_error());
      return 1;
    }
    if (orc_reduce_adam_shard((const void *const *)hg, 0, N, numel, RANK, th, m, v, out, lr, b1,
                              b2, eps, 0.f, t, 1) != 0) {
      fprintf(stderr, "oracle refused the arguments\n");
      return 1;
    }
  }
  float *gth = malloc(S * 4), *gm = malloc(S * 4), *gv = malloc(S * 4);
  uint16_t *gout = malloc(S * 2);
  check(cudaMemcpy(gth, dth, S * 4, cudaMemcpyDeviceToHost), "cudaMemcpy");
  check(cudaMemcpy(gm, dm, S * 4, cudaMemcpyDeviceToHost), "cudaMemcpy");
  check(cudaMemcpy(gv, dv, S * 4, cudaMemcpyDeviceToHost), "cudaMemcpy");
  check(cudaMemcpy(gout, dout, S * 2, cudaMemcpyDeviceToHost), "cudaMemcpy");
  /* fp32 states within 8 x 2.4e-7 relative, against a scale floored at 5 % of
     the array's largest magnitude (and lr for the master) so that cancellation
     in one element does not turn one rounding into many ulps; bf16 within one
     ulp.  The element-by-element tolerances of the parity tests are tighter. */
  double fth = lr, fm = 0.0, fv = 0.0;
  for (int64_t i = 0; i < S; ++i) {
    fm = fmax(fm, 0.05 * fabs(m[i]));
    fv = fmax(fv, 0.05 * fabs(v[i]));
  }
  double worst = 0.0;
  int64_t bad = 0;
  for (int64_t i = 0; i < S; ++i) {
    const double e1 = fabs((double)gth[i] - th[i]) / fmax(fabs(th[i]), fth);
    const double e2 = fabs((double)gm[i] - m[i]) / fmax(fabs(m[i]), fm);
    const double e3 = fabs((double)gv[i] - v[i]) / fmax(fabs(v[i]), fv);
    const double e = fmax(e1, fmax(e2, e3));
    if (e > worst) worst = e;
    if (e > 8 * 2.4e-7 || llabs(bf16_order(gout[i]) - bf16_order(out[i])) > 1) ++bad;
  }
  if (bad) {
    fprintf(stderr, "%lld of %d elements off (worst relative %.3e)\n", (long long)bad, S, worst);
    return 1;
  }
  printf("ok: N=%d, %d shard elements, 2 steps, worst relative %.2e, version %s\n", N, S, worst,
         dpopt_version());
  return 0;
}

/*
 * abi_step.c -- the C ABI used from plain C, with no Python and no PyTorch:
 * cudaMalloc'd buffers, a cudaStream_t, dpopt_reduce_adam for two steps on
 * one rank's shard, dpopt_stream_status, and the results checked against the
 * CPU oracle (oracle/oracle.c, linked as test infrastructure only); then a
 * third step through dpopt_reduce_adam_buckets_table with 159 separately
 * allocated bucket slices and a cudaMalloc'd launch table, bitwise against
 * the full-buffer entry; then three loss-scaled steps captured once into a
 * CUDA graph (cudaStreamBeginCapture) and replayed, bitwise against direct
 * calls.
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

  /* A third step twice, from the same states: once through the full-buffer
     entry, once through the one-launch bucket entry with every bucket slice in
     an allocation of its own (159 buckets of 63 elements, the last ragged: more
     than one launch's parameter space holds, so the launch table goes to the
     cudaMalloc'd memory). The two must leave the same bits. */
  enum { BL = 63, NB = (S + BL - 1) / BL };
  int64_t off[NB], len[NB];
  for (int b = 0; b < NB; ++b) {
    off[b] = (int64_t)b * BL;
    len[b] = S - off[b] < BL ? S - off[b] : BL;
  }
  float *st3[2][3];
  void *out3[2];
  for (int k = 0; k < 2; ++k) {
    for (int a = 0; a < 3; ++a) {
      check(cudaMalloc((void **)&st3[k][a], S * 4), "cudaMalloc");
      check(cudaMemcpy(st3[k][a], a == 0 ? dth : a == 1 ? dm : dv, S * 4,
                       cudaMemcpyDeviceToDevice), "cudaMemcpy");
    }
    check(cudaMalloc(&out3[k], S * 2), "cudaMalloc");
  }
  static const void *slices[NB * N];
  for (int b = 0; b < NB; ++b)
    for (int r = 0; r < N; ++r) {
      void *sl;
      check(cudaMalloc(&sl, len[b] * 2), "cudaMalloc");
      check(cudaMemcpy(sl, (const uint16_t *)dg[r] + (int64_t)RANK * S + off[b], len[b] * 2,
                       cudaMemcpyDeviceToDevice), "cudaMemcpy");
      slices[b * N + r] = sl;
    }
  int64_t tbytes = 0;
  void *table;
  if (dpopt_bucket_table_bytes(N, NB, &tbytes) != DPOPT_OK) return 1;
  check(cudaMalloc(&table, tbytes), "cudaMalloc");
  if (dpopt_reduce_adam_buckets_table(slices, DPOPT_GRAD_BF16, N, off, len, NB, st3[1][0],
                                      st3[1][1], st3[1][2], out3[1], lr, b1, b2, eps, 3, NULL,
                                      table, tbytes - 1, st) != DPOPT_ERR_INVALID_ARG) {
    fprintf(stderr, "a table one byte short was not rejected\n");
    return 1;
  }
  int rc = dpopt_reduce_adam((const void *const *)dg, N, numel, RANK, 4096, st3[0][0], st3[0][1],
                             st3[0][2], out3[0], lr, b1, b2, eps, 3, st);
  if (rc == DPOPT_OK)
    rc = dpopt_reduce_adam_buckets_table(slices, DPOPT_GRAD_BF16, N, off, len, NB, st3[1][0],
                                         st3[1][1], st3[1][2], out3[1], lr, b1, b2, eps, 3, NULL,
                                         table, tbytes, st);
  if (rc == DPOPT_OK) rc = dpopt_stream_status(st);
  if (rc != DPOPT_OK) {
    fprintf(stderr, "step 3: %s (%s)\n", dpopt_status_string(rc), dpopt_last_error());
    return 1;
  }
  for (int a = 0; a < 4; ++a) {
    const size_t bytes = a < 3 ? S * 4 : S * 2;
    unsigned char *x = malloc(bytes), *y = malloc(bytes);
    check(cudaMemcpy(x, a < 3 ? (void *)st3[0][a] : out3[0], bytes, cudaMemcpyDeviceToHost),
          "cudaMemcpy");
    check(cudaMemcpy(y, a < 3 ? (void *)st3[1][a] : out3[1], bytes, cudaMemcpyDeviceToHost),
          "cudaMemcpy");
    if (memcmp(x, y, bytes) != 0) {
      fprintf(stderr, "the bucket-table step differs from the full-buffer step (array %d)\n", a);
      return 1;
    }
    free(x);
    free(y);
  }
  /* Steps 4-6 captured once into a CUDA graph with the runtime API and replayed:
     the loss-scaled entry without a squared norm keeps the step count in the
     device state and reads the learning rate from device memory, so each replay
     is the next step at the rate written before it -- bitwise the direct calls
     that pass the same rates from the host. */
  const dpopt_loss_scale_config cfg = {1.0f, 1, 1, 1.0f};
  const float rates[3] = {1e-3f, 6e-4f, 2e-4f};
  float *st4[2][3];
  void *out4[2], *state4[2];
  for (int k = 0; k < 2; ++k) {
    for (int a = 0; a < 3; ++a) {
      check(cudaMalloc((void **)&st4[k][a], S * 4), "cudaMalloc");
      check(cudaMemcpy(st4[k][a], st3[0][a], S * 4, cudaMemcpyDeviceToDevice), "cudaMemcpy");
    }
    check(cudaMalloc(&out4[k], S * 2), "cudaMalloc");
    check(cudaMalloc(&state4[k], sizeof(dpopt_loss_scale_state)), "cudaMalloc");
    if (dpopt_loss_scale_init((dpopt_loss_scale_state *)state4[k], &cfg, st) != DPOPT_OK) return 1;
  }
  float *lr_dev;
  check(cudaMalloc((void **)&lr_dev, 4), "cudaMalloc");
  /* one direct call on spare arrays first: the kernels are loaded before the capture */
  void *state_w;
  check(cudaMalloc(&state_w, sizeof(dpopt_loss_scale_state)), "cudaMalloc");
  rc = dpopt_loss_scale_init((dpopt_loss_scale_state *)state_w, &cfg, st);
  if (rc == DPOPT_OK)
    rc = dpopt_amp_step((const void *const *)dg, DPOPT_GRAD_BF16, N, numel, RANK, 4096,
                        st3[1][0], st3[1][1], st3[1][2], out3[1], 1e-3f, b1, b2, eps, 0.01f, 0.f,
                        NULL, (dpopt_loss_scale_state *)state_w, &cfg, NULL, st);
  if (rc == DPOPT_OK) rc = dpopt_stream_status(st);
  if (rc != DPOPT_OK) {
    fprintf(stderr, "warm-up: %s (%s)\n", dpopt_status_string(rc), dpopt_last_error());
    return 1;
  }
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  check(cudaStreamBeginCapture(st, cudaStreamCaptureModeGlobal), "cudaStreamBeginCapture");
  rc = dpopt_amp_step((const void *const *)dg, DPOPT_GRAD_BF16, N, numel, RANK, 4096, st4[1][0],
                      st4[1][1], st4[1][2], out4[1], 0.f, b1, b2, eps, 0.01f, 0.f, NULL,
                      (dpopt_loss_scale_state *)state4[1], &cfg, lr_dev, st);
  check(cudaStreamEndCapture(st, &graph), "cudaStreamEndCapture");
  if (rc != DPOPT_OK) {
    fprintf(stderr, "capture: %s (%s)\n", dpopt_status_string(rc), dpopt_last_error());
    return 1;
  }
  check(cudaGraphInstantiate(&exec, graph, 0), "cudaGraphInstantiate");
  for (int k = 0; k < 3; ++k) {
    check(cudaMemcpy(lr_dev, &rates[k], 4, cudaMemcpyHostToDevice), "cudaMemcpy");
    check(cudaGraphLaunch(exec, st), "cudaGraphLaunch");
    rc = dpopt_amp_step((const void *const *)dg, DPOPT_GRAD_BF16, N, numel, RANK, 4096,
                        st4[0][0], st4[0][1], st4[0][2], out4[0], rates[k], b1, b2, eps, 0.01f,
                        0.f, NULL, (dpopt_loss_scale_state *)state4[0], &cfg, NULL, st);
    if (rc == DPOPT_OK) rc = dpopt_stream_status(st);
    if (rc != DPOPT_OK) {
      fprintf(stderr, "graph step %d: %s (%s)\n", k, dpopt_status_string(rc),
              dpopt_last_error());
      return 1;
    }
  }
  for (int a = 0; a < 5; ++a) {
    const size_t bytes = a < 3 ? S * 4 : a == 3 ? S * 2 : sizeof(dpopt_loss_scale_state);
    const void *src0 = a < 3 ? (void *)st4[0][a] : a == 3 ? out4[0] : state4[0];
    const void *src1 = a < 3 ? (void *)st4[1][a] : a == 3 ? out4[1] : state4[1];
    unsigned char *x = malloc(bytes), *y = malloc(bytes);
    check(cudaMemcpy(x, src0, bytes, cudaMemcpyDeviceToHost), "cudaMemcpy");
    check(cudaMemcpy(y, src1, bytes, cudaMemcpyDeviceToHost), "cudaMemcpy");
    if (memcmp(x, y, bytes) != 0) {
      fprintf(stderr, "the graph replays differ from the direct calls (array %d)\n", a);
      return 1;
    }
    if (a == 4 && ((const dpopt_loss_scale_state *)x)->step != 3) {
      fprintf(stderr, "the device step count is %lld after 3 steps\n",
              (long long)((const dpopt_loss_scale_state *)x)->step);
      return 1;
    }
    free(x);
    free(y);
  }
  check(cudaGraphExecDestroy(exec), "cudaGraphExecDestroy");
  check(cudaGraphDestroy(graph), "cudaGraphDestroy");

  printf("ok: N=%d, %d shard elements, 2 steps, worst relative %.2e; step 3 through the "
         "bucket table bitwise equal; steps 4-6 as graph replays bitwise equal; version %s\n",
         N, S, worst, dpopt_version());
  return 0;
}

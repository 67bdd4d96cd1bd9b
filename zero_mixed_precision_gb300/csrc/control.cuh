// control.cuh -- the single-CTA kernels around the step: loss-scale state
// initialisation and update, and the ordered final sum of the squared norm.
// Included by the C ABI unit only.
#pragma once

#include "kernels.cuh"

namespace dpopt {

__global__ void loss_scale_init_kernel(LossScaleState* st, LossScaleConfig cfg) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  LossScaleState s;
  s.scale = cfg.init_scale;
  s.good_steps = 0;
  s.hysteresis_left = cfg.hysteresis;
  s.last_overflow = 0;
  s.step = 0;
  s.skipped = 0;
  *st = s;
}

// After a step: skip bookkeeping, halving on every hysteresis-th overflow since
// the scale last changed (not below min_scale), doubling after `window` clean
// steps in a row.
__global__ void loss_scale_update_kernel(LossScaleState* st, const double* sqnorm,
                                         LossScaleConfig cfg) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  LossScaleState s = *st;
  const bool overflow = !isfinite(*sqnorm);
  s.last_overflow = overflow ? 1 : 0;
  if (overflow) {
    s.skipped += 1;
    s.good_steps = 0;
    s.hysteresis_left -= 1;
    if (s.hysteresis_left <= 0) {
      s.scale = fmaxf(s.scale * 0.5f, cfg.min_scale);
      s.hysteresis_left = cfg.hysteresis;
    }
  } else {
    s.step += 1;
    s.good_steps += 1;
    if (s.good_steps >= cfg.window) {
      s.scale = s.scale * 2.0f;
      s.good_steps = 0;
      s.hysteresis_left = cfg.hysteresis;
    }
  }
  *st = s;
}

// Sum of the partials in a fixed order: strided per thread, then a fixed tree.
__global__ void __launch_bounds__(kThreads)
    sqnorm_finish_kernel(const double* partials, int64_t nchunks, double* out) {
  __shared__ double red[kThreads];
  double acc = 0.0;
  for (int64_t c = threadIdx.x; c < nchunks; c += kThreads) acc = __dadd_rn(acc, partials[c]);
  red[threadIdx.x] = acc;
  __syncthreads();
#pragma unroll
  for (int w = kThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] = __dadd_rn(red[threadIdx.x], red[threadIdx.x + w]);
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = red[0];
}

}  // namespace dpopt

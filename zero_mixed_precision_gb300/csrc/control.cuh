// control.cuh -- the single-CTA kernels around the step: loss-scale state
// initialisation and update, and the ordered final sum of the squared norm.
// Included by the C ABI unit only.
#pragma once

#include "kernels.cuh"

namespace dpopt {

__global__ void loss_scale_init_kernel(LossScaleState* st, LossScaleConfig cfg) {
  pdl_enter();
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
// steps in a row.  Without a squared norm (null: a run without loss scaling)
// only the step count advances; the scale and its counters stay as they are.
__global__ void loss_scale_update_kernel(LossScaleState* st, const double* sqnorm,
                                         LossScaleConfig cfg) {
  pdl_enter();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  LossScaleState s = *st;
  if (sqnorm == nullptr) {
    s.last_overflow = 0;
    s.step += 1;
    *st = s;
    return;
  }
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

// Sum of the chunk partials (double-float pairs) in a fixed order: strided
// over 1024 threads, a shuffle tree in each warp, the warps' sums in warp
// order; the final pair is added once in fp64.
constexpr int kFinishThreads = 1024;

__global__ void __launch_bounds__(kFinishThreads)
    sqnorm_finish_kernel(const DFloat* partials, int64_t nchunks, double* out) {
  __shared__ DFloat warp_sum[kFinishThreads / 32];
  pdl_enter();
  DFloat acc{0.f, 0.f};
  for (int64_t c = threadIdx.x; c < nchunks; c += kFinishThreads) acc = df_add(acc, partials[c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const DFloat o{__shfl_down_sync(0xffffffffu, acc.hi, off),
                   __shfl_down_sync(0xffffffffu, acc.lo, off)};
    acc = df_add(acc, o);
  }
  if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    DFloat tot = warp_sum[0];
    for (int w = 1; w < kFinishThreads / 32; ++w) tot = df_add(tot, warp_sum[w]);
    *out = __dadd_rn((double)tot.hi, (double)tot.lo);
  }
}

}  // namespace dpopt

// norm.cuh -- the squared L2 norm of the averaged gradient, the pre-pass of
// global-norm clipping and of the loss-scale overflow test.  It forms each
// element's average exactly as the step does (the same replica loads and
// fixed-order compensated sum), so the norm is that of the gradient the step
// applies.
#pragma once

#include "kernels.cuh"

namespace dpopt {

// ---------------------------------------------------------------------------
// squared L2 norm of the averaged gradient (the clipping pre-pass)
// ---------------------------------------------------------------------------

// Elements per partial sum.  Fixed, so the partition -- and therefore the
// fp64 rounding of the total -- does not depend on the grid or the GPU.
constexpr int kNormChunk = 65536;

// The averaged gradient of one aligned 8-element group, as the step forms it.
template <int NR, int GK, int W>
__device__ __forceinline__ void norm_group(const void* const* gp, int64_t e0, uint64_t pol, int n,
                                           const Hyper& h, float (&g)[kGroup]) {
  const GlobalSource<GK, W> src{gp, e0, {nullptr, nullptr, nullptr}, pol};
  CompSum<float> cs[kGroup];
  reduce_group_x1<NR, GK>(src, n, cs);
#pragma unroll
  for (int j = 0; j < kGroup; ++j) g[j] = cs[j].average(h);
}

// One partial per chunk: sum over the chunk's elements of x^2, x = fl32(g *
// unscale) (exact for a power-of-two unscale) with g the same fixed-order
// average the step uses.  Each thread accumulates its elements in order as an
// fp32 pair (TwoProd for each square, TwoSum into the sum: about 2^-44
// relative), then the threads' sums are added in fp64 over a fixed tree.
// Seg::first_group holds the segment's first chunk here.
template <int NR, int GK, int MAXSEG, int MAXPTR>
__global__ void __launch_bounds__(kThreads, NR > 0 ? 4 : 2)
    grad_sqnorm_kernel(const __grid_constant__ LaunchParams<MAXSEG, MAXPTR> p, double* partials,
                       int64_t nchunks) {
  __shared__ double red[kThreads];
  const uint64_t pol = evict_first_policy();
  const float us = p.h.scale_dev ? __fdiv_rn(1.f, *p.h.scale_dev) : p.h.unscale;
  int si = 0;
  for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    while (c >= p.seg[si + 1].first_group) ++si;
    const Seg& sg = p.seg[si];
    const int64_t c0 = (c - sg.first_group) * (int64_t)kNormChunk;
    const void* const* gp = p.gptr + sg.ptr_base;
    float hi = 0.f, lo = 0.f;  // double-float running sum of the squares
    for (int k = threadIdx.x; k < kNormChunk / kGroup; k += kThreads) {
      const int64_t e0 = c0 + (int64_t)k * kGroup;
      if (e0 >= sg.len) break;
      const int64_t rem = sg.len - e0;
      float g[kGroup];
      int cnt = kGroup;
      if (GK == 1 && sg.vec == 2 && rem >= kGroup) {
        norm_group<NR, GK, 32>(gp, e0, pol, p.n_rep, p.h, g);
      } else if (sg.vec && rem >= kGroup) {
        norm_group<NR, GK, 16>(gp, e0, pol, p.n_rep, p.h, g);
      } else {
        cnt = (int)(rem < kGroup ? rem : kGroup);
        for (int j = 0; j < cnt; ++j) {
          CompSum<float> cs;
          cs.init(ld_grad1<GK>(gp[0], e0 + j));
          for (int r = 1; r < p.n_rep; ++r) cs.add(ld_grad1<GK>(gp[r], e0 + j));
          g[j] = cs.average(p.h);
        }
      }
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        if (j < cnt) {
          // x^2 exactly as p2 + pe (TwoProd), added with TwoSum
          const float x = __fmul_rn(g[j], us);
          const float p2 = __fmul_rn(x, x);
          const float pe = __fmaf_rn(x, x, -p2);
          float t, e;
          two_sum(hi, p2, t, e);
          hi = t;
          lo = __fadd_rn(lo, __fadd_rn(e, pe));
        }
      }
    }
    const double acc = __dadd_rn((double)hi, (double)lo);
    red[threadIdx.x] = acc;
    __syncthreads();
#pragma unroll
    for (int w = kThreads / 2; w > 0; w >>= 1) {
      if (threadIdx.x < w) red[threadIdx.x] = __dadd_rn(red[threadIdx.x], red[threadIdx.x + w]);
      __syncthreads();
    }
    if (threadIdx.x == 0) partials[c] = red[0];
    __syncthreads();
  }
}

}  // namespace dpopt

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

// Elements per partial sum: two 8-element groups per thread of a 256-thread
// CTA.  Fixed, so the partition -- and therefore the fp64 rounding of the
// total -- does not depend on the grid or the GPU; small, so that one CTA per
// chunk keeps every SM busy to the end (a 65536-element chunk per CTA left
// the last wave a quarter empty: 3.55 TB/s at N = 4).
constexpr int kNormChunk = 4096;
static_assert(sizeof(DFloat) == sizeof(double), "a chunk partial fills one 8-byte scratch slot");


// The stored average is read back by the step that follows, so its stores ask
// L2 to keep the lines (evict_last) while the replica loads pass through with
// evict_first: measured on GB300, +0.7-1.7 % on the clipped and loss-scaled
// lines (gpt2s, 1p3b) against plain stores.
__device__ __forceinline__ uint64_t evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void st_keep16(float* p, float4 a, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "f"(a.x),
               "f"(a.y), "f"(a.z), "f"(a.w), "l"(pol)
               : "memory");
}

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

// The same on packed f32x2 lanes: g[j] holds elements 2j and 2j+1.
template <int NR, int GK, int W>
__device__ __forceinline__ void norm_group_x2(const void* const* gp, int64_t e0, uint64_t pol,
                                              int n, const Hyper& h, float2 (&g)[kGroup / 2]) {
  const GlobalSource<GK, W> src{gp, e0, {nullptr, nullptr, nullptr}, pol};
  CompSum<float2> cs[kGroup / 2];
  reduce_group_x2<NR, GK>(src, n, cs);
#pragma unroll
  for (int j = 0; j < kGroup / 2; ++j) g[j] = cs[j].average(h);
}

// One partial per chunk: sum over the chunk's elements of x^2, x = fl32(g *
// unscale) (exact for a power-of-two unscale) with g the same fixed-order
// average the step uses.  Each thread accumulates its elements in order on
// packed f32x2 lanes -- even elements in one lane, odd in the other, each an
// fp32 pair (TwoProd for each square, TwoSum into the sum) -- and joins its
// two pairs; then the threads' pairs are added over a fixed tree of
// double-float additions -- a shuffle tree inside each warp, then the warps'
// sums in warp order -- and the chunk's pair is stored (8 bytes per chunk).
// No fp64 arithmetic: on GB300 an fp64 tree per 4096-element chunk kept the
// fp64 pipe half busy.  The packed lanes cut the pass from 61 to 42
// instructions per element at N = 4 (gpt2s: 67.7 -> 62.3 us).
// Seg::first_group holds the segment's first chunk here.
//
// STORE: the pass also writes each element's average g (fp32, before the
// unscale) to p.master[state_off + e] -- the reduced gradient shard -- so that
// a following step can read 4 bytes per element instead of N replicas.
// Five CTAs per SM for N <= 4 (at most 48 registers; the forms without STORE
// spill 16-40 bytes there, and measured no slower than at four CTAs without
// spills), four above.
template <int NR, int GK, bool STORE, int MAXSEG, int MAXPTR>
__global__ void __launch_bounds__(kThreads, NR > 0 ? (NR <= 4 ? 5 : 4) : 2)
    grad_sqnorm_kernel(const __grid_constant__ LaunchParams<MAXSEG, MAXPTR> p, DFloat* partials,
                       int64_t nchunks) {
  __shared__ DFloat warp_sum[kThreads / 32];
  pdl_enter();
  const uint64_t pol = evict_first_policy();
  const uint64_t keep = STORE ? evict_last_policy() : 0;
  const float us = p.h.scale_dev ? __fdiv_rn(1.f, *p.h.scale_dev) : p.h.unscale;
  int si = 0;
  for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    while (c >= p.seg[si + 1].first_group) ++si;
    const Seg& sg = p.seg[si];
    const int64_t c0 = (c - sg.first_group) * (int64_t)kNormChunk;
    const void* const* gp = p.gptr + sg.ptr_base;
    // double-float running sums of the squares, even and odd elements in the
    // two lanes
    float2 hi = make_float2(0.f, 0.f), lo = make_float2(0.f, 0.f);
    const float2 us2 = make_float2(us, us);
    for (int k = threadIdx.x; k < kNormChunk / kGroup; k += kThreads) {
      const int64_t e0 = c0 + (int64_t)k * kGroup;
      if (e0 >= sg.len) break;
      const int64_t rem = sg.len - e0;
      if (!dbg_ok(p.h, si < p.nseg && e0 >= 0) ||
          (STORE && !dbg_span(p.h, sg.state_off + e0,
                              sg.state_off + e0 + (rem < kGroup ? rem : kGroup))))
        break;
      float2 g[kGroup / 2];
      int cnt = kGroup;
      float* const avg = STORE ? p.master + sg.state_off + e0 : nullptr;
      if (GK == 1 && sg.vec == 2 && rem >= kGroup) {
        norm_group_x2<NR, GK, 32>(gp, e0, pol, p.n_rep, p.h, g);
      } else if (sg.vec && rem >= kGroup) {
        norm_group_x2<NR, GK, 16>(gp, e0, pol, p.n_rep, p.h, g);
      } else {
        // a partial or unaligned group: one element at a time, the missing
        // elements as zeros (whose squares add nothing)
        cnt = (int)(rem < kGroup ? rem : kGroup);
        float t[kGroup];
        for (int j = 0; j < kGroup; ++j) {
          t[j] = 0.f;
          if (j < cnt) {
            CompSum<float> cs;
            cs.init(ld_grad1<GK>(gp[0], e0 + j));
            for (int r = 1; r < p.n_rep; ++r) cs.add(ld_grad1<GK>(gp[r], e0 + j));
            t[j] = cs.average(p.h);
          }
        }
#pragma unroll
        for (int j = 0; j < kGroup / 2; ++j) g[j] = make_float2(t[2 * j], t[2 * j + 1]);
      }
      if constexpr (STORE) {
        const float4 lo4 = make_float4(g[0].x, g[0].y, g[1].x, g[1].y);
        const float4 hi4 = make_float4(g[2].x, g[2].y, g[3].x, g[3].y);
        if (sg.vec && cnt == kGroup) {
          st_keep16(avg, lo4, keep);
          st_keep16(avg + 4, hi4, keep);
        } else {
          for (int j = 0; j < cnt; ++j) avg[j] = (j & 1) ? g[j >> 1].y : g[j >> 1].x;
        }
      }
#pragma unroll
      for (int j = 0; j < kGroup / 2; ++j) {
        // x^2 exactly as p2 + pe (TwoProd), added with TwoSum
        const float2 x = vmul(g[j], us2);
        const float2 p2 = vmul(x, x);
        const float2 pe = vfma(x, x, vneg(p2));
        float2 t, e;
        two_sum(hi, p2, t, e);
        hi = t;
        lo = vadd(lo, vadd(e, pe));
      }
    }
    DFloat acc = df_add(DFloat{hi.x, lo.x}, DFloat{hi.y, lo.y});
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
#pragma unroll
      for (int w = 1; w < kThreads / 32; ++w) tot = df_add(tot, warp_sum[w]);
      partials[c] = tot;
    }
    __syncthreads();  // warp_sum is rewritten for the next chunk
  }
}

}  // namespace dpopt

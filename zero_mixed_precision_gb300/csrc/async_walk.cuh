// async_walk.cuh -- the step for many replicas of 16-bit gradients with the
// replica loads staged in shared memory by per-thread asynchronous copies.
//
// With N = 21..63 replicas the step is bound by how many gradient bytes each
// SM keeps in flight: the register-pipelined walk holds two chunks of 8
// 16-byte loads per thread (64 of its 126 registers), two CTAs per SM.  Here
// every thread copies its own 16-byte pieces of the next D chunks (three)
// straight into a ring of slots in shared memory (cp.async, no registers held
// while in flight), waits for the oldest chunk, adds it from shared memory in
// ascending replica order, and refills that slot with the chunk D
// further on.  A thread reads only the slots it filled itself, so no barrier
// is needed; cp.async.wait_group orders each slot's copy before its read.
// The arithmetic and the order are those of the other forms: the same bits.
#pragma once

#include "kernels.cuh"

namespace dpopt {

// One 16-byte asynchronous copy, global to shared, L1 bypassed, with an L2
// eviction policy (the gradients are read once).
__device__ __forceinline__ void cp_async16(uint32_t sdst, const void* gsrc, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(sdst),
               "l"(gsrc), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t ring_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Bytes between two consecutive replica rows of a slot: a row holds the
// 16 bytes of every thread of the CTA, so a warp's accesses are contiguous.
constexpr uint32_t kRowBytes = kThreads * 16;
constexpr uint32_t kSlotBytes = 8 * kRowBytes;  // one chunk of 8 replicas

template <int D>
constexpr uint32_t async_ring_bytes() { return D * kSlotBytes; }

// Replicas r0 .. min(r0 + 8, n) - 1 of this thread's group copied into the
// slot; one commit group per chunk (empty past the last replica, so that
// every chunk is one group).
__device__ __forceinline__ void issue_chunk(const void* const* gp, int64_t e0, int r0, int n,
                                            uint32_t slot, uint64_t pol) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (r0 + j < n) cp_async16(slot + j * kRowBytes, static_cast<const uint16_t*>(gp[r0 + j]) + e0,
                               pol);
  cp_async_commit();
}

// The fixed-order compensated sum of n >= 1 replicas of one group, D chunks
// of copies in flight.  `ring` is this thread's address in slot 0, row 0.
template <int D, int GK>
__device__ __forceinline__ void reduce_async(const void* const* gp, int64_t e0, int n,
                                             uint32_t ring, uint64_t pol,
                                             CompSum<float2> (&acc)[kGroup / 2]) {
  const int nch = (n + 7) >> 3;
#pragma unroll
  for (int c = 0; c < D; ++c) issue_chunk(gp, e0, 8 * c, n, ring + c * kSlotBytes, pol);
  for (int c = 0; c < nch; ++c) {
    cp_async_wait<D - 1>();  // chunk c has landed
    const uint32_t slot = ring + (uint32_t)(c % D) * kSlotBytes;
    GradLoad<GK> g[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) g[j].load_shared(slot + j * kRowBytes);
    const int r0 = 8 * c;
    const int cnt = n - r0 < 8 ? n - r0 : 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < cnt) {
#pragma unroll
        for (int k = 0; k < kGroup / 2; ++k) {
          if (c == 0 && j == 0) acc[k].init(g[j].pair(k));
          else acc[k].add(g[j].pair(k));
        }
      }
    }
    // the slot's values are in registers and added: refill it
    issue_chunk(gp, e0, r0 + 8 * D, n, slot, pol);
  }
}

// One 8-element group on packed lanes (group_vec_x2's arithmetic).
template <int D, int GK, bool EXT, class Out>
__device__ __forceinline__ void group_async(const void* const* gp, int64_t e0,
                                            const float* const (&st)[3], int n, uint32_t ring,
                                            uint64_t pol, const Hyper& h, const Out& o,
                                            float gscale) {
  constexpr int P = kGroup / 2;
  CompSum<float2> acc[P];
  float2 th[P], mm[P], vv[P];
  {
    float4 a, b;
    a = ld_state16(st[0]); b = ld_state16(st[0] + 4);
    th[0] = make_float2(a.x, a.y); th[1] = make_float2(a.z, a.w);
    th[2] = make_float2(b.x, b.y); th[3] = make_float2(b.z, b.w);
    a = ld_state16(st[1]); b = ld_state16(st[1] + 4);
    mm[0] = make_float2(a.x, a.y); mm[1] = make_float2(a.z, a.w);
    mm[2] = make_float2(b.x, b.y); mm[3] = make_float2(b.z, b.w);
    a = ld_state16(st[2]); b = ld_state16(st[2] + 4);
    vv[0] = make_float2(a.x, a.y); vv[1] = make_float2(a.z, a.w);
    vv[2] = make_float2(b.x, b.y); vv[3] = make_float2(b.z, b.w);
  }
  reduce_async<D, GK>(gp, e0, n, ring, pol, acc);
#pragma unroll
  for (int j = 0; j < P; ++j) {
    float2 g = acc[j].average(h);
    if constexpr (EXT) g = vmul(g, splat<float2>(gscale));
    adam_update<EXT>(g, th[j], mm[j], vv[j], h);
  }
  o.put(o.master, make_float4(th[0].x, th[0].y, th[1].x, th[1].y),
        make_float4(th[2].x, th[2].y, th[3].x, th[3].y));
  o.put(o.m, make_float4(mm[0].x, mm[0].y, mm[1].x, mm[1].y),
        make_float4(mm[2].x, mm[2].y, mm[3].x, mm[3].y));
  o.put(o.v, make_float4(vv[0].x, vv[0].y, vv[1].x, vv[1].y),
        make_float4(vv[2].x, vv[2].y, vv[3].x, vv[3].y));
  o.put_bf16(to_bf16x2(th[0].x, th[0].y), to_bf16x2(th[1].x, th[1].y),
             to_bf16x2(th[2].x, th[2].y), to_bf16x2(th[3].x, th[3].y));
}

// The step with the asynchronous walk (16-bit gradients, a runtime replica
// count, 16-byte state accesses): the walk of step_loop, whole vector groups
// through group_async, everything else one element at a time.
template <int D, int MINB, int GK, bool EXT, class LP>
__global__ void __launch_bounds__(kThreads, MINB) reduce_adam_async_kernel(const __grid_constant__ LP p) {
  extern __shared__ __align__(16) unsigned char async_ring[];
  pdl_wait();
  const Hyper& h = p.h;
  const float gscale = EXT ? grad_scale_of(h) : 1.f;
  const uint64_t pol = evict_first_policy();
  const uint32_t ring = ring_addr(async_ring) + threadIdx.x * 16u;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int si = 0;
  for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < p.total_groups;
       gi += stride) {
    while (gi >= p.seg[si + 1].first_group) ++si;
    const Seg& sg = p.seg[si];
    const int64_t e0 = (gi - sg.first_group) * kGroup;
    const int64_t rem = sg.len - e0;
    const int64_t so = sg.state_off + e0;
    if (!dbg_ok(h, si < p.nseg && e0 >= 0 && rem > 0) ||
        !dbg_span(h, so, so + (rem < kGroup ? rem : kGroup)))
      continue;
    if (sg.vec >= 1 && rem >= kGroup) {
      const float* const st[3] = {p.master + so, p.m + so, p.v + so};
      const GroupOutT<16> o{p.master + so, p.m + so, p.v + so, p.out + so};
      group_async<D, GK, EXT>(p.gptr + sg.ptr_base, e0, st, p.n_rep, ring, pol, h, o, gscale);
    } else {
      group_scalar<GK, EXT, false>(p, h, sg, e0, (int)(rem < kGroup ? rem : kGroup), gscale,
                                   nullptr);
    }
  }
}

}  // namespace dpopt

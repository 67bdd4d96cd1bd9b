// gather_bulk.cuh -- the fused step + ZeRO-3 all-gather whose bf16 copy is
// written to the replica buffers by bulk copies from shared memory.
//
// The step fused with the all-gather writes the shard's new bf16 values into
// the same position of every replica's parameter buffer ("Почему training 70B
// модели требует optimizer sharding (ZeRO-3)?", section 5: the parameters are
// all-gathered before the next forward pass).  Written by each thread, those
// are N 16-byte stores per 8-element group on top of the six state stores; on
// GB300 the store pipe, not DRAM, then sets the pace.  Here every thread puts
// its 16 bytes into the CTA's tile in shared memory and one thread hands the
// whole 4 KB tile to the bulk-copy engine once per replica buffer.  Measured
// on GB300 (G params/s, bulk copies against per-thread stores): gpt2s (N = 4)
// 161.4 against 146.9, 1p3b (N = 8) 115.0 against 100.9 -- 95 % of the
// measured copy bandwidth for 4N + 24 bytes per parameter, ahead of the step
// followed by a separate broadcast at every N measured.
#pragma once

#include "kernels.cuh"

namespace dpopt {

__device__ __forceinline__ uint32_t smem_u32_of(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The bf16 copy of a group staged in shared memory instead (the fused step +
// all-gather with bulk stores): the CTA's 2048-element tile of bf16 values is
// then written to every replica by bulk copies, not by N stores per thread.
template <int W = 16>
struct SmemBf16OutT : GroupOutT<W> {
  uint32_t saddr;  // this thread's 16 bytes of the CTA's tile
  __device__ __forceinline__ void put_bf16(uint32_t a, uint32_t b, uint32_t c, uint32_t d) const {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
  }
};

// Bulk stores from shared to global memory (PTX ISA: cp.async.bulk with
// bulk-group completion).  Both addresses 16-byte aligned, size a multiple of
// 16.  Shared-memory writes are made visible to the bulk copies' (async)
// proxy by fence.proxy.async before the copies are issued.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// The written lines carry an L2 eviction policy (evict-first: nothing here
// reads them again; 1p3b's fused step + all-gather 112.4 -> 115.0 G params/s).
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes,
                                           uint64_t pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
               ::"l"(gdst), "r"(ssrc), "r"(bytes), "l"(pol)
               : "memory");
}

// Shared-memory tiles a CTA cycles through (three measured the same as two).
constexpr int kGatherTiles = 2;
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Until at most N committed groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Until at most N committed groups are incomplete (their writes performed).
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// The same fused step + all-gather with the bf16 copy written by bulk
// copies.  The CTA walks the shard in tiles of kThreads groups (2048
// elements, 4 KB of bf16): every thread computes its group and writes master,
// m and v as usual, puts its 16 bf16 bytes into the tile in shared memory,
// and one thread then issues one 4 KB bulk copy of the tile per replica buffer
// (the own one and the N - 1 others).  Two tiles alternate: a tile is written
// again only once the copies of two tiles back have read it.  A tile that is
// not whole (the shard's tail, unaligned segments) takes the per-thread
// stores of step_loop.  Same values, same bytes in every buffer.
template <int NR, int GK, int PACK, int W, int MAXSEG, int MAXPTR>
__global__ void __launch_bounds__(kThreads, W == 32 ? wide_ctas<NR, GK>() : min_ctas<NR, PACK>())
    reduce_adam_gather_bulk_kernel(const __grid_constant__ LaunchParams<MAXSEG, MAXPTR> p,
                                   const __grid_constant__ GatherDst d) {
  __shared__ __align__(128) uint4 tile[kGatherTiles][kThreads];
  pdl_wait();
  constexpr int kLevel = W == 32 ? 2 : 1;
  const Hyper& h = p.h;
  const uint64_t pol = evict_first_policy();
  const Seg& sg = p.seg[0];  // the full-buffer call: one segment
  const int64_t cta_stride = (int64_t)gridDim.x * kThreads;
  int buf = 0;
  for (int64_t base = (int64_t)blockIdx.x * kThreads; base < p.total_groups;
       base += cta_stride) {
    // the same for every thread of the CTA: is this tile whole and vectorised?
    const bool whole = p.nseg == 1 && sg.vec >= kLevel && (base + kThreads) * kGroup <= sg.len;
    const int64_t gi = base + threadIdx.x;
    if (whole) {
      const int64_t e0 = gi * kGroup;
      const int64_t so = sg.state_off + e0;
      const int64_t so0 = sg.state_off + base * kGroup;  // the tile's first element
      const bool ok = dbg_ok(h, e0 >= 0 && e0 + kGroup <= sg.len) &&
                      dbg_span(h, so0, so0 + (int64_t)kThreads * kGroup);
      if (ok) {
        const GlobalSource<GK, W> src{p.gptr + sg.ptr_base, e0,
                                      {p.master + so, p.m + so, p.v + so}, pol};
        const SmemBf16OutT<W> o{{p.master + so, p.m + so, p.v + so, p.out + so},
                                smem_u32_of(&tile[buf][threadIdx.x])};
        if constexpr (PACK) group_vec_x2<NR, GK, false>(src, p.n_rep, h, o, 1.f);
        else group_vec_x1<NR, GK, false>(src, p.n_rep, h, o, 1.f);
      }
      fence_proxy_async_shared();
      __syncthreads();
      if (threadIdx.x == 0 && ok) {
        const uint32_t t = smem_u32_of(&tile[buf][0]);
        constexpr uint32_t kBytes = kThreads * kGroup * 2;
        bulk_store(p.out + so0, t, kBytes, pol);
        for (int i = 0; i < d.n; ++i) bulk_store(d.dst[i] + so0, t, kBytes, pol);
        bulk_commit();
      }
      // the next tile is free again once the copies that last read it are done
      if (threadIdx.x == 0) bulk_wait_read<kGatherTiles - 1>();
      __syncthreads();
      buf = buf + 1 == kGatherTiles ? 0 : buf + 1;
    } else if (gi < p.total_groups) {
      const int64_t e0 = (gi - sg.first_group) * kGroup;
      const int64_t rem = sg.len - e0;
      const int64_t so = sg.state_off + e0;
      if (!dbg_ok(h, rem > 0) || !dbg_span(h, so, so + (rem < kGroup ? rem : kGroup))) continue;
      if (sg.vec >= kLevel && rem >= kGroup) {
        const GlobalSource<GK, W> src{p.gptr + sg.ptr_base, e0,
                                      {p.master + so, p.m + so, p.v + so}, pol};
        const GatherOutT<W> o{{p.master + so, p.m + so, p.v + so, p.out + so}, &d, so};
        if constexpr (PACK) group_vec_x2<NR, GK, false>(src, p.n_rep, h, o, 1.f);
        else group_vec_x1<NR, GK, false>(src, p.n_rep, h, o, 1.f);
      } else {
        group_scalar<GK, false, true>(p, h, sg, e0, (int)(rem < kGroup ? rem : kGroup), 1.f, &d);
      }
    }
  }
  if (threadIdx.x == 0) bulk_wait<0>();  // every bulk copy performed before the CTA exits
}

}  // namespace dpopt

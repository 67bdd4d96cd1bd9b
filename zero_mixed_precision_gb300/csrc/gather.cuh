// gather.cuh -- ZeRO-3 parameter all-gather with every replica resident.
//
// After the step each rank holds the new bf16 copy of its own 1/N shard only;
// before the next forward pass every replica needs the full parameters
// ("Почему training 70B модели требует optimizer sharding (ZeRO-3)?", section
// 5: all-gather of the parameters, each GPU sends its shard to all others).
// With all N replica parameter buffers in this GPU's memory the all-gather of
// one rank's shard is a local broadcast: read the shard once, write it into
// the same position of every replica's buffer -- 2 + 2N bytes per parameter,
// an HBM-bound copy.
#pragma once

#include "gather_bulk.cuh"

namespace dpopt {

struct GatherParams {
  const uint16_t* src;                   // the shard's bf16 copy
  uint16_t* dst[DPOPT_MAX_REPLICAS];     // each replica's buffer at the shard's offset
  int64_t len;                           // elements
  int32_t n_dst;
  int32_t vec;                           // every pointer 16-byte aligned
#ifdef DPOPT_DEBUG_BOUNDS
  unsigned int* dbg_status;              // set when an index check fails (see dbg_ok)
#endif
};

// The CTA walks the shard in tiles of kThreads groups (2048 elements, 4 KB):
// every thread loads its 16 bytes into the tile in shared memory and one
// thread writes the whole tile to every replica buffer with bulk copies, so
// the N writes leave the store pipe (which otherwise sets the pace of this
// write-heavy copy) for the bulk-copy engine; two tiles alternate.  Tiles that
// are not whole, or not 16-byte aligned, go element group by group.
__global__ void __launch_bounds__(kThreads) allgather_bf16_kernel(const __grid_constant__ GatherParams p) {
  __shared__ __align__(128) uint4 tile[2][kThreads];
  pdl_wait();
  const uint64_t pol = evict_first_policy();
  const int64_t groups = (p.len + kGroup - 1) / kGroup;
  const int64_t cta_stride = (int64_t)gridDim.x * kThreads;
  int buf = 0;
  int64_t base = (int64_t)blockIdx.x * kThreads;
  for (; base < groups && p.vec && (base + kThreads) * kGroup <= p.len; base += cta_stride) {
    const int64_t e0 = (base + threadIdx.x) * kGroup;
    tile[buf][threadIdx.x] = ld_grad16(p.src + e0, pol);
    fence_proxy_async_shared();
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t t = smem_u32_of(&tile[buf][0]);
      constexpr uint32_t kBytes = kThreads * kGroup * 2;
      for (int r = 0; r < p.n_dst; ++r) bulk_store(p.dst[r] + base * kGroup, t, kBytes, pol);
      bulk_commit();
      bulk_wait_read<1>();  // the other tile is free again
    }
    __syncthreads();
    buf ^= 1;
  }
  // the remaining tile (not whole, or unaligned pointers): element groups
  for (int64_t gi = base + threadIdx.x; gi < groups; gi += cta_stride) {
    const int64_t e0 = gi * kGroup;
#ifdef DPOPT_DEBUG_BOUNDS
    if (e0 < 0 || e0 >= p.len) {
      if (p.dbg_status) atomicOr(p.dbg_status, 1u);
      continue;
    }
#endif
    if (p.vec && e0 + kGroup <= p.len) {
      const uint4 w = ld_grad16(p.src + e0, pol);
      for (int r = 0; r < p.n_dst; ++r) st_stream16u(p.dst[r] + e0, w.x, w.y, w.z, w.w);
    } else {
      const int64_t end = e0 + kGroup < p.len ? e0 + kGroup : p.len;
      for (int64_t e = e0; e < end; ++e) {
        const uint16_t x = p.src[e];
        for (int r = 0; r < p.n_dst; ++r) p.dst[r][e] = x;
      }
    }
  }
  if (threadIdx.x == 0) bulk_wait<0>();  // every bulk copy performed before the CTA exits
}

}  // namespace dpopt

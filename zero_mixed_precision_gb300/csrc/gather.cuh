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

#include "kernels.cuh"

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

__global__ void __launch_bounds__(kThreads) allgather_bf16_kernel(const __grid_constant__ GatherParams p) {
  pdl_wait();
  const uint64_t pol = evict_first_policy();
  const int64_t groups = (p.len + kGroup - 1) / kGroup;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < groups; gi += stride) {
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
}

}  // namespace dpopt

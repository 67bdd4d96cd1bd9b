// tma.cuh -- the fused reduce + Adam kernel, bulk-copy (TMA) staged form.
//
// A persistent CTA = one producer warp + kTmaConsumerWarps consumer warps.
// The producer's elected lane moves each tile of kTmaTile elements -- the N
// replica rows and the master/m/v rows -- from global to shared memory with
// 1-D bulk copies (cp.async.bulk, the Tensor Memory Accelerator's untiled
// form) into a ring of `stages` buffers, each guarded by a "full" mbarrier
// (transaction bytes) and an "empty" mbarrier (one arrival per consumer
// warp).  Consumers compute from shared memory with the same per-element
// arithmetic as the direct-load kernel and store the results straight to
// global memory.  The producer keeps several tiles in flight however long the
// arithmetic of the current one takes, so memory-level parallelism no longer
// depends on how many warps happen to be waiting on loads.
//
// Every wait is bounded: after `wait_limit` clock cycles a waiter sets the
// device status word and gives up; the producer then waits (bounded again)
// for the copies it has issued before its thread exits.  Results are
// bitwise identical to the direct-load kernel's.
#pragma once

#include "kernels.cuh"

namespace dpopt {

// Sticky status word of this library image: bit 0 is set when a bounded
// device-side wait gave up.  Read and cleared by dpopt_stream_status().
__device__ unsigned int g_status;

constexpr int kTmaConsumerWarps = 8;
constexpr int kTmaThreads = 32 * (kTmaConsumerWarps + 1);
constexpr int kTmaTile = kTmaConsumerWarps * 32 * kGroup;  // elements per tile (2048)
constexpr int kTmaMaxStages = 8;

struct TmaSeg {
  int64_t first_tile;  // tiles of all earlier segments (prefix sum)
  int64_t state_off;   // first shard element this segment updates
  int64_t body;        // elements moved by bulk copies: len rounded down to a multiple of 8
  int64_t len;         // elements (body + a scalar tail of < 8)
  int32_t ptr_base;    // index of replica 0's pointer in TmaParams::gptr
  int32_t pad_;
};

template <int MAXSEG, int MAXPTR>
struct TmaParams {
  Hyper h;
  float* master;
  float* m;
  float* v;
  uint16_t* out;
  int64_t total_tiles;
  long long wait_limit;  // clock cycles one bounded wait may take
  int32_t n_rep;
  int32_t nseg;
  int32_t stages;
  uint32_t stage_bytes;
  TmaSeg seg[MAXSEG + 1];  // seg[nseg].first_tile == total_tiles
  const void* gptr[MAXPTR];
};

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy primitives (PTX ISA: mbarrier, cp.async.bulk)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with `parity` has completed, for at most `limit`
// cycles.  Returns false (and sets the device status word) on time-out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (clock64() - t0 > limit) {
      atomicOr(&g_status, 1u);
      return false;
    }
  }
  return true;
}

// Global -> shared bulk copy completing `bytes` transaction bytes on `bar`.
// dst, src and bytes must all be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

// NR: the replica count (the ring holds two stages of N replica rows only
// for small N, so every eligible N has its own kernel).  W: the width of one
// state store to global memory (32: one 256-bit store per array and thread).
template <int NR, int GK, int W, int MAXSEG, int MAXPTR>
__global__ void __launch_bounds__(kTmaThreads, 1)
    reduce_adam_tma_kernel(const __grid_constant__ TmaParams<MAXSEG, MAXPTR> p) {
  static_assert(NR >= 1, "one kernel per replica count");
  pdl_wait();
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full_bar[kTmaMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kTmaMaxStages];

  constexpr uint32_t gsize = GK == 0 ? 2u : 4u;
  const int S = p.stages;
  constexpr int n = NR;
  const uint32_t row_bytes = (uint32_t)kTmaTile * gsize;     // one replica's row of a tile
  const uint32_t state_base = (uint32_t)n * row_bytes;      // master row, then m, then v
  const uint32_t smem0 = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kTmaConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = evict_first_policy();
      int si = 0;
      int64_t it = 0;
      for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
        while (t >= p.seg[si + 1].first_tile) ++si;
        const TmaSeg& sg = p.seg[si];
        const int s = (int)(it % S);
        const int64_t k = it / S;
        if (k > 0 && !mbar_wait_bounded(smem_u32(&empty_bar[s]), (uint32_t)((k - 1) & 1),
                                         p.wait_limit))
          break;
        const int64_t e0 = (t - sg.first_tile) * kTmaTile;
        const int64_t left = sg.body - e0;
        const uint32_t cnt = (uint32_t)(left < kTmaTile ? left : kTmaTile);
        const uint32_t sb = smem0 + (uint32_t)s * p.stage_bytes;
        const uint32_t fb = smem_u32(&full_bar[s]);
        const int64_t so = sg.state_off + e0;
        // (a tile that fails the bounds-checked build's test is armed without
        // copies: its phase completes on the arrival alone)
        const bool good = dbg_ok(p.h, si < p.nseg && e0 >= 0 && left > 0) &&
                          dbg_span(p.h, so, so + cnt);
        mbar_arrive_expect_tx(fb, good ? cnt * ((uint32_t)n * gsize + 12u) : 0u);
        if (good) {
          const void* const* gp = p.gptr + sg.ptr_base;
          for (int r = 0; r < n; ++r)
            bulk_g2s(sb + (uint32_t)r * row_bytes,
                     static_cast<const unsigned char*>(gp[r]) + e0 * gsize, cnt * gsize, fb, pol);
          bulk_g2s(sb + state_base, p.master + so, cnt * 4u, fb, pol);
          bulk_g2s(sb + state_base + kTmaTile * 4u, p.m + so, cnt * 4u, fb, pol);
          bulk_g2s(sb + state_base + kTmaTile * 8u, p.v + so, cnt * 4u, fb, pol);
        }
      }
      // drain: the last phase armed on every stage must complete before this
      // thread leaves (the copies write into this CTA's shared memory)
      for (int s = 0; s < S; ++s) {
        const int64_t uses = it / S + (s < it % S ? 1 : 0);
        if (uses > 0)
          mbar_wait_bounded(smem_u32(&full_bar[s]), (uint32_t)((uses - 1) & 1), p.wait_limit);
      }
    }
  } else {
    // ---------------- consumers ----------------
    const int c = threadIdx.x - 32;  // 0 .. 32*kTmaConsumerWarps-1
    int si = 0;
    int64_t it = 0;
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
      while (t >= p.seg[si + 1].first_tile) ++si;
      const TmaSeg& sg = p.seg[si];
      const int s = (int)(it % S);
      const int64_t k = it / S;
      bool ok = mbar_wait_bounded(smem_u32(&full_bar[s]), (uint32_t)(k & 1), p.wait_limit);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int64_t e0 = (t - sg.first_tile) * kTmaTile;
      const int64_t left = sg.body - e0;
      const int cnt = (int)(left < kTmaTile ? left : kTmaTile);
      const bool good = dbg_ok(p.h, si < p.nseg && e0 >= 0 && left > 0) &&
                        dbg_span(p.h, sg.state_off + e0, sg.state_off + e0 + cnt);
      if (good && c * kGroup < cnt) {
        const uint32_t sb = smem0 + (uint32_t)s * p.stage_bytes;
        const uint32_t sx = sb + state_base + (uint32_t)c * 32u;
        const SharedSource<GK> src{sb + (uint32_t)c * kGroup * gsize, row_bytes,
                                   {sx, sx + kTmaTile * 4u, sx + kTmaTile * 8u}};
        const int64_t so = sg.state_off + e0 + (int64_t)c * kGroup;
        const GroupOutT<W> o{p.master + so, p.m + so, p.v + so, p.out + so};
        group_vec_x1<NR, GK, false>(src, n, p.h, o, 1.f);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
    }
    // the (< 8)-element tail of each segment, one element at a time
    if (c == 0) {
      for (int j = blockIdx.x; j < p.nseg; j += gridDim.x) {
        const TmaSeg& sg = p.seg[j];
        if (sg.len > sg.body)
          group_scalar<GK, false, false>(p, p.h, sg, sg.body, (int)(sg.len - sg.body), 1.f,
                                        nullptr);
      }
    }
  }
}

// Exercises the bounded wait: one thread waits on an mbarrier that nothing
// ever arrives on; after `limit` cycles it gives up and sets the status word.
__global__ void selftest_wait_kernel(long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0u, limit);
}

}  // namespace dpopt

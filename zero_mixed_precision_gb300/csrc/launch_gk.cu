// launch_gk.cu -- the kernels of one gradient type and their launchers: the
// fused reduce + Adam step, the loss-scaled step and the squared-norm pass.
// The build compiles this file once per type (-DDPOPT_GK=0 bf16, 1 fp32,
// 2 fp16), so the three instantiation sets compile in parallel.
//
// Replica counts 1..8 each get a kernel with the replica loop unrolled: at
// most 64 registers, so four 256-thread CTAs share an SM and every thread has
// all N of its gradient loads in flight at once.  bf16 and fp16 gradients with
// 9..20 replicas get unrolled kernels too, reading the replicas in batches of
// 8 (the last one N mod 8) at the same four CTAs per SM: 100-102 % of the copy
// bandwidth at N = 9..14 against 85-92 % for the runtime-count packed body,
// and at N = 17..20 96.9-97.3 % against 94.1-96.9 % for the shared-memory
// walk (S = 256M).  Above 20 the 16-bit kernels walk the replicas at runtime
// count (the shared-memory walk to 63, the register-pipelined walk at 64);
// fp32 gradients take the runtime-count packed body above 8, where it already
// reaches the copy rate.  The accumulation order is the same in every form,
// so the choice changes speed only, never bits.

//
// The state access width of each kernel is wide_states() (kernels.cuh).
#include <algorithm>
#include <atomic>

#include "internal.h"
#include "async_walk.cuh"
#include "gather_bulk.cuh"
#include "norm.cuh"

#ifndef DPOPT_GK
#error "compile with -DDPOPT_GK=0 (bf16), 1 (fp32) or 2 (fp16)"
#endif

// The helpers below live in a namespace of their own per gradient type: nvcc
// names an anonymous namespace after the source file, and this file is
// compiled three times into one library.
#if DPOPT_GK == 0
#define DPOPT_GK_NS gk_bf16
#elif DPOPT_GK == 1
#define DPOPT_GK_NS gk_f32
#elif DPOPT_GK == 2
#define DPOPT_GK_NS gk_f16
#else
#error "DPOPT_GK must be 0, 1 or 2"
#endif

namespace dpopt {
namespace DPOPT_GK_NS {

constexpr int kGK = DPOPT_GK;

constexpr bool wide_states(int nr) { return dpopt::wide_states(kGK, nr); }

// Whether every segment's vector level allows the 32-byte accesses (level 0
// segments go one element at a time in either form).
template <int MS, int MP>
bool all_wide(const LaunchParams<MS, MP>& p) {
  for (int s = 0; s < p.nseg; ++s)
    if (p.seg[s].vec == 1) return false;
  return true;
}
// (a device-resident table was checked on the host while it was written)
bool all_wide(const TableParams& p) { return p.wide != 0; }

// Persistent grid: `want` CTAs of work, capped at the resident CTAs of every
// SM (occupancy looked up once per kernel).
template <class Kern>
int persistent_grid(Kern kern, std::atomic<int>& per_sm, int64_t want, unsigned* grid) {
  int sms = 0;
  int rc = sm_count(&sms);
  if (rc) return rc;
  int bps = per_sm.load(std::memory_order_relaxed);
  if (bps == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, kThreads, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (bps < 1) bps = 1;
    per_sm.store(bps, std::memory_order_relaxed);
  }
  *grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * bps));
  return DPOPT_OK;
}

int launched(cudaError_t e) {
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  count_launch();
  return DPOPT_OK;
}

// ---------------------------------------------------------------------------
// the step
// ---------------------------------------------------------------------------

// The step kernel for a parameter-space table, or for a device-resident one.
template <int NR, int PACK, bool EXT, int W, int MS, int MP>
auto step_kern(const LaunchParams<MS, MP>&) {
  return reduce_adam_ldg_kernel<NR, kGK, PACK, EXT, W, MS, MP>;
}
template <int NR, int PACK, bool EXT, int W>
auto step_kern(const TableParams&) {
  return reduce_adam_table_kernel<NR, kGK, PACK, EXT, W>;
}

template <int NR, int PACK, bool EXT, int W, class LP>
int step_kernel(const LP& p, cudaStream_t stream) {
  auto kern = step_kern<NR, PACK, EXT, W>(p);
  static std::atomic<int> per_sm{0};
  unsigned grid = 0;
  int rc = persistent_grid(kern, per_sm, (p.total_groups + kThreads - 1) / kThreads, &grid);
  if (rc) return rc;
  return launched(launch_pdl(kern, grid, kThreads, 0, stream, p));
}

// The runtime-count step for 16-bit gradients with the replica loads staged
// in shared memory by asynchronous copies (async_walk.cuh): `depth` chunks of
// 8 replicas in flight per thread, `min_blocks` CTAs per SM (96 KB of
// shared memory each).  Measured on GB300 (bf16, S = 256M, GB/s, asynchronous
// walk against the register-pipelined one): N = 17 6366 / 6356, 18 6428 /
// 6007, 20 6531 / 6268, 23 6644 / 6531, 24 6670 / 6521, 28 6670 / 6174,
// 31 6750 / 6217, 32 6835 / 6626, 40 6817 / 6357, 48 6816 / 6627, 56 6773 /
// 6530, 57 6809 / 6361, 63 6743 / 6263, 64 6617 / 6742.  Two chunks at three
// CTAs per SM (spilling) and four chunks at one CTA measured slower.
// max_replicas: replica counts from 21 up to this take the asynchronous walk
// (17..20 have unrolled kernels); N = 64 the register-pipelined walk of
// kernels.cuh, faster there.
struct AsyncWalk {
  static constexpr int depth = 3;
  static constexpr int min_blocks = 2;
  static constexpr int max_replicas = 63;
};

template <bool EXT, class LP>
int async_step(const LP& p, cudaStream_t stream) {
  auto kern = reduce_adam_async_kernel<AsyncWalk::depth, AsyncWalk::min_blocks, kGK, EXT, LP>;
  constexpr int smem = (int)async_ring_bytes<AsyncWalk::depth>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  static std::atomic<int> per_sm{0};
  int sms = 0;
  int rc = sm_count(&sms);
  if (rc) return rc;
  int bps = per_sm.load(std::memory_order_relaxed);
  if (bps == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, kThreads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (bps < 1) bps = 1;
    per_sm.store(bps, std::memory_order_relaxed);
  }
  const int64_t want = (p.total_groups + kThreads - 1) / kThreads;
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * bps));
  return launched(launch_pdl(kern, grid, kThreads, (size_t)smem, stream, p));
}

// Unrolled kernel for NR replicas in its measured width; a 32-byte kernel
// whose segments are not all 32-byte aligned hands over to the runtime-count
// 16-byte kernel.
template <int NR, bool EXT, class LP>
int step_nr(const LP& p, cudaStream_t s) {
  if constexpr (wide_states(NR)) {
    if (all_wide(p)) return step_kernel<NR, 0, EXT, 32>(p, s);
    return step_kernel<0, 1, EXT, 16>(p, s);
  } else {
    return step_kernel<NR, 0, EXT, 16>(p, s);
  }
}

template <bool EXT, class LP>
int step_n(const LP& p, cudaStream_t s) {
  switch (p.n_rep) {
    case 1: return step_nr<1, EXT>(p, s);
    case 2: return step_nr<2, EXT>(p, s);
    case 3: return step_nr<3, EXT>(p, s);
    case 4: return step_nr<4, EXT>(p, s);
    case 5: return step_nr<5, EXT>(p, s);
    case 6: return step_nr<6, EXT>(p, s);
    case 7: return step_nr<7, EXT>(p, s);
    case 8: return step_nr<8, EXT>(p, s);
    case 9: if constexpr (kGK != 1) return step_nr<9, EXT>(p, s); else break;
    case 10: if constexpr (kGK != 1) return step_nr<10, EXT>(p, s); else break;
    case 11: if constexpr (kGK != 1) return step_nr<11, EXT>(p, s); else break;
    case 12: if constexpr (kGK != 1) return step_nr<12, EXT>(p, s); else break;
    case 13: if constexpr (kGK != 1) return step_nr<13, EXT>(p, s); else break;
    case 14: if constexpr (kGK != 1) return step_nr<14, EXT>(p, s); else break;
    case 15: if constexpr (kGK != 1) return step_nr<15, EXT>(p, s); else break;
    case 16: if constexpr (kGK != 1) return step_nr<16, EXT>(p, s); else break;
    case 17: if constexpr (kGK != 1) return step_nr<17, EXT>(p, s); else break;
    case 18: if constexpr (kGK != 1) return step_nr<18, EXT>(p, s); else break;
    case 19: if constexpr (kGK != 1) return step_nr<19, EXT>(p, s); else break;
    case 20: if constexpr (kGK != 1) return step_nr<20, EXT>(p, s); else break;
    default: break;
  }
  if constexpr (kGK != 1) {
    if (p.n_rep >= 17 && p.n_rep <= AsyncWalk::max_replicas) return async_step<EXT>(p, s);
  }
  return step_kernel<0, 1, EXT, 16>(p, s);
}

// ---------------------------------------------------------------------------
// the step fused with the ZeRO-3 all-gather (one segment: the full-buffer call)
// ---------------------------------------------------------------------------

template <int NR, int PACK, int W>
int gather_kernel(const SmallParams& p, const GatherDst& d, cudaStream_t stream) {
  auto kern = reduce_adam_gather_bulk_kernel<NR, kGK, PACK, W, kSmallSegs, kSmallPtrs>;
  static std::atomic<int> per_sm{0};
  unsigned grid = 0;
  int rc = persistent_grid(kern, per_sm, (p.total_groups + kThreads - 1) / kThreads, &grid);
  if (rc) return rc;
  return launched(launch_pdl(kern, grid, kThreads, 0, stream, p, d));
}

// The same kernel forms as the plain step (widths by wide_states()).
template <int NR>
int gather_nr(const SmallParams& p, const GatherDst& d, cudaStream_t s) {
  if constexpr (wide_states(NR)) {
    if (all_wide(p)) return gather_kernel<NR, 0, 32>(p, d, s);
    return gather_kernel<0, 1, 16>(p, d, s);
  } else {
    return gather_kernel<NR, 0, 16>(p, d, s);
  }
}

// ---------------------------------------------------------------------------
// the loss-scaled step
// ---------------------------------------------------------------------------

template <int NR, int PACK, int W, int MS, int MP>
int amp_kernel(const LaunchParams<MS, MP>& p, const LossScaleState* st, const double* sq,
               cudaStream_t stream) {
  auto kern = reduce_adam_amp_kernel<NR, kGK, PACK, W, MS, MP>;
  static std::atomic<int> per_sm{0};
  unsigned grid = 0;
  int rc = persistent_grid(kern, per_sm, (p.total_groups + kThreads - 1) / kThreads, &grid);
  if (rc) return rc;
  return launched(launch_pdl(kern, grid, kThreads, 0, stream, p, st, sq));
}

// The loss-scaled kernels take the same widths as the step: their 256-bit
// forms spill 16..60 bytes at 64 registers (the per-step scalars sit in
// registers), yet measured faster than the 16-byte ones (fp32 N = 1: 5134
// against 4990 GB/s for the whole two-pass step).
template <int NR, int MS, int MP>
int amp_nr(const LaunchParams<MS, MP>& p, const LossScaleState* st, const double* sq,
           cudaStream_t s) {
  if constexpr (wide_states(NR)) {
    if (all_wide(p)) return amp_kernel<NR, 0, 32>(p, st, sq, s);
    return amp_kernel<0, 1, 16>(p, st, sq, s);
  } else {
    return amp_kernel<NR, 0, 16>(p, st, sq, s);
  }
}

// ---------------------------------------------------------------------------
// the squared-norm pass: one CTA per chunk, the hardware scheduler filling
// the SMs (a CTA loops over further chunks only beyond 2^24 of them)
// ---------------------------------------------------------------------------

template <int NR, bool STORE, int MS, int MP>
int norm_kernel(const LaunchParams<MS, MP>& p, double* partials, int64_t nchunks,
                cudaStream_t stream) {
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(nchunks, 1 << 24));
  return launched(launch_pdl(grad_sqnorm_kernel<NR, kGK, STORE, MS, MP>, grid, kThreads, 0,
                             stream, p, reinterpret_cast<DFloat*>(partials), nchunks));
}

template <bool STORE, int MS, int MP>
int norm_n(const LaunchParams<MS, MP>& p, double* partials, int64_t nchunks, cudaStream_t s) {
  switch (p.n_rep) {
    case 1: return norm_kernel<1, STORE>(p, partials, nchunks, s);
    case 2: return norm_kernel<2, STORE>(p, partials, nchunks, s);
    case 3: return norm_kernel<3, STORE>(p, partials, nchunks, s);
    case 4: return norm_kernel<4, STORE>(p, partials, nchunks, s);
    case 5: return norm_kernel<5, STORE>(p, partials, nchunks, s);
    case 6: return norm_kernel<6, STORE>(p, partials, nchunks, s);
    case 7: return norm_kernel<7, STORE>(p, partials, nchunks, s);
    case 8: return norm_kernel<8, STORE>(p, partials, nchunks, s);
    default: return norm_kernel<0, STORE>(p, partials, nchunks, s);
  }
}

}  // namespace DPOPT_GK_NS

using DPOPT_GK_NS::kGK;

template <int G, int MS, int MP>
int launch_step(const LaunchParams<MS, MP>& p, bool ext, cudaStream_t stream) {
  static_assert(G == kGK, "launch_step instantiated for another gradient type");
  return ext ? DPOPT_GK_NS::step_n<true>(p, stream) : DPOPT_GK_NS::step_n<false>(p, stream);
}

template <int G>
int launch_step_table(const TableParams& p, bool ext, cudaStream_t stream) {
  static_assert(G == kGK, "launch_step_table instantiated for another gradient type");
  return ext ? DPOPT_GK_NS::step_n<true>(p, stream) : DPOPT_GK_NS::step_n<false>(p, stream);
}

template <int G, int MS, int MP>
int launch_amp_step(const LaunchParams<MS, MP>& p, const LossScaleState* state,
                    const double* sqnorm, cudaStream_t stream) {
  static_assert(G == kGK, "launch_amp_step instantiated for another gradient type");
  switch (p.n_rep) {
    case 1: return DPOPT_GK_NS::amp_nr<1>(p, state, sqnorm, stream);
    case 2: return DPOPT_GK_NS::amp_nr<2>(p, state, sqnorm, stream);
    case 3: return DPOPT_GK_NS::amp_nr<3>(p, state, sqnorm, stream);
    case 4: return DPOPT_GK_NS::amp_nr<4>(p, state, sqnorm, stream);
    case 5: return DPOPT_GK_NS::amp_nr<5>(p, state, sqnorm, stream);
    case 6: return DPOPT_GK_NS::amp_nr<6>(p, state, sqnorm, stream);
    case 7: return DPOPT_GK_NS::amp_nr<7>(p, state, sqnorm, stream);
    case 8: return DPOPT_GK_NS::amp_nr<8>(p, state, sqnorm, stream);
    case 9: if constexpr (kGK != 1) return DPOPT_GK_NS::amp_nr<9>(p, state, sqnorm, stream); else break;
    case 10: if constexpr (kGK != 1) return DPOPT_GK_NS::amp_nr<10>(p, state, sqnorm, stream); else break;
    case 11: if constexpr (kGK != 1) return DPOPT_GK_NS::amp_nr<11>(p, state, sqnorm, stream); else break;
    case 12: if constexpr (kGK != 1) return DPOPT_GK_NS::amp_nr<12>(p, state, sqnorm, stream); else break;
    case 13: if constexpr (kGK != 1) return DPOPT_GK_NS::amp_nr<13>(p, state, sqnorm, stream); else break;
    case 14: if constexpr (kGK != 1) return DPOPT_GK_NS::amp_nr<14>(p, state, sqnorm, stream); else break;
    case 15: if constexpr (kGK != 1) return DPOPT_GK_NS::amp_nr<15>(p, state, sqnorm, stream); else break;
    case 16: if constexpr (kGK != 1) return DPOPT_GK_NS::amp_nr<16>(p, state, sqnorm, stream); else break;
    default: break;
  }
  return DPOPT_GK_NS::amp_kernel<0, 1, 16>(p, state, sqnorm, stream);
}

template <int G>
int launch_step_gather(const SmallParams& p, const GatherDst& d, cudaStream_t stream) {
  static_assert(G == kGK, "launch_step_gather instantiated for another gradient type");
  switch (p.n_rep) {
    case 1: return DPOPT_GK_NS::gather_nr<1>(p, d, stream);
    case 2: return DPOPT_GK_NS::gather_nr<2>(p, d, stream);
    case 3: return DPOPT_GK_NS::gather_nr<3>(p, d, stream);
    case 4: return DPOPT_GK_NS::gather_nr<4>(p, d, stream);
    case 5: return DPOPT_GK_NS::gather_nr<5>(p, d, stream);
    case 6: return DPOPT_GK_NS::gather_nr<6>(p, d, stream);
    case 7: return DPOPT_GK_NS::gather_nr<7>(p, d, stream);
    case 8: return DPOPT_GK_NS::gather_nr<8>(p, d, stream);
    case 9: if constexpr (kGK != 1) return DPOPT_GK_NS::gather_nr<9>(p, d, stream); else break;
    case 10: if constexpr (kGK != 1) return DPOPT_GK_NS::gather_nr<10>(p, d, stream); else break;
    case 11: if constexpr (kGK != 1) return DPOPT_GK_NS::gather_nr<11>(p, d, stream); else break;
    case 12: if constexpr (kGK != 1) return DPOPT_GK_NS::gather_nr<12>(p, d, stream); else break;
    case 13: if constexpr (kGK != 1) return DPOPT_GK_NS::gather_nr<13>(p, d, stream); else break;
    case 14: if constexpr (kGK != 1) return DPOPT_GK_NS::gather_nr<14>(p, d, stream); else break;
    case 15: if constexpr (kGK != 1) return DPOPT_GK_NS::gather_nr<15>(p, d, stream); else break;
    case 16: if constexpr (kGK != 1) return DPOPT_GK_NS::gather_nr<16>(p, d, stream); else break;
    default: break;
  }
  return DPOPT_GK_NS::gather_kernel<0, 1, 16>(p, d, stream);
}

template <int G, int MS, int MP>
int launch_sqnorm_pass(const LaunchParams<MS, MP>& p, double* partials, int64_t nchunks,
                       bool store_average, cudaStream_t stream) {
  static_assert(G == kGK, "launch_sqnorm_pass instantiated for another gradient type");
  if (!store_average) return DPOPT_GK_NS::norm_n<false>(p, partials, nchunks, stream);
  if constexpr (MS == kSmallSegs) return DPOPT_GK_NS::norm_n<true>(p, partials, nchunks, stream);
  return fail(DPOPT_ERR_UNSUPPORTED, "the averaged gradient is stored for one segment only");
}

template int launch_step<kGK>(const SmallParams&, bool, cudaStream_t);
template int launch_step<kGK>(const BigParams&, bool, cudaStream_t);
template int launch_step_table<kGK>(const TableParams&, bool, cudaStream_t);
template int launch_step_gather<kGK>(const SmallParams&, const GatherDst&, cudaStream_t);
template int launch_amp_step<kGK>(const SmallParams&, const LossScaleState*, const double*,
                                  cudaStream_t);
template int launch_sqnorm_pass<kGK>(const SmallParams&, double*, int64_t, bool, cudaStream_t);
template int launch_sqnorm_pass<kGK>(const BigParams&, double*, int64_t, bool, cudaStream_t);

}  // namespace dpopt

// internal.h -- what the library's translation units share: the launch
// parameter tables, the error helpers and the launchers each unit defines.
//
// The library is four units compiled in parallel: the C ABI and the small
// kernels (dpopt.cu), the bulk-copy kernel (tma.cu) and the step, mixed-
// precision step and squared-norm kernels of one gradient type
// (launch_gk.cu, compiled once per type with -DDPOPT_GK=0|1|2).  Nothing here
// allocates memory.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "dpopt.h"
#include "kernels.cuh"

namespace dpopt {

// Segment tables: one segment (a whole shard or one bucket), or a batch of
// buckets.  The batch table keeps a launch's parameters under 32 KB.
constexpr int kSmallSegs = 1;
constexpr int kSmallPtrs = DPOPT_MAX_REPLICAS;
constexpr int kBigSegs = 128;
constexpr int kBigPtrs = 2048;

using SmallParams = LaunchParams<kSmallSegs, kSmallPtrs>;
using BigParams = LaunchParams<kBigSegs, kBigPtrs>;
static_assert(kMaxGatherDst >= DPOPT_MAX_REPLICAS, "a gather table holds every replica");
static_assert(sizeof(BigParams) <= 32000, "kernel parameters must fit the 32 KB limit");

// One segment as the host sees it.
struct SegDesc {
  const void* const* ptrs;  // n_replicas gradient pointers at the segment start
  int64_t state_off;
  int64_t len;
};

// Error reporting (message kept per host thread for dpopt_last_error).
int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);
// Counts a kernel launch of this host thread (dpopt_launch_count).
void count_launch();
// SM count of the current device, cached per device.
int sm_count(int* out);

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the preceding kernel on the stream is finishing; every library kernel
// begins with pdl_enter() (kernels.cuh), which waits for that kernel before
// any global memory access.  Returns the launch's error code.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Per-gradient-type launchers (launch_gk.cu).  GK: 0 bf16, 1 fp32, 2 fp16.
// p must hold at least one non-empty segment.
template <int GK, int MS, int MP>
int launch_step(const LaunchParams<MS, MP>& p, bool ext, cudaStream_t stream);
// The step over a device-resident segment table (one launch for any number
// of buckets; direct loads only).
template <int GK>
int launch_step_table(const TableParams& p, bool ext, cudaStream_t stream);
// The plain step that also writes the bf16 copy into every buffer of d (the
// fused ZeRO-3 all-gather; one segment).
template <int GK>
int launch_step_gather(const SmallParams& p, const GatherDst& d, cudaStream_t stream);
template <int GK, int MS, int MP>
int launch_amp_step(const LaunchParams<MS, MP>& p, const LossScaleState* state,
                    const double* sqnorm, cudaStream_t stream);
// store_average: also write each element's average to p.master (one
// segment only).
template <int GK, int MS, int MP>
int launch_sqnorm_pass(const LaunchParams<MS, MP>& p, double* partials, int64_t nchunks,
                       bool store_average, cudaStream_t stream);

// Bulk-copy kernel (tma.cu).  tma_eligible: master/m/v 32-byte aligned, the
// other pointers 16-byte aligned, a supported gradient type and two stages of
// replica rows within the shared-memory budget.
bool tma_eligible(const SegDesc* segs, int s0, int s1, int n, int grad_dtype, const float* master,
                  const float* m, const float* v, const void* out);
int run_tma(const SegDesc* segs, int s0, int s1, int n, int grad_dtype, float* master, float* m,
            float* v, void* out, const Hyper& h, cudaStream_t stream);
// Reads and clears the sticky status word of the bounded waits: *timed_out
// is set when a wait gave up since the last call.
int take_wait_status(bool* timed_out);
// The bounded-wait self-test launch (a wait on a barrier nothing completes).
int launch_selftest_wait(long long limit_cycles, cudaStream_t stream);
// Longest bounded wait, in clock cycles (about one second).
constexpr long long kWaitLimitCycles = 2000000000LL;

}  // namespace dpopt

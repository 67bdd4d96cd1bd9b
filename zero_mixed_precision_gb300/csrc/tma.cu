// tma.cu -- launches of the bulk-copy (TMA) staged step kernel, the status
// word of the bounded device-side waits and their self-test.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "tma.cuh"

namespace dpopt {
namespace {

using SmallTma = TmaParams<kSmallSegs, kSmallPtrs>;
using BigTma = TmaParams<kBigSegs, kBigPtrs>;
static_assert(sizeof(BigTma) <= 32000, "kernel parameters must fit the 32 KB limit");

// Shared memory budget for the stage ring of one CTA (two CTAs of 8 consumer
// warps per SM measured best: 6386 GB/s at N = 4 against 4687 GB/s for one
// CTA with five stages).  Two stages of 2048 elements fit for bf16 N <= 6
// and fp32 N <= 3; each of those replica counts has its own kernel.
constexpr uint32_t kTmaSmemBudget = 100 * 1024;
constexpr int kTmaMaxReplicas = 6;

template <int NR, int GK, int W, int MS, int MP>
int launch_tma(const TmaParams<MS, MP>& p, cudaStream_t stream) {
  auto kern = reduce_adam_tma_kernel<NR, GK, W, MS, MP>;
  const size_t dyn = (size_t)p.stages * p.stage_bytes;
  // a function attribute belongs to the current device's context: set on
  // every call (a host-side call, no stream work), so that every device a
  // process drives gets it
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(kTmaSmemBudget + 1024));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  int sms = 0;
  int rc = sm_count(&sms);
  if (rc) return rc;
  int bps = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, kTmaThreads, dyn);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  if (bps < 1) return fail(DPOPT_ERR_UNSUPPORTED, "bulk-copy kernel does not fit an SM");
  const int64_t want = std::max<int64_t>(p.total_tiles, (int64_t)p.nseg);
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * bps));
  e = launch_pdl(kern, grid, kTmaThreads, dyn, stream, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  count_launch();
  return DPOPT_OK;
}

// Width of the consumers' state stores, by measurement on GB300 (256M-element
// shards): 256-bit stores for bf16 N <= 3 (6444 against 6059 GB/s at N = 3)
// and fp32 N = 1; two 16-byte stores above (bf16 N = 4: 6625 against 6356,
// fp32 N = 3: 6615 against 6432).
constexpr int tma_width(int gk, int nr) { return (gk == 0 ? nr <= 3 : nr <= 1) ? 32 : 16; }

template <int GK, int MS, int MP>
int dispatch_tma_gk(const TmaParams<MS, MP>& p, cudaStream_t stream) {
  switch (p.n_rep) {
    case 1: return launch_tma<1, GK, tma_width(GK, 1)>(p, stream);
    case 2: return launch_tma<2, GK, tma_width(GK, 2)>(p, stream);
    case 3: return launch_tma<3, GK, tma_width(GK, 3)>(p, stream);
    default: break;
  }
  if constexpr (GK == 0) {
    switch (p.n_rep) {
      case 4: return launch_tma<4, GK, tma_width(GK, 4)>(p, stream);
      case 5: return launch_tma<5, GK, tma_width(GK, 5)>(p, stream);
      case 6: return launch_tma<6, GK, tma_width(GK, 6)>(p, stream);
      default: break;
    }
  }
  return fail(DPOPT_ERR_UNSUPPORTED, "bulk-copy kernel: no ring for %d replicas", p.n_rep);
}

template <int MS, int MP>
int run_segments_tma(TmaParams<MS, MP>& p, const SegDesc* segs, int s0, int s1, int n,
                     cudaStream_t stream, int grad_dtype) {
  const uint32_t gsize = grad_dtype == DPOPT_GRAD_F32 ? 4u : 2u;
  int64_t tiles = 0;
  int nseg = 0;
  for (int s = s0; s < s1; ++s) {
    const SegDesc& d = segs[s];
    if (d.len == 0) continue;
    TmaSeg& sg = p.seg[nseg];
    sg.first_tile = tiles;
    sg.state_off = d.state_off;
    sg.len = d.len;
    sg.body = d.len & ~(int64_t)(kGroup - 1);
    sg.ptr_base = nseg * n;
    for (int r = 0; r < n; ++r) p.gptr[nseg * n + r] = d.ptrs[r];
    tiles += (sg.body + kTmaTile - 1) / kTmaTile;
    ++nseg;
  }
  if (nseg == 0) return DPOPT_OK;
  p.seg[nseg].first_tile = tiles;
  p.nseg = nseg;
  p.total_tiles = tiles;
  p.stage_bytes = (uint32_t)kTmaTile * ((uint32_t)n * gsize + 12u);
  p.stages = (int)std::min<uint32_t>(kTmaMaxStages, kTmaSmemBudget / p.stage_bytes);
  p.wait_limit = kWaitLimitCycles;
  if (p.stages < 2) return fail(DPOPT_ERR_UNSUPPORTED, "replica rows do not fit two stages");
  if (grad_dtype == DPOPT_GRAD_BF16) return dispatch_tma_gk<0>(p, stream);
  return dispatch_tma_gk<1>(p, stream);
}

template <class P>
void set_common(P& p, float* master, float* m, float* v, void* out, const Hyper& h, int n) {
  p.h = h;
  p.master = master;
  p.m = m;
  p.v = v;
  p.out = (uint16_t*)out;
  p.n_rep = n;
}

}  // namespace

bool tma_eligible(const SegDesc* segs, int s0, int s1, int n, int grad_dtype, const float* master,
                  const float* m, const float* v, const void* out) {
  if (n > kTmaMaxReplicas || grad_dtype == DPOPT_GRAD_F16) return false;
  const uint32_t gsize = grad_dtype == DPOPT_GRAD_F32 ? 4u : 2u;
  if (2u * (uint32_t)kTmaTile * ((uint32_t)n * gsize + 12u) > kTmaSmemBudget) return false;
  auto aligned32 = [](const void* q) { return ((uintptr_t)q & 31u) == 0; };
  for (int s = s0; s < s1; ++s) {
    const SegDesc& d = segs[s];
    if (d.len == 0) continue;
    if (!aligned32(master + d.state_off) || !aligned32(m + d.state_off) ||
        !aligned32(v + d.state_off) || !aligned16((const uint16_t*)out + d.state_off))
      return false;
    for (int r = 0; r < n; ++r)
      if (!aligned16(d.ptrs[r])) return false;
  }
  return true;
}

int run_tma(const SegDesc* segs, int s0, int s1, int n, int grad_dtype, float* master, float* m,
            float* v, void* out, const Hyper& h, cudaStream_t stream) {
  if (s1 - s0 == 1) {
    SmallTma p{};
    set_common(p, master, m, v, out, h, n);
    return run_segments_tma(p, segs, s0, s1, n, stream, grad_dtype);
  }
  static thread_local BigTma p;  // 20 KB: kept off the stack
  std::memset(&p, 0, sizeof p);
  set_common(p, master, m, v, out, h, n);
  return run_segments_tma(p, segs, s0, s1, n, stream, grad_dtype);
}

int take_wait_status(bool* timed_out) {
  unsigned int st = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&st, g_status, sizeof st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  *timed_out = st != 0;
  if (st != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
  }
  return DPOPT_OK;
}

int launch_selftest_wait(long long limit_cycles, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_cycles);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  count_launch();
  return DPOPT_OK;
}

}  // namespace dpopt

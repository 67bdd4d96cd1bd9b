// dpopt.cu -- the C ABI (include/dpopt.h): argument checks, the step's
// scalars, segment tables, the kernel choice and the small kernels (loss-scale
// bookkeeping, the norm's final sum, the all-gather).  The step, loss-scaled
// step and norm kernels live in launch_gk.cu, the bulk-copy kernel in tma.cu.
// No memory is allocated here.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "dpopt.h"
#include "control.cuh"
#include "gather.cuh"
#include "internal.h"
#include "norm.cuh"

namespace dpopt {
namespace {

constexpr int kMaxDevices = 64;

// Under DPOPT_KERNEL_AUTO the bulk-copy kernel carries the step where it
// measured faster than the direct-load kernel on GB300 (256M-element shards):
// fp32 N = 2 (6431 against 6163 GB/s) and fp32 N = 3 (6567 against 6218).
// Elsewhere the direct-load kernel is as fast or faster (bf16 N = 3: 6475
// against 6436; bf16 N = 1: 6439 against 6006; bf16 N = 4..6 by 0..4%).
bool auto_bulk(int n, int grad_dtype) {
  return grad_dtype == DPOPT_GRAD_F32 && (n == 2 || n == 3);
}

std::atomic<int> g_policy{DPOPT_KERNEL_AUTO};
std::atomic<int> g_gather_policy{DPOPT_GATHER_AUTO};

thread_local char g_last_error[512];
thread_local int64_t g_launches = 0;

struct DeviceCache {
  std::atomic<int> sms[kMaxDevices];
};
DeviceCache g_dev;

#ifdef DPOPT_DEBUG_BOUNDS
// Bounds-checked build: the word every failed index check sets (bit 0), read
// and cleared by dpopt_stream_status().  Its device address is looked up once
// per device; the kernels receive it in their Hyper block.
__device__ unsigned int g_bounds_status;
std::once_flag g_bounds_once[kMaxDevices];
unsigned int* g_bounds_addr[kMaxDevices];
cudaError_t g_bounds_err[kMaxDevices];

unsigned int* bounds_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_bounds_once[dev], [dev] {
    void* ptr = nullptr;
    g_bounds_err[dev] = cudaGetSymbolAddress(&ptr, g_bounds_status);
    g_bounds_addr[dev] = static_cast<unsigned int*>(ptr);
  });
  return g_bounds_err[dev] == cudaSuccess ? g_bounds_addr[dev] : nullptr;
}

__global__ void bounds_selftest_kernel(Hyper h, int64_t len) {
  // an index one past the end: the check fails, sets the word, and nothing
  // is accessed
  const int64_t idx = len;
  (void)dbg_ok(h, idx < len);
}
#endif

}  // namespace

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DPOPT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

void count_launch() { ++g_launches; }

int sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DPOPT_ERR_UNSUPPORTED, "device index too large");
  int s = g_dev.sms[dev].load(std::memory_order_relaxed);
  if (s == 0) {
    e = cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    g_dev.sms[dev].store(s, std::memory_order_relaxed);
  }
  *out = s;
  return DPOPT_OK;
}

namespace {

bool is_finite(float x) { return std::isfinite(x); }

// The span of shard elements a call may touch, for the bounds-checked build's
// kernels (a no-op in a release build).
void set_span(Hyper& h, int64_t lo, int64_t hi) {
#ifdef DPOPT_DEBUG_BOUNDS
  h.dbg_lo = lo;
  h.dbg_hi = hi;
#else
  (void)h; (void)lo; (void)hi;
#endif
}

// Scalars of step t, in fp64 on the host, split into fp32 pairs.
Hyper make_hyper(float lr, float beta1, float beta2, float eps, int64_t step, int n) {
  Hyper h{};
  const double b1 = beta1, b2 = beta2;
  auto split = [](double x, float& hi, float& lo) {
    hi = (float)x;
    lo = (float)(x - (double)hi);
  };
  h.beta1 = beta1;
  h.beta2 = beta2;
  split(1.0 - b1, h.c1_hi, h.c1_lo);
  split(1.0 - b2, h.c2_hi, h.c2_lo);
  const double bc1 = 1.0 - std::pow(b1, (double)step);
  const double bc2 = 1.0 - std::pow(b2, (double)step);
  split((double)lr / bc1, h.a_hi, h.a_lo);
  split(1.0 / std::sqrt(bc2), h.b_hi, h.b_lo);
  h.eps = eps;
  h.n_f = (float)n;
  h.inv_n = ((n & (n - 1)) == 0) ? (float)(1.0 / n) : 0.f;
  h.k_hi = 1.f;
  h.k_lo = 0.f;
  h.sqnorm = nullptr;
  h.max_norm = 0.0;
  h.unscale = 1.f;
  h.lr = lr;
  h.scale_dev = nullptr;
  h.lr_dev = nullptr;
  h.wd = 0.f;
#ifdef DPOPT_DEBUG_BOUNDS
  h.dbg_status = bounds_status_word();
  h.dbg_lo = 0;
  h.dbg_hi = INT64_MAX;
#endif
  return h;
}

int check_hyper(float lr, float beta1, float beta2, float eps, int64_t step) {
  if (!is_finite(lr)) return fail(DPOPT_ERR_INVALID_ARG, "lr must be finite");
  if (!is_finite(beta1) || beta1 < 0.f || beta1 >= 1.f)
    return fail(DPOPT_ERR_INVALID_ARG, "beta1 must lie in [0, 1)");
  if (!is_finite(beta2) || beta2 < 0.f || beta2 >= 1.f)
    return fail(DPOPT_ERR_INVALID_ARG, "beta2 must lie in [0, 1)");
  if (!is_finite(eps) || eps < 0.f) return fail(DPOPT_ERR_INVALID_ARG, "eps must be finite, >= 0");
  if (step < 1) return fail(DPOPT_ERR_INVALID_ARG, "step must be >= 1");
  return DPOPT_OK;
}

int check_replicas(int n_replicas, int grad_dtype) {
  if (n_replicas < 1) return fail(DPOPT_ERR_INVALID_ARG, "n_replicas must be >= 1");
  if (n_replicas > DPOPT_MAX_REPLICAS)
    return fail(DPOPT_ERR_UNSUPPORTED, "n_replicas %d exceeds %d", n_replicas, DPOPT_MAX_REPLICAS);
  if (grad_dtype != DPOPT_GRAD_BF16 && grad_dtype != DPOPT_GRAD_F32 &&
      grad_dtype != DPOPT_GRAD_F16)
    return fail(DPOPT_ERR_INVALID_ARG, "unknown grad_dtype %d", grad_dtype);
  return DPOPT_OK;
}

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi; }

// The four state/output ranges of elements [off, off+len) of the shard arrays.
int check_states(float* master, float* m, float* v, void* out, int64_t lo_elem, int64_t hi_elem,
                 Range st[4]) {
  if (!master || !m || !v || !out)
    return fail(DPOPT_ERR_INVALID_ARG, "master, m, v and param_bf16_out must be non-null");
  if (((uintptr_t)master | (uintptr_t)m | (uintptr_t)v) & 3u)
    return fail(DPOPT_ERR_INVALID_ARG, "fp32 state pointers must be 4-byte aligned");
  if ((uintptr_t)out & 1u) return fail(DPOPT_ERR_INVALID_ARG, "bf16 output must be 2-byte aligned");
  st[0] = {(uintptr_t)(master + lo_elem), (uintptr_t)(master + hi_elem)};
  st[1] = {(uintptr_t)(m + lo_elem), (uintptr_t)(m + hi_elem)};
  st[2] = {(uintptr_t)(v + lo_elem), (uintptr_t)(v + hi_elem)};
  st[3] = {(uintptr_t)((uint16_t*)out + lo_elem), (uintptr_t)((uint16_t*)out + hi_elem)};
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(st[i], st[j]))
        return fail(DPOPT_ERR_INVALID_ARG, "state/output arrays overlap");
  return DPOPT_OK;
}

int check_grad(const void* p, int64_t len, size_t esize, const Range* avoid, int navoid) {
  if (!p) return fail(DPOPT_ERR_INVALID_ARG, "null gradient pointer");
  if ((uintptr_t)p % esize) return fail(DPOPT_ERR_INVALID_ARG, "misaligned gradient pointer");
  Range g{(uintptr_t)p, (uintptr_t)p + (uintptr_t)len * esize};
  for (int i = 0; i < navoid; ++i)
    if (overlaps(g, avoid[i]))
      return fail(DPOPT_ERR_INVALID_ARG, "a gradient buffer overlaps a state, output or scratch "
                                         "range");
  return DPOPT_OK;
}

// The step for grad_dtype: the per-type launchers pick the kernel for N.
template <int MS, int MP>
int dispatch(const LaunchParams<MS, MP>& p, int grad_dtype, bool ext, cudaStream_t stream) {
  if (grad_dtype == DPOPT_GRAD_BF16) return launch_step<0>(p, ext, stream);
  if (grad_dtype == DPOPT_GRAD_F16) return launch_step<2>(p, ext, stream);
  return launch_step<1>(p, ext, stream);
}

// Fill the segment table of one LaunchParams from segments [s0, s1);
// `unit` is the element count one index of Seg::first_group stands for (8 for
// the update's groups, kNormChunk for the norm's chunks).  A segment's vector
// level: 2 when master/m/v (and fp32 gradients) are 32-byte aligned and
// everything else 16-byte aligned (one 256-bit access per state array per
// thread), 1 when everything is 16-byte aligned, else 0 (one element at a
// time).  Null state pointers (the norm) count as aligned.  Returns the index
// total (0 when every segment is empty).
int vec_level(const float* master, const float* m, const float* v, const uint16_t* out,
              const SegDesc& d, int n, int grad_dtype) {
  auto aligned32 = [](const void* q) { return ((uintptr_t)q & 31u) == 0; };
  bool v16 = aligned16(master + d.state_off) && aligned16(m + d.state_off) &&
             aligned16(v + d.state_off) && aligned16(out + d.state_off);
  bool v32 = aligned32(master + d.state_off) && aligned32(m + d.state_off) &&
             aligned32(v + d.state_off);
  for (int r = 0; r < n; ++r) {
    v16 = v16 && aligned16(d.ptrs[r]);
    if (grad_dtype == DPOPT_GRAD_F32) v32 = v32 && aligned32(d.ptrs[r]);
  }
  return v16 ? (v32 ? 2 : 1) : 0;
}

template <int MS, int MP>
int64_t fill_segments(LaunchParams<MS, MP>& p, const SegDesc* segs, int s0, int s1, int n,
                      int64_t unit, int grad_dtype) {
  int64_t units = 0;
  int nseg = 0;
  for (int s = s0; s < s1; ++s) {
    const SegDesc& d = segs[s];
    if (d.len == 0) continue;
    Seg& sg = p.seg[nseg];
    sg.first_group = units;
    sg.state_off = d.state_off;
    sg.len = d.len;
    sg.ptr_base = nseg * n;
    for (int r = 0; r < n; ++r) p.gptr[nseg * n + r] = d.ptrs[r];
    sg.vec = vec_level(p.master, p.m, p.v, p.out, d, n, grad_dtype);
    units += (d.len + unit - 1) / unit;
    ++nseg;
  }
  p.seg[nseg].first_group = units;
  p.seg[nseg].len = 0;
  p.nseg = nseg;
  p.total_groups = units;
  return units;
}

template <int MS, int MP>
int run_segments(LaunchParams<MS, MP>& p, const SegDesc* segs, int s0, int s1, int n,
                 cudaStream_t stream, int grad_dtype, bool ext) {
  if (fill_segments(p, segs, s0, s1, n, kGroup, grad_dtype) == 0) return DPOPT_OK;
  return dispatch(p, grad_dtype, ext, stream);
}

// Kernel choice: the bulk-copy kernel where it applies and the policy allows,
// else the direct-load kernel.
bool use_tma(const SegDesc* segs, int s0, int s1, int n, int grad_dtype, float* master,
             float* m, float* v, void* out) {
  const int pol = g_policy.load(std::memory_order_relaxed);
  if (pol == DPOPT_KERNEL_DIRECT) return false;
  if (!tma_eligible(segs, s0, s1, n, grad_dtype, master, m, v, out)) return false;
  if (pol == DPOPT_KERNEL_BULK) return true;
  return auto_bulk(n, grad_dtype);
}

int run(const SegDesc* segs, int nsegs, int grad_dtype, int n, float* master, float* m, float* v,
        void* out, const Hyper& h, bool ext, cudaStream_t stream) {
  if (nsegs == 1) {
    if (!ext && use_tma(segs, 0, 1, n, grad_dtype, master, m, v, out))
      return run_tma(segs, 0, 1, n, grad_dtype, master, m, v, out, h, stream);
    SmallParams p{};
    p.h = h;
    p.master = master; p.m = m; p.v = v; p.out = (uint16_t*)out;
    p.n_rep = n;
    return run_segments(p, segs, 0, 1, n, stream, grad_dtype, ext);
  }
  const int per_launch = std::min(kBigSegs, kBigPtrs / n);
  for (int s0 = 0; s0 < nsegs; s0 += per_launch) {
    const int s1 = std::min(nsegs, s0 + per_launch);
    int rc;
    if (!ext && use_tma(segs, s0, s1, n, grad_dtype, master, m, v, out)) {
      rc = run_tma(segs, s0, s1, n, grad_dtype, master, m, v, out, h, stream);
    } else {
      static thread_local BigParams p;  // 20 KB: kept off the stack
      std::memset(&p, 0, sizeof p);
      p.h = h;
      p.master = master; p.m = m; p.v = v; p.out = (uint16_t*)out;
      p.n_rep = n;
      rc = run_segments(p, segs, s0, s1, n, stream, grad_dtype, ext);
    }
    if (rc) return rc;
  }
  return DPOPT_OK;
}

// ---------------------------------------------------------------------------
// squared-norm pre-pass
// ---------------------------------------------------------------------------

int64_t norm_chunks(const SegDesc* segs, int nsegs) {
  int64_t c = 0;
  for (int s = 0; s < nsegs; ++s) c += (segs[s].len + kNormChunk - 1) / kNormChunk;
  return c;
}

template <int MS, int MP>
int launch_sqnorm(LaunchParams<MS, MP>& p, int64_t nchunks, double* partials, int grad_dtype,
                  bool store_average, cudaStream_t stream) {
  if (grad_dtype == DPOPT_GRAD_BF16)
    return launch_sqnorm_pass<0>(p, partials, nchunks, store_average, stream);
  if (grad_dtype == DPOPT_GRAD_F16)
    return launch_sqnorm_pass<2>(p, partials, nchunks, store_average, stream);
  return launch_sqnorm_pass<1>(p, partials, nchunks, store_average, stream);
}

// Squared norm of segments [0, nsegs) into *out (device), partials in scratch.
// avg_out (one segment only): also store each element's average there.
// The norm pass over one segment: its chunk partials from `partials` on, each
// element's average stored at its shard offset in avg_out when given.
int norm_segment(const SegDesc& seg, int grad_dtype, int n, const Hyper& h, double* partials,
                 float* avg_out, cudaStream_t stream, int64_t* chunks_out) {
  SmallParams p{};
  p.h = h;
  p.n_rep = n;
  p.master = avg_out;  // the average's destination (null: norm only)
  const int64_t chunks = fill_segments(p, &seg, 0, 1, n, kNormChunk, grad_dtype);
  *chunks_out = chunks;
  return chunks ? launch_sqnorm(p, chunks, partials, grad_dtype, avg_out != nullptr, stream)
                : DPOPT_OK;
}

// The ordered sum of `count` chunk partials (double-float pairs, one per 8-byte
// slot) into *out.
int norm_finish(const double* partials, int64_t count, double* out, cudaStream_t stream) {
  cudaError_t e = launch_pdl(sqnorm_finish_kernel, 1, kFinishThreads, 0, stream,
                             reinterpret_cast<const DFloat*>(partials), count, out);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  ++g_launches;
  return DPOPT_OK;
}

int run_sqnorm(const SegDesc* segs, int nsegs, int grad_dtype, int n, const Hyper& h,
               double* partials, double* out, cudaStream_t stream, float* avg_out = nullptr) {
  if (avg_out && nsegs != 1)
    return fail(DPOPT_ERR_UNSUPPORTED, "the averaged gradient is stored for one segment only");
  int64_t done = 0;
  if (nsegs == 1) {
    int rc = norm_segment(segs[0], grad_dtype, n, h, partials, avg_out, stream, &done);
    if (rc) return rc;
  } else {
    const int per_launch = std::min(kBigSegs, kBigPtrs / n);
    for (int s0 = 0; s0 < nsegs; s0 += per_launch) {
      const int s1 = std::min(nsegs, s0 + per_launch);
      static thread_local BigParams p;
      std::memset(&p, 0, sizeof p);
      p.h = h;
      p.n_rep = n;
      const int64_t chunks = fill_segments(p, segs, s0, s1, n, kNormChunk, grad_dtype);
      int rc = chunks ? launch_sqnorm(p, chunks, partials + done, grad_dtype, false, stream)
                      : DPOPT_OK;
      if (rc) return rc;
      done += chunks;
    }
  }
  return norm_finish(partials, done, out, stream);
}


// The segments of a full-buffer call (one: the whole shard), checked.  `avoid`
// lists extra ranges the gradients must not overlap (states, outputs, scratch).
int build_full(const void* const* grads, int grad_dtype, int n_replicas, int64_t numel,
               int shard_rank, int64_t bucket_elems, const Range* avoid, int navoid,
               const void* ptrs_out[DPOPT_MAX_REPLICAS], int64_t* S_out) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  if (!grads) return fail(DPOPT_ERR_INVALID_ARG, "grads must be non-null");
  if (numel < 0 || numel % n_replicas != 0)
    return fail(DPOPT_ERR_INVALID_ARG, "numel must be >= 0 and a multiple of n_replicas");
  if (shard_rank < 0 || shard_rank >= n_replicas)
    return fail(DPOPT_ERR_INVALID_ARG, "shard_rank must lie in [0, n_replicas)");
  if (bucket_elems < 1) return fail(DPOPT_ERR_INVALID_ARG, "bucket_elems must be >= 1");
  const int64_t S = numel / n_replicas;
  const int64_t base = (int64_t)shard_rank * S;
  const size_t esize = grad_dtype == DPOPT_GRAD_F32 ? 4 : 2;
  *S_out = S;
  if (S == 0) return DPOPT_OK;
  for (int r = 0; r < n_replicas; ++r) {
    if (!grads[r]) return fail(DPOPT_ERR_INVALID_ARG, "null gradient pointer");
    ptrs_out[r] = (const char*)grads[r] + (size_t)base * esize;
    rc = check_grad(ptrs_out[r], S, esize, avoid, navoid);
    if (rc) return rc;
  }
  return DPOPT_OK;
}

// The segments of a batched-bucket call, checked; lo/hi receive the span of
// shard elements they update.
int build_buckets(const void* const* slice_table, int grad_dtype, int n_replicas,
                  const int64_t* offsets, const int64_t* lens, int64_t n_buckets,
                  std::vector<SegDesc>& segs, int64_t* lo_out, int64_t* hi_out) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  if (n_buckets < 0) return fail(DPOPT_ERR_INVALID_ARG, "n_buckets must be >= 0");
  segs.clear();
  *lo_out = *hi_out = 0;
  if (n_buckets == 0) return DPOPT_OK;
  if (!slice_table || !offsets || !lens)
    return fail(DPOPT_ERR_INVALID_ARG, "slice_table, offsets and lens must be non-null");
  if (n_buckets > (int64_t)1 << 30) return fail(DPOPT_ERR_UNSUPPORTED, "too many buckets");
  int64_t lo = INT64_MAX, hi = 0;
  std::vector<std::pair<int64_t, int64_t>> spans;
  spans.reserve((size_t)n_buckets);
  for (int64_t b = 0; b < n_buckets; ++b) {
    if (offsets[b] < 0 || lens[b] < 0 || offsets[b] > INT64_MAX - lens[b])
      return fail(DPOPT_ERR_INVALID_ARG, "bucket %lld: bad offset/len", (long long)b);
    if (lens[b] == 0) continue;
    lo = std::min(lo, offsets[b]);
    hi = std::max(hi, offsets[b] + lens[b]);
    spans.emplace_back(offsets[b], offsets[b] + lens[b]);
  }
  if (spans.empty()) return DPOPT_OK;
  std::sort(spans.begin(), spans.end());
  for (size_t i = 1; i < spans.size(); ++i)
    if (spans[i].first < spans[i - 1].second)
      return fail(DPOPT_ERR_INVALID_ARG, "buckets overlap");
  segs.reserve((size_t)n_buckets);
  for (int64_t b = 0; b < n_buckets; ++b) {
    if (lens[b] == 0) continue;
    segs.push_back(SegDesc{slice_table + b * n_replicas, offsets[b], lens[b]});
  }
  *lo_out = lo;
  *hi_out = hi;
  return DPOPT_OK;
}

// Puts the buckets in shard order and joins those whose slices continue one
// another: bucket b + 1 starts where bucket b ends, in the shard and in every
// replica's gradient memory (the buckets of a flat, contiguous gradient
// buffer), whatever order the caller listed them in.  The step is
// elementwise, so the joined segments give the same bits in fewer segments
// (274 resident 4M-element buckets become one segment and one launch), and
// the norm's chunk partials then follow the shard order, so its bits do not
// depend on the listing order either.  Offsets are distinct (overlapping
// buckets were refused).
void coalesce(std::vector<SegDesc>& segs, int n, int grad_dtype) {
  std::sort(segs.begin(), segs.end(),
            [](const SegDesc& a, const SegDesc& b) { return a.state_off < b.state_off; });
  const uintptr_t esize = grad_dtype == DPOPT_GRAD_F32 ? 4 : 2;
  size_t w = 0;
  for (size_t s = 0; s < segs.size(); ++s) {
    if (w > 0) {
      SegDesc& a = segs[w - 1];
      const SegDesc& b = segs[s];
      bool joins = b.state_off == a.state_off + a.len;
      for (int r = 0; joins && r < n; ++r)
        joins = (uintptr_t)b.ptrs[r] == (uintptr_t)a.ptrs[r] + (uintptr_t)a.len * esize;
      if (joins) {
        a.len += b.len;
        continue;
      }
    }
    segs[w++] = segs[s];
  }
  segs.resize(w);
}

int check_bucket_grads(const std::vector<SegDesc>& segs, int n, int grad_dtype, const Range* avoid,
                       int navoid) {
  const size_t esize = grad_dtype == DPOPT_GRAD_F32 ? 4 : 2;
  for (const SegDesc& d : segs)
    for (int r = 0; r < n; ++r) {
      int rc = check_grad(d.ptrs[r], d.len, esize, avoid, navoid);
      if (rc) return rc;
    }
  return DPOPT_OK;
}

// Step options (null: plain Adam) -> the EXT fields of Hyper.  Returns
// whether the extended kernel is needed.
int apply_options(const dpopt_step_options* o, float lr, Hyper& h, bool* ext) {
  *ext = false;
  if (!o) return DPOPT_OK;
  if (!std::isfinite(o->weight_decay) || o->weight_decay < 0.f)
    return fail(DPOPT_ERR_INVALID_ARG, "weight_decay must be finite and >= 0");
  if (!std::isfinite(o->max_grad_norm) || o->max_grad_norm < 0.f)
    return fail(DPOPT_ERR_INVALID_ARG, "max_grad_norm must be finite and >= 0");
  if (!std::isfinite(o->grad_unscale) || o->grad_unscale < 0.f)
    return fail(DPOPT_ERR_INVALID_ARG, "grad_unscale must be finite and >= 0");
  if (o->max_grad_norm > 0.f) {
    if (!o->grad_sqnorm || ((uintptr_t)o->grad_sqnorm & 7u))
      return fail(DPOPT_ERR_INVALID_ARG, "clipping needs an 8-byte aligned grad_sqnorm");
    h.sqnorm = o->grad_sqnorm;
    h.max_norm = (double)o->max_grad_norm;
  }
  const double k = 1.0 - (double)lr * (double)o->weight_decay;
  h.k_hi = (float)k;
  h.k_lo = (float)(k - (double)h.k_hi);
  h.unscale = o->grad_unscale == 0.f ? 1.f : o->grad_unscale;
  *ext = true;
  return DPOPT_OK;
}

int full_impl(const void* const* grads, int grad_dtype, int n_replicas, int64_t numel,
              int shard_rank, int64_t bucket_elems, float* master, float* m, float* v, void* out,
              float lr, float beta1, float beta2, float eps, int64_t step,
              const dpopt_step_options* opts, cudaStream_t stream) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  rc = check_hyper(lr, beta1, beta2, eps, step);
  if (rc) return rc;
  Hyper h = make_hyper(lr, beta1, beta2, eps, step, n_replicas);
  bool ext = false;
  rc = apply_options(opts, lr, h, &ext);
  if (rc) return rc;
  if (numel > 0 && numel % n_replicas == 0 && numel / n_replicas > 0) {
    Range st[4];
    rc = check_states(master, m, v, out, 0, numel / n_replicas, st);
    if (rc) return rc;
    const void* ptrs[DPOPT_MAX_REPLICAS];
    int64_t S = 0;
    rc = build_full(grads, grad_dtype, n_replicas, numel, shard_rank, bucket_elems, st, 4, ptrs,
                    &S);
    if (rc) return rc;
    // Every contribution is resident and the buckets tile the shard
    // contiguously, so the whole shard is one segment: bucket_elems changes
    // neither the addresses nor the result, only what the iterator reports.
    SegDesc seg{ptrs, 0, S};
    set_span(h, 0, S);
    return run(&seg, 1, grad_dtype, n_replicas, master, m, v, out, h, ext, stream);
  }
  const void* ptrs[DPOPT_MAX_REPLICAS];
  int64_t S = 0;
  return build_full(grads, grad_dtype, n_replicas, numel, shard_rank, bucket_elems, nullptr, 0,
                    ptrs, &S);
}

int buckets_impl(const void* const* slice_table, int grad_dtype, int n_replicas,
                 const int64_t* offsets, const int64_t* lens, int64_t n_buckets, float* master,
                 float* m, float* v, void* out, float lr, float beta1, float beta2, float eps,
                 int64_t step, const dpopt_step_options* opts, cudaStream_t stream) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  rc = check_hyper(lr, beta1, beta2, eps, step);
  if (rc) return rc;
  Hyper h = make_hyper(lr, beta1, beta2, eps, step, n_replicas);
  bool ext = false;
  rc = apply_options(opts, lr, h, &ext);
  if (rc) return rc;
  std::vector<SegDesc> segs;
  int64_t lo = 0, hi = 0;
  rc = build_buckets(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets, segs, &lo, &hi);
  if (rc || segs.empty()) return rc;
  Range st[4];
  rc = check_states(master, m, v, out, lo, hi, st);
  if (rc) return rc;
  rc = check_bucket_grads(segs, n_replicas, grad_dtype, st, 4);
  if (rc) return rc;
  set_span(h, lo, hi);
  coalesce(segs, n_replicas, grad_dtype);
  return run(segs.data(), (int)segs.size(), grad_dtype, n_replicas, master, m, v, out, h, ext,
             stream);
}

// Bytes of a device-resident launch table for nb buckets of n replicas: nb + 1
// segment records (the last closes the prefix sums), then nb * n pointers.
int64_t table_bytes_for(int n, int64_t nb) {
  return (int64_t)sizeof(Seg) * (nb + 1) + (int64_t)sizeof(void*) * nb * n;
}

// The batched-bucket step in one launch for every bucket, however many:
// buckets that continue one another are joined first; if what remains fits
// one launch's parameter space it runs from there, else its launch table is
// written into the caller-owned device memory and the kernel reads it there.
int table_impl(const void* const* slice_table, int grad_dtype, int n_replicas,
               const int64_t* offsets, const int64_t* lens, int64_t n_buckets, float* master,
               float* m, float* v, void* out, float lr, float beta1, float beta2, float eps,
               int64_t step, const dpopt_step_options* opts, void* table, int64_t table_bytes,
               cudaStream_t stream) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  rc = check_hyper(lr, beta1, beta2, eps, step);
  if (rc) return rc;
  Hyper h = make_hyper(lr, beta1, beta2, eps, step, n_replicas);
  bool ext = false;
  rc = apply_options(opts, lr, h, &ext);
  if (rc) return rc;
  if (n_buckets < 0 || n_buckets > ((int64_t)1 << 30))
    return fail(DPOPT_ERR_INVALID_ARG, "n_buckets must lie in [0, 2^30]");
  const int64_t need = table_bytes_for(n_replicas, n_buckets);
  if (n_buckets > 0 && (!table || ((uintptr_t)table & 15u)))
    return fail(DPOPT_ERR_INVALID_ARG, "table must be a non-null, 16-byte aligned pointer");
  if (n_buckets > 0 && table_bytes < need)
    return fail(DPOPT_ERR_INVALID_ARG, "table holds %lld bytes, %lld needed",
                (long long)table_bytes, (long long)need);
  std::vector<SegDesc> segs;
  int64_t lo = 0, hi = 0;
  rc = build_buckets(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets, segs, &lo, &hi);
  if (rc || segs.empty()) return rc;
  Range avoid[5];
  rc = check_states(master, m, v, out, lo, hi, avoid);
  if (rc) return rc;
  const int64_t bytes = table_bytes_for(n_replicas, (int64_t)segs.size());
  avoid[4] = {(uintptr_t)table, (uintptr_t)table + (uintptr_t)bytes};
  for (int i = 0; i < 4; ++i)
    if (overlaps(avoid[4], avoid[i]))
      return fail(DPOPT_ERR_INVALID_ARG, "the table overlaps a state or output range");
  rc = check_bucket_grads(segs, n_replicas, grad_dtype, avoid, 5);
  if (rc) return rc;
  set_span(h, lo, hi);
  coalesce(segs, n_replicas, grad_dtype);
  if ((int64_t)segs.size() <= kBigSegs && (int64_t)segs.size() * n_replicas <= kBigPtrs)
    // the joined buckets fit one launch's parameter space: no table needed
    return run(segs.data(), (int)segs.size(), grad_dtype, n_replicas, master, m, v, out, h, ext,
               stream);

  // The records and pointers, packed on the host.  A copy from pageable host
  // memory returns once the bytes have left this buffer, so it is reused by
  // this thread's next call without waiting for the device.  A captured graph
  // would instead read the buffer at every replay, after later calls have
  // rewritten it: under capture the call is refused before anything is
  // enqueued.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing(stream, &cap);
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone)
    return fail(DPOPT_ERR_UNSUPPORTED,
                "the launch table is copied from reused host memory, which a captured graph "
                "cannot replay: capture buckets that fit one launch (%d segments, %d slice "
                "pointers)", kBigSegs, kBigPtrs);
  const int nseg = (int)segs.size();
  const int64_t used = table_bytes_for(n_replicas, nseg);
  static thread_local std::vector<unsigned char> staging;
  staging.assign((size_t)used, 0);
  Seg* rec = reinterpret_cast<Seg*>(staging.data());
  const void** ptrs = reinterpret_cast<const void**>(staging.data() + sizeof(Seg) * (nseg + 1));
  const uint16_t* out16 = static_cast<const uint16_t*>(out);
  int64_t units = 0;
  bool wide = true;
  for (int s = 0; s < nseg; ++s) {
    const SegDesc& d = segs[s];
    rec[s].first_group = units;
    rec[s].state_off = d.state_off;
    rec[s].len = d.len;
    rec[s].ptr_base = s * n_replicas;
    rec[s].vec = vec_level(master, m, v, out16, d, n_replicas, grad_dtype);
    wide = wide && rec[s].vec != 1;
    for (int r = 0; r < n_replicas; ++r) ptrs[(int64_t)s * n_replicas + r] = d.ptrs[r];
    units += (d.len + kGroup - 1) / kGroup;
  }
  rec[nseg].first_group = units;
  cudaError_t e = cudaMemcpyAsync(table, staging.data(), (size_t)used, cudaMemcpyHostToDevice,
                                  stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (launch table)");

  TableParams p{};
  p.h = h;
  p.master = master; p.m = m; p.v = v; p.out = (uint16_t*)out;
  p.total_groups = units;
  p.n_rep = n_replicas;
  p.nseg = nseg;
  p.seg = static_cast<const Seg*>(table);
  p.gptr = reinterpret_cast<const void* const*>(static_cast<const unsigned char*>(table) +
                                                sizeof(Seg) * (nseg + 1));
  p.wide = wide ? 1 : 0;
  if (grad_dtype == DPOPT_GRAD_BF16) return launch_step_table<0>(p, ext, stream);
  if (grad_dtype == DPOPT_GRAD_F16) return launch_step_table<2>(p, ext, stream);
  return launch_step_table<1>(p, ext, stream);
}

int check_norm_outputs(double* sqnorm_out, void* scratch, int64_t scratch_bytes, int64_t chunks,
                       Range avoid[2]) {
  if (!sqnorm_out || ((uintptr_t)sqnorm_out & 7u))
    return fail(DPOPT_ERR_INVALID_ARG, "sqnorm_out must be a non-null, 8-byte aligned pointer");
  if (chunks > 0 && (!scratch || ((uintptr_t)scratch & 7u)))
    return fail(DPOPT_ERR_INVALID_ARG, "scratch must be a non-null, 8-byte aligned pointer");
  if (scratch_bytes < chunks * 8)
    return fail(DPOPT_ERR_INVALID_ARG, "scratch holds %lld bytes, %lld needed",
                (long long)scratch_bytes, (long long)(chunks * 8));
  avoid[0] = {(uintptr_t)sqnorm_out, (uintptr_t)(sqnorm_out + 1)};
  avoid[1] = {(uintptr_t)scratch, (uintptr_t)scratch + (uintptr_t)(chunks * 8)};
  if (chunks > 0 && overlaps(avoid[0], avoid[1]))
    return fail(DPOPT_ERR_INVALID_ARG, "sqnorm_out lies inside the scratch partials");
  return DPOPT_OK;
}

int finish_empty_norm(double* sqnorm_out, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(sqnorm_out, 0, sizeof(double), stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return DPOPT_OK;
}

// The full-buffer squared norm: with `state` the unscale is 1/state->scale
// (read on the device), else grad_unscale (0: 1); with avg_out each element's
// average is also stored there (S floats, 4-byte aligned; the vector paths
// want 16 or 32 bytes).
int full_norm_impl(const void* const* grads, int grad_dtype, int n_replicas, int64_t numel,
                   int shard_rank, float grad_unscale, const LossScaleState* state,
                   float* avg_out, double* sqnorm_out, void* scratch, int64_t scratch_bytes,
                   cudaStream_t stream) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  if (!std::isfinite(grad_unscale) || grad_unscale < 0.f)
    return fail(DPOPT_ERR_INVALID_ARG, "grad_unscale must be finite and >= 0");
  if (numel < 0 || numel % n_replicas != 0)
    return fail(DPOPT_ERR_INVALID_ARG, "numel must be >= 0 and a multiple of n_replicas");
  const int64_t S = numel / n_replicas;
  const int64_t chunks = (S + kNormChunk - 1) / kNormChunk;
  Range avoid[3];
  rc = check_norm_outputs(sqnorm_out, scratch, scratch_bytes, chunks, avoid);
  if (rc) return rc;
  int navoid = chunks ? 2 : 1;
  if (avg_out && S > 0) {
    if ((uintptr_t)avg_out & 3u) return fail(DPOPT_ERR_INVALID_ARG, "avg_out must be 4-byte aligned");
    const Range a{(uintptr_t)avg_out, (uintptr_t)(avg_out + S)};
    for (int i = 0; i < navoid; ++i)
      if (overlaps(a, avoid[i]))
        return fail(DPOPT_ERR_INVALID_ARG, "avg_out overlaps sqnorm_out or the scratch partials");
    avoid[navoid++] = a;
  }
  const void* ptrs[DPOPT_MAX_REPLICAS];
  int64_t S2 = 0;
  rc = build_full(grads, grad_dtype, n_replicas, numel, shard_rank, 1, avoid, navoid, ptrs, &S2);
  if (rc) return rc;
  if (S == 0) return finish_empty_norm(sqnorm_out, stream);
  Hyper h = make_hyper(1.f, 0.f, 0.f, 0.f, 1, n_replicas);
  h.unscale = grad_unscale == 0.f ? 1.f : grad_unscale;
  if (state) h.scale_dev = &state->scale;
  set_span(h, 0, S);
  SegDesc seg{ptrs, 0, S};
  return run_sqnorm(&seg, 1, grad_dtype, n_replicas, h, (double*)scratch, sqnorm_out, stream,
                    avg_out);
}

// ---------------------------------------------------------------------------
// mixed-precision step with dynamic loss scaling
// ---------------------------------------------------------------------------

static_assert(sizeof(LossScaleState) == sizeof(dpopt_loss_scale_state), "state layout");
static_assert(sizeof(LossScaleConfig) == sizeof(dpopt_loss_scale_config), "config layout");

int check_scale_config(const dpopt_loss_scale_config* cfg, LossScaleConfig* out) {
  if (!cfg) return fail(DPOPT_ERR_INVALID_ARG, "loss-scale config must be non-null");
  if (!std::isfinite(cfg->init_scale) || cfg->init_scale <= 0.f || cfg->window < 1 ||
      cfg->hysteresis < 1 || !std::isfinite(cfg->min_scale) || cfg->min_scale <= 0.f)
    return fail(DPOPT_ERR_INVALID_ARG,
                "loss-scale config: scales must be finite and > 0, window and hysteresis >= 1");
  *out = LossScaleConfig{cfg->init_scale, cfg->window, cfg->hysteresis, cfg->min_scale};
  return DPOPT_OK;
}

int check_state_ptr(const void* st) {
  if (!st || ((uintptr_t)st & 7u))
    return fail(DPOPT_ERR_INVALID_ARG, "loss-scale state must be a non-null, 8-byte aligned pointer");
  return DPOPT_OK;
}

int dispatch_amp(const SmallParams& p, int grad_dtype, const LossScaleState* st, const double* sq,
                 cudaStream_t stream) {
  if (grad_dtype == DPOPT_GRAD_F16) return launch_amp_step<2>(p, st, sq, stream);
  if (grad_dtype == DPOPT_GRAD_BF16) return launch_amp_step<0>(p, st, sq, stream);
  return launch_amp_step<1>(p, st, sq, stream);
}

int launch_scale_update(LossScaleState* st, const double* sq, const LossScaleConfig& cfg,
                        cudaStream_t stream) {
  cudaError_t e = launch_pdl(loss_scale_update_kernel, 1, 32, 0, stream, st, sq, cfg);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  ++g_launches;
  return DPOPT_OK;
}

// ---------------------------------------------------------------------------
// allocation-free squared norm: partials in a fixed device array
// ---------------------------------------------------------------------------

// Chunk partials for dpopt_grad_sqnorm_noalloc: one fp64 per 4096-element
// chunk, so shards of up to kNoAllocMaxChunks * 4096 = 2^31 elements.  The
// array is part of the library image: every device that loads the library
// holds these 4 MB until the process exits.
constexpr int64_t kNoAllocMaxChunks = 524288;
static_assert(kNoAllocMaxChunks * kNormChunk == (int64_t)1 << 31, "noalloc covers 2^31 elements");
static __device__ __align__(256) double g_noalloc_partials[kNoAllocMaxChunks];

// Device address of g_noalloc_partials on the current device.  In host code
// the array's name only stands for the symbol, so the address is looked up
// once per device (with that device current) and cached.
std::once_flag g_noalloc_once[kMaxDevices];
double* g_noalloc_addr[kMaxDevices];
cudaError_t g_noalloc_err[kMaxDevices];

int noalloc_partials(double** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(DPOPT_ERR_UNSUPPORTED, "device index too large");
  std::call_once(g_noalloc_once[dev], [dev] {
    void* ptr = nullptr;
    g_noalloc_err[dev] = cudaGetSymbolAddress(&ptr, g_noalloc_partials);
    g_noalloc_addr[dev] = static_cast<double*>(ptr);
  });
  if (g_noalloc_err[dev] != cudaSuccess) return cuda_fail(g_noalloc_err[dev], "cudaGetSymbolAddress");
  *out = g_noalloc_addr[dev];
  return DPOPT_OK;
}

// The all-gather kernel over p.len elements into p.n_dst destinations.
int launch_gather(const GatherParams& p, cudaStream_t stream) {
  int sms = 0;
  int rc = sm_count(&sms);
  if (rc) return rc;
  const int64_t want = (p.len + (int64_t)kThreads * kGroup - 1) / ((int64_t)kThreads * kGroup);
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * 8));
  cudaError_t e = launch_pdl(allgather_bf16_kernel, grid, kThreads, 0, stream, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  ++g_launches;
  return DPOPT_OK;
}

// Whether the step fused with the all-gather runs, or the step into the own
// replica followed by the broadcast kernel.  With its bf16 tiles written by
// bulk copies the fused kernel measured faster at every N and size on GB300
// (G params/s, fused / two passes, bf16): S = 30M: N = 2 194.9 / 185.2,
// 3 177.7 / 165.3, 4 161.0 / 152.1, 5 144.8 / 138.4, 6 130.5 / 126.9,
// 8 114.3 / 111.3, 9 106.0 / 103.0, 12 88.0 / 86.3, 16 71.4 / 69.9,
// 24 51.9 / 50.4, 32 41.5 / 40.5; S = 4M: N = 2, 4, 8, 16, 64 likewise;
// fp32 S = 30M: N = 4 132.6 / 130.6, 8 89.6 / 88.8.  So the automatic policy
// always fuses; both forms write the same bits.
bool gather_fused(int n, int64_t shard, int grad_dtype) {
  (void)n; (void)shard; (void)grad_dtype;
  return g_gather_policy.load(std::memory_order_relaxed) != DPOPT_GATHER_SEPARATE;
}

}  // namespace
}  // namespace dpopt

using namespace dpopt;

extern "C" {

int dpopt_reduce_adam_ex(const void* const* grads, int grad_dtype, int n_replicas, int64_t numel,
                         int shard_rank, int64_t bucket_elems, float* master_f32, float* m_f32,
                         float* v_f32, void* param_bf16_out, float lr, float beta1, float beta2,
                         float eps, int64_t step, dpopt_stream_t stream) {
  return full_impl(grads, grad_dtype, n_replicas, numel, shard_rank, bucket_elems, master_f32,
                   m_f32, v_f32, param_bf16_out, lr, beta1, beta2, eps, step, nullptr,
                   (cudaStream_t)stream);
}

int dpopt_reduce_adam(const void* const* grads, int n_replicas, int64_t numel, int shard_rank,
                      int64_t bucket_elems, float* master_f32, float* m_f32, float* v_f32,
                      void* param_bf16_out, float lr, float beta1, float beta2, float eps,
                      int64_t step, dpopt_stream_t stream) {
  return dpopt_reduce_adam_ex(grads, DPOPT_GRAD_BF16, n_replicas, numel, shard_rank, bucket_elems,
                              master_f32, m_f32, v_f32, param_bf16_out, lr, beta1, beta2, eps,
                              step, stream);
}

int dpopt_reduce_adamw(const void* const* grads, int grad_dtype, int n_replicas, int64_t numel,
                       int shard_rank, int64_t bucket_elems, float* master_f32, float* m_f32,
                       float* v_f32, void* param_bf16_out, float lr, float beta1, float beta2,
                       float eps, int64_t step, const dpopt_step_options* opts,
                       dpopt_stream_t stream) {
  return full_impl(grads, grad_dtype, n_replicas, numel, shard_rank, bucket_elems, master_f32,
                   m_f32, v_f32, param_bf16_out, lr, beta1, beta2, eps, step, opts,
                   (cudaStream_t)stream);
}

int dpopt_bucket_count(int64_t shard_elems, int64_t bucket_elems, int64_t* count_out) {
  if (!count_out || shard_elems < 0 || bucket_elems < 1)
    return fail(DPOPT_ERR_INVALID_ARG, "bucket_count: invalid argument");
  *count_out = shard_elems / bucket_elems + (shard_elems % bucket_elems ? 1 : 0);
  return DPOPT_OK;
}

int dpopt_bucket_range(int64_t shard_elems, int64_t bucket_elems, int64_t idx,
                       int64_t* offset_out, int64_t* len_out) {
  int64_t count = 0;
  int rc = dpopt_bucket_count(shard_elems, bucket_elems, &count);
  if (rc) return rc;
  if (!offset_out || !len_out || idx < 0 || idx >= count)
    return fail(DPOPT_ERR_INVALID_ARG, "bucket_range: invalid argument");
  const int64_t off = idx * bucket_elems;
  *offset_out = off;
  *len_out = std::min(bucket_elems, shard_elems - off);
  return DPOPT_OK;
}

int dpopt_reduce_adam_buckets(const void* const* slice_table, int grad_dtype, int n_replicas,
                              const int64_t* offsets, const int64_t* lens, int64_t n_buckets,
                              float* master_f32, float* m_f32, float* v_f32, void* param_bf16_out,
                              float lr, float beta1, float beta2, float eps, int64_t step,
                              dpopt_stream_t stream) {
  return buckets_impl(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets, master_f32,
                      m_f32, v_f32, param_bf16_out, lr, beta1, beta2, eps, step, nullptr,
                      (cudaStream_t)stream);
}

int dpopt_reduce_adamw_buckets(const void* const* slice_table, int grad_dtype, int n_replicas,
                               const int64_t* offsets, const int64_t* lens, int64_t n_buckets,
                               float* master_f32, float* m_f32, float* v_f32,
                               void* param_bf16_out, float lr, float beta1, float beta2, float eps,
                               int64_t step, const dpopt_step_options* opts,
                               dpopt_stream_t stream) {
  return buckets_impl(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets, master_f32,
                      m_f32, v_f32, param_bf16_out, lr, beta1, beta2, eps, step, opts,
                      (cudaStream_t)stream);
}

int dpopt_bucket_table_bytes(int n_replicas, int64_t n_buckets, int64_t* bytes_out) {
  if (!bytes_out || n_replicas < 1 || n_replicas > DPOPT_MAX_REPLICAS || n_buckets < 0 ||
      n_buckets > ((int64_t)1 << 30))
    return fail(DPOPT_ERR_INVALID_ARG, "bucket_table_bytes: invalid argument");
  *bytes_out = table_bytes_for(n_replicas, n_buckets);
  return DPOPT_OK;
}

int dpopt_reduce_adam_buckets_table(const void* const* slice_table, int grad_dtype,
                                    int n_replicas, const int64_t* offsets, const int64_t* lens,
                                    int64_t n_buckets, float* master_f32, float* m_f32,
                                    float* v_f32, void* param_bf16_out, float lr, float beta1,
                                    float beta2, float eps, int64_t step,
                                    const dpopt_step_options* opts, void* table,
                                    int64_t table_bytes, dpopt_stream_t stream) {
  return table_impl(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets, master_f32,
                    m_f32, v_f32, param_bf16_out, lr, beta1, beta2, eps, step, opts, table,
                    table_bytes, (cudaStream_t)stream);
}

int dpopt_grad_sqnorm_scratch_bytes(int64_t elems, int64_t n_buckets, int64_t* bytes_out) {
  if (!bytes_out || elems < 0 || n_buckets < 0)
    return fail(DPOPT_ERR_INVALID_ARG, "grad_sqnorm_scratch_bytes: invalid argument");
  *bytes_out = 8 * ((elems + kNormChunk - 1) / kNormChunk + n_buckets);
  return DPOPT_OK;
}

int dpopt_grad_sqnorm(const void* const* grads, int grad_dtype, int n_replicas, int64_t numel,
                      int shard_rank, float grad_unscale, double* sqnorm_out, void* scratch,
                      int64_t scratch_bytes, dpopt_stream_t stream) {
  return full_norm_impl(grads, grad_dtype, n_replicas, numel, shard_rank, grad_unscale, nullptr,
                        nullptr, sqnorm_out, scratch, scratch_bytes, (cudaStream_t)stream);
}

int dpopt_grad_average_sqnorm(const void* const* grads, int grad_dtype, int n_replicas,
                              int64_t numel, int shard_rank, float grad_unscale, float* avg_out,
                              double* sqnorm_out, void* scratch, int64_t scratch_bytes,
                              dpopt_stream_t stream) {
  if (!avg_out) return fail(DPOPT_ERR_INVALID_ARG, "avg_out must be non-null");
  return full_norm_impl(grads, grad_dtype, n_replicas, numel, shard_rank, grad_unscale, nullptr,
                        avg_out, sqnorm_out, scratch, scratch_bytes, (cudaStream_t)stream);
}

// Same result as dpopt_grad_sqnorm, for callers that cannot hand the library
// a scratch buffer: the chunk partials live in g_noalloc_partials.  Nothing
// there has to start at zero -- each call writes every partial it later reads.
// All calls on a device share that one array, so calls whose kernels may run
// at the same time on the GPU (different streams, other host threads) race.
int dpopt_grad_sqnorm_noalloc(const void* const* grads, int grad_dtype, int n_replicas,
                              int64_t numel, int shard_rank, float grad_unscale,
                              double* sqnorm_out, dpopt_stream_t stream) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  if (!std::isfinite(grad_unscale) || grad_unscale < 0.f)
    return fail(DPOPT_ERR_INVALID_ARG, "grad_unscale must be finite and >= 0");
  if (numel < 0 || numel % n_replicas != 0)
    return fail(DPOPT_ERR_INVALID_ARG, "numel must be >= 0 and a multiple of n_replicas");
  const int64_t S = numel / n_replicas;
  const int64_t chunks = (S + kNormChunk - 1) / kNormChunk;
  if (chunks > kNoAllocMaxChunks)
    return fail(DPOPT_ERR_UNSUPPORTED,
                "dpopt_grad_sqnorm_noalloc: a shard of %lld elements needs %lld partials; the "
                "built-in array holds %lld (shards up to %lld elements)",
                (long long)S, (long long)chunks, (long long)kNoAllocMaxChunks,
                (long long)(kNoAllocMaxChunks * kNormChunk));
  if (!sqnorm_out || ((uintptr_t)sqnorm_out & 7u))
    return fail(DPOPT_ERR_INVALID_ARG, "sqnorm_out must be a non-null, 8-byte aligned pointer");
  Range avoid[1] = {{(uintptr_t)sqnorm_out, (uintptr_t)(sqnorm_out + 1)}};
  const void* ptrs[DPOPT_MAX_REPLICAS];
  int64_t S2 = 0;
  rc = build_full(grads, grad_dtype, n_replicas, numel, shard_rank, 1, avoid, 1, ptrs, &S2);
  if (rc) return rc;
  // the array's address is set up even for an empty shard, so that such a
  // call can serve as the device's set-up before any stream capture
  double* partials = nullptr;
  rc = noalloc_partials(&partials);
  if (rc) return rc;
  if (S == 0) return finish_empty_norm(sqnorm_out, (cudaStream_t)stream);
  Hyper h = make_hyper(1.f, 0.f, 0.f, 0.f, 1, n_replicas);
  h.unscale = grad_unscale == 0.f ? 1.f : grad_unscale;
  SegDesc seg{ptrs, 0, S};
  return run_sqnorm(&seg, 1, grad_dtype, n_replicas, h, partials, sqnorm_out,
                    (cudaStream_t)stream);
}

// The squared norm over bucket slices, buckets that continue one another
// joined first (so contiguous buckets take the chunk partition, and the bits,
// of one full-buffer call over the same elements); with avg_out each
// element's average is stored at its shard offset, which needs the buckets to
// join into one segment.  With `ready` (one event per bucket) the buckets are
// neither joined nor reordered: each one's pass is launched behind its own
// event, in the listed order, its partials placed at its rank in shard order,
// so the ordered finish gives the bits of the call without events over the
// same buckets kept apart; the average may then span any number of buckets.
int buckets_norm_impl(const void* const* slice_table, int grad_dtype, int n_replicas,
                      const int64_t* offsets, const int64_t* lens, int64_t n_buckets,
                      float grad_unscale, const LossScaleState* state, float* avg_out,
                      double* sqnorm_out, void* scratch, int64_t scratch_bytes,
                      cudaStream_t stream, const dpopt_event_t* ready = nullptr) {
  if (!std::isfinite(grad_unscale) || grad_unscale < 0.f)
    return fail(DPOPT_ERR_INVALID_ARG, "grad_unscale must be finite and >= 0");
  std::vector<SegDesc> segs;
  int64_t lo = 0, hi = 0;
  int rc = build_buckets(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets, segs, &lo,
                         &hi);
  if (rc) return rc;
  if (!ready) coalesce(segs, n_replicas, grad_dtype);
  if (!ready && avg_out && segs.size() > 1)
    return fail(DPOPT_ERR_UNSUPPORTED,
                "the average is stored for buckets that join into one segment (each bucket "
                "continuing the previous one in the shard and in every replica's gradients); "
                "these form %zu", segs.size());
  const int64_t chunks = norm_chunks(segs.data(), (int)segs.size());
  Range avoid[3];
  rc = check_norm_outputs(sqnorm_out, scratch, scratch_bytes, chunks, avoid);
  if (rc) return rc;
  int navoid = chunks ? 2 : 1;
  if (avg_out && hi > lo) {
    if ((uintptr_t)avg_out & 3u) return fail(DPOPT_ERR_INVALID_ARG, "avg_out must be 4-byte aligned");
    const Range a{(uintptr_t)(avg_out + lo), (uintptr_t)(avg_out + hi)};
    for (int i = 0; i < navoid; ++i)
      if (overlaps(a, avoid[i]))
        return fail(DPOPT_ERR_INVALID_ARG, "avg_out overlaps sqnorm_out or the scratch partials");
    avoid[navoid++] = a;
  }
  rc = check_bucket_grads(segs, n_replicas, grad_dtype, avoid, navoid);
  if (rc) return rc;
  if (segs.empty()) return finish_empty_norm(sqnorm_out, stream);
  Hyper h = make_hyper(1.f, 0.f, 0.f, 0.f, 1, n_replicas);
  h.unscale = grad_unscale == 0.f ? 1.f : grad_unscale;
  if (state) h.scale_dev = &state->scale;
  set_span(h, lo, hi);
  if (!ready)
    return run_sqnorm(segs.data(), (int)segs.size(), grad_dtype, n_replicas, h,
                      (double*)scratch, sqnorm_out, stream, avg_out);
  // each bucket's first partial: the chunks of the buckets before it in shard order
  std::vector<size_t> order(segs.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = i;
  std::sort(order.begin(), order.end(),
            [&](size_t a, size_t b) { return segs[a].state_off < segs[b].state_off; });
  std::vector<int64_t> base(segs.size());
  int64_t done = 0;
  for (size_t i : order) {
    base[i] = done;
    done += (segs[i].len + kNormChunk - 1) / kNormChunk;
  }
  size_t si = 0;
  for (int64_t b = 0; b < n_buckets; ++b) {
    if (lens[b] == 0) continue;
    if (ready[b]) {
      cudaError_t e = cudaStreamWaitEvent(stream, (cudaEvent_t)ready[b], 0);
      if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
    }
    int64_t launched_chunks = 0;
    rc = norm_segment(segs[si], grad_dtype, n_replicas, h, (double*)scratch + base[si], avg_out,
                      stream, &launched_chunks);
    if (rc) return rc;
    ++si;
  }
  return norm_finish((const double*)scratch, done, sqnorm_out, stream);
}

int dpopt_grad_sqnorm_buckets(const void* const* slice_table, int grad_dtype, int n_replicas,
                              const int64_t* offsets, const int64_t* lens, int64_t n_buckets,
                              float grad_unscale, double* sqnorm_out, void* scratch,
                              int64_t scratch_bytes, dpopt_stream_t stream) {
  return buckets_norm_impl(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets,
                           grad_unscale, nullptr, nullptr, sqnorm_out, scratch, scratch_bytes,
                           (cudaStream_t)stream);
}

int dpopt_grad_sqnorm_buckets_when_ready(const void* const* slice_table, int grad_dtype,
                                         int n_replicas, const int64_t* offsets,
                                         const int64_t* lens, int64_t n_buckets,
                                         const dpopt_event_t* ready, float grad_unscale,
                                         float* avg_out, double* sqnorm_out, void* scratch,
                                         int64_t scratch_bytes, dpopt_stream_t stream) {
  if (n_buckets > 0 && !ready) return fail(DPOPT_ERR_INVALID_ARG, "ready must be non-null");
  static const dpopt_event_t kNoEvents[1] = {nullptr};
  return buckets_norm_impl(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets,
                           grad_unscale, nullptr, avg_out, sqnorm_out, scratch, scratch_bytes,
                           (cudaStream_t)stream, n_buckets > 0 ? ready : kNoEvents);
}

int dpopt_grad_average_sqnorm_buckets(const void* const* slice_table, int grad_dtype,
                                      int n_replicas, const int64_t* offsets,
                                      const int64_t* lens, int64_t n_buckets, float grad_unscale,
                                      float* avg_out, double* sqnorm_out, void* scratch,
                                      int64_t scratch_bytes, dpopt_stream_t stream) {
  if (!avg_out) return fail(DPOPT_ERR_INVALID_ARG, "avg_out must be non-null");
  return buckets_norm_impl(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets,
                           grad_unscale, nullptr, avg_out, sqnorm_out, scratch, scratch_bytes,
                           (cudaStream_t)stream);
}

int dpopt_reduce_adam_bucket(const void* const* grad_slices, int grad_dtype, int n_replicas,
                             int64_t shard_offset, int64_t len, float* master_f32, float* m_f32,
                             float* v_f32, void* param_bf16_out, float lr, float beta1,
                             float beta2, float eps, int64_t step, dpopt_stream_t stream) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  if (!grad_slices) return fail(DPOPT_ERR_INVALID_ARG, "grad_slices must be non-null");
  if (shard_offset < 0 || len < 0)
    return fail(DPOPT_ERR_INVALID_ARG, "shard_offset and len must be >= 0");
  return dpopt_reduce_adam_buckets(grad_slices, grad_dtype, n_replicas, &shard_offset, &len, 1,
                                   master_f32, m_f32, v_f32, param_bf16_out, lr, beta1, beta2, eps,
                                   step, stream);
}

int dpopt_loss_scale_init(dpopt_loss_scale_state* state, const dpopt_loss_scale_config* cfg,
                          dpopt_stream_t stream) {
  int rc = check_state_ptr(state);
  if (rc) return rc;
  LossScaleConfig c;
  rc = check_scale_config(cfg, &c);
  if (rc) return rc;
  cudaError_t e = launch_pdl(loss_scale_init_kernel, 1, 32, 0, (cudaStream_t)stream,
                             (LossScaleState*)state, c);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  ++g_launches;
  return DPOPT_OK;
}

int dpopt_amp_sqnorm(const void* const* grads, int grad_dtype, int n_replicas, int64_t numel,
                     int shard_rank, const dpopt_loss_scale_state* state, double* sqnorm_out,
                     void* scratch, int64_t scratch_bytes, dpopt_stream_t stream) {
  int rc = check_state_ptr(state);
  if (rc) return rc;
  return full_norm_impl(grads, grad_dtype, n_replicas, numel, shard_rank, 0.f,
                        (const LossScaleState*)state, nullptr, sqnorm_out, scratch,
                        scratch_bytes, (cudaStream_t)stream);
}

int dpopt_amp_average_sqnorm(const void* const* grads, int grad_dtype, int n_replicas,
                             int64_t numel, int shard_rank, const dpopt_loss_scale_state* state,
                             float* avg_out, double* sqnorm_out, void* scratch,
                             int64_t scratch_bytes, dpopt_stream_t stream) {
  int rc = check_state_ptr(state);
  if (rc) return rc;
  if (!avg_out) return fail(DPOPT_ERR_INVALID_ARG, "avg_out must be non-null");
  return full_norm_impl(grads, grad_dtype, n_replicas, numel, shard_rank, 0.f,
                        (const LossScaleState*)state, avg_out, sqnorm_out, scratch, scratch_bytes,
                        (cudaStream_t)stream);
}

int dpopt_amp_average_sqnorm_buckets(const void* const* slice_table, int grad_dtype,
                                     int n_replicas, const int64_t* offsets, const int64_t* lens,
                                     int64_t n_buckets, const dpopt_loss_scale_state* state,
                                     float* avg_out, double* sqnorm_out, void* scratch,
                                     int64_t scratch_bytes, dpopt_stream_t stream) {
  int rc = check_state_ptr(state);
  if (rc) return rc;
  if (!avg_out) return fail(DPOPT_ERR_INVALID_ARG, "avg_out must be non-null");
  return buckets_norm_impl(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets, 0.f,
                           (const LossScaleState*)state, avg_out, sqnorm_out, scratch,
                           scratch_bytes, (cudaStream_t)stream);
}

int dpopt_amp_sqnorm_buckets_when_ready(const void* const* slice_table, int grad_dtype,
                                        int n_replicas, const int64_t* offsets,
                                        const int64_t* lens, int64_t n_buckets,
                                        const dpopt_event_t* ready,
                                        const dpopt_loss_scale_state* state, float* avg_out,
                                        double* sqnorm_out, void* scratch, int64_t scratch_bytes,
                                        dpopt_stream_t stream) {
  int rc = check_state_ptr(state);
  if (rc) return rc;
  if (n_buckets > 0 && !ready) return fail(DPOPT_ERR_INVALID_ARG, "ready must be non-null");
  static const dpopt_event_t kNoEvents[1] = {nullptr};
  return buckets_norm_impl(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets, 0.f,
                           (const LossScaleState*)state, avg_out, sqnorm_out, scratch,
                           scratch_bytes, (cudaStream_t)stream,
                           n_buckets > 0 ? ready : kNoEvents);
}

int dpopt_amp_step(const void* const* grads, int grad_dtype, int n_replicas, int64_t numel,
                   int shard_rank, int64_t bucket_elems, float* master_f32, float* m_f32,
                   float* v_f32, void* param_bf16_out, float lr, float beta1, float beta2,
                   float eps, float weight_decay, float max_grad_norm,
                   const double* global_sqnorm, dpopt_loss_scale_state* state,
                   const dpopt_loss_scale_config* cfg, const float* lr_dev,
                   dpopt_stream_t stream) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  if ((uintptr_t)lr_dev & 3u) return fail(DPOPT_ERR_INVALID_ARG, "lr_dev must be 4-byte aligned");
  if (lr_dev) lr = 0.f;  // not used: the kernel reads the rate from lr_dev
  rc = check_hyper(lr, beta1, beta2, eps, 1);
  if (rc) return rc;
  rc = check_state_ptr(state);
  if (rc) return rc;
  LossScaleConfig c;
  rc = check_scale_config(cfg, &c);
  if (rc) return rc;
  if (global_sqnorm ? ((uintptr_t)global_sqnorm & 7u) != 0 : max_grad_norm != 0.f)
    return fail(DPOPT_ERR_INVALID_ARG,
                "global_sqnorm must be 8-byte aligned, and non-null when clipping");
  Hyper h = make_hyper(lr, beta1, beta2, eps, 1, n_replicas);
  dpopt_step_options o{weight_decay, max_grad_norm, global_sqnorm, 0.f};
  bool ext = false;
  rc = apply_options(&o, lr, h, &ext);
  if (rc) return rc;
  h.max_norm = (double)max_grad_norm;
  h.lr_dev = lr_dev;
  h.wd = weight_decay;
  if (numel < 0 || numel % n_replicas != 0 || numel == 0) {
    const void* ptrs[DPOPT_MAX_REPLICAS];
    int64_t S = 0;
    rc = build_full(grads, grad_dtype, n_replicas, numel, shard_rank, bucket_elems, nullptr, 0,
                    ptrs, &S);
    if (rc) return rc;
    return launch_scale_update((LossScaleState*)state, global_sqnorm, c, (cudaStream_t)stream);
  }
  const int64_t S = numel / n_replicas;
  set_span(h, 0, S);
  Range st[5];
  rc = check_states(master_f32, m_f32, v_f32, param_bf16_out, 0, S, st);
  if (rc) return rc;
  st[4] = {(uintptr_t)state, (uintptr_t)state + sizeof(dpopt_loss_scale_state)};
  for (int i = 0; i < 4; ++i)
    if (overlaps(st[4], st[i]))
      return fail(DPOPT_ERR_INVALID_ARG, "the loss-scale state overlaps a state or output array");
  const void* ptrs[DPOPT_MAX_REPLICAS];
  int64_t S2 = 0;
  rc = build_full(grads, grad_dtype, n_replicas, numel, shard_rank, bucket_elems, st, 5, ptrs,
                  &S2);
  if (rc) return rc;
  SmallParams p{};
  p.h = h;
  p.master = master_f32; p.m = m_f32; p.v = v_f32; p.out = (uint16_t*)param_bf16_out;
  p.n_rep = n_replicas;
  SegDesc seg{ptrs, 0, S};
  if (fill_segments(p, &seg, 0, 1, n_replicas, kGroup, grad_dtype) > 0) {
    rc = dispatch_amp(p, grad_dtype, (const LossScaleState*)state, global_sqnorm,
                      (cudaStream_t)stream);
    if (rc) return rc;
  }
  return launch_scale_update((LossScaleState*)state, global_sqnorm, c, (cudaStream_t)stream);
}

int dpopt_reduce_adam_buckets_when_ready(const void* const* slice_table, int grad_dtype,
                                         int n_replicas, const int64_t* offsets,
                                         const int64_t* lens, int64_t n_buckets,
                                         const dpopt_event_t* ready, float* master_f32,
                                         float* m_f32, float* v_f32, void* param_bf16_out,
                                         float lr, float beta1, float beta2, float eps,
                                         int64_t step, dpopt_stream_t stream) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  rc = check_hyper(lr, beta1, beta2, eps, step);
  if (rc) return rc;
  if (n_buckets > 0 && !ready) return fail(DPOPT_ERR_INVALID_ARG, "ready must be non-null");
  std::vector<SegDesc> segs;
  int64_t lo = 0, hi = 0;
  rc = build_buckets(slice_table, grad_dtype, n_replicas, offsets, lens, n_buckets, segs, &lo, &hi);
  if (rc || segs.empty()) return rc;
  Range st[4];
  rc = check_states(master_f32, m_f32, v_f32, param_bf16_out, lo, hi, st);
  if (rc) return rc;
  rc = check_bucket_grads(segs, n_replicas, grad_dtype, st, 4);
  if (rc) return rc;
  Hyper h = make_hyper(lr, beta1, beta2, eps, step, n_replicas);
  set_span(h, lo, hi);
  // one launch per bucket, each behind its own readiness event, in bucket order
  size_t si = 0;
  for (int64_t b = 0; b < n_buckets; ++b) {
    if (lens[b] == 0) continue;
    if (ready[b]) {
      cudaError_t e = cudaStreamWaitEvent((cudaStream_t)stream, (cudaEvent_t)ready[b], 0);
      if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
    }
    rc = run(&segs[si], 1, grad_dtype, n_replicas, master_f32, m_f32, v_f32, param_bf16_out, h,
             false, (cudaStream_t)stream);
    if (rc) return rc;
    ++si;
  }
  return DPOPT_OK;
}

int dpopt_allgather_bf16(const void* shard_bf16, int64_t shard_elems, int shard_rank,
                         void* const* param_replicas, int n_replicas, dpopt_stream_t stream) {
  if (n_replicas < 1) return fail(DPOPT_ERR_INVALID_ARG, "n_replicas must be >= 1");
  if (n_replicas > DPOPT_MAX_REPLICAS)
    return fail(DPOPT_ERR_UNSUPPORTED, "n_replicas %d exceeds %d", n_replicas, DPOPT_MAX_REPLICAS);
  if (shard_elems < 0) return fail(DPOPT_ERR_INVALID_ARG, "shard_elems must be >= 0");
  if (shard_rank < 0 || shard_rank >= n_replicas)
    return fail(DPOPT_ERR_INVALID_ARG, "shard_rank must lie in [0, n_replicas)");
  if (shard_elems == 0) return DPOPT_OK;
  if (!shard_bf16 || !param_replicas)
    return fail(DPOPT_ERR_INVALID_ARG, "shard_bf16 and param_replicas must be non-null");
  if ((uintptr_t)shard_bf16 & 1u) return fail(DPOPT_ERR_INVALID_ARG, "misaligned shard pointer");
  GatherParams p{};
#ifdef DPOPT_DEBUG_BOUNDS
  p.dbg_status = bounds_status_word();
#endif
  p.src = static_cast<const uint16_t*>(shard_bf16);
  p.len = shard_elems;
  const uintptr_t bytes = (uintptr_t)shard_elems * 2u;
  const Range src{(uintptr_t)shard_bf16, (uintptr_t)shard_bf16 + bytes};
  Range dst[DPOPT_MAX_REPLICAS];
  bool vec = ((uintptr_t)shard_bf16 & 15u) == 0;
  int nd = 0;
  for (int r = 0; r < n_replicas; ++r) {
    if (!param_replicas[r]) return fail(DPOPT_ERR_INVALID_ARG, "null replica pointer");
    if ((uintptr_t)param_replicas[r] & 1u)
      return fail(DPOPT_ERR_INVALID_ARG, "misaligned replica pointer");
    uint16_t* d = static_cast<uint16_t*>(param_replicas[r]) + (int64_t)shard_rank * shard_elems;
    const Range dr{(uintptr_t)d, (uintptr_t)d + bytes};
    if ((const void*)d == shard_bf16) continue;  // the shard already sits in this replica
    if (overlaps(dr, src))
      return fail(DPOPT_ERR_INVALID_ARG, "a replica's destination overlaps the shard");
    for (int j = 0; j < nd; ++j)
      if (overlaps(dr, dst[j])) return fail(DPOPT_ERR_INVALID_ARG, "replica destinations overlap");
    dst[nd] = dr;
    p.dst[nd++] = d;
    vec = vec && (((uintptr_t)d & 15u) == 0);
  }
  p.n_dst = nd;
  p.vec = vec ? 1 : 0;
  if (nd == 0) return DPOPT_OK;
  return launch_gather(p, (cudaStream_t)stream);
}

int dpopt_reduce_adam_allgather(const void* const* grads, int grad_dtype, int n_replicas,
                                int64_t numel, int shard_rank, int64_t bucket_elems,
                                float* master_f32, float* m_f32, float* v_f32,
                                void* const* param_replicas, float lr, float beta1, float beta2,
                                float eps, int64_t step, dpopt_stream_t stream) {
  int rc = check_replicas(n_replicas, grad_dtype);
  if (rc) return rc;
  rc = check_hyper(lr, beta1, beta2, eps, step);
  if (rc) return rc;
  const void* ptrs[DPOPT_MAX_REPLICAS];
  int64_t S = 0;
  if (numel <= 0 || numel % n_replicas != 0)   // nothing to update: arguments checked only
    return build_full(grads, grad_dtype, n_replicas, numel, shard_rank, bucket_elems, nullptr, 0,
                      ptrs, &S);
  if (shard_rank < 0 || shard_rank >= n_replicas)
    return fail(DPOPT_ERR_INVALID_ARG, "shard_rank must lie in [0, n_replicas)");
  if (!param_replicas) return fail(DPOPT_ERR_INVALID_ARG, "param_replicas must be non-null");
  const int64_t shard = numel / n_replicas;
  const int64_t base = (int64_t)shard_rank * shard;
  for (int r = 0; r < n_replicas; ++r) {
    if (!param_replicas[r]) return fail(DPOPT_ERR_INVALID_ARG, "null replica pointer");
    if ((uintptr_t)param_replicas[r] & 1u)
      return fail(DPOPT_ERR_INVALID_ARG, "misaligned replica pointer");
  }
  // The rank's own replica buffer is the working copy; the others receive it.
  uint16_t* own = static_cast<uint16_t*>(param_replicas[shard_rank]) + base;
  Range avoid[4 + DPOPT_MAX_REPLICAS];
  rc = check_states(master_f32, m_f32, v_f32, own, 0, shard, avoid);
  if (rc) return rc;
  int navoid = 4;
  GatherDst d{};
  bool dst16 = true;
  for (int r = 0; r < n_replicas; ++r) {
    if (r == shard_rank) continue;
    uint16_t* q = static_cast<uint16_t*>(param_replicas[r]) + base;
    const Range dr{(uintptr_t)q, (uintptr_t)(q + shard)};
    for (int j = 0; j < navoid; ++j)
      if (overlaps(dr, avoid[j]))
        return fail(DPOPT_ERR_INVALID_ARG, "a replica's destination overlaps a state array or "
                                           "another replica's destination");
    avoid[navoid++] = dr;
    d.dst[d.n++] = q;
    dst16 = dst16 && aligned16(q);
  }
  rc = build_full(grads, grad_dtype, n_replicas, numel, shard_rank, bucket_elems, avoid, navoid,
                  ptrs, &S);
  if (rc) return rc;
  Hyper h = make_hyper(lr, beta1, beta2, eps, step, n_replicas);
  set_span(h, 0, S);
  SegDesc seg{ptrs, 0, S};
  SmallParams p{};
  p.h = h;
  p.master = master_f32; p.m = m_f32; p.v = v_f32; p.out = own;
  p.n_rep = n_replicas;
  cudaStream_t st = (cudaStream_t)stream;
  if (!gather_fused(n_replicas, S, grad_dtype)) {
    // the step into the own replica buffer, then its broadcast
    rc = run(&seg, 1, grad_dtype, n_replicas, master_f32, m_f32, v_f32, own, h, false, st);
    if (rc || d.n == 0) return rc;
    GatherParams g{};
#ifdef DPOPT_DEBUG_BOUNDS
    g.dbg_status = bounds_status_word();
#endif
    g.src = own;
    g.len = S;
    g.n_dst = d.n;
    bool vec = aligned16(own);
    for (int i = 0; i < d.n; ++i) {
      g.dst[i] = d.dst[i];
      vec = vec && aligned16(d.dst[i]);
    }
    g.vec = vec ? 1 : 0;
    return launch_gather(g, st);
  }
  if (fill_segments(p, &seg, 0, 1, n_replicas, kGroup, grad_dtype) == 0) return DPOPT_OK;
  if (!dst16) p.seg[0].vec = 0;  // the 16-byte bf16 stores need every destination aligned
  if (grad_dtype == DPOPT_GRAD_BF16) return launch_step_gather<0>(p, d, st);
  if (grad_dtype == DPOPT_GRAD_F16) return launch_step_gather<2>(p, d, st);
  return launch_step_gather<1>(p, d, st);
}

int dpopt_stream_status(dpopt_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  bool timed_out = false;
  const int rc = take_wait_status(&timed_out);
  if (rc) return rc;
  if (timed_out) return DPOPT_ERR_TIMEOUT;
#ifdef DPOPT_DEBUG_BOUNDS
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_bounds_status, sizeof word);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  if (word) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_bounds_status, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
    return fail(DPOPT_ERR_BOUNDS, "a kernel's index check failed (bounds-checked build)");
  }
#endif
  return DPOPT_OK;
}

int dpopt_selftest_bounds(dpopt_stream_t stream) {
#ifdef DPOPT_DEBUG_BOUNDS
  Hyper h = make_hyper(1.f, 0.f, 0.f, 0.f, 1, 1);
  if (!h.dbg_status) return fail(DPOPT_ERR_CUDA, "no device address for the bounds status word");
  bounds_selftest_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(h, 1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  ++g_launches;
  return DPOPT_OK;
#else
  (void)stream;
  return fail(DPOPT_ERR_UNSUPPORTED, "index checks exist in the bounds-checked build only");
#endif
}

const char* dpopt_status_string(int status) {
  switch (status) {
    case DPOPT_OK: return "DPOPT_OK";
    case DPOPT_ERR_INVALID_ARG: return "DPOPT_ERR_INVALID_ARG";
    case DPOPT_ERR_UNSUPPORTED: return "DPOPT_ERR_UNSUPPORTED";
    case DPOPT_ERR_CUDA: return "DPOPT_ERR_CUDA";
    case DPOPT_ERR_TIMEOUT: return "DPOPT_ERR_TIMEOUT";
    case DPOPT_ERR_BOUNDS: return "DPOPT_ERR_BOUNDS";
    default: return "DPOPT_UNKNOWN_STATUS";
  }
}

const char* dpopt_last_error(void) { return g_last_error; }

int dpopt_state_bytes(int64_t psi, int variant, int n_dp, int zero_stage, double* bytes_out) {
  if (!bytes_out || psi < 0 || n_dp < 1 || zero_stage < 0 || zero_stage > 3 ||
      (variant != 0 && variant != 1))
    return fail(DPOPT_ERR_INVALID_ARG, "state_bytes: invalid argument");
  const double p = 2.0, g = 2.0, o = variant == 0 ? 12.0 : 4.0;
  const double n = (double)n_dp, x = (double)psi;
  const double bp = x * p / (zero_stage >= 3 ? n : 1.0);
  const double bg = x * g / (zero_stage >= 2 ? n : 1.0);
  const double bo = x * o / (zero_stage >= 1 ? n : 1.0);
  *bytes_out = bp + bg + bo;
  return DPOPT_OK;
}

int64_t dpopt_launch_count(void) { return g_launches; }

int dpopt_set_kernel_policy(int policy) {
  if (policy != DPOPT_KERNEL_AUTO && policy != DPOPT_KERNEL_DIRECT && policy != DPOPT_KERNEL_BULK)
    return fail(DPOPT_ERR_INVALID_ARG, "unknown kernel policy %d", policy);
  g_policy.store(policy, std::memory_order_relaxed);
  return DPOPT_OK;
}

int dpopt_get_kernel_policy(void) { return g_policy.load(std::memory_order_relaxed); }

int dpopt_set_gather_policy(int policy) {
  if (policy != DPOPT_GATHER_AUTO && policy != DPOPT_GATHER_FUSED &&
      policy != DPOPT_GATHER_SEPARATE)
    return fail(DPOPT_ERR_INVALID_ARG, "unknown gather policy %d", policy);
  g_gather_policy.store(policy, std::memory_order_relaxed);
  return DPOPT_OK;
}

int dpopt_get_gather_policy(void) { return g_gather_policy.load(std::memory_order_relaxed); }

int dpopt_selftest_wait_timeout(int64_t limit_cycles, dpopt_stream_t stream) {
  if (limit_cycles < 1 || limit_cycles > kWaitLimitCycles)
    return fail(DPOPT_ERR_INVALID_ARG, "limit_cycles must lie in [1, %lld]",
                (long long)kWaitLimitCycles);
  return launch_selftest_wait((long long)limit_cycles, (cudaStream_t)stream);
}

const char* dpopt_version(void) {
#ifdef DPOPT_DEBUG_BOUNDS
  return "0.1.0+bounds";
#else
  return "0.1.0";
#endif
}

}  // extern "C"

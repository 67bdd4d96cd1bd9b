// kernels.cuh -- the fused reduce + Adam kernel, direct-load form.
//
// One launch walks a list of segments (a whole shard, one bucket, or a batch
// of buckets).  Each segment has its own N replica pointers and a range of the
// shard's state arrays.  The launch is persistent: gridDim.x is a multiple of
// the SM count and every thread strides over 8-element groups, so a warp
// reads 512 contiguous bytes of every bf16 replica and 1 KB of every fp32
// state array per iteration.  Each element belongs to exactly one thread and
// the replica order is fixed, so the result is bitwise reproducible.
//
// Memory traffic per element is the algorithmic minimum: N gradient reads,
// master/m/v read once and written once, the bf16 copy written once (no
// intermediate ever leaves registers).  Gradients are read once, so their
// loads carry an L2 evict-first policy and skip L1.
#pragma once

#include "numerics.cuh"

namespace dpopt {

constexpr int kGroup = 8;      // elements per thread per iteration
constexpr int kThreads = 256;  // threads per CTA

struct Seg {
  int64_t first_group;  // groups of all earlier segments (prefix sum)
  int64_t state_off;    // first shard element this segment updates
  int64_t len;          // elements
  int32_t ptr_base;     // index of replica 0's pointer in LaunchParams::gptr
  int32_t vec;          // 2: 32-byte accesses apply (see fill_segments), 1: 16-byte, 0: scalar
};

template <int MAXSEG, int MAXPTR>
struct LaunchParams {
  Hyper h;
  float* master;
  float* m;
  float* v;
  uint16_t* out;
  int64_t total_groups;
  int32_t n_rep;
  int32_t nseg;
  Seg seg[MAXSEG + 1];  // seg[nseg].first_group == total_groups
  const void* gptr[MAXPTR];
};

// The same launch with its segment and pointer tables in device memory (a
// caller-owned buffer the library writes before the launch), so one launch
// covers any number of buckets: seg holds nseg + 1 entries, gptr nseg * n_rep
// pointers.  The tables are read-only for the kernel's lifetime.
struct TableParams {
  Hyper h;
  float* master;
  float* m;
  float* v;
  uint16_t* out;
  int64_t total_groups;
  int32_t n_rep;
  int32_t nseg;
  const Seg* seg;
  const void* const* gptr;
  int32_t wide;  // every segment has vector level 2 (read on the host only)
};

// ---------------------------------------------------------------------------
// memory access helpers
// ---------------------------------------------------------------------------

// Programmatic dependent launch.  The library launches its kernels with
// programmatic stream serialization, so a kernel's CTAs may be scheduled while
// the kernel before it on the stream is still finishing.  Every kernel first
// waits (griddepcontrol.wait: until the preceding grid has completed and its
// memory is visible) before touching global memory.  The short passes that
// feed a step -- the norm pre-pass, its ordered finish, the loss-scale
// kernels -- also let their successor be scheduled at once
// (griddepcontrol.launch_dependents), so the step's launch and ramp-up hide
// behind their tail, and so does the loss-scaled step, whose successor is the
// one-thread scale update; the other step kernels do not, since back-to-back
// steps measured no faster that way.  Both instructions are no-ops for a kernel
// launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 16 bytes of a gradient buffer: read once, L1 bypassed, L2 evict-first.
__device__ __forceinline__ uint4 ld_grad16(const void* p, uint64_t pol) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "l"(pol));
  return r;
}

// 16 bytes of a state array (read here, written back by the same thread).
// A coherent load: the non-coherent (.nc) path is for data that stays
// read-only while the kernel runs, and these addresses are stored to by the
// same kernel.  L1 is skipped either way (every byte is read once).
__device__ __forceinline__ float4 ld_state16(const float* p) {
  float4 r;
  asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
      : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ void st_stream16(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

__device__ __forceinline__ void st_stream16u(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.global.cs.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// 32 bytes in one 256-bit access (sm_100 and later; the address must be
// 32-byte aligned).  A warp then moves 1 KB of contiguous, whole 32-byte
// sectors per instruction, where two 16-byte accesses per thread would each
// touch every sector of that KB by halves.
__device__ __forceinline__ void ld_state32(const float* p, float4& lo, float4& hi) {
  asm volatile("ld.global.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=f"(lo.x), "=f"(lo.y), "=f"(lo.z), "=f"(lo.w), "=f"(hi.x), "=f"(hi.y), "=f"(hi.z),
        "=f"(hi.w)
      : "l"(p));
}

__device__ __forceinline__ void ld_grad32(const void* p, uint64_t pol, uint4& a, uint4& b) {
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
      : "l"(p), "l"(pol));
}

__device__ __forceinline__ void st_stream32(float* p, float4 lo, float4 hi) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(lo.x),
               "f"(lo.y), "f"(lo.z), "f"(lo.w), "f"(hi.x), "f"(hi.y), "f"(hi.z), "f"(hi.w)
               : "memory");
}

// Stores that keep the line in L2 (a value the next kernel reads back).
__device__ __forceinline__ void st_global16(float* p, float4 a) {
  asm volatile("st.global.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(a.x), "f"(a.y), "f"(a.z),
               "f"(a.w)
               : "memory");
}

__device__ __forceinline__ void st_global32(float* p, float4 lo, float4 hi) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(lo.x),
               "f"(lo.y), "f"(lo.z), "f"(lo.w), "f"(hi.x), "f"(hi.y), "f"(hi.z), "f"(hi.w)
               : "memory");
}

// 8 gradient values of one replica as fp32.  GK 0: bf16 (one 16-byte load),
// GK 1: fp32 (one 32-byte load, or two 16-byte ones: W), GK 2: fp16.
template <int GK>
struct GradLoad;

__device__ __forceinline__ uint4 ld_shared16(uint32_t saddr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(saddr));
  return r;
}

template <>
struct GradLoad<0> {
  uint4 w;
  template <int W = 16>
  __device__ __forceinline__ void load(const void* base, int64_t e0, uint64_t pol) {
    w = ld_grad16(static_cast<const uint16_t*>(base) + e0, pol);
  }
  __device__ __forceinline__ void load_shared(uint32_t saddr) { w = ld_shared16(saddr); }
  __device__ __forceinline__ void zero() { w = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ float get(int k) const {
    uint32_t x = (k < 2) ? w.x : (k < 4) ? w.y : (k < 6) ? w.z : w.w;
    return (k & 1) ? bf16_hi(x) : bf16_lo(x);
  }
  // elements 2j and 2j+1
  __device__ __forceinline__ float2 pair(int j) const {
    return bf16x2_to_float2(j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w);
  }
};

template <>
struct GradLoad<1> {
  uint4 a, b;
  template <int W = 16>
  __device__ __forceinline__ void load(const void* base, int64_t e0, uint64_t pol) {
    const float* p = static_cast<const float*>(base) + e0;
    if constexpr (W == 32) {
      ld_grad32(p, pol, a, b);
    } else {
      a = ld_grad16(p, pol);
      b = ld_grad16(p + 4, pol);
    }
  }
  __device__ __forceinline__ void load_shared(uint32_t saddr) {
    a = ld_shared16(saddr);
    b = ld_shared16(saddr + 16);
  }
  __device__ __forceinline__ void zero() { a = b = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ float get(int k) const {
    const uint4& q = (k < 4) ? a : b;
    int j = k & 3;
    return __uint_as_float(j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w);
  }
  __device__ __forceinline__ float2 pair(int j) const {
    const uint4& q = (j < 2) ? a : b;
    return (j & 1) ? make_float2(__uint_as_float(q.z), __uint_as_float(q.w))
                   : make_float2(__uint_as_float(q.x), __uint_as_float(q.y));
  }
};

// fp16: binary16 words; widening to fp32 is exact (PTX cvt.f32.f16).
__device__ __forceinline__ float f16_to_f32(uint32_t bits16) {
  float f;
  asm("{ .reg .b16 h; cvt.u16.u32 h, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "r"(bits16));
  return f;
}

template <>
struct GradLoad<2> {
  uint4 w;
  template <int W = 16>
  __device__ __forceinline__ void load(const void* base, int64_t e0, uint64_t pol) {
    w = ld_grad16(static_cast<const uint16_t*>(base) + e0, pol);
  }
  __device__ __forceinline__ void load_shared(uint32_t saddr) { w = ld_shared16(saddr); }
  __device__ __forceinline__ void zero() { w = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ float get(int k) const {
    uint32_t x = (k < 2) ? w.x : (k < 4) ? w.y : (k < 6) ? w.z : w.w;
    return f16_to_f32((k & 1) ? (x >> 16) : (x & 0xFFFFu));
  }
  __device__ __forceinline__ float2 pair(int j) const {
    uint32_t x = j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w;
    return make_float2(f16_to_f32(x & 0xFFFFu), f16_to_f32(x >> 16));
  }
};

template <int GK>
__device__ __forceinline__ float ld_grad1(const void* base, int64_t e) {
  if constexpr (GK == 0) {
    uint16_t h = static_cast<const uint16_t*>(base)[e];
    return __uint_as_float(((uint32_t)h) << 16);
  } else if constexpr (GK == 2) {
    return f16_to_f32(static_cast<const uint16_t*>(base)[e]);
  } else {
    return static_cast<const float*>(base)[e];
  }
}

// ---------------------------------------------------------------------------
// where one 8-element group's inputs come from, where its outputs go
// ---------------------------------------------------------------------------

// Inputs read straight from global memory (the direct-load kernel).  W: the
// width of one state access (32: one 256-bit load per array, 16: two).
template <int GK, int W = 16>
struct GlobalSource {
  const void* const* gp;  // the segment's replica pointers
  int64_t e0;             // group's first element within the segment
  const float* st[3];     // master, m, v at the group's first element
  uint64_t pol;
  __device__ __forceinline__ void grad(GradLoad<GK>& g, int r) const {
    g.template load<W>(gp[r], e0, pol);
  }
  __device__ __forceinline__ void state8(int a, float4& lo, float4& hi) const {
    if constexpr (W == 32) {
      ld_state32(st[a], lo, hi);
    } else {
      lo = ld_state16(st[a]);
      hi = ld_state16(st[a] + 4);
    }
  }
};

// Inputs staged in shared memory by bulk copies (the bulk-copy kernel).
template <int GK>
struct SharedSource {
  uint32_t g0;       // shared address of replica 0's 8 values for this thread
  uint32_t rstride;  // bytes between consecutive replicas' rows
  uint32_t st[3];    // shared addresses of master, m, v for this thread
  __device__ __forceinline__ void grad(GradLoad<GK>& g, int r) const {
    g.load_shared(g0 + (uint32_t)r * rstride);
  }
  __device__ __forceinline__ void state8(int a, float4& lo, float4& hi) const {
    const uint4 u = ld_shared16(st[a]), w = ld_shared16(st[a] + 16u);
    lo = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                     __uint_as_float(u.w));
    hi = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                     __uint_as_float(w.w));
  }
};

// Outputs, at the group's first element; W as for GlobalSource.
template <int W = 16>
struct GroupOutT {
  float* master;
  float* m;
  float* v;
  uint16_t* out;
  __device__ __forceinline__ void put(float* p, float4 lo, float4 hi) const {
    if constexpr (W == 32) {
      st_stream32(p, lo, hi);
    } else {
      st_stream16(p, lo.x, lo.y, lo.z, lo.w);
      st_stream16(p + 4, hi.x, hi.y, hi.z, hi.w);
    }
  }
  // the group's 8 bf16 values, packed two to a word
  __device__ __forceinline__ void put_bf16(uint32_t a, uint32_t b, uint32_t c, uint32_t d) const {
    st_stream16u(out, a, b, c, d);
  }
};
using GroupOut = GroupOutT<16>;

// Further destinations of the bf16 copy: the step fused with the ZeRO-3
// all-gather writes the shard's new bf16 values into the same position of
// every other replica's parameter buffer.  dst[i] points at the shard's first
// element in replica buffer i.
constexpr int kMaxGatherDst = 64;
struct GatherDst {
  uint16_t* dst[kMaxGatherDst];
  int32_t n;
};

template <int W = 16>
struct GatherOutT : GroupOutT<W> {
  const GatherDst* gd;
  int64_t so;  // the group's first shard element
  __device__ __forceinline__ void put_bf16(uint32_t a, uint32_t b, uint32_t c, uint32_t d) const {
    st_stream16u(this->out, a, b, c, d);
    for (int i = 0; i < gd->n; ++i) st_stream16u(gd->dst[i] + so, a, b, c, d);
  }
};

// ---------------------------------------------------------------------------
// one 8-element group, vector path
// ---------------------------------------------------------------------------

// The fixed-order compensated replica sum of one 8-element group (scalar
// lanes), shared by the step and the squared-norm pre-pass so both see the
// same bits of g.
// Replicas R0 .. R0+REM-1 added in order, in batches of at most 8 whose loads
// are issued together.
template <int REM, int R0, int GK, class Src>
__device__ __forceinline__ void add_batches_x1(const Src& src, CompSum<float> (&acc)[kGroup]) {
  constexpr int B = REM < 8 ? REM : 8;
  GradLoad<GK> gl[B];
#pragma unroll
  for (int r = 0; r < B; ++r) src.grad(gl[r], R0 + r);
#pragma unroll
  for (int r = 0; r < B; ++r) {
#pragma unroll
    for (int k = 0; k < kGroup; ++k) acc[k].add(gl[r].get(k));
  }
  if constexpr (REM > 8) add_batches_x1<REM - 8, R0 + 8, GK>(src, acc);
}

template <int NR, int GK, class Src>
__device__ __forceinline__ void reduce_group_x1(const Src& src, int n, CompSum<float> (&acc)[kGroup]) {
  if constexpr (NR > 8) {
    // batches of 8 (the last one NR mod 8) so that at most 8 loads are held at once
    {
      GradLoad<GK> gl[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) src.grad(gl[r], r);
#pragma unroll
      for (int k = 0; k < kGroup; ++k) acc[k].init(gl[0].get(k));
#pragma unroll
      for (int r = 1; r < 8; ++r) {
#pragma unroll
        for (int k = 0; k < kGroup; ++k) acc[k].add(gl[r].get(k));
      }
    }
    add_batches_x1<NR - 8, 8, GK>(src, acc);
  } else if constexpr (NR > 0) {
    GradLoad<GK> gl[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) src.grad(gl[r], r);
#pragma unroll
    for (int k = 0; k < kGroup; ++k) acc[k].init(gl[0].get(k));
#pragma unroll
    for (int r = 1; r < NR; ++r) {
#pragma unroll
      for (int k = 0; k < kGroup; ++k) acc[k].add(gl[r].get(k));
    }
  } else {
    // runtime replica count: chunks of 8 replicas, loads of a chunk in flight together
    constexpr int C = 8;
    for (int r0 = 0; r0 < n; r0 += C) {
      GradLoad<GK> gl[C];
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (r0 + j < n) src.grad(gl[j], r0 + j);
        else gl[j].zero();
      }
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (r0 + j < n) {
          if (r0 + j == 0) {
#pragma unroll
            for (int k = 0; k < kGroup; ++k) acc[k].init(gl[j].get(k));
          } else {
#pragma unroll
            for (int k = 0; k < kGroup; ++k) acc[k].add(gl[j].get(k));
          }
        }
      }
    }
  }
}

// Scalar-lane form: 8 elements per thread, one element per operation.  Fewer
// register pairings; faster when the optimizer arithmetic dominates (small N).
template <int NR, int GK, bool EXT, class Src, class Out>
__device__ __forceinline__ void group_vec_x1(const Src& src, int n, const Hyper& h, const Out& o,
                                             float gscale) {
  float th[kGroup], mm[kGroup], vv[kGroup];
  {
    float4 a, b;
    src.state8(0, a, b);
    th[0] = a.x; th[1] = a.y; th[2] = a.z; th[3] = a.w;
    th[4] = b.x; th[5] = b.y; th[6] = b.z; th[7] = b.w;
    src.state8(1, a, b);
    mm[0] = a.x; mm[1] = a.y; mm[2] = a.z; mm[3] = a.w;
    mm[4] = b.x; mm[5] = b.y; mm[6] = b.z; mm[7] = b.w;
    src.state8(2, a, b);
    vv[0] = a.x; vv[1] = a.y; vv[2] = a.z; vv[3] = a.w;
    vv[4] = b.x; vv[5] = b.y; vv[6] = b.z; vv[7] = b.w;
  }
  CompSum<float> acc[kGroup];
  reduce_group_x1<NR, GK>(src, n, acc);
#pragma unroll
  for (int k = 0; k < kGroup; ++k) {
    float g = acc[k].average(h);
    if constexpr (EXT) g = __fmul_rn(g, gscale);
    adam_update<EXT>(g, th[k], mm[k], vv[k], h);
  }
  o.put(o.master, make_float4(th[0], th[1], th[2], th[3]), make_float4(th[4], th[5], th[6], th[7]));
  o.put(o.m, make_float4(mm[0], mm[1], mm[2], mm[3]), make_float4(mm[4], mm[5], mm[6], mm[7]));
  o.put(o.v, make_float4(vv[0], vv[1], vv[2], vv[3]), make_float4(vv[4], vv[5], vv[6], vv[7]));
  o.put_bf16(to_bf16x2(th[0], th[1]), to_bf16x2(th[2], th[3]), to_bf16x2(th[4], th[5]),
             to_bf16x2(th[6], th[7]));
}

// Replicas r0 .. r0+C-1 of one 8-element group added, in order, to packed
// running sums (FIRST: replica r0 starts them); all C loads issued before the
// first addition.
template <int C, bool FIRST, int GK, class Src>
__device__ __forceinline__ void add_chunk_x2(const Src& src, int r0,
                                             CompSum<float2> (&acc)[kGroup / 2]) {
  GradLoad<GK> gl[C];
#pragma unroll
  for (int j = 0; j < C; ++j) src.grad(gl[j], r0 + j);
#pragma unroll
  for (int j = 0; j < C; ++j) {
#pragma unroll
    for (int k = 0; k < kGroup / 2; ++k) {
      if (FIRST && j == 0) acc[k].init(gl[j].pair(k));
      else acc[k].add(gl[j].pair(k));
    }
  }
}

// Replicas r .. r+K-1 of one 8-element group loaded into g[0 .. K-1].
template <int K, int GK, class Src>
__device__ __forceinline__ void load_chunk(const Src& src, int r, GradLoad<GK> (&g)[8]) {
#pragma unroll
  for (int j = 0; j < K; ++j) src.grad(g[j], r + j);
}

// g[0 .. K-1] added, in order, to packed running sums (FIRST: g[0] starts them).
template <int K, bool FIRST, int GK>
__device__ __forceinline__ void sum_chunk(const GradLoad<GK> (&g)[8],
                                          CompSum<float2> (&acc)[kGroup / 2]) {
#pragma unroll
  for (int j = 0; j < K; ++j) {
#pragma unroll
    for (int k = 0; k < kGroup / 2; ++k) {
      if (FIRST && j == 0) acc[k].init(g[j].pair(k));
      else acc[k].add(g[j].pair(k));
    }
  }
}

// The end of a pipelined replica walk: `cur` holds the last full chunk of 8
// (loaded, not yet added); the remaining rem < 8 replicas from r are loaded
// into `spare` before `cur` is added, so their loads overlap that addition.
template <int GK, class Src>
__device__ __forceinline__ void finish_chunks(const Src& src, int r, int rem,
                                              const GradLoad<GK> (&cur)[8],
                                              GradLoad<GK> (&spare)[8],
                                              CompSum<float2> (&acc)[kGroup / 2]) {
  switch (rem) {
#define DPOPT_REM(K)                          \
  case K:                                     \
    load_chunk<K>(src, r, spare);             \
    sum_chunk<8, false>(cur, acc);            \
    sum_chunk<K, false>(spare, acc);          \
    break;
    DPOPT_REM(1) DPOPT_REM(2) DPOPT_REM(3) DPOPT_REM(4) DPOPT_REM(5) DPOPT_REM(6) DPOPT_REM(7)
#undef DPOPT_REM
    default: sum_chunk<8, false>(cur, acc); break;
  }
}

// The fixed-order compensated replica sum of one 8-element group on packed
// f32x2 lanes (element pairs 2j, 2j+1): the same operations per element as
// reduce_group_x1, so the same bits.
template <int NR, int GK, class Src>
__device__ __forceinline__ void reduce_group_x2(const Src& src, int n,
                                                CompSum<float2> (&acc)[kGroup / 2]) {
  constexpr int P = kGroup / 2;
  if constexpr (NR == 0 && GK != 1) {
    if (n >= 16) {
      // Runtime replica count of 16 or more, 16-bit gradients, software-
      // pipelined: the next chunk of 8 replicas is loaded into one register
      // set while the chunk before it, in the other set, is added -- up to 16
      // loads of a thread in flight instead of 8, at the same two CTAs per SM
      // (126 registers).  Same replica order, same bits.  Measured on GB300
      // (bf16, S = 256M): N = 64 6608 -> 6842 GB/s, 32 6600 -> 6708, 31
      // 6200 -> 6432, 24 6452 -> 6560, 17 6093 -> 6025; the 70B shard
      // (N = 64) 43.0 -> 44.5 G params/s.  fp32 gradients keep the chunked
      // walk below: two 8-replica sets of 32-byte loads would not fit the
      // registers (fp32 N = 32: 7053 against 6953 GB/s pipelined).
      GradLoad<GK> ga[8], gb[8];
      load_chunk<8>(src, 0, ga);
      load_chunk<8>(src, 8, gb);
      sum_chunk<8, true>(ga, acc);
      int r = 16;  // gb holds replicas r-8 .. r-1
      while (true) {
        if (r + 8 > n) {
          finish_chunks(src, r, n - r, gb, ga, acc);
          return;
        }
        load_chunk<8>(src, r, ga);
        sum_chunk<8, false>(gb, acc);
        r += 8;      // ga holds replicas r-8 .. r-1
        if (r + 8 > n) {
          finish_chunks(src, r, n - r, ga, gb, acc);
          return;
        }
        load_chunk<8>(src, r, gb);
        sum_chunk<8, false>(ga, acc);
        r += 8;
      }
    }
  }
  if constexpr (NR > 0) {
    GradLoad<GK> gl[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) src.grad(gl[r], r);
#pragma unroll
    for (int j = 0; j < P; ++j) acc[j].init(gl[0].pair(j));
#pragma unroll
    for (int r = 1; r < NR; ++r) {
#pragma unroll
      for (int j = 0; j < P; ++j) acc[j].add(gl[r].pair(j));
    }
  } else {
    // runtime replica count: chunks of 8 replicas, then the remainder (1..7)
    // as one more chunk; all loads of a chunk in flight together, every chunk
    // fully unrolled, replicas in ascending order.  (A predicated 8-wide
    // remainder left N = 9..15 at 78-85 % of the copy bandwidth, remainders
    // split 4 + 2 + 1 paid one load latency per piece, and balancing all
    // chunks slowed the multiples of 8.)
    constexpr int C = 8;
    int r0;
    if (n >= C) {
      add_chunk_x2<C, true, GK>(src, 0, acc);
      r0 = C;
    } else {
      GradLoad<GK> gl[C];
#pragma unroll
      for (int j = 0; j < C; ++j) {
        if (j < n) src.grad(gl[j], j);
        else gl[j].zero();
      }
#pragma unroll
      for (int k = 0; k < P; ++k) acc[k].init(gl[0].pair(k));
#pragma unroll
      for (int j = 1; j < C; ++j) {
        if (j < n) {
#pragma unroll
          for (int k = 0; k < P; ++k) acc[k].add(gl[j].pair(k));
        }
      }
      r0 = n;
    }
    for (; r0 + C <= n; r0 += C) add_chunk_x2<C, false, GK>(src, r0, acc);
    switch (n - r0) {
      case 1: add_chunk_x2<1, false, GK>(src, r0, acc); break;
      case 2: add_chunk_x2<2, false, GK>(src, r0, acc); break;
      case 3: add_chunk_x2<3, false, GK>(src, r0, acc); break;
      case 4: add_chunk_x2<4, false, GK>(src, r0, acc); break;
      case 5: add_chunk_x2<5, false, GK>(src, r0, acc); break;
      case 6: add_chunk_x2<6, false, GK>(src, r0, acc); break;
      case 7: add_chunk_x2<7, false, GK>(src, r0, acc); break;
      default: break;
    }
  }
}

// Packed form: 4 element pairs per thread, every operation on f32x2 lanes.
// Pays off when the replica sum dominates (large N).
template <int NR, int GK, bool EXT, class Src, class Out>
__device__ __forceinline__ void group_vec_x2(const Src& src, int n, const Hyper& h, const Out& o,
                                             float gscale) {
  constexpr int P = kGroup / 2;  // element pairs per group
  float2 th[P], mm[P], vv[P];
  {
    float4 a, b;
    src.state8(0, a, b);
    th[0] = make_float2(a.x, a.y); th[1] = make_float2(a.z, a.w);
    th[2] = make_float2(b.x, b.y); th[3] = make_float2(b.z, b.w);
    src.state8(1, a, b);
    mm[0] = make_float2(a.x, a.y); mm[1] = make_float2(a.z, a.w);
    mm[2] = make_float2(b.x, b.y); mm[3] = make_float2(b.z, b.w);
    src.state8(2, a, b);
    vv[0] = make_float2(a.x, a.y); vv[1] = make_float2(a.z, a.w);
    vv[2] = make_float2(b.x, b.y); vv[3] = make_float2(b.z, b.w);
  }
  CompSum<float2> acc[P];
  reduce_group_x2<NR, GK>(src, n, acc);
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

// ---------------------------------------------------------------------------
// a partial or unaligned group, one element at a time
// ---------------------------------------------------------------------------

template <int GK, bool EXT, bool GATHER, class LP, class SegT>
__device__ __noinline__ void group_scalar(const LP& p, const Hyper& h, const SegT& sg, int64_t e0,
                                          int count, float gscale, const GatherDst* gd) {
  if (!dbg_ok(h, e0 >= 0 && count >= 0 && e0 + count <= sg.len) ||
      !dbg_span(h, sg.state_off + e0, sg.state_off + e0 + count))
    return;
  const void* const* gp = p.gptr + sg.ptr_base;
  const int n = p.n_rep;
  for (int k = 0; k < count; ++k) {
    const int64_t e = e0 + k;
    const int64_t so = sg.state_off + e;
    CompSum<float> acc;
    acc.init(ld_grad1<GK>(gp[0], e));
    for (int r = 1; r < n; ++r) acc.add(ld_grad1<GK>(gp[r], e));
    float th = p.master[so], mm = p.m[so], vv = p.v[so];
    float g = acc.average(h);
    if constexpr (EXT) g = __fmul_rn(g, gscale);
    adam_update<EXT>(g, th, mm, vv, h);
    p.master[so] = th;
    p.m[so] = mm;
    p.v[so] = vv;
    const uint16_t b = to_bf16(th);
    p.out[so] = b;
    if constexpr (GATHER)
      for (int i = 0; i < gd->n; ++i) gd->dst[i][so] = b;
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

// Resident CTAs per SM the register budget is sized for: 4 x 256 threads
// (<= 64 registers) with an unrolled replica count (N <= 8); the runtime-count
// bodies take what they need (2 CTAs for the packed one).
template <int NR, int PACK>
constexpr int min_ctas() { return NR > 0 ? 4 : (PACK ? 2 : 1); }

// State access width of the unrolled kernels, by measurement on GB300
// (256M-element shards): one 256-bit access per state array and thread
// (W = 32: whole sectors, half the load/store instructions) is faster for
// fp32 gradients at every N <= 8 (+0..8%) and for bf16/fp16 gradients with
// N <= 3 (N = 2: 6395 against 5601 GB/s); for bf16/fp16 N >= 4 two 16-byte
// accesses (W = 16) are faster (N = 4: 6627 against 6363).  gk: 0 bf16,
// 1 fp32, 2 fp16.
constexpr bool wide_states(int gk, int nr) {
  return nr >= 1 && (gk == 1 ? nr <= 8 : nr <= 3);
}

// Resident CTAs per SM of a 256-bit kernel: its accesses need aligned
// 8-register tuples, and at four CTAs (64 registers) most forms spill, so
// they run three (up to 85 registers; bf16 N = 2: 6395 against 5884 GB/s,
// fp32 N = 5: 6722 against 6240).  bf16/fp16 with one replica fits 64
// registers without spills and keeps four (6439 against 5925).
template <int NR, int GK>
constexpr int wide_ctas() { return (NR == 1 && GK != 1) ? 4 : 3; }

// The grid-stride walk over the 8-element groups of every segment.  W is the
// width of one state access (32: one 256-bit access per array, for segments
// of vector level 2; 16: two 16-byte accesses, level >= 1); other groups go
// one element at a time.
template <int NR, int GK, int PACK, bool EXT, int W, class LP>
__device__ __forceinline__ void step_loop(const LP& p, const Hyper& h, float gscale) {
  constexpr int kLevel = W == 32 ? 2 : 1;
  const uint64_t pol = evict_first_policy();
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
    if (sg.vec >= kLevel && rem >= kGroup) {
      const GlobalSource<GK, W> src{p.gptr + sg.ptr_base, e0,
                                    {p.master + so, p.m + so, p.v + so}, pol};
      const GroupOutT<W> o{p.master + so, p.m + so, p.v + so, p.out + so};
      if constexpr (PACK) group_vec_x2<NR, GK, EXT>(src, p.n_rep, h, o, gscale);
      else group_vec_x1<NR, GK, EXT>(src, p.n_rep, h, o, gscale);
    } else {
      group_scalar<GK, EXT, false>(p, h, sg, e0, (int)(rem < kGroup ? rem : kGroup), gscale,
                                   nullptr);
    }
  }
}

// PACK selects the lane form of the vector body (0: scalar, 1: f32x2); the
// two forms give identical bits, so the choice is made by speed alone.  EXT
// adds the AdamW decay and the gradient multiplier (clipping, unscaling).
template <int NR, int GK, int PACK, bool EXT, int W, int MAXSEG, int MAXPTR>
__global__ void __launch_bounds__(kThreads, W == 32 ? wide_ctas<NR, GK>() : min_ctas<NR, PACK>())
    reduce_adam_ldg_kernel(const __grid_constant__ LaunchParams<MAXSEG, MAXPTR> p) {
  pdl_wait();
  const float gscale = EXT ? grad_scale_of(p.h) : 1.f;
  step_loop<NR, GK, PACK, EXT, W>(p, p.h, gscale);
}

// The step over a device-resident segment table: the same walk, the tables
// read through L1 instead of the parameter space.
template <int NR, int GK, int PACK, bool EXT, int W>
__global__ void __launch_bounds__(kThreads, W == 32 ? wide_ctas<NR, GK>() : min_ctas<NR, PACK>())
    reduce_adam_table_kernel(const __grid_constant__ TableParams p) {
  pdl_wait();
  const float gscale = EXT ? grad_scale_of(p.h) : 1.f;
  step_loop<NR, GK, PACK, EXT, W>(p, p.h, gscale);
}

// ---------------------------------------------------------------------------
// mixed-precision step with dynamic loss scaling
// ---------------------------------------------------------------------------

// Device-resident loss-scale state (the layout of dpopt_loss_scale_state).
struct LossScaleState {
  float scale;
  int32_t good_steps;
  int32_t hysteresis_left;
  int32_t last_overflow;
  int64_t step;
  int64_t skipped;
};

struct LossScaleConfig {
  float init_scale;
  int32_t window;
  int32_t hysteresis;
  float min_scale;
};

// The step of a loss-scaled run: skipped entirely when the global squared norm
// of the unscaled gradient is not finite (an overflow somewhere); otherwise
// the bias corrections of step state->step + 1 and the multiplier 1/scale
// (times the clip coefficient) are formed here, from device state, so no host
// synchronisation is needed between steps and the launch replays unchanged
// from a captured CUDA graph.  A null sqnorm means no overflow test and no
// clipping (a run without loss scaling that keeps its step count on the
// device).
// The 256-bit forms run three CTAs per SM at every N (up to 85 registers): the
// per-step scalars held in registers make even the one-replica form spill at
// four (loss-scaled gpt2s step through the stored average: 130.7 against
// 122.2 G params/s).
template <int NR, int GK, int PACK, int W, int MAXSEG, int MAXPTR>
__global__ void __launch_bounds__(kThreads, W == 32 ? 3 : min_ctas<NR, PACK>())
    reduce_adam_amp_kernel(const __grid_constant__ LaunchParams<MAXSEG, MAXPTR> p,
                           const LossScaleState* state, const double* sqnorm) {
  // The one-thread loss-scale update that follows is scheduled at once and
  // waits (griddepcontrol.wait) for this grid to complete.
  pdl_enter();
  // Thread 0 forms the step's scalars once; every thread then takes a copy of
  // the grid-constant Hyper with only those overwritten, so the untouched
  // fields stay constant-bank operands instead of occupying registers.
  __shared__ float s_ab[6];
  __shared__ float s_gscale;
  __shared__ int skip;
  if (threadIdx.x == 0) {
    Hyper h = p.h;
    const double sq = sqnorm ? *sqnorm : 0.0;
    skip = isfinite(sq) ? 0 : 1;
    const LossScaleState st = *state;
    const double t = (double)(st.step + 1);
    const double bc1 = 1.0 - pow((double)h.beta1, t);
    const double bc2 = 1.0 - pow((double)h.beta2, t);
    // the learning rate of this step: from device memory when given (a
    // schedule a captured graph replays), and then the AdamW factor
    // 1 - lr*wd too, rounded as the host forms it
    const float lr = h.lr_dev ? *h.lr_dev : h.lr;
    const double a = (double)lr / bc1;
    const double b = 1.0 / sqrt(bc2);
    s_ab[0] = __double2float_rn(a);
    s_ab[1] = __double2float_rn(a - (double)s_ab[0]);
    s_ab[2] = __double2float_rn(b);
    s_ab[3] = __double2float_rn(b - (double)s_ab[2]);
    if (h.lr_dev) {
      const double k = __dsub_rn(1.0, __dmul_rn((double)lr, (double)h.wd));
      s_ab[4] = __double2float_rn(k);
      s_ab[5] = __double2float_rn(__dsub_rn(k, (double)s_ab[4]));
    }
    h.unscale = __fdiv_rn(1.f, st.scale);
    h.sqnorm = sqnorm;
    s_gscale = grad_scale_of(h);
  }
  __syncthreads();
  if (skip) return;
  Hyper h = p.h;
  h.a_hi = s_ab[0];
  h.a_lo = s_ab[1];
  h.b_hi = s_ab[2];
  h.b_lo = s_ab[3];
  if (p.h.lr_dev) {
    h.k_hi = s_ab[4];
    h.k_lo = s_ab[5];
  }
  step_loop<NR, GK, PACK, true, W>(p, h, s_gscale);
}

}  // namespace dpopt

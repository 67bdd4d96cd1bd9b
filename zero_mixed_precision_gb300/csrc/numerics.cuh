// numerics.cuh -- per-element arithmetic of the fused reduce + Adam step.
//
// The step is specified against an fp64 evaluation: the replica sum exact and
// rounded once to fp32, m' and v' rounded once to fp32, and the master update
// computed from the stored m' and v' and rounded once.  fp64 is far too slow
// on this part (its fp64 rate is a small fraction of its fp32 rate), so every
// quantity is carried as fp32 plus an fp32 error term where one rounding
// would not be enough, using error-free transformations:
//   TwoSum  (Knuth, TAOCP vol. 2, 4.2.2): s + e == a + b exactly;
//   TwoProd (with FMA, e.g. Muller et al., Handbook of Floating-Point
//           Arithmetic, 4.4): p + e == a * b exactly;
//   one Newton correction of an approximate square root and quotient whose
//           residual is formed exactly with an FMA (Markstein 1990; Karp &
//           Markstein 1997).
// When an input or a result is not finite, the element falls back to the
// plain IEEE fp32 formula, which propagates Inf and NaN the way the fp64
// evaluation does.
//
// Every routine is a template over the lane type V: `float` (one element) or
// `float2` (two elements, evaluated with the packed f32x2 instructions of
// sm_100+).  Both instantiations perform the same sequence of correctly
// rounded IEEE operations on every element, so an element gets bit-identical
// results whichever path (vector body, scalar tail, unaligned range) handles
// it.  Only explicitly rounded intrinsics are used: nothing is contracted or
// reordered by the compiler.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace dpopt {

// Scalars of one step, prepared on the host in fp64 and split into
// unevaluated (hi, lo) fp32 pairs where a single fp32 would lose accuracy.
struct Hyper {
  float beta1, beta2;  // exponential decay rates
  float c1_hi, c1_lo;  // 1 - beta1
  float c2_hi, c2_lo;  // 1 - beta2
  float a_hi, a_lo;    // lr / (1 - beta1^t)
  float b_hi, b_lo;    // 1 / sqrt(1 - beta2^t)
  float eps;
  float inv_n;         // 1/N when N is a power of two (exact scaling), else 0
  float n_f;           // N
  float k_hi, k_lo;    // 1 - lr*weight_decay (AdamW), used by the extended step only
  // gradient scale of the extended step: g <- fl32(g * c), c an fp32 scalar
  // computed once per launch from these (see grad_scale_of)
  const double* sqnorm;  // device: squared global L2 norm of the averaged gradient, or null
  double max_norm;       // clip threshold (clipping when > 0 and sqnorm is non-null)
  float unscale;         // multiplier applied first (1/loss scale; 1 when unused)
  float lr;              // learning rate (for bias corrections formed on the device)
  const float* scale_dev;  // device loss scale: the norm pre-pass unscales by 1/*scale_dev
  const float* lr_dev;     // device learning rate of the loss-scaled step (null: lr above),
  float wd;                // with the weight decay its 1 - lr*wd is formed from
#ifdef DPOPT_DEBUG_BOUNDS
  // bounds-checked builds only: the status word a failed index check sets, and
  // the span [dbg_lo, dbg_hi) of shard elements the call may touch
  unsigned int* dbg_status;
  int64_t dbg_lo, dbg_hi;
#endif
};

// Index checks of the bounds-checked build (-DDPOPT_DEBUG_BOUNDS).  A kernel
// asks dbg_ok(h, cond) before every access whose index it derived from the
// launch's tables; a false condition sets bit 0 of *h.dbg_status and the
// caller skips the access, so a wrong index is reported by
// dpopt_stream_status() as DPOPT_ERR_BOUNDS instead of touching memory.  In a
// release build dbg_ok is the constant true and compiles away.
#ifdef DPOPT_DEBUG_BOUNDS
__device__ __forceinline__ bool dbg_ok(const Hyper& h, bool cond) {
  if (!cond && h.dbg_status) atomicOr(h.dbg_status, 1u);
  return cond;
}
// [lo, hi) of shard elements lies inside the call's span
__device__ __forceinline__ bool dbg_span(const Hyper& h, int64_t lo, int64_t hi) {
  return dbg_ok(h, lo >= h.dbg_lo && lo <= hi && hi <= h.dbg_hi);
}
#else
__device__ __forceinline__ constexpr bool dbg_ok(const Hyper&, bool) { return true; }
__device__ __forceinline__ constexpr bool dbg_span(const Hyper&, int64_t, int64_t) { return true; }
#endif

// The extended step's gradient multiplier: c = unscale * min(1, max_norm /
// (sqrt(sqnorm) + 1e-6)), evaluated in fp64 and rounded once to fp32.
// The same value in every thread (one device scalar read).
__device__ __forceinline__ float grad_scale_of(const Hyper& h) {
  double c = (double)h.unscale;
  if (h.sqnorm != nullptr && h.max_norm > 0.0) {
    const double nrm = __dsqrt_rn(*h.sqnorm);
    const double coef = __ddiv_rn(h.max_norm, __dadd_rn(nrm, 1e-6));
    if (coef < 1.0) c = __dmul_rn(c, coef);
  }
  return __double2float_rn(c);
}

// ---------------------------------------------------------------------------
// lane-generic IEEE operations (round to nearest even)
// ---------------------------------------------------------------------------

__device__ __forceinline__ float vadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float vmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float vfma(float a, float b, float c) { return __fmaf_rn(a, b, c); }
__device__ __forceinline__ float vneg(float a) { return -a; }

__device__ __forceinline__ float2 vadd(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 vmul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 vfma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 vneg(float2 a) { return make_float2(-a.x, -a.y); }

// a - b, rounded once.  On f32x2 lanes as fma(b, -1, a): the exact a - b
// rounded once, the same bits as a subtraction, in one packed instruction.
__device__ __forceinline__ float vsub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float2 vsub(float2 a, float2 b) {
  return __ffma2_rn(b, make_float2(-1.f, -1.f), a);
}

template <class V> __device__ __forceinline__ V splat(float s);
template <> __device__ __forceinline__ float splat<float>(float s) { return s; }
template <> __device__ __forceinline__ float2 splat<float2>(float s) { return make_float2(s, s); }

template <class V> struct Lanes;
template <> struct Lanes<float> {
  static constexpr int n = 1;
  __device__ static __forceinline__ float& at(float& v, int) { return v; }
  __device__ static __forceinline__ float get(const float& v, int) { return v; }
};
template <> struct Lanes<float2> {
  static constexpr int n = 2;
  __device__ static __forceinline__ float& at(float2& v, int i) { return i ? v.y : v.x; }
  __device__ static __forceinline__ float get(const float2& v, int i) { return i ? v.y : v.x; }
};

__device__ __forceinline__ bool finite(float x) { return fabsf(x) <= 3.402823466e38f; }

__device__ __forceinline__ float rsqrt_approx(float x) {
  float y;
  asm("rsqrt.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <class V>
__device__ __forceinline__ void two_sum(V a, V b, V& s, V& e) {
  s = vadd(a, b);
  V bp = vsub(s, a);
  V ap = vsub(s, bp);
  e = vadd(vsub(a, ap), vsub(b, bp));
}

// A double-float: hi + lo with |lo| <= ulp(hi)/2, about 48 significant bits.
struct DFloat {
  float hi, lo;
};

// a + b for non-negative double-floats (sums of squares): TwoSum of the high
// parts, the low parts added to its error, then renormalised.  Relative error
// about 2^-47; fp32 operations only (GB300's fp64 rate is a small fraction of
// its fp32 rate).
__device__ __forceinline__ DFloat df_add(DFloat a, DFloat b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  const float hi = __fadd_rn(s, e);
  return DFloat{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}

// ---------------------------------------------------------------------------
// Reduce: running compensated sum over the replicas in ascending order.
// ---------------------------------------------------------------------------

template <class V>
struct CompSum {
  V s, c;  // s + c carries the partial sum with ~48 significant bits
  __device__ __forceinline__ void init(V x0) {
    s = x0;
    c = splat<V>(0.f);
  }
  __device__ __forceinline__ void add(V x) {
    V t, e;
    two_sum(s, x, t, e);
    s = t;
    c = vadd(c, e);
  }
  // fl32(sum) then / N.  A non-finite running sum is returned as it is.
  __device__ __forceinline__ V average(const Hyper& h) const {
    V tot = vadd(s, c);
#pragma unroll
    for (int i = 0; i < Lanes<V>::n; ++i)
      if (!finite(Lanes<V>::get(s, i))) Lanes<V>::at(tot, i) = Lanes<V>::get(s, i);
    if (h.inv_n != 0.f) return vmul(tot, splat<V>(h.inv_n));
#pragma unroll
    for (int i = 0; i < Lanes<V>::n; ++i)
      Lanes<V>::at(tot, i) = __fdiv_rn(Lanes<V>::get(tot, i), h.n_f);
    return tot;
  }
};

// ---------------------------------------------------------------------------
// Adam moments, each rounded (nearly always correctly) once to fp32.
// ---------------------------------------------------------------------------

// m' = beta1*m + (1-beta1)*g
template <class V>
__device__ __forceinline__ V moment1(V m, V g, const Hyper& h) {
  const V b1 = splat<V>(h.beta1), c1h = splat<V>(h.c1_hi), c1l = splat<V>(h.c1_lo);
  V p1 = vmul(b1, m);
  V e1 = vfma(b1, m, vneg(p1));
  V p2 = vmul(c1h, g);
  V e2 = vfma(c1l, g, vfma(c1h, g, vneg(p2)));
  V s, e3;
  two_sum(p1, p2, s, e3);
  V r = vadd(s, vadd(vadd(e1, e2), e3));
#pragma unroll
  for (int i = 0; i < Lanes<V>::n; ++i)
    if (!finite(Lanes<V>::get(r, i)))
      Lanes<V>::at(r, i) = __fmaf_rn(h.beta1, Lanes<V>::get(m, i), Lanes<V>::get(p2, i));
  return r;
}

// v' = beta2*v + (1-beta2)*g*g, formed as ((1-beta2)*g)*g so that the square
// overflows only where the rounded result itself would.
template <class V>
__device__ __forceinline__ V moment2(V v, V g, const Hyper& h) {
  const V b2 = splat<V>(h.beta2), c2h = splat<V>(h.c2_hi), c2l = splat<V>(h.c2_lo);
  V P = vmul(c2h, g);
  V Pe = vfma(c2l, g, vfma(c2h, g, vneg(P)));
  V p2 = vmul(P, g);
  V e2 = vfma(Pe, g, vfma(P, g, vneg(p2)));
  V p1 = vmul(b2, v);
  V e1 = vfma(b2, v, vneg(p1));
  V s, e3;
  two_sum(p1, p2, s, e3);
  V r = vadd(s, vadd(vadd(e1, e2), e3));
#pragma unroll
  for (int i = 0; i < Lanes<V>::n; ++i)
    if (!finite(Lanes<V>::get(r, i)))
      Lanes<V>::at(r, i) = __fmaf_rn(h.beta2, Lanes<V>::get(v, i), Lanes<V>::get(p2, i));
  return r;
}

// theta' = k*theta - lr * (m'/bc1) / (sqrt(v'/bc2) + eps), the plain fp32 form
// (k = 1 - lr*weight_decay, 1 for plain Adam), used for non-finite inputs or
// results.
static __device__ __noinline__ float master_update_plain(float theta, float m_new, float v_new,
                                                  float a_hi, float b_hi, float eps, float k) {
  float d = __fadd_rn(__fmul_rn(__fsqrt_rn(v_new), b_hi), eps);
  float delta = __fdiv_rn(__fmul_rn(a_hi, m_new), d);
  return __fsub_rn(__fmul_rn(theta, k), delta);
}

// theta' = theta - a*m' / (b*sqrt(v') + eps) with a = lr/bc1, b = 1/sqrt(bc2),
// the quotient carried as q + q_lo and the subtraction rounded once.  With
// EXT the decoupled weight decay of AdamW (Loshchilov & Hutter 2019) is
// folded in: theta' = k*theta - a*m'/(...), k = 1 - lr*weight_decay carried
// as a (hi, lo) pair and k*theta as an exact product.
template <class V, bool EXT>
__device__ __forceinline__ V master_update(V theta, V m_new, V v_new, const Hyper& h) {
  constexpr int L = Lanes<V>::n;
  // sqrt(v') as s + s_lo: approximate reciprocal square root, one correction
  V y;
#pragma unroll
  for (int i = 0; i < L; ++i) Lanes<V>::at(y, i) = rsqrt_approx(Lanes<V>::get(v_new, i));
  V s = vmul(v_new, y);
  V rr = vfma(vneg(s), s, v_new);
  V s_lo = vmul(rr, vmul(splat<V>(0.5f), y));
#pragma unroll
  for (int i = 0; i < L; ++i) {
    const float vi = Lanes<V>::get(v_new, i);
    if (!(vi >= 0x1p-100f && vi <= 3.402823466e38f)) {  // zero, tiny, Inf, NaN
      Lanes<V>::at(s, i) = __fsqrt_rn(vi);
      Lanes<V>::at(s_lo, i) = 0.f;
    }
  }
  // D = b*sqrt(v') + eps as D + D_lo
  const V bh = splat<V>(h.b_hi), bl = splat<V>(h.b_lo);
  V p = vmul(s, bh);
  V pe = vfma(s, bh, vneg(p));
  V lo = vfma(s, bl, vfma(s_lo, bh, pe));
  V D, de;
  two_sum(p, splat<V>(h.eps), D, de);
  V D_lo = vadd(lo, de);
  // numerator a*m' as n + n_lo
  const V ah = splat<V>(h.a_hi), al = splat<V>(h.a_lo);
  V n = vmul(ah, m_new);
  V n_lo = vfma(al, m_new, vfma(ah, m_new, vneg(n)));
  // quotient q + q_lo = (n + n_lo) / (D + D_lo): approximate reciprocal, one correction
  V rD;
#pragma unroll
  for (int i = 0; i < L; ++i) Lanes<V>::at(rD, i) = rcp_approx(Lanes<V>::get(D, i));
  V q = vmul(n, rD);
  V r = vfma(vneg(q), D, n);
  r = vfma(vneg(q), D_lo, vadd(r, n_lo));
  V q_lo = vmul(r, rD);
  // (k*)theta - (q + q_lo), rounded once
  V t, te, th;
  if constexpr (EXT) {
    const V kh = splat<V>(h.k_hi), kl = splat<V>(h.k_lo);
    V P = vmul(theta, kh);
    V Pe = vfma(theta, kl, vfma(theta, kh, vneg(P)));
    two_sum(P, vneg(q), t, te);
    th = vadd(t, vadd(vadd(te, Pe), vneg(q_lo)));
  } else {
    two_sum(theta, vneg(q), t, te);
    th = vadd(t, vadd(te, vneg(q_lo)));
  }
#pragma unroll
  for (int i = 0; i < L; ++i)
    if (!finite(Lanes<V>::get(th, i)) || !finite(Lanes<V>::get(q_lo, i)))
      Lanes<V>::at(th, i) =
          master_update_plain(Lanes<V>::get(theta, i), Lanes<V>::get(m_new, i),
                              Lanes<V>::get(v_new, i), h.a_hi, h.b_hi, h.eps, EXT ? h.k_hi : 1.f);
  return th;
}

// The single-lane form of master_update, written with a branch instead of
// lane selects (fewer live registers); the same operations on every element.
template <bool EXT>
__device__ __forceinline__ float master_update_x1(float theta, float m_new, float v_new,
                                                  const Hyper& h) {
  float s, s_lo;
  if (v_new >= 0x1p-100f && v_new <= 3.402823466e38f) {
    float y = rsqrt_approx(v_new);
    s = __fmul_rn(v_new, y);
    float rr = __fmaf_rn(-s, s, v_new);
    s_lo = __fmul_rn(rr, __fmul_rn(0.5f, y));
  } else {
    s = __fsqrt_rn(v_new);
    s_lo = 0.f;
  }
  float p = __fmul_rn(s, h.b_hi);
  float pe = __fmaf_rn(s, h.b_hi, -p);
  float lo = __fmaf_rn(s, h.b_lo, __fmaf_rn(s_lo, h.b_hi, pe));
  float D, de;
  two_sum(p, h.eps, D, de);
  float D_lo = __fadd_rn(lo, de);
  float n = __fmul_rn(h.a_hi, m_new);
  float n_lo = __fmaf_rn(h.a_lo, m_new, __fmaf_rn(h.a_hi, m_new, -n));
  float rD = rcp_approx(D);
  float q = __fmul_rn(n, rD);
  float r = __fmaf_rn(-q, D, n);
  r = __fmaf_rn(-q, D_lo, __fadd_rn(r, n_lo));
  float q_lo = __fmul_rn(r, rD);
  float t, te, th;
  if constexpr (EXT) {
    float P = __fmul_rn(theta, h.k_hi);
    float Pe = __fmaf_rn(theta, h.k_lo, __fmaf_rn(theta, h.k_hi, -P));
    two_sum(P, -q, t, te);
    th = __fadd_rn(t, __fadd_rn(__fadd_rn(te, Pe), -q_lo));
  } else {
    two_sum(theta, -q, t, te);
    th = __fadd_rn(t, __fadd_rn(te, -q_lo));
  }
  if (!finite(th) || !finite(q_lo))
    th = master_update_plain(theta, m_new, v_new, h.a_hi, h.b_hi, h.eps, EXT ? h.k_hi : 1.f);
  return th;
}

// One step after the reduce: updates theta, m, v in place.
template <bool EXT, class V>
__device__ __forceinline__ void adam_update(V g, V& theta, V& m, V& v, const Hyper& h) {
  m = moment1(m, g, h);
  v = moment2(v, g, h);
  if constexpr (Lanes<V>::n == 1) theta = master_update_x1<EXT>(theta, m, v, h);
  else theta = master_update<V, EXT>(theta, m, v, h);
}

// bf16 bits of x, round to nearest, ties to even (PTX cvt.rn.bf16.f32).
__device__ __forceinline__ uint16_t to_bf16(float x) {
  unsigned short b;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(b) : "f"(x));
  return b;
}

// Two bf16 (RNE) packed in one word: lo in bits 0..15, hi in bits 16..31.
__device__ __forceinline__ uint32_t to_bf16x2(float lo, float hi) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
  return w;
}

// bf16 -> fp32 is exact: the 16 bits become the top half of a binary32.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(bf16_lo(w), bf16_hi(w));
}

}  // namespace dpopt

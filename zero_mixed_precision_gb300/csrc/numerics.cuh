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
// All operations use the explicitly rounded intrinsics so that the compiler
// neither contracts a multiply-add nor reorders anything.  When an input or a
// result is not finite, the element falls back to the plain IEEE fp32
// formula, which propagates Inf and NaN the way the fp64 evaluation does.
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
  float pad_;
};

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bp = __fsub_rn(s, a);
  float ap = __fsub_rn(s, bp);
  e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

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

// ---------------------------------------------------------------------------
// Reduce: running compensated sum over the replicas in ascending order.
// ---------------------------------------------------------------------------

struct CompSum {
  float s, c;  // s + c carries the partial sum with ~48 significant bits
  __device__ __forceinline__ void init(float x0) { s = x0; c = 0.f; }
  __device__ __forceinline__ void add(float x) {
    float t, e;
    two_sum(s, x, t, e);
    s = t;
    c = __fadd_rn(c, e);
  }
  // fl32(sum) then / N.  A non-finite running sum is returned as it is.
  __device__ __forceinline__ float average(const Hyper& h) const {
    float tot = finite(s) ? __fadd_rn(s, c) : s;
    return h.inv_n != 0.f ? __fmul_rn(tot, h.inv_n) : __fdiv_rn(tot, h.n_f);
  }
};

// ---------------------------------------------------------------------------
// Adam moments, each rounded (nearly always correctly) once to fp32.
// ---------------------------------------------------------------------------

// m' = beta1*m + (1-beta1)*g
__device__ __forceinline__ float moment1(float m, float g, const Hyper& h) {
  float p1 = __fmul_rn(h.beta1, m);
  float e1 = __fmaf_rn(h.beta1, m, -p1);
  float p2 = __fmul_rn(h.c1_hi, g);
  float e2 = __fmaf_rn(h.c1_lo, g, __fmaf_rn(h.c1_hi, g, -p2));
  float s, e3;
  two_sum(p1, p2, s, e3);
  float r = __fadd_rn(s, __fadd_rn(__fadd_rn(e1, e2), e3));
  if (!finite(r)) r = __fmaf_rn(h.beta1, m, __fmul_rn(h.c1_hi, g));
  return r;
}

// v' = beta2*v + (1-beta2)*g*g, formed as ((1-beta2)*g)*g so that the square
// overflows only where the rounded result itself would.
__device__ __forceinline__ float moment2(float v, float g, const Hyper& h) {
  float P = __fmul_rn(h.c2_hi, g);
  float Pe = __fmaf_rn(h.c2_lo, g, __fmaf_rn(h.c2_hi, g, -P));
  float p2 = __fmul_rn(P, g);
  float e2 = __fmaf_rn(Pe, g, __fmaf_rn(P, g, -p2));
  float p1 = __fmul_rn(h.beta2, v);
  float e1 = __fmaf_rn(h.beta2, v, -p1);
  float s, e3;
  two_sum(p1, p2, s, e3);
  float r = __fadd_rn(s, __fadd_rn(__fadd_rn(e1, e2), e3));
  if (!finite(r)) r = __fmaf_rn(h.beta2, v, p2);
  return r;
}

// theta' = theta - lr * (m'/bc1) / (sqrt(v'/bc2) + eps), the plain fp32 form,
// used for non-finite inputs or results.
__device__ __noinline__ float master_update_plain(float theta, float m_new, float v_new,
                                                  Hyper h) {
  float d = __fadd_rn(__fmul_rn(__fsqrt_rn(v_new), h.b_hi), h.eps);
  float delta = __fdiv_rn(__fmul_rn(h.a_hi, m_new), d);
  return __fsub_rn(theta, delta);
}

// theta' = theta - a*m' / (b*sqrt(v') + eps) with a = lr/bc1, b = 1/sqrt(bc2),
// the quotient carried as q + q_lo and the subtraction rounded once.
__device__ __forceinline__ float master_update(float theta, float m_new, float v_new,
                                               const Hyper& h) {
  float s, s_lo;
  if (v_new >= 0x1p-100f && v_new <= 3.402823466e38f) {
    float y = rsqrt_approx(v_new);
    s = __fmul_rn(v_new, y);
    float r = __fmaf_rn(-s, s, v_new);
    s_lo = __fmul_rn(r, __fmul_rn(0.5f, y));
  } else {
    s = __fsqrt_rn(v_new);
    s_lo = 0.f;
  }
  // D = b*sqrt(v') + eps as D + D_lo
  float p = __fmul_rn(s, h.b_hi);
  float pe = __fmaf_rn(s, h.b_hi, -p);
  float lo = __fmaf_rn(s, h.b_lo, __fmaf_rn(s_lo, h.b_hi, pe));
  float D, de;
  two_sum(p, h.eps, D, de);
  float D_lo = __fadd_rn(lo, de);
  // numerator a*m' as n + n_lo
  float n = __fmul_rn(h.a_hi, m_new);
  float n_lo = __fmaf_rn(h.a_lo, m_new, __fmaf_rn(h.a_hi, m_new, -n));
  // quotient q + q_lo = (n + n_lo) / (D + D_lo)
  float rD = rcp_approx(D);
  float q = __fmul_rn(n, rD);
  float r = __fmaf_rn(-q, D, n);
  r = __fmaf_rn(-q, D_lo, __fadd_rn(r, n_lo));
  float q_lo = __fmul_rn(r, rD);
  // theta - (q + q_lo), rounded once
  float t, te;
  two_sum(theta, -q, t, te);
  float th = __fadd_rn(t, __fsub_rn(te, q_lo));
  if (!finite(th) || !finite(q_lo)) th = master_update_plain(theta, m_new, v_new, h);
  return th;
}

// One element of the step after the reduce: updates theta, m, v in place.
__device__ __forceinline__ void adam_element(float g, float& theta, float& m, float& v,
                                             const Hyper& h) {
  m = moment1(m, g, h);
  v = moment2(v, g, h);
  theta = master_update(theta, m, v, h);
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

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace dpopt

/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the fused ZeRO gradient
 * reduce + mixed-precision Adam step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; it exists so that tests, the smoke check and the CPU
 * baseline of the benchmark can check the CUDA path against an independent
 * restatement of what the method computes.  It shares no code, header,
 * constant or helper with the CUDA library.
 *
 * Sources restated here (no code is printed on these pages for the update):
 *  - "Data Parallelism 数据并行（二）" (translation of "Data-Parallel
 *    Distributed Training of Deep Learning Models"), section "数据并行训练
 *    (DP)": the synchronised gradient is the sum of the local gradients
 *    times 1/#Nodes, and the floating-point summation order is a choice
 *    that changes the result.
 *  - "Почему training 70B модели требует optimizer sharding (ZeRO-3)?",
 *    section 5 (the ZeRO-3 step): reduce-scatter sums the gradients over all
 *    GPUs and each GPU keeps only its own shard; the optimizer then updates
 *    only that shard from its own gradient and optimizer-state shards.
 *  - "Глава 4.4 -- Распределённое обучение", section 2, and the appendix
 *    "DNN 训练的内存需求" of the DP page: fp32 master copy, fp32 first and
 *    second Adam moments, 16-bit working copy of the parameters.
 *  - The Adam equations themselves are not printed on any of the pages; the
 *    textbook bias-corrected form (Kingma & Ba, 2015, Algorithm 1) with eps
 *    added outside the square root is used.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *  - The replica sum runs in ascending replica order, in fp64.  For up to 64
 *    bf16 inputs this fp64 sum is exact unless the exponents span more than
 *    39 binades; it is then rounded once to fp32 ("the synchronised
 *    gradient") and divided by N, the quotient rounded to fp32.
 *  - Hyper-parameters are the fp32 values passed in, widened exactly to fp64.
 *  - m' and v' are formed in fp64 from the fp32 states and rounded to fp32
 *    for storage; the update is then computed in fp64 from the STORED fp32
 *    m' and v' (the state the optimizer keeps), theta' = fl32(theta - delta).
 *  - The bf16 working copy is the round-to-nearest-even bf16 of the stored
 *    fp32 master.
 *
 * Build: cc -O2 -ffp-contract=off -fPIC -shared [-fopenmp] oracle.c -lm
 * (no fast-math: every step must be the IEEE operation it says it is).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* bf16 and fp32 encodings                                              */
/* ------------------------------------------------------------------ */

/* bf16 is the upper 16 bits of an IEEE-754 binary32 (1 sign bit, 8 exponent
 * bits, 7 fraction bits), so widening it is exact: put the 16 bits on top of
 * 16 zero bits and read the result as a binary32. */
double orc_bf16_to_f64(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a binary32 to the nearest bf16, ties to even (IEEE-754 default
 * rounding).  For a fixed sign the binary32 encodings are ordered like their
 * magnitudes, so the two bf16 neighbours of x are the truncated upper half
 * (toward zero) and that plus one (away from zero); the discarded low 16
 * bits say how far x lies between them: below half -> truncate, above half
 * -> away, exactly half -> whichever neighbour has an even last bit.  A
 * carry out of the fraction moves to the next binade, and past the largest
 * finite value it lands on the infinity encoding, as it should.  NaN stays a
 * NaN (quiet bit set, sign kept). */
uint16_t orc_f32_to_bf16_rne(float x) {
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    if ((bits & 0x7F800000u) == 0x7F800000u && (bits & 0x007FFFFFu) != 0u) {
        return (uint16_t)((bits >> 16) | 0x0040u);
    }
    uint32_t upper = bits >> 16;
    uint32_t lower = bits & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) {
        upper += 1u;
    }
    return (uint16_t)upper;
}

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent field 0 holds zero and the subnormals f * 2^-24, field 31
 * the infinities and NaNs; otherwise the value is (1024 + f) * 2^(e - 25). */
double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double x;
    if (e == 0) x = ldexp((double)f, -24);
    else if (e == 31) x = f ? NAN : INFINITY;
    else x = ldexp((double)(1024 + f), e - 25);
    return sign ? -x : x;
}

/* ------------------------------------------------------------------ */
/* Reduce: fixed-order average of N replica gradients                   */
/* ------------------------------------------------------------------ */

#define ORC_GRAD_BF16 0
#define ORC_GRAD_F32 1
#define ORC_GRAD_F16 2

static double grad_at(const void *buf, int dtype, int64_t i) {
    if (dtype == ORC_GRAD_BF16) {
        return orc_bf16_to_f64(((const uint16_t *)buf)[i]);
    }
    if (dtype == ORC_GRAD_F16) {
        return orc_f16_to_f64(((const uint16_t *)buf)[i]);
    }
    return (double)((const float *)buf)[i];
}

/* g_i = fl32( fl32( sum_{r=0}^{N-1} x_r[i] ) / N ), the sum taken in fp64 in
 * ascending replica order.  Restates the gradient-averaging equation of the
 * DP page ("数据并行训练 (DP)": sum of the local gradients times
 * 1/#Nodes) with the order fixed (the same section says the order is a
 * choice that changes the floating-point result). */
float orc_average_one(const void *const *grads, int dtype, int n, int64_t i) {
    double s = 0.0;
    for (int r = 0; r < n; ++r) {
        s += grad_at(grads[r], dtype, i);
    }
    float s32 = (float)s;             /* one rounding of the (exact) sum */
    return (float)((double)s32 / (double)n); /* fp64 quotient rounded to fp32 */
}

/* ------------------------------------------------------------------ */
/* Adam on one element (textbook, bias-corrected, eps outside the sqrt)  */
/* ------------------------------------------------------------------ */

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    double bc1, bc2; /* 1 - beta1^t, 1 - beta2^t */
} orc_hyper;

static orc_hyper make_hyper(float lr, float beta1, float beta2, float eps,
                            float weight_decay, int64_t step) {
    orc_hyper h;
    h.lr = (double)lr;
    h.beta1 = (double)beta1;
    h.beta2 = (double)beta2;
    h.eps = (double)eps;
    h.weight_decay = (double)weight_decay;
    h.bc1 = 1.0 - pow(h.beta1, (double)step);
    h.bc2 = 1.0 - pow(h.beta2, (double)step);
    return h;
}

/* One Adam step on one element.  m_t = b1 m + (1-b1) g ; v_t = b2 v +
 * (1-b2) g^2 ; m_hat = m_t / (1-b1^t) ; v_hat = v_t / (1-b2^t) ;
 * theta -= lr m_hat / (sqrt(v_hat) + eps).  Moments are stored in fp32 and
 * the update uses the stored values.  With weight_decay != 0 the decay is
 * decoupled (AdamW, Loshchilov & Hutter 2019): theta -= lr * wd * theta,
 * applied to the pre-update theta, as the DeepSpeed example on the ZeRO-3
 * page configures ("optimizer": AdamW, weight_decay 0.01). */
static void adam_one(double g, float *theta, float *m, float *v, uint16_t *out,
                     const orc_hyper *h) {
    double m_new = h->beta1 * (double)(*m) + (1.0 - h->beta1) * g;
    double v_new = h->beta2 * (double)(*v) + (1.0 - h->beta2) * g * g;
    float m32 = (float)m_new;
    float v32 = (float)v_new;
    double m_hat = (double)m32 / h->bc1;
    double v_hat = (double)v32 / h->bc2;
    double delta = h->lr * m_hat / (sqrt(v_hat) + h->eps);
    double th = (double)(*theta);
    double th_new = th - delta;
    if (h->weight_decay != 0.0) { /* plain Adam has no decay term at all */
        th_new -= h->lr * h->weight_decay * th;
    }
    float th32 = (float)th_new;
    *m = m32;
    *v = v32;
    *theta = th32;
    if (out) {
        *out = orc_f32_to_bf16_rne(th32);
    }
}

/* ------------------------------------------------------------------ */
/* The composed step on a range of the flattened buffers                */
/* ------------------------------------------------------------------ */

/* Average the N replicas over elements [offset, offset+count) of the
 * flattened gradient buffers and apply one Adam step to the matching
 * count-element state arrays (state element j <-> gradient element
 * offset+j).  Returns 0, or -1 on a bad argument.  nthreads > 1 splits the
 * independent elements over OpenMP threads (no arithmetic is reordered). */
int orc_reduce_adam_range(const void *const *grads, int dtype, int n,
                          int64_t offset, int64_t count, float *master,
                          float *m, float *v, uint16_t *out, float lr,
                          float beta1, float beta2, float eps,
                          float weight_decay, int64_t step, int nthreads) {
    if (n < 1 || count < 0 || offset < 0 || step < 1) return -1;
    if (dtype != ORC_GRAD_BF16 && dtype != ORC_GRAD_F32 && dtype != ORC_GRAD_F16) return -1;
    orc_hyper h = make_hyper(lr, beta1, beta2, eps, weight_decay, step);
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
    for (int64_t j = 0; j < count; ++j) {
        float g = orc_average_one(grads, dtype, n, offset + j);
        adam_one((double)g, &master[j], &m[j], &v[j], out ? &out[j] : 0, &h);
    }
    (void)nthreads;
    return 0;
}

/* ZeRO form: rank `shard_rank` of N owns [shard_rank*S, (shard_rank+1)*S) of
 * every flattened replica buffer, S = numel / N ("Почему training 70B ...",
 * sections 3 and 5: each GPU keeps 1/N, reduce-scatter keeps its own shard,
 * the optimizer updates only that shard).  numel must be a multiple of N. */
int orc_reduce_adam_shard(const void *const *grads, int dtype, int n,
                          int64_t numel, int shard_rank, float *master, float *m,
                          float *v, uint16_t *out, float lr, float beta1,
                          float beta2, float eps, float weight_decay,
                          int64_t step, int nthreads) {
    if (n < 1 || numel < 0 || numel % n != 0) return -1;
    if (shard_rank < 0 || shard_rank >= n) return -1;
    int64_t s = numel / n;
    return orc_reduce_adam_range(grads, dtype, n, (int64_t)shard_rank * s, s,
                                 master, m, v, out, lr, beta1, beta2, eps,
                                 weight_decay, step, nthreads);
}

/* Element-wise gather form used for sampled checks of large workloads: the
 * gradients are given already gathered, grads[r][j] = replica r at the j-th
 * sampled element; states are the sampled elements' states. */
int orc_reduce_adam_gathered(const void *const *grads, int dtype, int n,
                             int64_t count, float *master, float *m, float *v,
                             uint16_t *out, float lr, float beta1, float beta2,
                             float eps, float weight_decay, int64_t step) {
    return orc_reduce_adam_range(grads, dtype, n, 0, count, master, m, v, out,
                                 lr, beta1, beta2, eps, weight_decay, step, 1);
}

/* ------------------------------------------------------------------ */
/* Global-norm gradient clipping (the clipping config of the ZeRO-3     */
/* answer's DeepSpeed example: gradient_clipping 1.0)                    */
/* ------------------------------------------------------------------ */

/* sum_i (g_i * unscale)^2 over elements [offset, offset+count), in fp64,
 * g_i the fixed-order average above.  The global squared norm of a model is
 * the sum of these over every rank's shard. */
double orc_grad_sqnorm(const void *const *grads, int dtype, int n, int64_t offset,
                       int64_t count, float unscale) {
    double acc = 0.0;
    for (int64_t j = 0; j < count; ++j) {
        double x = (double)orc_average_one(grads, dtype, n, offset + j) * (double)unscale;
        acc += x * x;
    }
    return acc;
}

/* The gradient multiplier: unscale * min(1, max_norm / (sqrt(sqnorm) + 1e-6))
 * evaluated in fp64 and rounded once to fp32 (max_norm <= 0: no clipping). */
float orc_grad_scale(double sqnorm, float max_norm, float unscale) {
    double c = (double)unscale;
    if (max_norm > 0.0f) {
        double coef = (double)max_norm / (sqrt(sqnorm) + 1e-6);
        if (coef < 1.0) c *= coef;
    }
    return (float)c;
}

/* One step with the averaged gradient multiplied by gscale first:
 * g' = fl32(g * gscale), then (Adam)W as above. */
int orc_reduce_adamw_range(const void *const *grads, int dtype, int n, int64_t offset,
                           int64_t count, float *master, float *m, float *v, uint16_t *out,
                           float lr, float beta1, float beta2, float eps, float weight_decay,
                           float gscale, int64_t step) {
    if (n < 1 || count < 0 || offset < 0 || step < 1) return -1;
    orc_hyper h = make_hyper(lr, beta1, beta2, eps, weight_decay, step);
    for (int64_t j = 0; j < count; ++j) {
        float g = orc_average_one(grads, dtype, n, offset + j);
        float gs = (float)((double)g * (double)gscale);
        adam_one((double)gs, &master[j], &m[j], &v[j], out ? &out[j] : 0, &h);
    }
    return 0;
}

/* Widen an array of binary16 bit patterns (pinned against a library). */
void orc_f16_to_f64_array(const uint16_t *h, int64_t count, double *out) {
    for (int64_t j = 0; j < count; ++j) out[j] = orc_f16_to_f64(h[j]);
}

/* Average only (no optimizer), for pinning the reduce half on its own. */
int orc_average(const void *const *grads, int dtype, int n, int64_t count,
                float *g_out) {
    if (n < 1 || count < 0) return -1;
    for (int64_t j = 0; j < count; ++j) {
        g_out[j] = orc_average_one(grads, dtype, n, j);
    }
    return 0;
}

/* Adam only, from an fp32 averaged gradient (pins the optimizer half). */
int orc_adam(const float *g, int64_t count, float *master, float *m, float *v,
             uint16_t *out, float lr, float beta1, float beta2, float eps,
             float weight_decay, int64_t step) {
    if (count < 0 || step < 1) return -1;
    orc_hyper h = make_hyper(lr, beta1, beta2, eps, weight_decay, step);
    for (int64_t j = 0; j < count; ++j) {
        adam_one((double)g[j], &master[j], &m[j], &v[j], out ? &out[j] : 0, &h);
    }
    return 0;
}

/* bf16 rounding of a whole array (pinned against a library routine). */
void orc_f32_to_bf16_array(const float *x, int64_t count, uint16_t *out) {
    for (int64_t j = 0; j < count; ++j) out[j] = orc_f32_to_bf16_rne(x[j]);
}

int orc_threads_available(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

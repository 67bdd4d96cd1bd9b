/*
 * synth.c -- seeded, counter-based synthetic input generator (host side).
 *
 * This module holds none of the method's arithmetic: it only draws the
 * gradients and optimizer states that both the CPU oracle and the CUDA path
 * are fed with.  The device-side twin (synth_dev.cu) implements the same
 * definition, so a large workload can be generated in device memory while the
 * host regenerates any sampled element bit-for-bit.
 *
 * Definition (every step is an exact integer operation or a single IEEE
 * binary64 operation, so both sides agree bit-for-bit):
 *   mix(z)      = SplitMix64 output function (Steele, Lea & Flood 2014):
 *                 z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                 z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31
 *   key         = mix(seed * GAMMA + mix(stream + 0x632BE59BD9B4E019))
 *   draw(i, j)  = mix(key + (8*i + j + 1) * GAMMA),  GAMMA = 0x9E3779B97F4A7C15
 *   uniforms    : draws j = 0..5 give twelve 32-bit halves k, u = (k + 1/2) 2^-32
 *   z           = (u_0 + ... + u_11) - 6      (Irwin-Hall(12): mean 0, var 1)
 *               = (k_0 + ... + k_11 + 6 - 6*2^32) * 2^-32, formed in 64-bit
 *                 integers and converted once (|.| < 2^36: exact in binary64)
 *   outlier     : draw j = 6, top 53 bits * 2^-53 < p  -> x *= outlier_scale
 *   x           = mu + sigma * z   (two roundings, never fused), |x| if asked
 *   fp32 value  = x rounded to nearest binary32; bf16 value = that binary32
 *                 rounded to nearest-even bf16; fp16 value = that binary32
 *                 rounded to nearest-even binary16 (subnormals kept, overflow
 *                 to infinity).
 * z is therefore exact; only mu + sigma*z rounds.
 *
 * Build: cc -O2 -ffp-contract=off -fPIC -shared synth.c
 */
#include <stdint.h>
#include <string.h>

#define SYN_GAMMA 0x9E3779B97F4A7C15ull

static uint64_t syn_mix(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z;
}

uint64_t syn_key(uint64_t seed, uint64_t stream) {
    return syn_mix(seed * SYN_GAMMA + syn_mix(stream + 0x632BE59BD9B4E019ull));
}

static uint64_t syn_draw(uint64_t key, uint64_t i, uint64_t j) {
    return syn_mix(key + (8u * i + j + 1u) * SYN_GAMMA);
}

typedef struct {
    double mu, sigma, outlier_p, outlier_scale;
    int absval;
} syn_dist;

static double syn_value(uint64_t key, uint64_t i, const syn_dist *d) {
    int64_t ksum = 0;
    for (uint64_t j = 0; j < 6; ++j) {
        uint64_t w = syn_draw(key, i, j);
        ksum += (int64_t)(w >> 32);
        ksum += (int64_t)(w & 0xFFFFFFFFull);
    }
    double z = (double)(ksum + 6 - 6 * (int64_t)0x100000000ll) * 0x1p-32;
    double prod = d->sigma * z;
    double x = d->mu + prod;
    if (d->outlier_p > 0.0) {
        uint64_t w = syn_draw(key, i, 6);
        double u = (double)(w >> 11) * 0x1p-53;
        if (u < d->outlier_p) x = x * d->outlier_scale;
    }
    if (d->absval && x < 0.0) x = -x;
    return x;
}

static uint16_t syn_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    uint32_t up = b >> 16, lowbits = b & 0xFFFFu;
    if (lowbits > 0x8000u || (lowbits == 0x8000u && (up & 1u))) up += 1u;
    return (uint16_t)up;
}

/* binary32 -> binary16, round to nearest even.  The binary16 value of a
 * binary32 f is f's significand cut to 11 bits (fewer for subnormal results)
 * at the bit position set by f's exponent; the cut-off bits decide the
 * rounding as usual: above half up, below half down, exactly half to even. */
static uint16_t syn_f16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    uint32_t sign = (b >> 16) & 0x8000u;
    uint32_t ex = (b >> 23) & 0xFFu;
    uint32_t man = b & 0x7FFFFFu;
    if (ex == 0xFFu) return (uint16_t)(sign | 0x7C00u | (man ? 0x200u : 0u));
    int e = (int)ex - 127;                 /* unbiased exponent */
    if (e > 15) return (uint16_t)(sign | 0x7C00u);
    if (ex == 0 || e < -25) return (uint16_t)sign; /* |f| < 2^-25 rounds to zero */
    uint32_t sig = man | 0x800000u;        /* 24-bit significand, value sig * 2^(e-23) */
    int shift;                             /* bits of sig to drop */
    uint32_t base;                         /* exponent field of the result */
    if (e >= -14) { shift = 13; base = (uint32_t)(e + 15) << 10; sig &= 0x7FFFFFu; sig |= 0x800000u; }
    else { shift = 13 + (-14 - e); base = 0; }
    uint32_t kept = sig >> shift;
    uint32_t rest = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (e >= -14) kept &= 0x3FFu;          /* the implicit bit lives in the exponent field */
    uint32_t r = base + kept;
    if (rest > half || (rest == half && (kept & 1u))) r += 1u;  /* carries into the exponent */
    return (uint16_t)(sign | r);
}

/* out[k] = value of element start+k, k < count.  kind 0: bf16, 1: fp32, 2: fp16. */
void syn_fill(void *out, int kind, int64_t start, int64_t count, uint64_t seed,
              uint64_t stream, double mu, double sigma, double outlier_p,
              double outlier_scale, int absval) {
    syn_dist d = {mu, sigma, outlier_p, outlier_scale, absval};
    uint64_t key = syn_key(seed, stream);
    for (int64_t k = 0; k < count; ++k) {
        float f = (float)syn_value(key, (uint64_t)(start + k), &d);
        if (kind == 0) ((uint16_t *)out)[k] = syn_bf16_rne(f);
        else if (kind == 2) ((uint16_t *)out)[k] = syn_f16_rne(f);
        else ((float *)out)[k] = f;
    }
}

/* out[k] = value of element idx[k]. */
void syn_gather(void *out, int kind, const int64_t *idx, int64_t count,
                uint64_t seed, uint64_t stream, double mu, double sigma,
                double outlier_p, double outlier_scale, int absval) {
    syn_dist d = {mu, sigma, outlier_p, outlier_scale, absval};
    uint64_t key = syn_key(seed, stream);
    for (int64_t k = 0; k < count; ++k) {
        float f = (float)syn_value(key, (uint64_t)idx[k], &d);
        if (kind == 0) ((uint16_t *)out)[k] = syn_bf16_rne(f);
        else if (kind == 2) ((uint16_t *)out)[k] = syn_f16_rne(f);
        else ((float *)out)[k] = f;
    }
}

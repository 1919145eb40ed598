/*
 * qwgen.c - seeded synthetic inputs for the batch-one Qwen3 decoder.
 *
 * This file holds none of the decoder's arithmetic.  It only draws random
 * numbers and lays them out as the tensors a Qwen3-0.6B-shape checkpoint
 * would hold (bf16 weights, uniform token ids, bf16 K/V fills), plus the
 * Q8 group-32 quantiser that turns bf16 weights into int8 codes and fp16
 * scales.  Both the CPU oracle and the CUDA path consume exactly these bytes.
 *
 * Random source: the PCG32 generator as frozen in "Portable WebAssembly
 * Runtime Architecture for TinyRustLM", section "Deterministic sampling
 * contract" (transition, output function, seeding, and the 24-bit uniform
 * u = (r >> 8) * 2^-24).  Jump-ahead uses the LCG stride method of
 * F. Brown, "Random Number Generation with Arbitrary Strides" (1994), so
 * that threads can start at any offset of one stream and produce the same
 * sequence as a single thread.
 *
 * Normal deviates: Box-Muller (1958) on consecutive uniform pairs, in
 * double, rounded to float and then to bf16 (round to nearest even).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PCG_MULT 6364136223846793005ULL

typedef struct {
    uint64_t state;
    uint64_t inc;
} qwg_pcg32;

static uint32_t pcg_next(qwg_pcg32 *r) {
    uint64_t old = r->state;
    r->state = old * PCG_MULT + r->inc;
    uint32_t xs = (uint32_t)(((old >> 18) ^ old) >> 27);
    uint32_t rot = (uint32_t)(old >> 59);
    return (xs >> rot) | (xs << ((32u - rot) & 31u));
}

static void pcg_seed(qwg_pcg32 *r, uint64_t seed, uint64_t stream) {
    r->state = 0;
    r->inc = (stream << 1) | 1u;
    pcg_next(r);
    r->state += seed;
    pcg_next(r);
}

/* Advance the LCG state by `delta` steps in O(log delta). */
static void pcg_advance(qwg_pcg32 *r, uint64_t delta) {
    uint64_t acc_mult = 1, acc_plus = 0;
    uint64_t cur_mult = PCG_MULT, cur_plus = r->inc;
    while (delta > 0) {
        if (delta & 1u) {
            acc_mult *= cur_mult;
            acc_plus = acc_plus * cur_mult + cur_plus;
        }
        cur_plus = (cur_mult + 1) * cur_plus;
        cur_mult *= cur_mult;
        delta >>= 1;
    }
    r->state = acc_mult * r->state + acc_plus;
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* IEEE binary32 -> binary16, round to nearest even (finite inputs). */
static uint16_t f32_to_f16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t a = u & 0x7fffffffu;
    if (a >= 0x7f800000u) return (uint16_t)(sign | 0x7c00u | (a > 0x7f800000u ? 0x200u : 0));
    if (a >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u); /* rounds to >= 65520 -> inf */
    int e = (int)(a >> 23) - 127;
    uint32_t mant = (a & 0x7fffffu) | 0x800000u;
    if (e >= -14) {
        /* normal half: keep 10 of 23 fraction bits */
        uint32_t h = ((uint32_t)(e + 15) << 10) | ((a >> 13) & 0x3ffu);
        uint32_t rest = a & 0x1fffu;
        if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1; /* carry may bump exponent: correct */
        return (uint16_t)(sign | h);
    }
    if (a < 0x33000000u) return (uint16_t)sign; /* below half of the smallest subnormal */
    /* subnormal half: value = mant * 2^(e-23); unit = 2^-24 -> shift = -(e-23) - 24 */
    int shift = -e - 1; /* number of bits dropped from the 24-bit significand, 14..24 */
    uint32_t h = mant >> shift;
    uint32_t rest = mant & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rest > half || (rest == half && (h & 1u))) h += 1;
    return (uint16_t)(sign | h);
}

static float f16_bits_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    float out;
    if (e == 0) {
        out = ldexpf((float)m, -24);
        if (sign) out = -out;
        return out;
    }
    uint32_t u = e == 31 ? (sign | 0x7f800000u | (m << 13)) : (sign | ((e + 112u) << 23) | (m << 13));
    memcpy(&out, &u, 4);
    return out;
}

/* ---------------------------------------------------------------- threads */

typedef struct {
    uint16_t *out;
    int64_t begin_pair, end_pair, n;
    uint64_t seed, stream;
    double mean, std;
} normal_job;

static void *normal_worker(void *p) {
    normal_job *j = (normal_job *)p;
    qwg_pcg32 r;
    pcg_seed(&r, j->seed, j->stream);
    pcg_advance(&r, (uint64_t)(2 * j->begin_pair));
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t pidx = j->begin_pair; pidx < j->end_pair; ++pidx) {
        uint32_t r1 = pcg_next(&r), r2 = pcg_next(&r);
        double u1 = (double)(r1 >> 8) * (1.0 / 16777216.0);
        double u2 = (double)(r2 >> 8) * (1.0 / 16777216.0);
        double rad = sqrt(-2.0 * log(1.0 - u1));
        double z0 = rad * cos(two_pi * u2), z1 = rad * sin(two_pi * u2);
        int64_t i0 = 2 * pidx;
        j->out[i0] = f32_to_bf16_rne((float)(j->mean + j->std * z0));
        if (i0 + 1 < j->n) j->out[i0 + 1] = f32_to_bf16_rne((float)(j->mean + j->std * z1));
    }
    return NULL;
}

/* n bf16 values ~ N(mean, std^2) from stream (seed, stream); identical for any nthreads. */
void qwgen_normal_bf16(uint16_t *out, int64_t n, uint64_t seed, uint64_t stream, double mean, double std,
                       int nthreads) {
    int64_t pairs = (n + 1) / 2;
    if (nthreads < 1) nthreads = 1;
    if (pairs < 65536) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    normal_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].out = out;
        jobs[t].n = n;
        jobs[t].begin_pair = pairs * t / nthreads;
        jobs[t].end_pair = pairs * (t + 1) / nthreads;
        jobs[t].seed = seed;
        jobs[t].stream = stream;
        jobs[t].mean = mean;
        jobs[t].std = std;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, normal_worker, &jobs[t]);
    normal_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* Raw PCG32 words (for checking the generator itself). */
void qwgen_pcg32_words(uint32_t *out, int64_t n, uint64_t seed, uint64_t stream, uint64_t skip) {
    qwg_pcg32 r;
    pcg_seed(&r, seed, stream);
    pcg_advance(&r, skip);
    for (int64_t i = 0; i < n; ++i) out[i] = pcg_next(&r);
}

/* Uniform token ids in [0, vocab): multiply-shift of one 32-bit word per id. */
void qwgen_tokens(int32_t *out, int64_t n, uint64_t seed, uint64_t stream, int32_t vocab) {
    qwg_pcg32 r;
    pcg_seed(&r, seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(((uint64_t)pcg_next(&r) * (uint64_t)vocab) >> 32);
}

/*
 * Symmetric int8 quantiser, one fp16 scale per row per group of 32 input
 * columns: s = fp16(maxabs / 127), q = clamp(round_half_away(w / f32(s)), -127, 127),
 * an all-zero group gets s = 0 and q = 0.  w is bf16 [rows, cols], cols % 32 == 0.
 */
void qwgen_quantize_q8_g32(const uint16_t *w, int64_t rows, int64_t cols, int8_t *q, uint16_t *s) {
    int64_t groups = cols / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < groups; ++g) {
            const uint16_t *src = w + r * cols + g * 32;
            float vals[32];
            float maxabs = 0.0f;
            for (int i = 0; i < 32; ++i) {
                uint32_t u = (uint32_t)src[i] << 16;
                memcpy(&vals[i], &u, 4);
                float a = fabsf(vals[i]);
                if (a > maxabs) maxabs = a;
            }
            uint16_t sh = f32_to_f16_rne(maxabs / 127.0f);
            float sf = f16_bits_to_f32(sh);
            s[r * groups + g] = sh;
            for (int i = 0; i < 32; ++i) {
                float v = 0.0f;
                if (sf != 0.0f) {
                    v = roundf(vals[i] / sf);
                    if (v > 127.0f) v = 127.0f;
                    if (v < -127.0f) v = -127.0f;
                }
                q[r * cols + g * 32 + i] = (int8_t)v;
            }
        }
    }
}

/* Elementwise helpers exposed for the generator's own tests. */
uint16_t qwgen_f32_to_f16(float f) { return f32_to_f16_rne(f); }
uint16_t qwgen_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }

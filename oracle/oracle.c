/*
 * oracle.c - plain fp32 CPU oracle of the batch-one Qwen3 decoder forward.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
 * baseline leg may load this library.  It shares no code, header, table or
 * helper with the CUDA path; the two meet only in the seeded input bytes.
 *
 * Numerical policy ("Scalar-Native Qwen3 Reference Runtime As The Numerical
 * Authority", section 4 "Floating-Point and Determinism Policy"): every
 * activation, accumulation and non-linearity is IEEE binary32; no fused
 * multiply-add (built with -ffp-contract=off, no fast-math); gradual
 * underflow; a NaN or infinity aborts the token with an error code.
 *
 * Operator sequence: the same page, section 2 "Decoder-Layer Mathematical
 * Formulation" steps 1-7 and the decode_layer walk-through of section 5:
 *   x0 = E[id]
 *   per layer: h = RMSNorm(x); q,k,v = W h; per-head QK-Norm; RoPE;
 *              append k,v; grouped-query attention; x += Wo o;
 *              h2 = RMSNorm(x); a = silu(Wg h2) * (Wu h2); x += Wd a
 *   logits = E RMSNorm(x) (tied head); greedy argmax, ties to the lowest id.
 * Dot products accumulate sequentially in k order (section 5 q8_dot:
 * acc += act[k] * (q * scale)).  Each output row is owned by exactly one
 * thread ("Portable WebAssembly Runtime Architecture", "Threads, Scheduling"
 * partitioning decision), so results do not depend on the thread count.
 *
 * Readings where the pages' equations were lost in extraction (each is also
 * listed with its reason in the repository's design notes):
 *   RMSNorm      y_i = w_i * (x_i * r),  r = 1 / sqrtf(sum(x^2)/n + eps)
 *   RoPE         half-split pairs (i, i + d/2), i < d/2:
 *                x'_i = x_i cos(p t_i) - x_{i+d/2} sin(p t_i)
 *                x'_{i+d/2} = x_{i+d/2} cos(p t_i) + x_i sin(p t_i)
 *                t_i = theta^(-2i/d); the angle, cos and sin in double, rounded to f32
 *   attention    s_j = (q . k_j) * (1/sqrt(d)); m = max s; e_j = expf(s_j - m);
 *                z = sum e_j (j order); o = sum_j (e_j / z) v_j (j order)
 *   SiLU         silu(g) = g * (1 / (1 + expf(-g)));  a = silu(g) * u
 *   Q8 x Q8      (weight format 2, "Real-Browser WASM Qwen3 Execution", section 5
 *                "Q8_0 Mixed-Precision Matrix Multiplication": the f32 input of every
 *                projection is quantized per 32-element block before the dot product):
 *                d = amax / 127; q_i = clamp(round-half-away(a_i / d), -127, 127)
 *                (all 0 when amax = 0); the block scale kept as fp16(d) (round to
 *                nearest even).  Per row, per block b in order: isum = sum of the 32
 *                products q_w q_a in i32 (|isum| <= 32 * 127 * 127 < 2^31, the
 *                "Integer-overflow rule" of "Portable WebAssembly Runtime
 *                Architecture"), acc += f32(isum) * (f32(s_w) * f32(s_a)).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
    ORA_OK = 0,
    ORA_INVALID_ARGUMENT = 1,
    ORA_UNSUPPORTED_QUANTIZATION = 12,
    ORA_UNSUPPORTED_SHAPE = 13,
    ORA_CONTEXT_EXCEEDED = 14,
    ORA_OUT_OF_MEMORY = 9,
    ORA_NUMERICAL_FAILURE = 18,
};

enum { ORA_W_BF16 = 0, ORA_W_INT8_G32 = 1, ORA_W_Q8Q8 = 2 };

typedef struct {
    int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab;
    float rms_eps;
    double rope_theta;
    int32_t max_ctx;
    int32_t weight_format;
    int32_t nthreads;
} ora_config;

/* Matrices in checkpoint order: q, k, v, o, gate, up, down. */
enum { M_Q = 0, M_K, M_V, M_O, M_GATE, M_UP, M_DOWN, M_COUNT };

typedef struct {
    const uint16_t *input_norm, *q_norm, *k_norm, *post_norm; /* bf16 */
    const void *w[M_COUNT];       /* bf16 [out,in], or int8 [out,in] (ORA_W_INT8_G32, ORA_W_Q8Q8) */
    const uint16_t *s[M_COUNT];   /* fp16 [out, in/32] scales (int8 formats only) */
} ora_layer;

typedef struct {
    int fmt;             /* ORA_W_BF16, ORA_W_INT8_G32 or ORA_W_Q8Q8 */
    int rows, cols;
    const void *w;
    const uint16_t *s;
} ora_mat;

typedef struct ora_model {
    ora_config cfg;
    const uint16_t *embed, *final_norm;
    ora_layer *layers;
    float *k_cache, *v_cache;   /* f32 [L][Hkv][max_ctx][d] */
    int32_t len;
    float *cos_t, *sin_t;       /* f32 [max_ctx][d/2] */
    int kv_round_bf16;          /* error attribution only: store K/V rounded to bf16 */
} ora_model;

/* ------------------------------------------------------------ scalars */

float ora_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE 754 binary16 -> binary32 (exact). */
float ora_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t e = (uint32_t)(h >> 10) & 0x1fu;
    uint32_t m = (uint32_t)h & 0x3ffu;
    float v;
    if (e == 0) {
        v = ldexpf((float)m, -24); /* subnormal: m * 2^-24, exact */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexpf((float)(1024u + m), (int)e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* IEEE 754 binary32 -> binary16, round to nearest even (overflow to infinity, gradual
 * underflow to subnormals). */
uint16_t ora_f32_to_f16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    const uint32_t e = (u >> 23) & 0xffu, m = u & 0x7fffffu;
    if (e == 0xffu) return (uint16_t)(sign | 0x7c00u | (m ? 0x200u : 0u));
    const float a = fabsf(f);
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7c00u);  /* rounds past the largest finite half */
    if (a < ldexpf(1.0f, -14)) {                          /* subnormal half: a multiple of 2^-24 */
        const float t = a * ldexpf(1.0f, 24);               /* exact: a power-of-two scaling */
        float r = rintf(t);                                 /* the default mode: nearest even */
        return (uint16_t)(sign | (uint16_t)r);              /* r = 1024 becomes the smallest normal */
    }
    /* normal: keep 10 mantissa bits, round the 13 dropped ones to nearest even */
    uint32_t he = e - 127 + 15, hm = m >> 13, rest = m & 0x1fffu;
    if (rest > 0x1000u || (rest == 0x1000u && (hm & 1u))) {
        hm += 1;
        if (hm == 0x400u) {
            hm = 0;
            he += 1;
        }
    }
    if (he >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (he << 10) | hm);
}

/* One 32-element activation block to int8 codes and its fp16 scale (the Q8 x Q8 reading above). */
void ora_quantize_q8_block(const float *a, int8_t *q, uint16_t *scale) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) amax = fabsf(a[i]) > amax ? fabsf(a[i]) : amax;
    const float d = amax / 127.0f;
    for (int i = 0; i < 32; ++i) {
        float v = d > 0.0f ? roundf(a[i] / d) : 0.0f;  /* roundf: halves away from zero */
        if (v > 127.0f) v = 127.0f;
        if (v < -127.0f) v = -127.0f;
        q[i] = (int8_t)v;
    }
    *scale = ora_f32_to_f16(d);
}

/* Integer dot product of one block: sum of 32 int8 x int8 products in i32. */
int32_t ora_q8_block_dot(const int8_t *w, const int8_t *a) {
    int32_t s = 0;
    for (int i = 0; i < 32; ++i) s += (int32_t)w[i] * (int32_t)a[i];
    return s;
}

float ora_silu(float g) {
    float sig = 1.0f / (1.0f + expf(-g));
    return g * sig;
}

static int finite_all(const float *x, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        if (!isfinite(x[i])) return 0;
    return 1;
}

/* ------------------------------------------------------- parallel rows */

typedef void (*row_fn)(void *ctx, int64_t begin, int64_t end);

typedef struct {
    row_fn fn;
    void *ctx;
    int64_t begin, end;
} row_job;

static void *row_worker(void *p) {
    row_job *j = (row_job *)p;
    j->fn(j->ctx, j->begin, j->end);
    return NULL;
}

static void parallel_rows(int nthreads, int64_t n, row_fn fn, void *ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < 64 || nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    if (nthreads > n) nthreads = (int)n;
    pthread_t th[256];
    row_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].begin = n * t / nthreads;
        jobs[t].end = n * (t + 1) / nthreads;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, row_worker, &jobs[t]);
    row_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------ dot rows */

/* y = W[row,:] . x, accumulated sequentially over k (int8: act * (q * scale)); Q8 x Q8: block by
 * block over the quantized input (xq codes, xs fp16 scales). */
static float mat_row_dot(const ora_mat *m, int64_t row, const float *x, const int8_t *xq, const uint16_t *xs) {
    float acc = 0.0f;
    if (m->fmt == ORA_W_Q8Q8) {
        const int8_t *q = (const int8_t *)m->w + row * m->cols;
        const uint16_t *s = m->s + row * (m->cols / 32);
        for (int b = 0; b < m->cols / 32; ++b) {
            const int32_t isum = ora_q8_block_dot(q + b * 32, xq + b * 32);
            acc += (float)isum * (ora_f16_to_f32(s[b]) * ora_f16_to_f32(xs[b]));
        }
    } else if (m->fmt == ORA_W_BF16) {
        const uint16_t *w = (const uint16_t *)m->w + row * m->cols;
        for (int k = 0; k < m->cols; ++k) acc += x[k] * ora_bf16_to_f32(w[k]);
    } else {
        const int8_t *q = (const int8_t *)m->w + row * m->cols;
        const uint16_t *s = m->s + row * (m->cols / 32);
        for (int b = 0; b < m->cols / 32; ++b) {
            float scale = ora_f16_to_f32(s[b]);
            for (int i = 0; i < 32; ++i) {
                float qv = (float)q[b * 32 + i];
                acc += x[b * 32 + i] * (qv * scale);
            }
        }
    }
    return acc;
}

typedef struct {
    const ora_mat *m;
    const float *x;
    float *y;
    const float *residual; /* NULL or residual added as y = residual + dot */
    const int8_t *xq;      /* Q8 x Q8: the quantized input */
    const uint16_t *xs;
} matvec_ctx;

static void matvec_rows(void *p, int64_t b, int64_t e) {
    matvec_ctx *c = (matvec_ctx *)p;
    for (int64_t r = b; r < e; ++r) {
        float d = mat_row_dot(c->m, r, c->x, c->xq, c->xs);
        c->y[r] = c->residual ? c->residual[r] + d : d;
    }
}

static void matvec(int nthreads, const ora_mat *m, const float *x, float *y, const float *residual) {
    matvec_ctx c = {m, x, y, residual, NULL, NULL};
    int8_t *xq = NULL;
    uint16_t *xs = NULL;
    if (m->fmt == ORA_W_Q8Q8) {  /* the input is quantized once, then every row reads it */
        xq = (int8_t *)malloc((size_t)m->cols);
        xs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(m->cols / 32));
        for (int b = 0; b < m->cols / 32; ++b) ora_quantize_q8_block(x + b * 32, xq + b * 32, xs + b);
        c.xq = xq;
        c.xs = xs;
    }
    parallel_rows(nthreads, m->rows, matvec_rows, &c);
    free(xq);
    free(xs);
}

/* Exposed for tests: y[r] = W[r,:] . x for one bf16 or int8 matrix. */
int ora_matvec(int fmt, const void *w, const uint16_t *s, int rows, int cols, const float *x, float *y,
               int nthreads) {
    if (fmt != ORA_W_BF16 && cols % 32) return ORA_UNSUPPORTED_QUANTIZATION;
    ora_mat m = {fmt, rows, cols, w, s};
    matvec(nthreads, &m, x, y, NULL);
    return ORA_OK;
}

/* --------------------------------------------------------- operators */

/* RMSNorm over n elements with bf16 weight w (w == NULL means unit weight). */
void ora_rmsnorm(const float *x, const uint16_t *w, int n, float eps, float *y) {
    float ss = 0.0f;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    float ms = ss / (float)n;
    float r = 1.0f / sqrtf(ms + eps);
    for (int i = 0; i < n; ++i) {
        float wi = w ? ora_bf16_to_f32(w[i]) : 1.0f;
        y[i] = wi * (x[i] * r);
    }
}

/* cos/sin of pos * theta^(-2i/d) for i < d/2, computed in double, rounded to f32. */
void ora_rope_angles(int pos, int d, double theta, float *cos_out, float *sin_out) {
    for (int i = 0; i < d / 2; ++i) {
        double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
        double ang = (double)pos * inv_freq;
        cos_out[i] = (float)cos(ang);
        sin_out[i] = (float)sin(ang);
    }
}

/* Rotate the half-split pairs (i, i + d/2) of one head vector in place. */
void ora_rope_apply(float *v, int d, const float *c, const float *s) {
    int half = d / 2;
    for (int i = 0; i < half; ++i) {
        float a = v[i], b = v[i + half];
        v[i] = a * c[i] - b * s[i];
        v[i + half] = b * c[i] + a * s[i];
    }
}

/*
 * QK-Norm then RoPE on one head vector (length d) in place: the head is
 * RMS-normalised with the shared per-dimension weight w, then rotated at
 * the position whose angles are c, s ("RoPE acts on the normalized queries
 * and keys", section 2 steps 3-4).
 */
void ora_qk_norm_rope(float *v, const uint16_t *w, int d, float eps, const float *c, const float *s,
                      float *tmp /* [d] */) {
    ora_rmsnorm(v, w, d, eps, tmp);
    memcpy(v, tmp, sizeof(float) * (size_t)d);
    ora_rope_apply(v, d, c, s);
}

/*
 * One attention head over n cached positions: q [d], K,V [n][d] (row stride
 * ld floats) -> o [d].  Returns ORA_NUMERICAL_FAILURE on a non-finite score
 * or normaliser, ORA_INVALID_ARGUMENT for n == 0.
 */
int ora_attention_head(const float *q, const float *K, const float *V, int n, int d, int64_t ld, float *o,
                       float *scratch /* [n] */) {
    if (n <= 0) return ORA_INVALID_ARGUMENT;
    float scale = (float)(1.0 / sqrt((double)d));
    float m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        float dot = 0.0f;
        const float *kj = K + (int64_t)j * ld;
        for (int t = 0; t < d; ++t) dot += q[t] * kj[t];
        float sj = dot * scale;
        if (!isfinite(sj)) return ORA_NUMERICAL_FAILURE;
        scratch[j] = sj;
        if (sj > m) m = sj;
    }
    float z = 0.0f;
    for (int j = 0; j < n; ++j) {
        scratch[j] = expf(scratch[j] - m);
        z += scratch[j];
    }
    if (!(z > 0.0f) || !isfinite(z)) return ORA_NUMERICAL_FAILURE;
    for (int t = 0; t < d; ++t) o[t] = 0.0f;
    for (int j = 0; j < n; ++j) {
        float p = scratch[j] / z;
        const float *vj = V + (int64_t)j * ld;
        for (int t = 0; t < d; ++t) o[t] += p * vj[t];
    }
    return ORA_OK;
}

/* Greedy pick: largest logit, lowest id on ties; any NaN/inf is an error. */
int ora_argmax(const float *logits, int64_t n, int32_t *out) {
    if (n <= 0) return ORA_INVALID_ARGUMENT;
    int64_t best = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (!isfinite(logits[i])) return ORA_NUMERICAL_FAILURE;
        if (logits[i] > logits[best]) best = i;
    }
    *out = (int32_t)best;
    return ORA_OK;
}

/* ------------------------------------------------------------- model */

static ora_mat layer_mat(const ora_model *md, const ora_layer *ly, int which) {
    const ora_config *c = &md->cfg;
    int qd = c->n_heads * c->head_dim, kvd = c->n_kv_heads * c->head_dim;
    int rows = 0, cols = 0;
    switch (which) {
        case M_Q: rows = qd; cols = c->hidden; break;
        case M_K: rows = kvd; cols = c->hidden; break;
        case M_V: rows = kvd; cols = c->hidden; break;
        case M_O: rows = c->hidden; cols = qd; break;
        case M_GATE: rows = c->intermediate; cols = c->hidden; break;
        case M_UP: rows = c->intermediate; cols = c->hidden; break;
        case M_DOWN: rows = c->hidden; cols = c->intermediate; break;
    }
    ora_mat m = {c->weight_format, rows, cols, ly->w[which], ly->s[which]};
    return m;
}

static int check_config(const ora_config *c) {
    if (c->n_layers < 1 || c->hidden < 1 || c->n_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 2 ||
        c->intermediate < 1 || c->vocab < 1 || c->max_ctx < 1)
        return ORA_INVALID_ARGUMENT;
    if (c->n_heads % c->n_kv_heads || c->head_dim % 2) return ORA_UNSUPPORTED_SHAPE;
    if (c->weight_format != ORA_W_BF16 &&
        (c->hidden % 32 || c->intermediate % 32 || (c->n_heads * c->head_dim) % 32))
        return ORA_UNSUPPORTED_QUANTIZATION;
    if (c->weight_format != ORA_W_BF16 && c->weight_format != ORA_W_INT8_G32 && c->weight_format != ORA_W_Q8Q8)
        return ORA_UNSUPPORTED_QUANTIZATION;
    return ORA_OK;
}

int ora_create(const ora_config *cfg, const uint16_t *embed, const uint16_t *final_norm, const ora_layer *layers,
               ora_model **out) {
    *out = NULL;
    int rc = check_config(cfg);
    if (rc) return rc;
    ora_model *m = (ora_model *)calloc(1, sizeof(ora_model));
    m->cfg = *cfg;
    m->embed = embed;
    m->final_norm = final_norm;
    m->layers = (ora_layer *)malloc(sizeof(ora_layer) * (size_t)cfg->n_layers);
    memcpy(m->layers, layers, sizeof(ora_layer) * (size_t)cfg->n_layers);
    size_t kv = (size_t)cfg->n_layers * cfg->n_kv_heads * (size_t)cfg->max_ctx * cfg->head_dim;
    m->k_cache = (float *)malloc(kv * sizeof(float));
    m->v_cache = (float *)malloc(kv * sizeof(float));
    int half = cfg->head_dim / 2;
    m->cos_t = (float *)malloc(sizeof(float) * (size_t)cfg->max_ctx * half);
    m->sin_t = (float *)malloc(sizeof(float) * (size_t)cfg->max_ctx * half);
    if (!m->k_cache || !m->v_cache || !m->cos_t || !m->sin_t) {
        free(m->k_cache); free(m->v_cache); free(m->cos_t); free(m->sin_t); free(m->layers); free(m);
        return ORA_INVALID_ARGUMENT;
    }
    for (int p = 0; p < cfg->max_ctx; ++p)
        ora_rope_angles(p, cfg->head_dim, cfg->rope_theta, m->cos_t + (size_t)p * half, m->sin_t + (size_t)p * half);
    m->len = 0;
    *out = m;
    return ORA_OK;
}

void ora_destroy(ora_model *m) {
    if (!m) return;
    free(m->k_cache); free(m->v_cache); free(m->cos_t); free(m->sin_t); free(m->layers); free(m);
}

int32_t ora_length(const ora_model *m) { return m->len; }

void ora_kv_reset(ora_model *m) { m->len = 0; }

static float *kv_row(const ora_model *m, float *base, int l, int kvh, int pos) {
    const ora_config *c = &m->cfg;
    return base + (((size_t)l * c->n_kv_heads + kvh) * (size_t)c->max_ctx + pos) * c->head_dim;
}

/* Replace the cache with n_pos positions of bf16 K/V, layout [L][Hkv][n_pos][d]. */
int ora_kv_import(ora_model *m, const uint16_t *k, const uint16_t *v, int32_t n_pos) {
    const ora_config *c = &m->cfg;
    if (n_pos < 0 || n_pos > c->max_ctx) return ORA_CONTEXT_EXCEEDED;
    for (int l = 0; l < c->n_layers; ++l)
        for (int h = 0; h < c->n_kv_heads; ++h)
            for (int p = 0; p < n_pos; ++p) {
                size_t src = (((size_t)l * c->n_kv_heads + h) * (size_t)n_pos + p) * c->head_dim;
                float *kd = kv_row(m, m->k_cache, l, h, p), *vd = kv_row(m, m->v_cache, l, h, p);
                for (int t = 0; t < c->head_dim; ++t) {
                    kd[t] = ora_bf16_to_f32(k[src + t]);
                    vd[t] = ora_bf16_to_f32(v[src + t]);
                }
            }
    m->len = n_pos;
    return ORA_OK;
}

/*
 * Error attribution switch (not part of the reference computation): when set,
 * K/V rows are rounded to bf16 (nearest even) as they are stored, which
 * isolates the effect of a bf16 cache from every other source of difference.
 */
void ora_set_kv_round_bf16(ora_model *m, int on) { m->kv_round_bf16 = on; }

static float round_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    u &= 0xffff0000u;
    memcpy(&f, &u, 4);
    return f;
}

/* Copy the cached f32 key and value rows of (layer, kv head, position). */
int ora_kv_row(const ora_model *m, int l, int kvh, int pos, float *k, float *v) {
    const ora_config *c = &m->cfg;
    if (l < 0 || l >= c->n_layers || kvh < 0 || kvh >= c->n_kv_heads || pos < 0 || pos >= m->len)
        return ORA_INVALID_ARGUMENT;
    memcpy(k, kv_row(m, m->k_cache, l, kvh, pos), sizeof(float) * (size_t)c->head_dim);
    memcpy(v, kv_row(m, m->v_cache, l, kvh, pos), sizeof(float) * (size_t)c->head_dim);
    return ORA_OK;
}

typedef struct {
    const ora_model *m;
    int l, pos;
    const float *q; /* [Hq][d] roped */
    float *o;       /* [Hq][d] */
    float *scratch; /* [Hq][pos+1] */
    int rc[256];
} attn_ctx;

static void attn_heads(void *p, int64_t b, int64_t e) {
    attn_ctx *a = (attn_ctx *)p;
    const ora_config *c = &a->m->cfg;
    int g = c->n_heads / c->n_kv_heads;
    for (int64_t h = b; h < e; ++h) {
        int kvh = (int)h / g;
        const float *K = kv_row(a->m, a->m->k_cache, a->l, kvh, 0);
        const float *V = kv_row(a->m, a->m->v_cache, a->l, kvh, 0);
        a->rc[h] = ora_attention_head(a->q + h * c->head_dim, K, V, a->pos + 1, c->head_dim, c->head_dim,
                                      a->o + h * c->head_dim, a->scratch + h * (int64_t)(a->pos + 1));
    }
}

/*
 * One token through one decoder layer at position pos; x [H] updated in place.
 * k and v of this position are written into the cache.
 */
static int layer_step(ora_model *md, int l, float *x, int pos, float *buf) {
    const ora_config *c = &md->cfg;
    const ora_layer *ly = &md->layers[l];
    int H = c->hidden, d = c->head_dim, Hq = c->n_heads, Hkv = c->n_kv_heads, I = c->intermediate;
    int nt = c->nthreads;
    float *h = buf;                 /* [max(H, I)] */
    float *q = h + (H > I ? H : I); /* [Hq*d] */
    float *k = q + Hq * d;          /* [Hkv*d] */
    float *v = k + Hkv * d;         /* [Hkv*d] */
    float *o = v + Hkv * d;         /* [Hq*d] */
    float *g = o + Hq * d;          /* [I] */
    float *u = g + I;               /* [I] */
    float *tmp = u + I;             /* [d] */
    float *scratch = tmp + d;       /* [Hq*(pos+1)] */

    /* 1. pre-attention RMSNorm */
    ora_rmsnorm(x, ly->input_norm, H, c->rms_eps, h);
    /* 2. bias-free projections */
    ora_mat mq = layer_mat(md, ly, M_Q), mk = layer_mat(md, ly, M_K), mv = layer_mat(md, ly, M_V);
    matvec(nt, &mq, h, q, NULL);
    matvec(nt, &mk, h, k, NULL);
    matvec(nt, &mv, h, v, NULL);
    /* 3. QK-Norm per head, 4. RoPE at this position */
    const float *cs = md->cos_t + (size_t)pos * (d / 2), *sn = md->sin_t + (size_t)pos * (d / 2);
    for (int hh = 0; hh < Hq; ++hh) ora_qk_norm_rope(q + hh * d, ly->q_norm, d, c->rms_eps, cs, sn, tmp);
    for (int hh = 0; hh < Hkv; ++hh) ora_qk_norm_rope(k + hh * d, ly->k_norm, d, c->rms_eps, cs, sn, tmp);
    /* 5. K/V append at [l][kvh][pos][:] */
    for (int hh = 0; hh < Hkv; ++hh) {
        float *kd = kv_row(md, md->k_cache, l, hh, pos), *vd = kv_row(md, md->v_cache, l, hh, pos);
        memcpy(kd, k + hh * d, sizeof(float) * d);
        memcpy(vd, v + hh * d, sizeof(float) * d);
        if (md->kv_round_bf16)
            for (int t = 0; t < d; ++t) {
                kd[t] = round_bf16(kd[t]);
                vd[t] = round_bf16(vd[t]);
            }
    }
    /* 6. grouped-query attention over positions 0..pos */
    attn_ctx ac;
    ac.m = md; ac.l = l; ac.pos = pos; ac.q = q; ac.o = o; ac.scratch = scratch;
    memset(ac.rc, 0, sizeof(ac.rc));
    parallel_rows(Hq >= 4 ? nt : 1, Hq, attn_heads, &ac);
    for (int hh = 0; hh < Hq; ++hh)
        if (ac.rc[hh]) return ac.rc[hh];
    /* 7. output projection with residual */
    ora_mat mo = layer_mat(md, ly, M_O);
    matvec(nt, &mo, o, x, x);
    /* 8. SwiGLU MLP with residual */
    ora_rmsnorm(x, ly->post_norm, H, c->rms_eps, h);
    ora_mat mg = layer_mat(md, ly, M_GATE), mu = layer_mat(md, ly, M_UP), mdn = layer_mat(md, ly, M_DOWN);
    matvec(nt, &mg, h, g, NULL);
    matvec(nt, &mu, h, u, NULL);
    for (int i = 0; i < I; ++i) g[i] = ora_silu(g[i]) * u[i];
    matvec(nt, &mdn, g, x, x);
    if (!finite_all(x, H)) return ORA_NUMERICAL_FAILURE;
    return ORA_OK;
}

static size_t step_buf_floats(const ora_config *c, int pos) {
    int H = c->hidden, I = c->intermediate, d = c->head_dim;
    return (size_t)(H > I ? H : I) + (size_t)2 * c->n_heads * d + (size_t)2 * c->n_kv_heads * d + 2 * (size_t)I +
           (size_t)d + (size_t)c->n_heads * (pos + 1);
}

/* Final RMSNorm and tied lm_head: logits[v] = E[v,:] . RMSNorm(x). */
static int head_logits(const ora_model *md, const float *x, float *logits, float *hf) {
    const ora_config *c = &md->cfg;
    ora_rmsnorm(x, md->final_norm, c->hidden, c->rms_eps, hf);
    ora_mat e = {ORA_W_BF16, c->vocab, c->hidden, md->embed, NULL};
    matvec(c->nthreads, &e, hf, logits, NULL);
    return finite_all(logits, c->vocab) ? ORA_OK : ORA_NUMERICAL_FAILURE;
}

/*
 * Decode one token at position len: logits [V] and, if hidden != NULL, the
 * residual stream [L+1][H] (index 0 = embedding row, l+1 = after layer l).
 * logits == NULL skips the final norm and head: a prompt row other than the
 * last only has to leave its K/V in the cache (final norm, head and argmax act
 * on the last prompt row, "Portable WebAssembly Runtime Architecture for
 * TinyRustLM", section "Prefill versus decode").  On an error the cache length
 * is unchanged.
 */
int ora_step(ora_model *md, int32_t token, float *logits, float *hidden) {
    const ora_config *c = &md->cfg;
    if (token < 0 || token >= c->vocab) return ORA_INVALID_ARGUMENT;
    if (md->len + 1 > c->max_ctx) return ORA_CONTEXT_EXCEEDED;
    int pos = md->len, H = c->hidden;
    float *x = (float *)malloc(sizeof(float) * (size_t)H * 2);
    float *buf = (float *)malloc(sizeof(float) * step_buf_floats(c, pos));
    const uint16_t *e = md->embed + (size_t)token * H;
    for (int i = 0; i < H; ++i) x[i] = ora_bf16_to_f32(e[i]);
    if (hidden) memcpy(hidden, x, sizeof(float) * H);
    int rc = ORA_OK;
    for (int l = 0; l < c->n_layers && !rc; ++l) {
        rc = layer_step(md, l, x, pos, buf);
        if (hidden) memcpy(hidden + (size_t)(l + 1) * H, x, sizeof(float) * H);
    }
    if (!rc && logits) rc = head_logits(md, x, logits, x + H);
    free(x);
    free(buf);
    if (!rc) md->len = pos + 1;
    return rc;
}

/*
 * Full-sequence recomputation with no cache reuse: all T positions pass
 * through each layer together and attention applies the causal mask
 * explicitly (position t sees j <= t).  logits [T][V].  Uses private K/V
 * arrays; the model's own cache and length are untouched.
 */
int ora_full(const ora_model *md, const int32_t *tokens, int32_t T, float *logits) {
    const ora_config *c = &md->cfg;
    if (T <= 0 || T > c->max_ctx) return ORA_INVALID_ARGUMENT;
    int H = c->hidden, d = c->head_dim, Hq = c->n_heads, Hkv = c->n_kv_heads, I = c->intermediate;
    int g = Hq / Hkv, nt = c->nthreads;
    float *X = (float *)malloc(sizeof(float) * (size_t)T * H);
    float *h = (float *)malloc(sizeof(float) * (size_t)(H > I ? H : I));
    float *Q = (float *)malloc(sizeof(float) * (size_t)T * Hq * d);
    float *K = (float *)malloc(sizeof(float) * (size_t)T * Hkv * d);
    float *V = (float *)malloc(sizeof(float) * (size_t)T * Hkv * d);
    float *Kh = (float *)malloc(sizeof(float) * (size_t)T * d);
    float *Vh = (float *)malloc(sizeof(float) * (size_t)T * d);
    float *O = (float *)malloc(sizeof(float) * (size_t)T * Hq * d);
    float *G = (float *)malloc(sizeof(float) * (size_t)I);
    float *U = (float *)malloc(sizeof(float) * (size_t)I);
    float *tmp = (float *)malloc(sizeof(float) * (size_t)d);
    float *scr = (float *)malloc(sizeof(float) * (size_t)T);
    int rc = ORA_OK;
    for (int t = 0; t < T; ++t) {
        if (tokens[t] < 0 || tokens[t] >= c->vocab) { rc = ORA_INVALID_ARGUMENT; goto done; }
        for (int i = 0; i < H; ++i) X[(size_t)t * H + i] = ora_bf16_to_f32(md->embed[(size_t)tokens[t] * H + i]);
    }
    for (int l = 0; l < c->n_layers; ++l) {
        const ora_layer *ly = &md->layers[l];
        ora_mat mq = layer_mat(md, ly, M_Q), mk = layer_mat(md, ly, M_K), mv = layer_mat(md, ly, M_V);
        ora_mat mo = layer_mat(md, ly, M_O), mg = layer_mat(md, ly, M_GATE), mu = layer_mat(md, ly, M_UP);
        ora_mat mdn = layer_mat(md, ly, M_DOWN);
        for (int t = 0; t < T; ++t) {
            float *x = X + (size_t)t * H;
            float *q = Q + (size_t)t * Hq * d, *k = K + (size_t)t * Hkv * d, *v = V + (size_t)t * Hkv * d;
            ora_rmsnorm(x, ly->input_norm, H, c->rms_eps, h);
            matvec(nt, &mq, h, q, NULL);
            matvec(nt, &mk, h, k, NULL);
            matvec(nt, &mv, h, v, NULL);
            const float *cs = md->cos_t + (size_t)t * (d / 2), *sn = md->sin_t + (size_t)t * (d / 2);
            for (int hh = 0; hh < Hq; ++hh) ora_qk_norm_rope(q + hh * d, ly->q_norm, d, c->rms_eps, cs, sn, tmp);
            for (int hh = 0; hh < Hkv; ++hh) ora_qk_norm_rope(k + hh * d, ly->k_norm, d, c->rms_eps, cs, sn, tmp);
        }
        for (int hh = 0; hh < Hq; ++hh) {
            int kvh = hh / g;
            for (int j = 0; j < T; ++j) {
                memcpy(Kh + (size_t)j * d, K + ((size_t)j * Hkv + kvh) * d, sizeof(float) * d);
                memcpy(Vh + (size_t)j * d, V + ((size_t)j * Hkv + kvh) * d, sizeof(float) * d);
            }
            for (int t = 0; t < T; ++t) {
                /* causal mask: position t attends to positions 0..t only */
                rc = ora_attention_head(Q + ((size_t)t * Hq + hh) * d, Kh, Vh, t + 1, d, d,
                                        O + ((size_t)t * Hq + hh) * d, scr);
                if (rc) goto done;
            }
        }
        for (int t = 0; t < T; ++t) {
            float *x = X + (size_t)t * H;
            matvec(nt, &mo, O + (size_t)t * Hq * d, x, x);
            ora_rmsnorm(x, ly->post_norm, H, c->rms_eps, h);
            matvec(nt, &mg, h, G, NULL);
            matvec(nt, &mu, h, U, NULL);
            for (int i = 0; i < I; ++i) G[i] = ora_silu(G[i]) * U[i];
            matvec(nt, &mdn, G, x, x);
        }
    }
    for (int t = 0; t < T && !rc; ++t) rc = head_logits(md, X + (size_t)t * H, logits + (size_t)t * c->vocab, h);
done:
    free(X); free(h); free(Q); free(K); free(V); free(Kh); free(Vh); free(O); free(G); free(U); free(tmp); free(scr);
    return rc;
}

/* ------------------------------------------------------------- sampling
 *
 * The sampler of "Portable WebAssembly Runtime Architecture for TinyRustLM",
 * sections "Deterministic sampling contract" (PCG32: transition, seeding and the
 * f32 uniform) and "Sampling order", with the repetition penalty of "Scalar-Native
 * Qwen3 Reference Runtime ...", section 7 (a repeated positive logit is divided by
 * the penalty, a repeated negative one multiplied).  Readings where the two pages
 * differ or stay open: the nucleus keeps the minimal prefix whose cumulative
 * probability is at least top_p (the former page; the latter says "exceeds");
 * probabilities of the top-k survivors are renormalised before the nucleus and the
 * nucleus is renormalised before the draw; a draw u picks the first candidate whose
 * cumulative probability exceeds u (the last one if rounding leaves none); every
 * sampled (temperature > 0) step consumes exactly one PCG32 word, a greedy step
 * none; top_k <= 0 keeps every token.  All arithmetic is binary32 in candidate
 * order. */

typedef struct {
    uint64_t state, inc;
} ora_pcg32;

static uint32_t ora_pcg32_next(ora_pcg32 *r) {
    const uint64_t old = r->state;
    r->state = old * 6364136223846793005ULL + r->inc;
    const uint32_t xorshifted = (uint32_t)(((old >> 18) ^ old) >> 27);
    const uint32_t rot = (uint32_t)(old >> 59);
    return (xorshifted >> rot) | (xorshifted << ((32u - rot) & 31u));
}

/* Seeded state: state 0, increment (stream << 1) | 1, advance, add the seed, advance. */
void ora_pcg32_seed(uint64_t seed, uint64_t stream, uint64_t out[2]) {
    ora_pcg32 r = {0, (stream << 1) | 1u};
    (void)ora_pcg32_next(&r);
    r.state += seed;
    (void)ora_pcg32_next(&r);
    out[0] = r.state;
    out[1] = r.inc;
}

static int cand_before(float xa, int32_t ia, float xb, int32_t ib) {
    return xa > xb || (xa == xb && ia < ib);  /* descending value, ascending id */
}

/*
 * logits [V] (unchanged), history [n_hist] token ids (each present token penalised
 * once), rng [2] = (state, increment) updated in place.  Outputs: the token; and,
 * when the arrays are given, the retained candidates in draw order (ids), their
 * cumulative probabilities, their count, and the draw u (-1 for a greedy step).
 * Errors: INVALID_ARGUMENT for V <= 0, a token id out of range, a non-positive or
 * non-finite penalty or a negative / non-finite temperature, top_p outside (0, 1];
 * NUMERICAL_FAILURE when every logit is -inf (nothing can be drawn).
 */
int ora_sample(const float *logits, int32_t V, const int32_t *history, int32_t n_hist, float temperature,
               int32_t top_k, float top_p, float penalty, uint64_t rng[2], int32_t *token, int32_t *ids_out,
               float *cum_out, int32_t *n_out, float *u_out) {
    if (V <= 0 || n_hist < 0 || !token || !rng) return ORA_INVALID_ARGUMENT;
    if (!(penalty > 0.0f) || !isfinite(penalty)) return ORA_INVALID_ARGUMENT;
    if (!(temperature >= 0.0f) || !isfinite(temperature)) return ORA_INVALID_ARGUMENT;
    if (!(top_p > 0.0f) || top_p > 1.0f) return ORA_INVALID_ARGUMENT;
    float *x = (float *)malloc(sizeof(float) * (size_t)V);
    int32_t *ord = (int32_t *)malloc(sizeof(int32_t) * (size_t)V);
    unsigned char *seen = (unsigned char *)calloc((size_t)V, 1);
    float *p = (float *)malloc(sizeof(float) * (size_t)V);
    int rc = ORA_OK;
    if (!x || !ord || !seen || !p) {
        rc = ORA_OUT_OF_MEMORY;
        goto out;
    }
    /* 1. logits in token-id order */
    memcpy(x, logits, sizeof(float) * (size_t)V);
    /* 3. repetition penalty, once per distinct token of the history */
    for (int32_t i = 0; i < n_hist; ++i) {
        const int32_t t = history[i];
        if (t < 0 || t >= V) {
            rc = ORA_INVALID_ARGUMENT;
            goto out;
        }
        if (seen[t]) continue;
        seen[t] = 1;
        if (x[t] > 0.0f)
            x[t] = x[t] / penalty;
        else if (x[t] < 0.0f)
            x[t] = x[t] * penalty;
    }
    /* NaN -> -inf, -0 -> +0 */
    int any = 0;
    for (int32_t i = 0; i < V; ++i) {
        if (isnan(x[i])) x[i] = -INFINITY;
        if (x[i] == 0.0f) x[i] = 0.0f;
        if (x[i] != -INFINITY) any = 1;
    }
    if (!any) {
        rc = ORA_NUMERICAL_FAILURE;
        goto out;
    }
    /* temperature 0: the greatest logit, lowest id on ties, no draw */
    if (temperature == 0.0f) {
        int32_t best = 0;
        for (int32_t i = 1; i < V; ++i)
            if (cand_before(x[i], i, x[best], best)) best = i;
        *token = best;
        if (ids_out) ids_out[0] = best;
        if (cum_out) cum_out[0] = 1.0f;
        if (n_out) *n_out = 1;
        if (u_out) *u_out = -1.0f;
        goto out;
    }
    for (int32_t i = 0; i < V; ++i) x[i] = x[i] / temperature;
    /* top-k: descending logit, ascending id (insertion into a sorted prefix of k) */
    const int32_t k = (top_k <= 0 || top_k > V) ? V : top_k;
    int32_t nk = 0;
    for (int32_t i = 0; i < V; ++i) {
        if (nk == k && !cand_before(x[i], i, x[ord[k - 1]], ord[k - 1])) continue;
        int32_t j = nk < k ? nk++ : k - 1;
        while (j > 0 && cand_before(x[i], i, x[ord[j - 1]], ord[j - 1])) {
            ord[j] = ord[j - 1];
            --j;
        }
        ord[j] = i;
    }
    /* stable probabilities over the survivors (max-shifted exp, sum in order) */
    const float m = x[ord[0]];
    float s = 0.0f;
    for (int32_t j = 0; j < nk; ++j) {
        p[j] = expf(x[ord[j]] - m);
        s = s + p[j];
    }
    for (int32_t j = 0; j < nk; ++j) p[j] = p[j] / s;
    /* top-p: the minimal prefix whose cumulative probability is at least top_p */
    int32_t n = nk;
    if (top_p < 1.0f) {
        float c = 0.0f;
        for (int32_t j = 0; j < nk; ++j) {
            c = c + p[j];
            if (c >= top_p) {
                n = j + 1;
                break;
            }
        }
    }
    /* renormalise the nucleus; cumulative scan in the same order */
    float z = 0.0f;
    for (int32_t j = 0; j < n; ++j) z = z + p[j];
    /* one PCG32 word -> u = (w >> 8) * 2^-24 in [0, 1) */
    ora_pcg32 g = {rng[0], rng[1]};
    const uint32_t w = ora_pcg32_next(&g);
    rng[0] = g.state;
    const float u = (float)(w >> 8) * (1.0f / 16777216.0f);
    /* the first candidate whose cumulative probability exceeds u */
    int32_t pick = -1;
    float c = 0.0f;
    for (int32_t j = 0; j < n; ++j) {
        c = c + p[j] / z;
        if (cum_out) cum_out[j] = c;
        if (ids_out) ids_out[j] = ord[j];
        if (pick < 0 && c > u) pick = j;
    }
    if (pick < 0) pick = n - 1;
    *token = ord[pick];
    if (n_out) *n_out = n;
    if (u_out) *u_out = u;
out:
    free(x);
    free(ord);
    free(seen);
    free(p);
    return rc;
}

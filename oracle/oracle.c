/*
 * oracle.c -- plain FP64 CPU oracle of the BF16Optimizer step (see oracle.h).
 *
 * TEST INFRASTRUCTURE: loaded only by the tests, the smoke check and the
 * benchmark's CPU leg.  Built with -std=c11 -ffp-contract=off so that every
 * FP64 operation is rounded separately, on x86 and on Arm alike.
 *
 * Parity pins (closed forms, invariants, library special cases and brute force)
 * live in tests/test_oracle_pins.py and tests/test_oracle_xcheck.py.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#include "../synth/synth.h"

/* ---------------------------------------------------------------- helpers */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bf16 is the upper half of an IEEE binary32.  Round to nearest, ties to even
 * (IEEE 754-2008 section 4.3.1) on the 16 dropped bits; NaN stays a quiet NaN. */
uint16_t orc_f32_to_bf16(float x) {
    uint32_t u = f32_bits(x);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

float orc_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Generic fixed-partition parallel loop over [0, n). */
typedef void (*orc_body_fn)(void *ctx, uint64_t lo, uint64_t hi);
typedef struct { orc_body_fn fn; void *ctx; uint64_t lo, hi; } orc_task_t;

static void *orc_task_main(void *a) {
    orc_task_t *t = (orc_task_t *)a;
    t->fn(t->ctx, t->lo, t->hi);
    return NULL;
}

static void orc_parallel(orc_body_fn fn, void *ctx, uint64_t n, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((uint64_t)nthreads > n) nthreads = n ? (int)n : 1;
    if (nthreads == 1) { fn(ctx, 0, n); return; }
    orc_task_t task[256];
    pthread_t th[256];
    int ok[256];
    for (int w = 0; w < nthreads; ++w) {
        task[w].fn = fn; task[w].ctx = ctx;
        task[w].lo = n * (uint64_t)w / (uint64_t)nthreads;
        task[w].hi = n * (uint64_t)(w + 1) / (uint64_t)nthreads;
        ok[w] = pthread_create(&th[w], NULL, orc_task_main, &task[w]) == 0;
        if (!ok[w]) fn(ctx, task[w].lo, task[w].hi);
    }
    for (int w = 0; w < nthreads; ++w)
        if (ok[w]) pthread_join(th[w], NULL);
}

/* ------------------------------------------------------------- bf16 array */

typedef struct { const float *x; uint16_t *out; } cast_ctx;
static void cast_body(void *c, uint64_t lo, uint64_t hi) {
    cast_ctx *k = (cast_ctx *)c;
    for (uint64_t i = lo; i < hi; ++i) k->out[i] = orc_f32_to_bf16(k->x[i]);
}
void orc_f32_to_bf16_array(const float *x, uint16_t *out, uint64_t n, int nthreads) {
    cast_ctx c = {x, out};
    orc_parallel(cast_body, &c, n, nthreads);
}

/* ------------------------------------------------------------- accumulate */

/* "BLOOM 176B 训练技术概览", section "BF16 优化器": micro-batch gradients are
 * accumulated in FP32.  One micro-batch: a = first ? g : RN32(a + g), the sum
 * taken in FP64 (exact for an FP32 plus a bf16 of comparable range, and in any
 * case rounded once more to FP32 only: FP64 carries 53 >= 2*24+2 bits, so this
 * double rounding equals the correctly rounded FP32 sum -- S. A. Figueroa,
 * "When is double rounding innocuous?", SIGNUM Newsl. 1995). */
static float orc_acc_one(float a, uint16_t g, int first) {
    double gd = (double)orc_bf16_to_f32(g);
    if (first) return (float)gd;
    return (float)((double)a + gd);
}

typedef struct { float *acc; const uint16_t *g; int first; } acc_ctx;
static void acc_body(void *c, uint64_t lo, uint64_t hi) {
    acc_ctx *k = (acc_ctx *)c;
    for (uint64_t i = lo; i < hi; ++i) k->acc[i] = orc_acc_one(k->acc[i], k->g[i], k->first);
}
void orc_accumulate(float *acc, const uint16_t *g, uint64_t n, int first, int nthreads) {
    acc_ctx c = {acc, g, first};
    orc_parallel(acc_body, &c, n, nthreads);
}

/* The gradient the norm and the update see: the accumulated FP32 gradient times
 * grad_scale, rounded to FP32 (the product of two FP32 values is exact in FP64). */
static float orc_effective(float acc, float grad_scale) {
    if (grad_scale == 1.0f) return acc;
    return (float)((double)acc * (double)grad_scale);
}

/* ------------------------------------------------------------------- norm */

/* The squared global L2 norm of the accumulated gradient over every element
 * of every parameter group ("企业官网建设流程全解析" (cf-1.com), section 4.3:
 * clipping by the global gradient norm).
 * Fixed summation order: sequential FP64 sums over chunks of ORC_CHUNK
 * elements, then a sequential FP64 sum of the chunk sums in index order.
 * Squares of FP32 values are exact in FP64.  The result does not depend on
 * the thread count. */
#define ORC_CHUNK 65536ULL

typedef struct { const float *acc; float gs; double *part; uint64_t n; } ss_ctx;
static void ss_body(void *c, uint64_t lo, uint64_t hi) {
    ss_ctx *k = (ss_ctx *)c;
    for (uint64_t ch = lo; ch < hi; ++ch) {
        uint64_t b = ch * ORC_CHUNK, e = b + ORC_CHUNK;
        if (e > k->n) e = k->n;
        double s = 0.0;
        for (uint64_t i = b; i < e; ++i) {
            double x = (double)orc_effective(k->acc[i], k->gs);
            s += x * x;
        }
        k->part[ch] = s;
    }
}

static double orc_sum_parts(const double *part, uint64_t nch) {
    double s = 0.0;
    for (uint64_t ch = 0; ch < nch; ++ch) s += part[ch];
    return s;
}

double orc_sumsq(const float *acc, uint64_t n, float grad_scale, int nthreads) {
    uint64_t nch = (n + ORC_CHUNK - 1) / ORC_CHUNK;
    if (nch == 0) return 0.0;
    double *part = (double *)malloc(nch * sizeof(double));
    if (!part) return NAN;
    ss_ctx c = {acc, grad_scale, part, n};
    orc_parallel(ss_body, &c, nch, nthreads);
    double s = orc_sum_parts(part, nch);
    free(part);
    return s;
}

/* "企业官网建设流程全解析" (cf-1.com), section 4.3: the global gradient norm is
 * clipped at a threshold of 1.0.  Coefficient c = max_norm / ||g|| when
 * ||g|| > max_norm, otherwise 1 (gradients left unchanged); max_norm <= 0
 * turns clipping off.  Not rounded. */
double orc_clip_coef(double sumsq, double max_norm) {
    double norm = sqrt(sumsq);
    if (max_norm > 0.0 && norm > max_norm) return max_norm / norm;
    return 1.0;
}

/* ------------------------------------------------------------------ AdamW */

/* "企业官网建设流程全解析", section 1: FP32 master weights, momentum and variance
 * next to the 16-bit parameters; section 3.3: AdamW (lr 6e-5, weight decay 0.01).
 * One element of one AdamW step (Kingma & Ba Algorithm 1 with decoupled,
 * lr-scaled weight decay, Loshchilov & Hutter), FP64 throughout, from the
 * FP32-stored m, v and master; the results are stored as FP32 and the bf16
 * parameter is cast from the stored FP32 master.
 *   gc = e * c
 *   m' = b1 m + (1 - b1) gc
 *   v' = b2 v + (1 - b2) gc^2
 *   p' = p - lr wd p - lr (m'/bc1) / (sqrt(v'/bc2) + eps)
 * with bc1 = 1 - b1^t and bc2 = 1 - b2^t. */
static void orc_adamw_one(float *p, float *m, float *v, uint16_t *pb, float e, double c,
                          const orc_group_t *G, double bc1, double bc2) {
    double gc = (double)e * c;
    double m1 = G->beta1 * (double)*m + (1.0 - G->beta1) * gc;
    double v1 = G->beta2 * (double)*v + (1.0 - G->beta2) * gc * gc;
    double mhat = m1 / bc1;
    double vhat = v1 / bc2;
    double p0 = (double)*p;
    double p1 = p0 - G->lr * G->weight_decay * p0 - G->lr * mhat / (sqrt(vhat) + G->eps);
    *m = (float)m1;
    *v = (float)v1;
    *p = (float)p1;
    *pb = orc_f32_to_bf16(*p);
}

static void orc_bias_corr(const orc_group_t *G, int64_t t, double *bc1, double *bc2) {
    *bc1 = 1.0 - pow(G->beta1, (double)t);
    *bc2 = 1.0 - pow(G->beta2, (double)t);
}

typedef struct {
    float *p, *m, *v; uint16_t *pb; const float *acc; float gs; double c;
    const orc_group_t *G; double bc1, bc2;
} adam_ctx;
static void adam_body(void *c, uint64_t lo, uint64_t hi) {
    adam_ctx *k = (adam_ctx *)c;
    for (uint64_t i = lo; i < hi; ++i)
        orc_adamw_one(&k->p[i], &k->m[i], &k->v[i], &k->pb[i], orc_effective(k->acc[i], k->gs), k->c,
                      k->G, k->bc1, k->bc2);
}

void orc_adamw(float *p, float *m, float *v, uint16_t *p_bf16, const float *acc, uint64_t n,
               float grad_scale, double clip, const orc_group_t *grp, int64_t t, int nthreads) {
    adam_ctx c = {p, m, v, p_bf16, acc, grad_scale, clip, grp, 0.0, 0.0};
    orc_bias_corr(grp, t, &c.bc1, &c.bc2);
    orc_parallel(adam_body, &c, n, nthreads);
}

/* ------------------------------------------------------- streamed inputs */

static uint64_t orc_grad_key(const orc_stream_t *s, uint32_t step, uint32_t micro) {
    return synth_key(s->seed, s->workload, SYNTH_KIND_GRAD, step, micro);
}
static uint64_t orc_zero_key(const orc_stream_t *s) {
    return synth_key(s->seed, s->workload, SYNTH_KIND_ZERO_MASK, 0, 0);
}

/* Accumulated gradient of element i at step `step`, micro-batches in order. */
static float orc_stream_acc(const orc_stream_t *s, const uint64_t *keys, uint64_t zkey, uint64_t i) {
    float a = 0.0f;
    for (uint32_t k = 0; k < s->gas; ++k) {
        uint16_t g = synth_grad_bf16(keys[k], i, s->grad_sigma_scale, zkey, s->zero_thresh);
        a = orc_acc_one(a, g, k == 0);
    }
    return a;
}

typedef struct { const orc_stream_t *s; const uint64_t *keys; uint64_t zkey, n; double *part; } sss_ctx;
static void sss_body(void *c, uint64_t lo, uint64_t hi) {
    sss_ctx *k = (sss_ctx *)c;
    for (uint64_t ch = lo; ch < hi; ++ch) {
        uint64_t b = ch * ORC_CHUNK, e = b + ORC_CHUNK;
        if (e > k->n) e = k->n;
        double sum = 0.0;
        for (uint64_t i = b; i < e; ++i) {
            double x = (double)orc_effective(orc_stream_acc(k->s, k->keys, k->zkey, i), k->s->grad_scale);
            sum += x * x;
        }
        k->part[ch] = sum;
    }
}

double orc_stream_sumsq(const orc_stream_t *s, uint32_t step, uint64_t n, int nthreads) {
    uint64_t nch = (n + ORC_CHUNK - 1) / ORC_CHUNK;
    if (nch == 0 || s->gas == 0) return 0.0;
    double *part = (double *)malloc(nch * sizeof(double));
    uint64_t *keys = (uint64_t *)malloc(s->gas * sizeof(uint64_t));
    if (!part || !keys) { free(part); free(keys); return NAN; }
    for (uint32_t k = 0; k < s->gas; ++k) keys[k] = orc_grad_key(s, step, k);
    sss_ctx c = {s, keys, orc_zero_key(s), n, part};
    orc_parallel(sss_body, &c, nch, nthreads);
    double r = orc_sum_parts(part, nch);
    free(part);
    free(keys);
    return r;
}

void orc_sample_run(const orc_stream_t *s, const uint64_t *idx, uint64_t k, const float *p0,
                    const orc_group_t *groups, const uint32_t *group_of, uint32_t steps,
                    const double *clip, int64_t t0, float *p, float *m, float *v, uint16_t *p_bf16,
                    float *acc_out) {
    uint64_t zkey = orc_zero_key(s);
    uint64_t *keys = (uint64_t *)malloc((s->gas ? s->gas : 1) * sizeof(uint64_t));
    if (!keys) return;
    for (uint64_t j = 0; j < k; ++j) { p[j] = p0[j]; m[j] = 0.0f; v[j] = 0.0f; p_bf16[j] = orc_f32_to_bf16(p0[j]); }
    for (uint32_t st = 0; st < steps; ++st) {
        for (uint32_t q = 0; q < s->gas; ++q) keys[q] = orc_grad_key(s, st, q);
        int64_t t = t0 + (int64_t)st + 1;
        for (uint64_t j = 0; j < k; ++j) {
            const orc_group_t *G = &groups[group_of[j]];
            double bc1, bc2;
            orc_bias_corr(G, t, &bc1, &bc2);
            float a = orc_stream_acc(s, keys, zkey, idx[j]);
            if (acc_out && st + 1 == steps) acc_out[j] = a;
            orc_adamw_one(&p[j], &m[j], &v[j], &p_bf16[j], orc_effective(a, s->grad_scale), clip[st], G, bc1,
                          bc2);
        }
    }
    free(keys);
}

/* ------------------------------------------------------------- LR schedule */

/* "单机多卡实战：Megatron-DeepSpeed训练类BLOOM模型全流程解析", section 3: lr 6e-5,
 * min_lr 1e-6, lr_decay_style cosine, warmup_iters 500.
 * Warmup: lr grows linearly and reaches lr at step `warmup`.  Decay: the
 * cosine half-wave from lr (just after warmup) to min_lr (at step `decay`):
 * lr_t = min_lr + (lr - min_lr) (1 + cos(pi s)) / 2, s = (t - warmup)/(decay - warmup). */
double orc_lr_at(double lr, double min_lr, int64_t warmup, int64_t decay, int64_t t) {
    if (t <= warmup) return lr * (double)t / (double)warmup;
    if (t > decay) return min_lr;
    double s = (double)(t - warmup) / (double)(decay - warmup);
    return min_lr + (lr - min_lr) * (1.0 + cos(3.14159265358979323846 * s)) / 2.0;
}

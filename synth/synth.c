/*
 * synth.c -- exported, multi-threaded fill/gather routines over synth.h.
 *
 * Harness code: builds libsynth.so, which the tests and the benchmark use to
 * create seeded inputs (micro-batch gradients, initial master weights) in host
 * memory before they are copied to the device.  No optimizer arithmetic here.
 */
#include "synth.h"

#include <pthread.h>
#include <stdlib.h>

typedef struct {
    int kind;                 /* 0 grad bf16, 1 normal f32, 2 loguniform f32 */
    void *out;
    const uint64_t *idx;      /* gather mode when non-NULL */
    uint64_t n, first;
    uint64_t key, zero_key, zero_thresh;
    double scale;
    int e_lo, e_hi;
    uint64_t lo, hi;          /* this worker's [lo, hi) */
} synth_job_t;

static void synth_run_range(const synth_job_t *j) {
    for (uint64_t t = j->lo; t < j->hi; ++t) {
        uint64_t i = j->idx ? j->idx[t] : j->first + t;
        switch (j->kind) {
        case 0:
            ((uint16_t *)j->out)[t] = synth_grad_bf16(j->key, i, j->scale, j->zero_key, j->zero_thresh);
            break;
        case 1:
            ((float *)j->out)[t] = synth_normal_f32(j->key, i, j->scale);
            break;
        default:
            ((float *)j->out)[t] = synth_loguniform_f32(j->key, i, j->e_lo, j->e_hi);
            break;
        }
    }
}

static void *synth_worker(void *arg) {
    synth_run_range((const synth_job_t *)arg);
    return NULL;
}

static void synth_parallel(synth_job_t base, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (base.n < (1u << 16)) nthreads = 1;
    if (nthreads == 1) {
        base.lo = 0;
        base.hi = base.n;
        synth_run_range(&base);
        return;
    }
    synth_job_t jobs[256];
    pthread_t th[256];
    int started[256];
    for (int w = 0; w < nthreads; ++w) {
        jobs[w] = base;
        jobs[w].lo = base.n * (uint64_t)w / (uint64_t)nthreads;
        jobs[w].hi = base.n * (uint64_t)(w + 1) / (uint64_t)nthreads;
        started[w] = pthread_create(&th[w], NULL, synth_worker, &jobs[w]) == 0;
        if (!started[w]) synth_run_range(&jobs[w]);
    }
    for (int w = 0; w < nthreads; ++w)
        if (started[w]) pthread_join(th[w], NULL);
}

uint64_t synth_stream_key(uint64_t seed, uint32_t workload, uint32_t kind, uint32_t step, uint32_t micro) {
    return synth_key(seed, workload, kind, step, micro);
}

double synth_sigma_scale(double sigma) { return synth_scale_for_sigma(sigma); }

void synth_fill_grad_bf16(uint16_t *out, uint64_t n, uint64_t first, uint64_t key, double scale,
                          uint64_t zero_key, uint64_t zero_thresh, int nthreads) {
    synth_job_t j = {0};
    j.kind = 0; j.out = out; j.n = n; j.first = first; j.key = key; j.scale = scale;
    j.zero_key = zero_key; j.zero_thresh = zero_thresh;
    synth_parallel(j, nthreads);
}

void synth_fill_normal_f32(float *out, uint64_t n, uint64_t first, uint64_t key, double scale, int nthreads) {
    synth_job_t j = {0};
    j.kind = 1; j.out = out; j.n = n; j.first = first; j.key = key; j.scale = scale;
    synth_parallel(j, nthreads);
}

void synth_fill_loguniform_f32(float *out, uint64_t n, uint64_t first, uint64_t key, int e_lo, int e_hi,
                               int nthreads) {
    synth_job_t j = {0};
    j.kind = 2; j.out = out; j.n = n; j.first = first; j.key = key; j.e_lo = e_lo; j.e_hi = e_hi;
    synth_parallel(j, nthreads);
}

void synth_gather_grad_bf16(uint16_t *out, const uint64_t *idx, uint64_t n, uint64_t key, double scale,
                            uint64_t zero_key, uint64_t zero_thresh) {
    synth_job_t j = {0};
    j.kind = 0; j.out = out; j.idx = idx; j.n = n; j.key = key; j.scale = scale;
    j.zero_key = zero_key; j.zero_thresh = zero_thresh;
    synth_parallel(j, 1);
}

void synth_gather_normal_f32(float *out, const uint64_t *idx, uint64_t n, uint64_t key, double scale) {
    synth_job_t j = {0};
    j.kind = 1; j.out = out; j.idx = idx; j.n = n; j.key = key; j.scale = scale;
    synth_parallel(j, 1);
}

void synth_gather_loguniform_f32(float *out, const uint64_t *idx, uint64_t n, uint64_t key, int e_lo, int e_hi) {
    synth_job_t j = {0};
    j.kind = 2; j.out = out; j.idx = idx; j.n = n; j.key = key; j.e_lo = e_lo; j.e_hi = e_hi;
    synth_parallel(j, 1);
}

/*
 * step_parity.c -- the C ABI driven from plain C, checked against the oracle.
 *
 * Test program, not part of the library.  Two optimizer steps over 100,003
 * elements in two parameter groups (weight decay 0.01 and 0), GAS 3 with the
 * last micro-batch deferred, run through include/bf16opt.h with device memory
 * from the CUDA runtime -- no Python, no PyTorch -- twice: as one FLAT shard
 * (every buffer one element past a 256-byte boundary) and as a LIST of three
 * separately allocated tensors (offsets of 1, 2 and 3 elements; the gradient
 * list points into one flat buffer per micro-batch); as two FLAT partitions
 * of the shard standing for two ZeRO ranks, whose local sums of squares are
 * summed in rank order by bf16opt_set_rank_sumsqs; and as an offload handle
 * whose master and moments live in ordinary host memory.  The same two steps
 * run through the FP64 CPU oracle (oracle/oracle.h) on the same seeded inputs
 * (synth/synth.h).
 *
 * Tolerances are those of the parity tests: the norm within 1e-6 relative;
 * m within 1e-6 of max(|m_ref|, M_t) and the master within 1e-6 of
 * max(|p_ref|, A_t), where M_t = b1 M_{t-1} + (1 - b1)|gc_t| and
 * A_t = A_{t-1}(1 - lr wd) + lr |u_t| (A_0 = |p_0|) are the sums of the
 * magnitudes of the terms of each recurrence; v within 1e-6 relative; and
 * every bf16 parameter the round-to-nearest-even bf16 of the GPU's master.
 *
 * Exit status: 0 when everything agrees, 1 on a parity failure, 2 on an API
 * or CUDA error.
 */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "bf16opt.h"
#include "oracle.h"
#include "synth.h"

#define N 100003u
#define SPLIT 70001u      /* [0, SPLIT) decays, [SPLIT, N) does not */
#define PART 50000u       /* two-partition mode: rank 0 owns [0, PART), rank 1 [PART, N) */

enum { MODE_FLAT = 0, MODE_LIST = 1, MODE_RANKS = 2, MODE_OFFLOAD = 3 };
static const char *const MODE_NAME[4] = {"FLAT", "LIST, 3 tensors", "2 partitions, rank-ordered norm",
                                         "offload, state in host memory"};
#define GAS 3u
#define STEPS 2u
#define WORKLOAD 31u
#define REL 1e-6

static int api(int rc, const char *what, const bf16opt_t *h) {
    if (rc < 0) {
        fprintf(stderr, "%s: %s (%s)\n", what, bf16opt_error_string(rc), bf16opt_last_error(h));
        exit(2);
    }
    return rc;
}

static void cuda(cudaError_t e, const char *what) {
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        exit(2);
    }
}

/* Device buffer of `count` elements of `size` bytes, one element past the
 * allocation's (256-byte aligned) start; *base receives what to free. */
static void *dev_offset(size_t count, size_t size, void **base) {
    cuda(cudaMalloc(base, (count + 64) * size), "cudaMalloc");
    return (char *)*base + size;
}

static int run(int mode) {
    const int list_mode = mode == MODE_LIST;
    const bf16opt_group_t groups[2] = {{6e-5f, 0.9f, 0.95f, 1e-8f, 0.01f}, {6e-5f, 0.9f, 0.95f, 1e-8f, 0.0f}};
    orc_group_t ogroups[2];
    for (int g = 0; g < 2; ++g) {   /* the oracle gets the same FP32-rounded values */
        ogroups[g].lr = groups[g].lr;
        ogroups[g].beta1 = groups[g].beta1;
        ogroups[g].beta2 = groups[g].beta2;
        ogroups[g].eps = groups[g].eps;
        ogroups[g].weight_decay = groups[g].weight_decay;
    }
    const bf16opt_range_t ranges[2] = {{0, SPLIT, 0, 0}, {SPLIT, N, 1, 0}};

    /* host inputs and oracle state */
    float *p = malloc(N * sizeof(float)), *m = calloc(N, sizeof(float)), *v = calloc(N, sizeof(float));
    float *acc = calloc(N, sizeof(float));
    uint16_t *pb = calloc(N, sizeof(uint16_t));
    uint16_t *grads[GAS];
    double *M = calloc(N, sizeof(double)), *A = malloc(N * sizeof(double));
    const uint64_t kmaster = synth_key(0, WORKLOAD, SYNTH_KIND_MASTER, 0, 0);
    for (uint32_t i = 0; i < N; ++i) {
        p[i] = synth_normal_f32(kmaster, i, synth_scale_for_sigma(0.02));
        A[i] = fabs((double)p[i]);
    }
    for (uint32_t k = 0; k < GAS; ++k) grads[k] = malloc(N * sizeof(uint16_t));

    /* device state: FLAT = five shard buffers; LIST = five per tensor */
    enum { NT = 3 };
    const uint32_t tb[NT + 1] = {0, 40000, SPLIT, N};     /* tensor i = elements [tb[i], tb[i+1]) */
    const uint32_t tgroup[NT] = {0, 0, 1};
    void *bases[5 * NT + GAS];
    int nb = 0;
    float *d_p[NT], *d_m[NT], *d_v[NT], *d_acc[NT];
    uint16_t *d_pb[NT];
    const int parts = list_mode ? NT : 1;
    for (int i = 0; i < parts; ++i) {
        const uint32_t lo = list_mode ? tb[i] : 0, cnt = list_mode ? tb[i + 1] - tb[i] : N;
        const size_t off = list_mode ? (size_t)i + 1 : 1;   /* elements past a 256-byte boundary */
        void *b0, *b1, *b2, *b3, *b4;
        cuda(cudaMalloc(&b0, (cnt + 64) * 4), "cudaMalloc");
        cuda(cudaMalloc(&b1, (cnt + 64) * 4), "cudaMalloc");
        cuda(cudaMalloc(&b2, (cnt + 64) * 4), "cudaMalloc");
        cuda(cudaMalloc(&b3, (cnt + 64) * 4), "cudaMalloc");
        cuda(cudaMalloc(&b4, (cnt + 64) * 2), "cudaMalloc");
        bases[nb++] = b0; bases[nb++] = b1; bases[nb++] = b2; bases[nb++] = b3; bases[nb++] = b4;
        d_p[i] = (float *)b0 + off;
        d_m[i] = (float *)b1 + off;
        d_v[i] = (float *)b2 + off;
        d_acc[i] = (float *)b3 + off;
        d_pb[i] = (uint16_t *)b4 + off;
        cuda(cudaMemcpy(d_p[i], p + lo, (size_t)cnt * sizeof(float), cudaMemcpyHostToDevice), "upload masters");
        cuda(cudaMemset(d_m[i], 0, (size_t)cnt * sizeof(float)), "memset");
        cuda(cudaMemset(d_v[i], 0, (size_t)cnt * sizeof(float)), "memset");
    }
    /* offload: master and moments in ordinary (pageable) host memory */
    float *h_p = NULL, *h_m = NULL, *h_v = NULL;
    if (mode == MODE_OFFLOAD) {
        h_p = malloc(N * sizeof(float));
        h_m = calloc(N, sizeof(float));
        h_v = calloc(N, sizeof(float));
        memcpy(h_p, p, N * sizeof(float));
    }
    uint16_t *d_g[GAS];
    for (uint32_t k = 0; k < GAS; ++k) d_g[k] = dev_offset(N, 2, &bases[nb++]);

    bf16opt_desc_t d;
    memset(&d, 0, sizeof d);
    d.n_groups = 2;
    d.groups = groups;
    d.max_grad_norm = 1.0f;
    d.grad_scale = 1.0f;
    bf16opt_tensor_t tens[NT];
    bf16opt_t *h = NULL, *h1 = NULL;      /* h1: rank 1 in the two-partition mode */
    if (mode == MODE_FLAT || mode == MODE_OFFLOAD) {
        d.mode = BF16OPT_FLAT;
        d.n = N;
        d.master = mode == MODE_OFFLOAD ? h_p : d_p[0];
        d.exp_avg = mode == MODE_OFFLOAD ? h_m : d_m[0];
        d.exp_avg_sq = mode == MODE_OFFLOAD ? h_v : d_v[0];
        d.grad_accum = d_acc[0];
        d.param_bf16 = d_pb[0];
        d.ranges = ranges;
        d.n_ranges = 2;
        if (mode == MODE_OFFLOAD) api(bf16opt_create_offload(&d, 2, &h), "bf16opt_create_offload", NULL);
        else api(bf16opt_create(&d, &h), "bf16opt_create", NULL);
    } else if (mode == MODE_LIST) {
        memset(tens, 0, sizeof tens);
        for (int i = 0; i < NT; ++i) {
            tens[i].master = d_p[i];
            tens[i].exp_avg = d_m[i];
            tens[i].exp_avg_sq = d_v[i];
            tens[i].grad_accum = d_acc[i];
            tens[i].param_bf16 = d_pb[i];
            tens[i].numel = tb[i + 1] - tb[i];
            tens[i].group = tgroup[i];
        }
        d.mode = BF16OPT_LIST;
        d.n_tensors = NT;
        d.tensors = tens;
        api(bf16opt_create(&d, &h), "bf16opt_create", NULL);
    } else {
        /* rank 0: [0, PART), all in group 0; rank 1: [PART, N), groups 0 then 1 */
        const bf16opt_range_t r0[1] = {{0, PART, 0, 0}};
        const bf16opt_range_t r1[2] = {{0, SPLIT - PART, 0, 0}, {SPLIT - PART, N - PART, 1, 0}};
        d.mode = BF16OPT_FLAT;
        d.n = PART;
        d.master = d_p[0];
        d.exp_avg = d_m[0];
        d.exp_avg_sq = d_v[0];
        d.grad_accum = d_acc[0];
        d.param_bf16 = d_pb[0];
        d.ranges = r0;
        d.n_ranges = 1;
        api(bf16opt_create(&d, &h), "bf16opt_create (rank 0)", NULL);
        d.n = N - PART;
        d.master = d_p[0] + PART;
        d.exp_avg = d_m[0] + PART;
        d.exp_avg_sq = d_v[0] + PART;
        d.grad_accum = d_acc[0] + PART;
        d.param_bf16 = d_pb[0] + PART;
        d.ranges = r1;
        d.n_ranges = 2;
        api(bf16opt_create(&d, &h1), "bf16opt_create (rank 1)", NULL);
    }

    int bad = 0;
    double worst_norm = 0.0;
    for (uint32_t s = 0; s < STEPS; ++s) {
        for (uint32_t k = 0; k < GAS; ++k) {
            const uint64_t key = synth_key(0, WORKLOAD, SYNTH_KIND_GRAD, s, k);
            for (uint32_t i = 0; i < N; ++i) grads[k][i] = synth_grad_bf16(key, i, synth_scale_for_sigma(0.05), 0, 0);
            cuda(cudaMemcpy(d_g[k], grads[k], N * sizeof(uint16_t), cudaMemcpyHostToDevice), "upload gradient");
            unsigned flags = (k == 0 ? BF16OPT_FIRST : 0u) | (k == GAS - 1 ? BF16OPT_LAST | BF16OPT_DEFER : 0u);
            if (mode == MODE_LIST) {
                const uint16_t *glist[NT] = {d_g[k] + tb[0], d_g[k] + tb[1], d_g[k] + tb[2]};
                api(bf16opt_accumulate(h, NULL, glist, flags, NULL), "bf16opt_accumulate", h);
            } else if (mode == MODE_RANKS) {
                api(bf16opt_accumulate(h, d_g[k], NULL, flags, NULL), "bf16opt_accumulate (rank 0)", h);
                api(bf16opt_accumulate(h1, d_g[k] + PART, NULL, flags, NULL), "bf16opt_accumulate (rank 1)", h1);
            } else {
                api(bf16opt_accumulate(h, d_g[k], NULL, flags, NULL), "bf16opt_accumulate", h);
            }
            orc_accumulate(acc, grads[k], N, k == 0, 1);
        }
        double norm = 0.0;
        if (mode == MODE_RANKS) {
            /* each rank's sum of squares; the "all-gather" is this array, in rank order */
            double local[2], swapped[2], norm1 = -1.0;
            api(bf16opt_grad_norm_local(h, NULL, &local[0]), "bf16opt_grad_norm_local (rank 0)", h);
            api(bf16opt_grad_norm_local(h1, NULL, &local[1]), "bf16opt_grad_norm_local (rank 1)", h1);
            swapped[0] = local[1];
            swapped[1] = local[0];
            if (local[0] != local[1] &&
                bf16opt_set_rank_sumsqs(h, swapped, 2, 0, NULL, &norm) != BF16OPT_ERR_INVALID_ARG) {
                fprintf(stderr, "a gather out of rank order was accepted\n");
                bad = 1;
            }
            api(bf16opt_set_rank_sumsqs(h, local, 2, 0, NULL, &norm), "bf16opt_set_rank_sumsqs (rank 0)", h);
            api(bf16opt_set_rank_sumsqs(h1, local, 2, 1, NULL, &norm1), "bf16opt_set_rank_sumsqs (rank 1)", h1);
            if (norm != norm1) {
                fprintf(stderr, "step %u: the ranks' norms differ: %.17g vs %.17g\n", s, norm, norm1);
                bad = 1;
            }
            api(bf16opt_step(h1, NULL, NULL), "bf16opt_step (rank 1)", h1);
        } else {
            api(bf16opt_grad_norm(h, NULL, &norm), "bf16opt_grad_norm", h);
        }
        api(bf16opt_step(h, NULL, NULL), "bf16opt_step", h);

        const double S = orc_sumsq(acc, N, 1.0f, 1), c = orc_clip_coef(S, 1.0);
        const int64_t t = (int64_t)s + 1;
        orc_adamw(p, m, v, pb, acc, SPLIT, 1.0f, c, &ogroups[0], t, 1);
        orc_adamw(p + SPLIT, m + SPLIT, v + SPLIT, pb + SPLIT, acc + SPLIT, N - SPLIT, 1.0f, c, &ogroups[1], t, 1);
        const double rel = fabs(norm - sqrt(S)) / sqrt(S);
        if (rel > worst_norm) worst_norm = rel;
        if (!(rel <= REL)) {
            fprintf(stderr, "step %u: norm %.17g vs %.17g\n", s, norm, sqrt(S));
            bad = 1;
        }
        /* operand scales of the recurrences (from the oracle's stored state) */
        for (uint32_t i = 0; i < N; ++i) {
            const orc_group_t *G = &ogroups[i < SPLIT ? 0 : 1];
            M[i] = G->beta1 * M[i] + (1.0 - G->beta1) * fabs((double)acc[i]) * c;
            const double u = fabs((double)m[i] / (1.0 - pow(G->beta1, (double)t))) /
                             (sqrt((double)v[i] / (1.0 - pow(G->beta2, (double)t))) + G->eps);
            A[i] = A[i] * (1.0 - G->lr * G->weight_decay) + G->lr * u;
        }
    }
    cuda(cudaDeviceSynchronize(), "device sync");

    float *gp = malloc(N * sizeof(float)), *gm = malloc(N * sizeof(float)), *gv = malloc(N * sizeof(float));
    uint16_t *gpb = malloc(N * sizeof(uint16_t));
    for (int i = 0; i < parts; ++i) {
        const uint32_t lo = list_mode ? tb[i] : 0, cnt = list_mode ? tb[i + 1] - tb[i] : N;
        if (mode == MODE_OFFLOAD) {     /* the new state is in the host arrays */
            memcpy(gp, h_p, N * sizeof(float));
            memcpy(gm, h_m, N * sizeof(float));
            memcpy(gv, h_v, N * sizeof(float));
        } else {
            cuda(cudaMemcpy(gp + lo, d_p[i], (size_t)cnt * sizeof(float), cudaMemcpyDeviceToHost), "download");
            cuda(cudaMemcpy(gm + lo, d_m[i], (size_t)cnt * sizeof(float), cudaMemcpyDeviceToHost), "download");
            cuda(cudaMemcpy(gv + lo, d_v[i], (size_t)cnt * sizeof(float), cudaMemcpyDeviceToHost), "download");
        }
        cuda(cudaMemcpy(gpb + lo, d_pb[i], (size_t)cnt * sizeof(uint16_t), cudaMemcpyDeviceToHost), "download");
    }
    int64_t steps_done = 0;
    api(bf16opt_get_step(h, &steps_done), "bf16opt_get_step", h);
    if (steps_done != STEPS) {
        fprintf(stderr, "step counter %lld, expected %u\n", (long long)steps_done, STEPS);
        bad = 1;
    }
    if (h1) {
        api(bf16opt_get_step(h1, &steps_done), "bf16opt_get_step (rank 1)", h1);
        if (steps_done != STEPS) bad = 1;
    }

    double worst_m = 0.0, worst_v = 0.0, worst_p = 0.0;
    for (uint32_t i = 0; i < N; ++i) {
        const double sm = fmax(fabs((double)m[i]), M[i]), sv = fabs((double)v[i]), sp = fmax(fabs((double)p[i]), A[i]);
        const double em = fabs((double)gm[i] - m[i]), ev = fabs((double)gv[i] - v[i]), ep = fabs((double)gp[i] - p[i]);
        if (!(em <= REL * sm) || !(ev <= REL * sv) || !(ep <= REL * sp) || gpb[i] != orc_f32_to_bf16(gp[i])) {
            if (bad < 10)
                fprintf(stderr, "element %u: m %.9g/%.9g v %.9g/%.9g p %.9g/%.9g bf16 %04x\n", i, gm[i], m[i], gv[i],
                        v[i], gp[i], p[i], gpb[i]);
            bad += 1;
        }
        if (sm > 0 && em / sm > worst_m) worst_m = em / sm;
        if (sv > 0 && ev / sv > worst_v) worst_v = ev / sv;
        if (sp > 0 && ep / sp > worst_p) worst_p = ep / sp;
    }
    printf("c-abi step parity (%s): %u elements, %u steps, GAS %u; norm rel err %.3g; scaled err m %.3g v %.3g "
           "p %.3g; %s\n", MODE_NAME[mode], N, STEPS, GAS, worst_norm, worst_m, worst_v, worst_p, bad ? "FAIL" : "ok");

    api(bf16opt_destroy(h), "bf16opt_destroy", NULL);
    if (h1) api(bf16opt_destroy(h1), "bf16opt_destroy (rank 1)", NULL);
    free(h_p); free(h_m); free(h_v);
    for (int k = 0; k < nb; ++k) cudaFree(bases[k]);
    free(p); free(m); free(v); free(acc); free(pb); free(M); free(A);
    free(gp); free(gm); free(gv); free(gpb);
    for (uint32_t k = 0; k < GAS; ++k) free(grads[k]);
    return bad ? 1 : 0;
}

int main(void) {
    int failed = 0;
    for (int mode = MODE_FLAT; mode <= MODE_OFFLOAD; ++mode) failed |= run(mode);
    return failed ? 1 : 0;
}

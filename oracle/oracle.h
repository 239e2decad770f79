/*
 * oracle.h -- plain FP64 CPU oracle of the BF16Optimizer step.
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline / reference leg load liboracle.so.  It shares no
 * code with the CUDA path; it reads its inputs from synth/synth.h (the seeded
 * input generators) and from caller arrays only.
 *
 * Every function evaluates the textbook definition once per element in FP64
 * and rounds at the storage points the method fixes:
 *   - "BLOOM 176B 训练技术概览", section "BF16 优化器": gradients of the pipeline
 *     micro-batches are accumulated in FP32 and all accumulation is FP32;
 *   - "企业官网建设流程全解析" (cf-1.com; body "千亿级大模型训练的挑战与并行化策略"),
 *     section 1: FP32 master weights, momentum and variance next to 16-bit
 *     parameters and gradients; section 3.3: AdamW, lr 6e-5, weight_decay 0.01;
 *     section 4.3: clipping of the global gradient norm at 1.0;
 *   - "单机多卡实战：Megatron-DeepSpeed训练类BLOOM模型全流程解析", section 3:
 *     gradient_accumulation_steps 4, clip_grad 1.0, weight_decay 0.01, bf16.
 * Readings where the pages are silent:
 *   - micro-batch gradients are SUMMED (no 1/GAS), in ascending micro-batch
 *     order, the FP32 sum stored after every add;
 *   - the norm is the L2 norm over every element of every group; the clip
 *     coefficient is max_norm / norm when norm > max_norm, else exactly 1,
 *     and max_norm <= 0 disables clipping;
 *   - AdamW is Adam with bias correction (Kingma & Ba, arXiv:1412.6980,
 *     Algorithm 1; t starts at 1) and decoupled weight decay scaled by lr
 *     (Loshchilov & Hutter, arXiv:1711.05101), eps added after the square
 *     root of the bias-corrected variance;
 *   - m, v and the master are stored as FP32 (round to nearest even) after
 *     every step and the bf16 parameter is the round-to-nearest-even bf16 of
 *     the stored FP32 master.
 */
#ifndef BF16OPT_ORACLE_H
#define BF16OPT_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
} orc_group_t;

/* A seeded gradient stream (inputs only; see synth/synth.h). */
typedef struct {
    uint64_t seed;
    uint32_t workload;        /* workload id used in the stream keys */
    uint32_t gas;             /* micro-batches per step */
    double grad_sigma_scale;  /* synth_scale_for_sigma(sigma) */
    uint64_t zero_thresh;     /* forced-zero fraction * 2^64, 0 = none */
    float grad_scale;         /* multiplier on the accumulated gradient, 1 = none */
    uint32_t pad;
} orc_stream_t;

/* bf16 <-> FP32. */
uint16_t orc_f32_to_bf16(float x);
float orc_bf16_to_f32(uint16_t h);
void orc_f32_to_bf16_array(const float *x, uint16_t *out, uint64_t n, int nthreads);

/* acc <- (first ? 0 : acc) + fp32(g), stored FP32. */
void orc_accumulate(float *acc, const uint16_t *g, uint64_t n, int first, int nthreads);

/* S = sum_i e_i^2 with e_i = RN32(acc_i * grad_scale); fixed chunk order. */
double orc_sumsq(const float *acc, uint64_t n, float grad_scale, int nthreads);

/* Clip coefficient for sum of squares S. */
double orc_clip_coef(double sumsq, double max_norm);

/* One AdamW step at step number t (>= 1) over n elements of one group. */
void orc_adamw(float *p, float *m, float *v, uint16_t *p_bf16, const float *acc, uint64_t n,
               float grad_scale, double clip, const orc_group_t *grp, int64_t t, int nthreads);

/* Sum of squares of step `step`'s accumulated gradient over [0, n) of the stream,
 * regenerating every micro-batch from its counters. */
double orc_stream_sumsq(const orc_stream_t *s, uint32_t step, uint64_t n, int nthreads);

/* Runs `steps` whole optimizer steps on k sampled elements of the stream.
 * idx: element indices; p0: their initial masters (m = v = 0);
 * group_of: index into groups[] per sample; clip[s]: step s's clip coefficient;
 * the step number of step s is t0 + s + 1.  Outputs the final FP32 states, the
 * bf16 parameter and the last step's accumulated gradient (acc_out may be NULL). */
void orc_sample_run(const orc_stream_t *s, const uint64_t *idx, uint64_t k, const float *p0,
                    const orc_group_t *groups, const uint32_t *group_of, uint32_t steps,
                    const double *clip, int64_t t0, float *p, float *m, float *v, uint16_t *p_bf16,
                    float *acc_out);

/* Learning rate at step number t >= 1 ("单机多卡实战：Megatron-DeepSpeed训练类BLOOM
 * 模型全流程解析", section 3: lr, min_lr, lr_decay_style cosine, warmup_iters):
 * linear warmup 0 -> lr over `warmup` steps, cosine lr -> min_lr until step `decay`,
 * then min_lr. */
double orc_lr_at(double lr, double min_lr, int64_t warmup, int64_t decay, int64_t t);

#ifdef __cplusplus
}
#endif
#endif

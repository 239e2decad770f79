/*
 * bf16opt.h -- C ABI of the BF16 mixed-precision optimizer step for one GPU.
 *
 * What the library computes, per optimizer step over one rank's parameter
 * shard (the BF16Optimizer of BLOOM-176B training):
 *   1. the bf16 gradients of the GAS micro-batches are summed into an FP32
 *      accumulator, in micro-batch order, stored as FP32 after every add
 *      ("BLOOM 176B 训练技术概览", section "BF16 优化器": all accumulation in
 *      FP32, gradients accumulated in FP32 across pipeline micro-batches);
 *   2. the global L2 norm of the accumulated gradient is reduced
 *      deterministically and the gradient is clipped to max_grad_norm
 *      ("企业官网建设流程全解析" (cf-1.com), section 4.3: global-norm threshold 1.0;
 *      "单机多卡实战：Megatron-DeepSpeed训练类BLOOM模型全流程解析", section 3: clip_grad 1.0);
 *   3. AdamW with decoupled, lr-scaled weight decay and bias correction
 *      updates the FP32 master weights and the FP32 first/second moments
 *      ("企业官网建设流程全解析", section 1: FP32 master, momentum and variance;
 *      section 3.3: AdamW lr 6e-5, weight_decay 0.01) and the bf16 working
 *      parameters are written as the round-to-nearest-even bf16 of the FP32
 *      master, all in one pass.
 *
 * Conventions.
 *   - Every buffer is caller-owned device memory (e.g. from PyTorch) that must
 *     outlive the handle; buffers must not overlap.  The library owns only
 *     its scratch (segment/chunk tables, norm partials, norm scalars, the
 *     step counter and the per-step scalars).
 *   - FP32 buffers must be 4-byte aligned and bf16 buffers 2-byte aligned
 *     (BF16OPT_ERR_ALIGNMENT otherwise).  Any offset modulo 16 bytes works;
 *     full speed needs every buffer of a tensor to share the same element
 *     offset modulo 16 bytes, and the last few percent the same offset
 *     modulo 128 bytes (any such offset runs as fast as an aligned one).
 *   - Elements are counted in uint64_t; a tensor or shard may exceed 2^32.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All device work is enqueued on it; no call synchronises
 *     except bf16opt_grad_norm with a non-NULL host_norm.
 *   - Every call returns 0 on success, a positive warning, or a negative
 *     error code; no C++ exception crosses the ABI.  On an error nothing is
 *     enqueued and the handle's sequence state is unchanged.
 *     bf16opt_last_error() gives a one-line message.
 *   - A handle is bound to the device that was current at bf16opt_create and
 *     is not thread-safe: use one handle from one host thread at a time.
 *     The library keeps a registry of live handles: a pointer that
 *     bf16opt_create did not return, or a handle already destroyed, is
 *     rejected with BF16OPT_ERR_INVALID_ARG by every call (bf16opt_destroy
 *     included) and never dereferenced.  bf16opt_destroy frees all the
 *     handle's memory but a small host record, so no later handle ever
 *     receives a destroyed handle's address.
 *   - Results are deterministic and do not depend on the launch grid (the
 *     environment variable BF16OPT_MAX_GRID, read at create, caps the CTAs
 *     per launch; it exists to test exactly that).
 *
 * Sequence per optimizer step (checked on the host; BF16OPT_ERR_SEQUENCE):
 *   accumulate(FIRST) ... accumulate(LAST) -> grad_norm -> step
 *   FIRST marks the first micro-batch (the accumulator is overwritten, not
 *   added to); LAST marks the last one (the norm's partial sums are fused
 *   into that pass).  FIRST|LAST is a single micro-batch.  grad_norm (or
 *   grad_norm_local) needs the LAST micro-batch: after FIRST without LAST it
 *   returns BF16OPT_ERR_SEQUENCE.  Any micro-batch may carry BF16OPT_DEFER (see
 *   there); LAST|DEFER is the plain "fuse the last micro-batch into the step"
 *   case.
 */
#ifndef BF16OPT_H
#define BF16OPT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define BF16OPT_OK 0
#define BF16OPT_WARN_NONFINITE 1       /* grad_norm: the norm is Inf or NaN */
#define BF16OPT_ERR_INVALID_ARG (-1)   /* NULL handle/pointer, bad size, bad hyper-parameter, overlap */
#define BF16OPT_ERR_ALIGNMENT (-2)     /* FP32 pointer not 4-B aligned or bf16 pointer not 2-B aligned */
#define BF16OPT_ERR_SEQUENCE (-3)      /* call out of the accumulate -> grad_norm -> step order */
#define BF16OPT_ERR_OOM (-4)           /* the library's scratch could not be allocated */
#define BF16OPT_ERR_CUDA (-5)          /* a CUDA runtime call or kernel launch failed */
#define BF16OPT_ERR_UNSUPPORTED (-6)   /* e.g. no usable CUDA device */

/* ---- ABI version -------------------------------------------------------
 * Raised whenever a declaration, a constant or a struct layout of this header
 * changes.  bf16opt_abi_version() returns the value the library was built
 * with; code compiled against a header with another value must not use it.
 * No CUDA call; never fails. */
#define BF16OPT_ABI_VERSION 2
int bf16opt_abi_version(void);

/* ---- modes and flags --------------------------------------------------- */
#define BF16OPT_FLAT 0   /* one contiguous shard: five flat buffers + group ranges */
#define BF16OPT_LIST 1   /* ragged list: five buffers per tensor (separate allocations) */

#define BF16OPT_FIRST 1u /* first micro-batch of the step: acc = fp32(g) */
#define BF16OPT_LAST 2u  /* last micro-batch: fuse the norm's partial sums into this pass */
#define BF16OPT_DEFER 4u /* keep this micro-batch's gradient instead of folding it into the
                            FP32 accumulator now: it is folded (in micro-batch order) by
                            the next pass that reads gradients -- the next accumulate
                            without DEFER, or, if none follows before LAST, the norm and
                            the step kernels, so the accumulator is never stored for it.
                            The buffer must stay valid and unchanged until that pass has
                            run on the stream (until bf16opt_step for deferred micro-
                            batches of the last run).  At most BF16OPT_MAX_DEFERRED may be
                            pending.  Same FP32 adds in the same order: bit-identical to
                            not deferring; it trades 2 bytes/element of gradient memory
                            per pending micro-batch for 8 bytes/element of HBM traffic */

#define BF16OPT_MAX_DEFERRED 8

#define BF16OPT_MAX_GROUPS 16

/* ---- descriptors (host memory; copied by bf16opt_create) ---------------- */

/* FLAT mode: elements [begin, end) of the shard belong to parameter group `group`. */
typedef struct {
    uint64_t begin, end;
    uint32_t group;
    uint32_t reserved;     /* must be 0 */
} bf16opt_range_t;

/* LIST mode: one tensor; every pointer is device memory of `numel` elements. */
typedef struct {
    float *master;         /* FP32 master weights */
    float *exp_avg;        /* FP32 first moment m */
    float *exp_avg_sq;     /* FP32 second moment v */
    float *grad_accum;     /* FP32 gradient accumulator */
    uint16_t *param_bf16;  /* bf16 working parameters (bit patterns) */
    uint64_t numel;
    uint32_t group;
    uint32_t reserved;     /* must be 0 */
} bf16opt_tensor_t;

/* AdamW hyper-parameters of one parameter group. */
typedef struct {
    float lr;              /* >= 0 */
    float beta1, beta2;    /* in [0, 1) */
    float eps;             /* > 0 */
    float weight_decay;    /* >= 0; decoupled: p -= lr * weight_decay * p */
} bf16opt_group_t;

typedef struct {
    int32_t mode;                    /* BF16OPT_FLAT or BF16OPT_LIST */
    uint32_t n_groups;               /* 1 .. BF16OPT_MAX_GROUPS */
    const bf16opt_group_t *groups;   /* n_groups entries */
    /* FLAT */
    uint64_t n;                      /* shard elements (0 allowed) */
    float *master, *exp_avg, *exp_avg_sq, *grad_accum;
    uint16_t *param_bf16;
    const bf16opt_range_t *ranges;   /* must tile [0, n) in order; NULL/0 = one range, group 0 */
    uint32_t n_ranges;
    /* LIST */
    uint32_t n_tensors;
    const bf16opt_tensor_t *tensors;
    /* clipping */
    float max_grad_norm;             /* global L2 clip threshold; <= 0 disables clipping */
    float grad_scale;                /* multiplies the accumulated gradient before norm and
                                        update (rounded to FP32); 1 = none; finite, != 0 */
} bf16opt_desc_t;

typedef struct bf16opt bf16opt_t;    /* opaque handle */

/* ---- entry points ------------------------------------------------------- */

/* One handle per rank's parameter shard ("BLOOM 176B 训练技术概览", section
 * 并行细节 / ZeRO: each GPU holds only its part of the parameters, gradients
 * and optimizer states).  Validates `d` before any CUDA call, copies its host
 * arrays (the caller may free them on return), builds the segment and chunk
 * tables on the device and allocates the library's scratch; the device
 * buffers stay the caller's.  *out receives the handle (NULL on error).  The
 * step counter starts at 0.  Errors: INVALID_ARG (NULL d or out, bad mode,
 * 0 or more than BF16OPT_MAX_GROUPS groups, a hyper-parameter out of range,
 * non-finite max_grad_norm, zero or non-finite grad_scale, NULL buffers,
 * ranges that do not tile [0, n) in order, overlapping buffers, more than
 * 2^32 - 1 chunks), ALIGNMENT, UNSUPPORTED (no CUDA device), OOM, CUDA;
 * bf16opt_last_error(NULL) has the message. */
int bf16opt_create(const bf16opt_desc_t *d, bf16opt_t **out);

/* ZeRO-Offload variant ("企业官网建设流程全解析" (cf-1.com), section 3.3: the
 * DeepSpeed configuration with offload_optimizer on the CPU; "单机多卡实战：
 * Megatron-DeepSpeed训练类BLOOM模型全流程解析", section 6: offloading optimizer
 * state to host memory to fit larger models).  Explicitly selected, never a
 * fallback: a FLAT handle whose FP32 master, exp_avg and exp_avg_sq are HOST
 * memory (12 bytes per element off the device), while grad_accum and
 * param_bf16 are memory of the current device.  accumulate, grad_norm (and the
 * multi-rank calls), get/set_step, the LR schedule and skipping work as for
 * bf16opt_create.  bf16opt_step then: completes the accumulator if
 * micro-batches are still deferred; computes the step's scalars, advances the
 * step counter and takes the skip decision on the device (the same kernel as
 * the device step); copies the accumulator to the host in blocks of 2^24
 * elements, updates master and moments with the same FP32 operations as the
 * device step on n_threads host threads (<= 0: one per core) while the next
 * block is copied, and enqueues the copy of each block's bf16 parameters back
 * to param_bf16 on `stream`.  It returns when the host arrays hold the new
 * state; the bf16 parameters are on the device when `stream` reaches those
 * copies.  Results: the same bits as a device handle over the same values.
 * The library allocates 192 MiB of page-locked staging (less for a smaller
 * shard) and the threads.  Not during a stream capture.  Errors: as
 * bf16opt_create, and INVALID_ARG (not FLAT; master/moments not host memory;
 * grad_accum/param_bf16 not memory of the current device), OOM. */
int bf16opt_create_offload(const bf16opt_desc_t *d, int n_threads, bf16opt_t **out);

/* Adds one micro-batch of bf16 gradients into the FP32 accumulator
 * ("BLOOM 176B 训练技术概览", "BF16 优化器").
 *   FLAT: grad_flat = device bf16 buffer of n elements, grad_list = NULL.
 *   LIST: grad_flat = NULL, grad_list = HOST array of n_tensors device
 *         pointers (read during the call only).
 *   flags: BF16OPT_FIRST / BF16OPT_LAST / BF16OPT_DEFER (see above).
 * The gradient buffer is read on `stream`; it may be reused after the work
 * on `stream` is done, except under BF16OPT_DEFER (until the pass that folds
 * it).  Errors: SEQUENCE (no FIRST outside an accumulation), INVALID_ARG
 * (not a live handle, unknown flag, a NULL or wrong-mode gradient pointer, a
 * DEFER beyond BF16OPT_MAX_DEFERRED pending), ALIGNMENT (a gradient pointer
 * not 2-byte aligned), CUDA. */
int bf16opt_accumulate(bf16opt_t *h, const uint16_t *grad_flat, const uint16_t *const *grad_list,
                       unsigned flags, void *stream);

/* Finishes the deterministic global L2 norm of the accumulated gradient
 * (times grad_scale) and the clip coefficient c = max_grad_norm / norm if
 * norm > max_grad_norm, else 1 ("企业官网建设流程全解析", section 4.3).  Both stay
 * on the device for bf16opt_step.  host_norm == NULL: fully asynchronous.
 * host_norm != NULL: waits for `stream` and stores the norm (FP64); returns
 * BF16OPT_WARN_NONFINITE if it is Inf or NaN (the caller decides whether to
 * call bf16opt_step; the library skips nothing unless bf16opt_set_skip_nonfinite
 * asked it to).  Errors: SEQUENCE (no completed accumulation FIRST ... LAST
 * since the last step), INVALID_ARG (not a live handle), CUDA. */
int bf16opt_grad_norm(bf16opt_t *h, void *stream, double *host_norm);

/* Multi-rank use.  Under ZeRO every rank owns one partition of the parameters
 * and the clipping norm is global over all of them ("BLOOM 176B 训练技术概览",
 * section 并行细节 / ZeRO: each GPU holds only its part; "企业官网建设流程全解析",
 * section 4.3: the global norm).  The exchange is one FP64 scalar per rank;
 * moving it belongs to the caller's communication library, the arithmetic to
 * this one:
 *   1. bf16opt_grad_norm_local: in place of bf16opt_grad_norm, finishes this
 *      rank's sum of squares, waits for `stream` and stores it in *local_sumsq;
 *   2. the caller gathers every rank's value into an array in rank order
 *      (an all-gather);
 *   3. bf16opt_set_rank_sumsqs: sums that array in rank order (FP64, rank 0
 *      first: every rank gets the same bits, so every rank clips alike) and
 *      turns the sum into the norm and clip coefficient on the device
 *      (enqueued on `stream`); bf16opt_step follows.
 * Sequence: local needs a completed accumulation (as grad_norm); set_rank
 * and set_global need local.  A non-finite local or global sum is passed
 * through unchanged and reported as BF16OPT_WARN_NONFINITE (the caller decides
 * whether to step). */
int bf16opt_grad_norm_local(bf16opt_t *h, void *stream, double *local_sumsq);

/* per_rank: HOST array of the n_ranks gathered local sums, in rank order;
 * rank: this handle's rank, whose entry must equal, bit for bit, the value
 * bf16opt_grad_norm_local returned (a gather that put the values out of order
 * is refused).  global_norm: NULL, or receives sqrt of the rank-ordered sum
 * (no synchronisation).  Errors: INVALID_ARG (not a live handle, NULL
 * per_rank, n_ranks == 0, rank >= n_ranks, per_rank[rank] not this rank's
 * value), SEQUENCE (no grad_norm_local since the accumulation), CUDA. */
int bf16opt_set_rank_sumsqs(bf16opt_t *h, const double *per_rank, uint32_t n_ranks, uint32_t rank, void *stream,
                            double *global_norm);

/* The rank-ordered sum that bf16opt_set_rank_sumsqs uses:
 * *global_sumsq = ((per_rank[0] + per_rank[1]) + ...) + per_rank[n_ranks-1]
 * in FP64.  Host-only; needs no device or handle.  Errors: INVALID_ARG (NULL
 * pointer, n_ranks == 0). */
int bf16opt_sum_rank_sumsqs(const double *per_rank, uint32_t n_ranks, double *global_sumsq);

/* For callers that reduce the sums themselves: sets the norm and clip
 * coefficient from an already summed global_sumsq (enqueued on `stream`).
 * Every rank must pass the same bits.  Errors as bf16opt_set_rank_sumsqs. */
int bf16opt_set_global_sumsq(bf16opt_t *h, double global_sumsq, void *stream);

/* CUDA graphs.  The step counter, the hyper-parameters and the LR schedule
 * live on the device and bf16opt_step computes its scalars there, so the
 * sequence accumulate ... -> grad_norm (host_norm = NULL) -> step, captured
 * once on a stream, replays as later steps (same gradient buffers; lr_override
 * values are frozen into the capture).  Calls that synchronise (grad_norm with
 * host_norm, grad_norm_local, get/set_step, set_lr_schedule,
 * set_skip_nonfinite, debug_faults, create, create_offload, destroy, and step
 * on an offload handle) must stay outside a capture. */

/* One fused pass: clip, AdamW (t = t + 1, bias-corrected, decoupled
 * weight decay), FP32 master/moment update and bf16 parameter write
 * ("企业官网建设流程全解析", sections 1 and 3.3).
 * lr_override: NULL, or a HOST array of n_groups learning rates that
 * replaces the groups' lr for this step only (for an LR schedule; read during
 * the call only).  Errors: SEQUENCE (no grad_norm or set_global_sumsq since
 * the accumulation), INVALID_ARG (not a live handle, a negative or non-finite
 * lr_override entry), CUDA. */
int bf16opt_step(bf16opt_t *h, const float *lr_override, void *stream);

/* Learning-rate schedule of the training configuration ("单机多卡实战：
 * Megatron-DeepSpeed训练类BLOOM模型全流程解析", section 3: lr 6e-5, min_lr 1e-6,
 * lr_decay_style cosine, warmup_iters 500): linear warmup from 0 to the group's
 * lr over warmup_steps, then cosine decay to min_lr_ratio * lr at decay_steps,
 * then constant.  For the step number t >= 1 the factor on every group's lr is
 *   t <= warmup_steps:                f = t / warmup_steps
 *   warmup_steps < t <= decay_steps:  f = r + (1 - r) (1 + cos(pi (t - warmup_steps)
 *                                              / (decay_steps - warmup_steps))) / 2
 *   t > decay_steps:                  f = r                      (r = min_lr_ratio)
 * evaluated in FP64. */
typedef struct {
    int64_t warmup_steps;  /* >= 0 */
    int64_t decay_steps;   /* >= warmup_steps */
    float min_lr_ratio;    /* in [0, 1] */
    uint32_t reserved;     /* must be 0 */
} bf16opt_lr_schedule_t;

/* f(t) of the schedule above into *factor.  Host-only; needs no device or handle.
 * Errors: INVALID_ARG for NULL pointers, t < 1 or an invalid schedule. */
int bf16opt_lr_factor(const bf16opt_lr_schedule_t *s, int64_t t, double *factor);

/* Attaches a copy of schedule `s` to the handle (NULL detaches it).  Every later
 * bf16opt_step then uses lr = (lr_override[g] or the group's lr) * f(t) with t
 * the step number of that step (the step counter plus one, so a resumed run
 * that restored its counter with bf16opt_set_step continues the schedule).
 * Waits for all work on the handle's device first, so steps already enqueued
 * keep the old schedule; not during a stream capture.  Errors: INVALID_ARG
 * (not a live handle, an invalid schedule as for bf16opt_lr_factor), CUDA. */
int bf16opt_set_lr_schedule(bf16opt_t *h, const bf16opt_lr_schedule_t *s);

/* Opt-in guard for steps whose global norm is Inf or NaN (enable != 0): the
 * decision is taken on the device by bf16opt_step's first kernel, which then
 * leaves the step counter unchanged, and the fused kernel returns without
 * touching master, moments or bf16 parameters -- so it also holds inside a
 * captured CUDA graph, where the host cannot read the norm before the step.
 * Off by default: the method has no skip logic (bf16 does not overflow the
 * way fp16 does; "企业官网建设流程全解析", section 4.1) and grad_norm reports
 * BF16OPT_WARN_NONFINITE for the caller to act on.  Waits for all work on the
 * handle's device first, so steps already enqueued keep the old setting; not
 * during a stream capture.  Errors: INVALID_ARG (NULL handle), CUDA. */
int bf16opt_set_skip_nonfinite(bf16opt_t *h, int enable);

/* Frees the library's scratch (waits for the device); the caller's buffers
 * are untouched.  NULL is accepted.  A pointer that is not a live handle
 * (never created, or already destroyed) gives BF16OPT_ERR_INVALID_ARG. */
int bf16opt_destroy(bf16opt_t *h);

/* Step counter t (number of completed steps, kept on the device), for
 * checkpoint and resume: restore the caller's buffers and set_step(t) to
 * continue.  Both calls first wait for all work on the handle's device
 * (cudaDeviceSynchronize), so they are ordered after every step already
 * enqueued, on any stream (non-blocking ones included); not during a stream
 * capture.  Errors: INVALID_ARG (NULL, t < 0), CUDA. */
int bf16opt_get_step(const bf16opt_t *h, int64_t *t);
int bf16opt_set_step(bf16opt_t *h, int64_t t);

/* ---- allocation-free one-shot norm -----------------------------------------
 * No counterpart in the paper: a service entry point for callers that cannot
 * call cudaMalloc -- code inside another framework's launch path that is given
 * only a stream and a pre-planned workspace (plugins, custom-op launchers),
 * processes whose device memory is held by a caching allocator (a raw
 * cudaMalloc can then fail), and latency-sensitive loops that cannot take the
 * device synchronisation cudaMalloc/cudaFree imply.
 *
 * Computes, without a handle and without allocating anything, the global L2
 * norm of a flat FP32 gradient accumulator `grad_accum` of n elements (each
 * element times grad_scale, rounded to FP32), with the same deterministic
 * chunked reduction as bf16opt_grad_norm on a one-range FLAT shard over an
 * accumulator with the same offset modulo 128 bytes, and the
 * clip coefficient c = max_grad_norm / norm if norm > max_grad_norm (> 0),
 * else 1.  `out` is owned by the caller; the result is written there on
 * `stream` (nothing is synchronised).  `out` and `grad_accum` must be memory
 * the current device can use: its own device memory, managed memory, or
 * page-locked host memory (cudaMallocHost / cudaHostRegister, used through
 * its mapped device address); anything else (pageable host memory, another
 * device's memory) is refused with BF16OPT_ERR_INVALID_ARG before any work is
 * enqueued.
 *
 * Scratch: one FP64 partial per chunk of up to 32,768 elements, kept in a file-scope
 * device array of 65,536 entries (512 KiB) that every GPU loading this
 * library holds until the process exits; hence n is limited to
 * BF16OPT_STATIC_NORM_MAX_ELEMS (2^30) elements and larger n is rejected with
 * BF16OPT_ERR_INVALID_ARG before any work is enqueued.  Every call writes the
 * partials it later reads, so nothing has to start at zero.  All calls on a
 * device share that one array: calls whose work overlaps on the GPU (e.g. on
 * two streams without ordering between them) race and give wrong results.
 * The array's device address belongs to the context that loaded the library's
 * kernels: the first call on each device, and the first call after that
 * device's context was reset (cudaDeviceReset), looks it up
 * (cudaGetSymbolAddress) with the device current; make those calls before any
 * stream capture.  Errors: INVALID_ARG (NULL pointers, n too large,
 * non-finite or zero grad_scale, non-finite max_grad_norm, memory the device
 * cannot use), ALIGNMENT (grad_accum not 4-B aligned, out not 8-B aligned),
 * UNSUPPORTED (no device), CUDA (symbol lookup or launch failed);
 * bf16opt_last_error(NULL) has the message. */
#define BF16OPT_STATIC_NORM_MAX_ELEMS (((uint64_t)1) << 30)

typedef struct {
    double sumsq;      /* sum of squares of the (scaled) accumulated gradient */
    double norm;       /* sqrt(sumsq) */
    double clip_coef;  /* max_grad_norm / norm if norm > max_grad_norm, else 1 */
} bf16opt_norm_result_t;

int bf16opt_grad_norm_static(const float *grad_accum, uint64_t n, float grad_scale, float max_grad_norm,
                             bf16opt_norm_result_t *out, void *stream);

/* ---- data path of the step -------------------------------------------------
 * No counterpart in the paper.  Which kernel the handle's most recent
 * bf16opt_step ran (enqueued): NONE (no step yet, or the shard is empty),
 * VECTOR (per-thread 16-byte vector loads and stores), PIPELINE (bulk
 * asynchronous copies through shared memory; see below), HOST (an offload
 * handle: the host cores update the master and moments).  Errors: INVALID_ARG
 * (not a live handle, path NULL). */
#define BF16OPT_PATH_NONE 0
#define BF16OPT_PATH_VECTOR 1
#define BF16OPT_PATH_PIPELINE 2
#define BF16OPT_PATH_HOST 3
int bf16opt_step_path(const bf16opt_t *h, int *path);

/* ---- pipeline health ----------------------------------------------------
 * No counterpart in the paper: a health check of the copy pipeline.  On
 * shards of 2^25 elements and more whose buffers are aligned alike (per
 * segment: the FP32 streams at one element index modulo 4, the bf16 streams
 * at one modulo 8, agreeing modulo 4), bf16opt_step and the accumulate passes
 * after FIRST that store the accumulator move their traffic with bulk
 * asynchronous copies through a ring of shared-memory stages.  The
 * environment variable BF16OPT_PIPE=1 / 0, read when a handle is created,
 * forces this on / off.  Every wait on a stage is bounded (2 s; a stage
 * normally turns over in microseconds).  A wait that gives up is counted in
 * a device word and its CTA stops, leaving the rest of its units of that
 * pass not updated.  This call waits for the current device, stores that
 * device's count into *count (0 = every pass completed) and clears it.
 * Errors: INVALID_ARG (count NULL), UNSUPPORTED (no device), CUDA. */
int bf16opt_pipeline_timeouts(uint32_t *count);

/* ---- checked build -------------------------------------------------------
 * No counterpart in the paper: a debugging aid standing in for a memory
 * checker.  In a build compiled with -DBF16K_CHECKS the kernels test, before
 * each chunk's accesses, that the chunk lies inside its segment, that its
 * scalar head and vector body stay inside the chunk and that every vector
 * pointer is 16-byte (FP32) / 8-byte (bf16) aligned; a violation sets a bit in
 * a device word (1 = chunk outside its segment, 2 = body outside the chunk,
 * 4 = misaligned vector pointer) and the chunk is skipped instead of accessed.
 * This call waits for the device, stores the word into *bits and clears it.
 * Release builds: *bits = 0 and BF16OPT_ERR_UNSUPPORTED.
 * Errors: INVALID_ARG (bits NULL), UNSUPPORTED, CUDA. */
int bf16opt_debug_faults(uint32_t *bits);

/* Static message of a status code; one-line message of the handle's last error. */
const char *bf16opt_error_string(int code);
const char *bf16opt_last_error(const bf16opt_t *h);

#ifdef __cplusplus
}
#endif
#endif /* BF16OPT_H */

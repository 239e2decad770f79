// kernels.cuh -- sm_103a kernels of the BF16 mixed-precision optimizer step.
//
// Bandwidth-bound kernels (no tensor cores: nothing here is a contraction)
// over a table of chunks, and three single-CTA kernels:
//   k_accum          folds bf16 micro-batch gradients into the FP32 accumulator,
//                    optionally with the per-chunk partial sums of squares of the
//                    global norm fused in ("BLOOM 176B 训练技术概览", section
//                    "BF16 优化器": FP32 accumulation of gradients across pipeline
//                    micro-batches);
//   k_norm_final     fixed-order FP64 sum of the chunk partials, norm and clip
//                    coefficient ("企业官网建设流程全解析" (cf-1.com), section 4.3: global
//                    norm clipped at 1.0), and the next step's per-group AdamW
//                    scalars and skip decision;
//   k_norm_from_sumsq the same from an all-rank sum handed in by the host (ZeRO);
//   k_step_scalars   t <- t + 1 and the scalars of step t again, for a step with a
//                    learning-rate override or settings changed since the norm;
//   k_step           clip x AdamW x FP32 master/moment update x bf16 cast in one pass
//                    ("企业官网建设流程全解析", sections 1 and 3.3); advances the step
//                    counter when the norm kernel prepared the scalars;
//   k_step_pipe, k_accum_pipe  the fused step and the accumulate passes after
//                    FIRST with the same arithmetic, their traffic moved by
//                    bulk copies through shared memory (pipe_run, at the end).
//
// Work decomposition.  A segment is one run of elements with one parameter
// group and one set of base pointers (a flat range or a list tensor).  The
// host cuts each segment into chunks of at most kChunk elements (the first one
// shortened so that later chunks start on a 128-byte line of the
// accumulator); a persistent grid takes the chunks by a fixed stride or claims
// them from a counter (see the chunk schedule below).  Inside a chunk, thread
// t handles 4-element quads t, t+T, ... so that every warp-wide access
// is contiguous: FP32 as 16-byte and bf16 as 8-byte vectors.  Leading elements
// up to the lead pointer's next kHeadAlign-element boundary, and the ragged
// tail, are done one element at a time by a warp chosen per chunk.  If the
// buffers of a segment do not share their offset modulo 16 bytes the whole
// chunk runs element-wise (correct, slower).
//
// Determinism.  The norm's partial of chunk c depends only on the chunk's
// data and on the fixed thread->element map, so the result does not depend
// on the grid size, on scheduling or on which CTA takes which chunk; the final
// sum runs in chunk order.
#pragma once

#include <cuda_bf16.h>
#include <type_traits>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bf16k {

// Launch shape; the defaults were chosen by measurement on GB300 and can be
// overridden at build time (-DBF16K_ACC_THREADS=..., -DBF16K_CHUNK=...).
#ifndef BF16K_ACC_THREADS
#define BF16K_ACC_THREADS 256
#endif
#ifndef BF16K_STEP_THREADS
#define BF16K_STEP_THREADS 512
#endif
#ifndef BF16K_STEP_MIN_BLOCKS
#define BF16K_STEP_MIN_BLOCKS 1
#endif
#ifndef BF16K_CHUNK
#define BF16K_CHUNK 32768
#endif
#ifndef BF16K_HEAD_ALIGN
#define BF16K_HEAD_ALIGN 32
#endif
// Quads (4 elements) in flight per thread, by pass, and the cap on resident
// CTAs per SM a launch is sized for.
#ifndef BF16K_ACC_U
#define BF16K_ACC_U 8         // accumulate family
#endif
#ifndef BF16K_STEP_U
#define BF16K_STEP_U 2        // fused step
#endif
#ifndef BF16K_FOLD4_ACC_U
#define BF16K_FOLD4_ACC_U 4   // passes folding 2-4 gradients
#endif
#ifndef BF16K_FOLD8_ACC_U
#define BF16K_FOLD8_ACC_U 1   // passes folding 5-8 gradients
#endif
#ifndef BF16K_FOLD4_STEP_U
#define BF16K_FOLD4_STEP_U 2  // fused step folding 2-4 gradients
#endif
#ifndef BF16K_FOLD8_STEP_U
#define BF16K_FOLD8_STEP_U 1  // fused step folding 5-8 gradients
#endif
#ifndef BF16K_MAX_CTAS_PER_SM
#define BF16K_MAX_CTAS_PER_SM 64
#endif
constexpr int kAccThreads = BF16K_ACC_THREADS;    // threads per CTA, accumulate / norm passes
constexpr int kStepThreads = BF16K_STEP_THREADS;  // threads per CTA, fused step
constexpr int kThreads = kAccThreads;
constexpr uint32_t kChunk = BF16K_CHUNK;          // elements per chunk (multiple of 4)
// The vector body of a chunk starts where the lead pointer's element index is
// a multiple of kHeadAlign (power of two, >= 4): 128-byte FP32 / 64-byte bf16
// boundaries at 32, so that no warp's 512-byte access starts or ends inside a
// 32-byte sector when the buffers are offset from those boundaries.
constexpr uint32_t kHeadAlign = BF16K_HEAD_ALIGN;
static_assert(kHeadAlign >= 4 && (kHeadAlign & (kHeadAlign - 1)) == 0, "kHeadAlign: a power of two >= 4");
constexpr int kMaxGroups = 16;
constexpr int kListSlots = 1024;     // gradient pointers per LIST-mode launch
constexpr int kFinalThreads = 1024;

struct Seg {
    float *acc, *p, *m, *v;   // already offset to the segment's first element
    uint16_t *bf;
    uint64_t numel;
    uint64_t grad_off;        // element offset of the segment in its gradient buffer
    uint32_t grad_slot;       // which per-call gradient pointer
    uint32_t group;
};

struct Chunk {
    uint64_t start;           // first element, relative to the segment
    uint32_t seg;
    uint32_t len;
};

struct NormState {
    double sumsq;             // sum of squares of the (scaled) accumulated gradient
    double norm;              // sqrt(sumsq)
    float c_hi, c_lo;         // clip coefficient c = c_hi + c_lo (float-float)
    int32_t finite;
    int32_t pad;
};

// Per-group scalars of one step, FP32, computed in FP64 on the device
// (group_scalars: by the norm kernel, or by k_step_scalars).
struct GroupK {
    float b1, omb1, b2, omb2;
    float eps;
    float decay;              // lr * weight_decay
    float step_size;          // lr / (1 - b1^t)
    float inv_sqrt_bc2;       // 1 / sqrt(1 - b2^t)
};
struct GroupTable {
    GroupK g[kMaxGroups];
};

// Hyper-parameters of the handle, kept on the device so that a captured
// step (CUDA graph) computes the scalars of whatever step it replays.
struct StepParams {
    float lr[kMaxGroups], beta1[kMaxGroups], beta2[kMaxGroups], eps[kMaxGroups], wd[kMaxGroups];
    int32_t n_groups;
    int32_t has_sched;             // warmup + cosine factor on every lr
    int64_t warmup, decay;
    float min_ratio;
    int32_t skip_nonfinite;        // leave the state alone when the norm is not finite
};

// Device step counter and the scalars of the current step.
struct StepState {
    int64_t t;                     // completed steps
    int32_t skip;                  // this step is skipped (non-finite norm, skipping enabled)
    int32_t pad;
    GroupTable gtab;
};

// Per-call learning rates (optional), by value.
struct LrOverride {
    float lr[kMaxGroups];
    int32_t use;
};

// Gradient sources passed by value as kernel parameters.  A pass folds k
// micro-batch gradients (k <= kMaxFold) into the value in micro-batch order.
constexpr int kMaxFold = 8;
struct FlatGrads {
    const uint16_t *base[kMaxFold];   // micro-batch j's flat gradient buffer
    uint32_t k;
    uint32_t pad;
    __device__ __forceinline__ const uint16_t *get(uint32_t, int j) const { return base[j]; }
};
struct ListGrads {
    uint32_t slot_base;               // first tensor of this launch
    uint32_t nslots;                  // tensors in this launch (k * nslots <= kListSlots)
    uint32_t k;
    uint32_t pad;
    const uint16_t *ptr[kListSlots];  // ptr[j * nslots + (tensor - slot_base)]
    __device__ __forceinline__ const uint16_t *get(uint32_t s, int j) const { return ptr[j * nslots + (s - slot_base)]; }
};

// ------------------------------------------------------------ checked build
// Built with -DBF16K_CHECKS, the kernels also test what the host guarantees by
// construction -- every chunk lies inside its segment, the scalar head and the
// vector body stay inside the chunk, every vector pointer is 16-byte (FP32) /
// 8-byte (bf16) aligned -- and on a violation set a bit in g_check_faults and
// skip the chunk instead of making the access (no trap, no fault).  The tests
// are uniform across a CTA, so a skipped chunk never splits a barrier.
// Release builds compile them away.
enum : uint32_t { kFaultChunkRange = 1u, kFaultBody = 2u, kFaultAlign = 4u };
#ifdef BF16K_CHECKS
__device__ uint32_t g_check_faults;
#endif
__device__ __forceinline__ bool check_fails(bool bad, uint32_t bit) {
#ifdef BF16K_CHECKS
    if (bad) {
        atomicOr(&g_check_faults, bit);
        return true;
    }
#else
    (void)bad;
    (void)bit;
#endif
    return false;
}
__device__ __forceinline__ bool mis16(const void *p) { return ((uintptr_t)p & 15u) != 0; }
__device__ __forceinline__ bool mis8(const void *p) { return ((uintptr_t)p & 7u) != 0; }

// -------------------------------------------------- programmatic dependent launch
// Every kernel of a step is launched with programmatic stream serialization:
// it may be scheduled while its predecessor on the stream is still draining,
// so its CTAs are resident and past their launch latency when that work ends.
// It therefore waits here, before its first global-memory access, until every
// prerequisite grid has completed with its writes visible (a no-op when it was
// launched the ordinary way), and at once allows its own successor to be
// scheduled.  The wait is the hardware's; no kernel spins on a flag.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ chunk schedule
// Under a fixed chunk stride a pass lasts as long as its slowest CTAs, and on
// GB300 some CTAs stream from HBM measurably slower than others: on the
// 1.72B-element shard the write-heavy FIRST pass ran at 0.93 of the copy peak
// with fixed strides and at 1.01 with the CTAs claiming chunks from a counter
// (the whole step 16.5 -> 15.8 ms).  Giving only the last quarter of the
// chunks out by claims was slower (15.96 ms): the CTAs' speed difference is
// larger than such a pool.  A chunk's results depend only on the chunk (the
// norm's partials are indexed by chunk), so they are bit-identical whatever
// CTA takes which chunk.
// The counter resets itself: every CTA makes exactly one claim past the last
// chunk, and the CTA whose claim is the very last one (nch + gridDim.x - 1)
// stores 0 -- after it no CTA of the grid touches the counter, and the next
// kernel on the stream starts after this grid has completed.  Hence no memset
// between passes, also inside a captured graph.
// ctr == nullptr: the fixed stride c0 + b, c0 + b + G, ...
struct ClaimSched {
    unsigned *ctr;
    uint32_t c0, c1;
    uint32_t *sh;          // shared slot for the claimed index

    __device__ __forceinline__ ClaimSched(unsigned *q, uint32_t a, uint32_t b, uint32_t *slot)
        : ctr(q), c0(a), c1(b), sh(slot) {}
    // All threads of the CTA call it; `ahead`: the value thread 0 claimed
    // while the previous chunk ran (use_ahead), else claimed now.
    __device__ __forceinline__ uint32_t claim(bool use_ahead, uint32_t ahead) {
        __syncthreads();                           // every thread is done with the previous index
        if (threadIdx.x == 0) *sh = use_ahead ? ahead : atomicAdd(ctr, 1u);
        __syncthreads();
        return c0 + *sh;
    }
    __device__ __forceinline__ uint32_t first() { return ctr ? claim(false, 0) : c0 + blockIdx.x; }
    __device__ __forceinline__ bool claims() const { return ctr != nullptr; }
    __device__ __forceinline__ uint32_t next(uint32_t c, bool use_ahead = false, uint32_t ahead = 0) {
        return ctr ? claim(use_ahead, ahead) : c + gridDim.x;
    }
    // c_end: the chunk index that ended the CTA's loop, i.e. its claim past the end
    __device__ __forceinline__ void release(uint32_t c_end) {
        if (ctr && threadIdx.x == 0 && c_end - c0 == (c1 - c0) + gridDim.x - 1) atomicExch(ctr, 0u);
    }
};
// The fixed stride alone, for the passes that fold several deferred gradients
// (they run at two or three CTAs per SM, and the claiming code's registers
// would cost them a resident CTA; measured slower).
struct StrideSched {
    uint32_t c0;
    __device__ __forceinline__ StrideSched(unsigned *, uint32_t a, uint32_t, uint32_t *) : c0(a) {}
    __device__ __forceinline__ uint32_t first() const { return c0 + blockIdx.x; }
    __device__ __forceinline__ bool claims() const { return false; }
    __device__ __forceinline__ uint32_t next(uint32_t c, bool = false, uint32_t = 0) const { return c + gridDim.x; }
    __device__ __forceinline__ void release(uint32_t) const {}
};
template <int KMAX>
using SchedFor = typename std::conditional<(KMAX <= 1), ClaimSched, StrideSched>::type;

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Compensated sum of squares in FP32: x*x split exactly into p + e (fma), p
// added by TwoSum (Knuth; Ogita, Rump & Oishi, "Accurate sum and dot
// product", SIAM J. Sci. Comput. 26(6), 2005).  The _rn intrinsics keep
// the compiler from contracting the error-free transformations into FMAs.
struct Comp {
    float s, c;
};
__device__ __forceinline__ void comp_add_sq(Comp &a, float x) {
    const float p = __fmul_rn(x, x);
    const float e = __fmaf_rn(x, x, -p);
    const float t = __fadd_rn(a.s, p);
    const float bp = __fsub_rn(t, a.s);
    const float err = __fadd_rn(__fsub_rn(a.s, __fsub_rn(t, bp)), __fsub_rn(p, bp));
    a.s = t;
    a.c = __fadd_rn(a.c, __fadd_rn(err, e));
}

// Gradient pointers of one pass, by value (for the out-of-line rescaled sum).
template <int KA>
struct GradPtrs {
    const uint16_t *p[KA];
};

// Deterministic CTA sum of one double per thread (kThreads threads); result valid in thread 0.
__device__ __forceinline__ double cta_sum(double x, double *sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) sh[w] = x;
    __syncthreads();
    double r = 0.0;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < kThreads / 32; ++i) r += sh[i];
    }
    __syncthreads();
    return r;
}

// A pointer's FP32/bf16 element index modulo 4 (16-byte FP32 / 8-byte bf16
// boundary) and modulo kHeadAlign.
__device__ __forceinline__ uint32_t phase4_f32(const void *p) { return (uint32_t)(((uintptr_t)p >> 2) & 3u); }
__device__ __forceinline__ uint32_t phase4_b16(const void *p) { return (uint32_t)(((uintptr_t)p >> 1) & 3u); }
__device__ __forceinline__ uint32_t phaseA_f32(const void *p) { return (uint32_t)(((uintptr_t)p >> 2) & (kHeadAlign - 1)); }
__device__ __forceinline__ uint32_t phaseA_b16(const void *p) { return (uint32_t)(((uintptr_t)p >> 1) & (kHeadAlign - 1)); }

// ---------------------------------------------------------------- accumulate

// Folds the pass's gradients into one FP32 value per element, in micro-batch
// order: v = acc (HAS_ACC) or the first gradient, then v = RN32(v + g_j) for
// each further gradient -- the same FP32 adds, in the same order, as one
// accumulate per micro-batch.
template <bool HAS_ACC, int KMAX>
__device__ __forceinline__ float fold_scalar(const float *a, const uint16_t *const *g, int K, uint32_t i) {
    float v = HAS_ACC ? a[i] : __uint_as_float((uint32_t)g[0][i] << 16);
#pragma unroll
    for (int j = HAS_ACC ? 0 : 1; j < KMAX; ++j)
        if (j < K) v = __fadd_rn(v, __uint_as_float((uint32_t)g[j][i] << 16));
    return v;
}

template <bool HAS_ACC, int KMAX>
__device__ __forceinline__ float4 fold_quad(const float4 &av, const uint2 *gv, int K) {
    float4 r;
    if (HAS_ACC) {
        r = av;
    } else {
        r = make_float4(bf_lo(gv[0].x), bf_hi(gv[0].x), bf_lo(gv[0].y), bf_hi(gv[0].y));
    }
#pragma unroll
    for (int j = HAS_ACC ? 0 : 1; j < KMAX; ++j) {
        if (j < K) {
            r.x = __fadd_rn(r.x, bf_lo(gv[j].x));
            r.y = __fadd_rn(r.y, bf_hi(gv[j].x));
            r.z = __fadd_rn(r.z, bf_lo(gv[j].y));
            r.w = __fadd_rn(r.w, bf_hi(gv[j].y));
        }
    }
    return r;
}

// A thread's sum of squares over its elements of a chunk, for a thread whose
// plain FP32 sum came out non-finite.  bf16 has FP32's exponent range, so a
// gradient above ~1.8e19 is an ordinary value whose square overflows FP32 but
// not the FP64 sum of squares of the definition.  Each value is multiplied by
// 2^-96 first (exact for every value above 2^-30), squared and summed the
// same compensated way, and the sum is scaled back by 2^192 in FP64.  Scaled
// squares that underflow stand for less than 2^43 each, against a thread sum
// above FP32's maximum (~2^128): relative 2^-78 even for 128 of them.  The
// scaled sum of finite values cannot overflow, so an infinite sum here means
// an infinite element and is returned as +Inf (the compensation term is NaN
// then, Inf - Inf); a NaN element gives NaN -- as the definition's FP64 sum
// would.  Visits the same
// elements as the vector pass: head (from rh), tail (from rt), then quads
// threadIdx.x + k * NT.
// FOLD: the value is fold(acc?, g...) (not stored by the pass); otherwise
// acc[i] (stored by the pass, or read alone).
template <bool FOLD, bool HAS_ACC, int KMAX, int KA, int NT>
__device__ __noinline__ double sumsq_rescaled(const float *a, GradPtrs<KA> gp, int K, uint32_t head, uint32_t nq,
                                              uint32_t len, float gscale, uint32_t rh, uint32_t rt) {
    Comp cs = {0.f, 0.f};
    auto add = [&](uint32_t i) {
        const float v = FOLD ? fold_scalar<HAS_ACC, KMAX>(a, gp.p, K, i) : a[i];
        comp_add_sq(cs, __fmul_rn(__fmul_rn(v, gscale), 0x1p-96f));
    };
    const uint32_t tail0 = head + (nq << 2);
    for (uint32_t i = rh; i < head; i += NT) add(i);
    for (uint32_t i = tail0 + rt; i < len; i += NT) add(i);
    for (uint32_t q = threadIdx.x; q < nq; q += NT)
        for (uint32_t r = 0; r < 4; ++r) add(head + 4 * q + r);
    const double s = isinf(cs.s) ? (double)cs.s : (double)cs.s + (double)cs.c;
    return s * 0x1p192;
}

__host__ __device__ constexpr int ilog2(uint32_t x) { return x <= 1 ? 0 : 1 + ilog2(x >> 1); }

// Thread index, rotated by whole warps, that takes a chunk's scalar head
// (half = 0) or tail (half = 1) elements.  The scalar elements cost a dependent
// load -> store round trip; always giving them to warp 0 made that warp lag
// further behind with every chunk (nothing re-synchronises the warps between
// chunks) and left the SM nearly idle while it caught up at the end.  The warp
// is the top bits of a Fibonacci hash of the chunk index (Knuth, TAOCP vol. 3,
// section 6.4), which spreads the chunks b, b + G, b + 2G, ... of one CTA over
// all warps for any grid size G; the tail goes to the warp half-way round.
// The map depends only on the chunk index, so results stay grid-independent.
template <int NT>
__device__ __forceinline__ uint32_t scalar_lane(uint32_t c, uint32_t half) {
    constexpr uint32_t W = NT / 32;
    static_assert(W >= 2 && (W & (W - 1)) == 0, "scalar_lane: a power-of-two number of warps");
    constexpr int kShift = 32 - ilog2(W);
    const uint32_t w = (c * 2654435761u + (half ? 0x80000000u : 0u)) >> kShift;
    return (threadIdx.x + NT - w * 32) % NT;
}

// Leading scalar elements of the chunk: up to the first element at which the
// lead pointer (the FP32 one if used, else the first gradient) sits on a
// kHeadAlign-element boundary; every other pointer is then at least on a
// 16-byte FP32 / 8-byte bf16 boundary, because all must share their element
// index modulo 4 -- or `len` when they do not (the chunk runs element-wise).
template <int KMAX>
__device__ __forceinline__ uint32_t chunk_head(const void *fp32_ptr, bool use_fp32, const uint16_t *const *g, int K,
                                               uint32_t len) {
    uint32_t ph = 0, lead = 0;
    bool have = false, vec = true;
    if (use_fp32) {
        ph = phase4_f32(fp32_ptr);
        lead = phaseA_f32(fp32_ptr);
        have = true;
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (j < K) {
            const uint32_t pg = phase4_b16(g[j]);
            if (have && pg != ph) vec = false;
            if (!have) lead = phaseA_b16(g[j]);
            ph = pg;
            have = true;
        }
    }
    uint32_t head = vec ? ((kHeadAlign - lead) & (kHeadAlign - 1)) : len;
    return head > len ? len : head;
}

// One pass over chunks [c0, c1): v = fold(acc?, g_0..g_{K-1}), stored back to
// acc if WRITE, and its per-chunk sum of squares (times gscale, rounded to
// FP32 first) written to partials[c] if NORM.  KMAX = 0 reads acc alone.
// Resident CTAs per SM the single-gradient passes are built for (the register
// budget of their measured launch shape, which the chunk-claiming code would
// otherwise exceed): 8 for the FIRST pass, 4 for the other stored pass, 3 for
// a norm pass.  0 for the passes that fold several deferred gradients: no
// minimum, the compiler's own choice (a minimum of 1 is not the same -- it
// lets the compiler spend registers up to one CTA per SM, and those passes
// lost a resident CTA).
template <bool HAS_ACC, int KMAX, bool WRITE, bool NORM>
constexpr int accum_min_blocks() {
    return KMAX == 1 ? ((!HAS_ACC && WRITE && !NORM) ? 8 : (NORM ? 3 : 4)) : 0;
}

template <bool HAS_ACC, int KMAX, bool WRITE, bool NORM, class GT, int U>
__global__ void __launch_bounds__(kThreads, (accum_min_blocks<HAS_ACC, KMAX, WRITE, NORM>()))
k_accum(const Seg *__restrict__ segs, const Chunk *__restrict__ chunks, uint32_t c0, uint32_t c1, GT gt,
        double *__restrict__ partials, float gscale, unsigned *queue) {
    __shared__ double sh[kThreads / 32];
    __shared__ uint32_t sh_claim;
    constexpr int KA = KMAX > 0 ? KMAX : 1;
    const int K = KMAX <= 1 ? KMAX : (int)gt.k;
    pdl_enter();
    SchedFor<KMAX> sch(queue, c0, c1, &sh_claim);
    uint32_t c = sch.first();
    for (; c < c1; c = sch.next(c)) {
        const Chunk ch = chunks[c];
        const Seg s = segs[ch.seg];
        float *a = s.acc + ch.start;
        const uint16_t *g[KA];
#pragma unroll
        for (int j = 0; j < KA; ++j) g[j] = (j < K) ? gt.get(s.grad_slot, j) + s.grad_off + ch.start : nullptr;
        const uint32_t len = ch.len;
        const uint32_t head = chunk_head<KMAX>(a, HAS_ACC || WRITE, g, K, len);
        const uint32_t nq = (len - head) >> 2;
        const uint32_t tail0 = head + (nq << 2);
        if (check_fails(ch.start + len > s.numel, kFaultChunkRange) || check_fails(tail0 > len, kFaultBody))
            continue;
        if (nq != 0) {
            bool bad = (HAS_ACC || WRITE) && mis16(a + head);
#pragma unroll
            for (int j = 0; j < KA; ++j)
                if (j < K) bad = bad || mis8(g[j] + head);
            if (check_fails(bad, kFaultAlign)) continue;
        }

        Comp cs = {0.f, 0.f};
        auto scalar = [&](uint32_t i) {
            const float v = fold_scalar<HAS_ACC, KMAX>(a, g, K, i);
            if (WRITE) a[i] = v;
            if (NORM) comp_add_sq(cs, __fmul_rn(v, gscale));
        };
        const uint32_t rh = scalar_lane<kThreads>(c, 0), rt = scalar_lane<kThreads>(c, 1);
        for (uint32_t i = rh; i < head; i += kThreads) scalar(i);
        for (uint32_t i = tail0 + rt; i < len; i += kThreads) scalar(i);

        const uint2 *g4[KA];
#pragma unroll
        for (int j = 0; j < KA; ++j) g4[j] = reinterpret_cast<const uint2 *>(g[j] + head);
        float4 *a4 = reinterpret_cast<float4 *>(a + head);
        for (uint32_t base = threadIdx.x; base < nq; base += kThreads * U) {
            uint2 gv[U][KA];
            float4 av[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t q = base + u * kThreads;
                if (q < nq) {
#pragma unroll
                    for (int j = 0; j < KMAX; ++j)
                        if (j < K) gv[u][j] = __ldcs(g4[j] + q);
                    if (HAS_ACC) av[u] = __ldcs(a4 + q);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t q = base + u * kThreads;
                if (q < nq) {
                    const float4 r = fold_quad<HAS_ACC, KMAX>(av[u], gv[u], K);
                    if (WRITE) __stcs(a4 + q, r);
                    if (NORM) {
                        comp_add_sq(cs, __fmul_rn(r.x, gscale));
                        comp_add_sq(cs, __fmul_rn(r.y, gscale));
                        comp_add_sq(cs, __fmul_rn(r.z, gscale));
                        comp_add_sq(cs, __fmul_rn(r.w, gscale));
                    }
                }
            }
        }
        if (NORM) {
            double mine = (double)cs.s + (double)cs.c;
            if (!isfinite(mine)) {                      // rare: a square overflowed FP32
                GradPtrs<KA> gp;
#pragma unroll
                for (int j = 0; j < KA; ++j) gp.p[j] = g[j];
                mine = sumsq_rescaled<!WRITE, HAS_ACC, KMAX, KA, kThreads>(a, gp, K, head, nq, len, gscale, rh, rt);
            }
            const double tot = cta_sum(mine, sh);
            if (threadIdx.x == 0) partials[c] = tot;
        }
    }
    sch.release(c);
}

// ---------------------------------------------------------------- norm final

// Fixed-order FP64 sum of n partials by one CTA of kFinalThreads threads:
// thread i adds partials i, i + kFinalThreads, ... in index order, then a
// halving tree over the threads.  The order depends only on n, so every call
// over the same partials gives the same bits.  Result valid in thread 0.
__device__ __forceinline__ double final_sum(const double *__restrict__ partials, uint32_t n, double *sh) {
    double s = 0.0;
    for (uint32_t i = threadIdx.x; i < n; i += kFinalThreads) s += partials[i];
    sh[threadIdx.x] = s;
    __syncthreads();
    for (int w = kFinalThreads / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
        __syncthreads();
    }
    return sh[0];
}

// norm = sqrt(S) and the clip coefficient c = max_norm / norm if norm >
// max_norm (max_norm > 0), else exactly 1 ("企业官网建设流程全解析", section 4.3).
struct NormClip {
    double sumsq, norm, c;
};
__device__ __forceinline__ NormClip norm_and_clip(double S, float max_norm) {
    NormClip r;
    r.sumsq = S;
    r.norm = sqrt(S);
    r.c = 1.0;
    if (max_norm > 0.0f && r.norm > (double)max_norm) r.c = (double)max_norm / r.norm;
    return r;
}

// The handle's norm state from a norm and clip coefficient: c kept as a
// float-float pair so that acc * c is rounded once in the step.
__device__ __forceinline__ void store_norm_state(const NormClip &r, NormState *__restrict__ out) {
    const float hi = __double2float_rn(r.c);
    out->sumsq = r.sumsq;
    out->norm = r.norm;
    out->c_hi = hi;
    out->c_lo = __double2float_rn(r.c - (double)hi);
    out->finite = isfinite(r.sumsq) ? 1 : 0;
    out->pad = 0;
}

// b^t for an integer t >= 0 by binary exponentiation in FP64: about 2 log2(t)
// multiplications (GB300's FP64 pipe is slow; a general pow costs far more),
// a fixed function of t, so every path that reaches step t -- eager, replayed
// graph, resumed run -- gets the same bits.  Relative error below
// 2 log2(t) units of 2^-53, far inside what the FP32 scalars keep.
__device__ __forceinline__ double pow_int(double b, int64_t t) {
    double r = 1.0, x = b;
    for (uint64_t e = (uint64_t)t; e != 0; e >>= 1) {
        if (e & 1) r *= x;
        x *= x;
    }
    return r;
}

// The per-group FP32 scalars of step t, computed in FP64 from the FP32
// hyper-parameters: bias corrections 1 - b^t (Kingma & Ba, Algorithm 1),
// step_size = lr / bc1, 1 / sqrt(bc2), decay = lr * wd, with lr times the
// warmup + cosine factor when a schedule is attached.
__device__ __forceinline__ void group_scalars(const StepParams *__restrict__ P, int64_t t, float lr_g, int g,
                                              GroupK &o) {
    double f = 1.0;
    if (P->has_sched) {
        const double r = (double)P->min_ratio;
        if (t <= P->warmup) {
            f = (double)t / (double)P->warmup;
        } else if (t <= P->decay) {
            const double x = (double)(t - P->warmup) / (double)(P->decay - P->warmup);
            f = r + (1.0 - r) * 0.5 * (1.0 + cos(3.141592653589793 * x));
        } else {
            f = r;
        }
    }
    const double lr = (double)lr_g * f;
    const double b1 = (double)P->beta1[g], b2 = (double)P->beta2[g];
    const double bc1 = 1.0 - pow_int(b1, t);
    const double bc2 = 1.0 - pow_int(b2, t);
    o.b1 = (float)b1;
    o.omb1 = (float)(1.0 - b1);
    o.b2 = (float)b2;
    o.omb2 = (float)(1.0 - b2);
    o.eps = P->eps[g];
    o.decay = (float)(lr * (double)P->wd[g]);
    o.step_size = (float)(lr / bc1);
    o.inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
}

// The scalars of the next step (t + 1, the groups' own learning rates) and its
// skip decision, prepared as soon as the norm is known so that the step needs
// no kernel of its own: thread g < n_groups writes group g, thread 0 the skip
// flag.  The step counter itself advances only when the step runs.
__device__ __forceinline__ void prepare_step(const StepParams *__restrict__ P, StepState *S, double sumsq) {
    const int g = threadIdx.x;
    const int64_t t = S->t + 1;
    if (g < P->n_groups && g < kMaxGroups) group_scalars(P, t, P->lr[g], g, S->gtab.g[g]);
    if (g == 0) S->skip = (P->skip_nonfinite && !isfinite(sumsq)) ? 1 : 0;
}

// Sum of the chunk partials in a fixed order, then norm and clip coefficient,
// and the scalars of the step that follows.
// Warp 0 computes the group scalars, warp 1 the norm and clip coefficient, at
// the same time.
__global__ void __launch_bounds__(kFinalThreads)
k_norm_final(const double *__restrict__ partials, uint32_t n, float max_norm, NormState *__restrict__ out,
             const StepParams *__restrict__ P, StepState *S) {
    __shared__ double sh[kFinalThreads];
    pdl_enter();
    const double sumsq = final_sum(partials, n, sh);
    if (threadIdx.x < 32) prepare_step(P, S, sumsq);
    else if (threadIdx.x == 32) store_norm_state(norm_and_clip(sumsq, max_norm), out);
}

// Norm and clip coefficient from a sum of squares given by the host (the
// all-rank sum under ZeRO): same formula as k_norm_final.  Two warps.
__global__ void k_norm_from_sumsq(double sumsq, float max_norm, NormState *__restrict__ out,
                                  const StepParams *__restrict__ P, StepState *S) {
    pdl_enter();
    if (threadIdx.x < 32) prepare_step(P, S, sumsq);
    else if (threadIdx.x == 32) store_norm_state(norm_and_clip(sumsq, max_norm), out);
}

// t <- t + 1 (unless the step is skipped) and the per-group scalars of step t
// with the per-call learning rates, for a step whose scalars were not prepared
// with the norm (a learning-rate override, settings changed since the norm, or
// an empty shard).  One warp.
__global__ void k_step_scalars(const StepParams *__restrict__ P, StepState *S, LrOverride ov,
                               const NormState *__restrict__ ns) {
    pdl_enter();
    const int skip = (P->skip_nonfinite && !ns->finite) ? 1 : 0;
    const int64_t t = S->t + 1;
    const int g = threadIdx.x;
    if (g < P->n_groups && g < kMaxGroups) group_scalars(P, t, ov.use ? ov.lr[g] : P->lr[g], g, S->gtab.g[g]);
    __syncwarp();
    if (g == 0) {
        S->skip = skip;
        if (!skip) S->t = t;
    }
}

// ---------------------------------------------------------------------- step

struct AdamOut {
    float p, m, v;
};

__device__ __forceinline__ AdamOut adam_elem(float e, float p, float m, float v, float c_hi, float c_lo,
                                             const GroupK &G) {
    const float gc = fmaf(e, c_hi, e * c_lo);                 // clipped gradient
    const float m1 = fmaf(G.b1, m, G.omb1 * gc);
    const float v1 = fmaf(G.b2, v, G.omb2 * gc * gc);
    const float den = fmaf(sqrtf(v1), G.inv_sqrt_bc2, G.eps); // sqrt(v_hat) + eps
    const float upd = __fdiv_rn(m1, den);
    // p - (lr wd p + step_size upd): the decay and the update are summed first
    // (both are small next to p), so p itself is rounded once.
    const float delta = fmaf(G.decay, p, G.step_size * upd);
    const float p1 = __fsub_rn(p, delta);
    return {p1, m1, v1};
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Fused clip + AdamW + master update + bf16 cast over chunks [c0, c1).  The
// gradient is fold(acc?, g_0..g_{K-1}): the stored accumulator (KMAX = 0), or
// the accumulator plus deferred micro-batches, or deferred micro-batches alone.
template <bool HAS_ACC, int KMAX, class GT, int U>
__global__ void __launch_bounds__(kStepThreads, BF16K_STEP_MIN_BLOCKS)
k_step(const Seg *__restrict__ segs, const Chunk *__restrict__ chunks, uint32_t c0, uint32_t c1, GT gt,
       StepState *st, const NormState *__restrict__ ns, float gscale, int commit_t, unsigned *queue) {
    __shared__ uint32_t sh_claim;
    constexpr int KA = KMAX > 0 ? KMAX : 1;
    const int K = KMAX <= 1 ? KMAX : (int)gt.k;
    pdl_enter();
    if (st->skip) return;                   // non-finite norm, skipping enabled (no CTA claims a chunk)
    // the step counter advances with the step whose scalars the norm prepared
    // (nothing in this kernel reads it)
    if (commit_t && blockIdx.x == 0 && threadIdx.x == 0) st->t += 1;
    const GroupTable *__restrict__ gtab = &st->gtab;
    const float c_hi = ns->c_hi, c_lo = ns->c_lo;
    // one CTA per SM: the next pooled chunk is claimed when the current one
    // starts, so the atomic's round trip overlaps the chunk's work
    SchedFor<KMAX> sch(queue, c0, c1, &sh_claim);
    uint32_t ahead = 0;
    uint32_t c = sch.first();
    for (; c < c1; c = sch.next(c, true, ahead)) {
        if (sch.claims() && threadIdx.x == 0) ahead = atomicAdd(queue, 1u);
        const Chunk ch = chunks[c];
        const Seg s = segs[ch.seg];
        const GroupK G = gtab->g[s.group];
        const float *a = s.acc + ch.start;
        const uint16_t *g[KA];
#pragma unroll
        for (int j = 0; j < KA; ++j) g[j] = (j < K) ? gt.get(s.grad_slot, j) + s.grad_off + ch.start : nullptr;
        float *p = s.p + ch.start;
        float *m = s.m + ch.start;
        float *v = s.v + ch.start;
        uint16_t *bf = s.bf + ch.start;
        const uint32_t len = ch.len;

        uint32_t head = chunk_head<KMAX>(p, true, g, K, len);
        const uint32_t ph = phase4_f32(p);
        if (!(phase4_f32(m) == ph && phase4_f32(v) == ph && phase4_b16(bf) == ph && (!HAS_ACC || phase4_f32(a) == ph)))
            head = len;
        const uint32_t nq = (len - head) >> 2;
        const uint32_t tail0 = head + (nq << 2);
        if (check_fails(ch.start + len > s.numel, kFaultChunkRange) || check_fails(tail0 > len, kFaultBody))
            continue;
        if (nq != 0) {
            bool bad = mis16(p + head) || mis16(m + head) || mis16(v + head) || mis8(bf + head) ||
                       (HAS_ACC && mis16(a + head));
#pragma unroll
            for (int j = 0; j < KA; ++j)
                if (j < K) bad = bad || mis8(g[j] + head);
            if (check_fails(bad, kFaultAlign)) continue;
        }

        auto scalar = [&](uint32_t i) {
            const float e = __fmul_rn(fold_scalar<HAS_ACC, KMAX>(a, g, K, i), gscale);
            const AdamOut o = adam_elem(e, p[i], m[i], v[i], c_hi, c_lo, G);
            p[i] = o.p;
            m[i] = o.m;
            v[i] = o.v;
            bf[i] = __bfloat16_as_ushort(__float2bfloat16_rn(o.p));
        };
        const uint32_t rh = scalar_lane<kStepThreads>(c, 0), rt = scalar_lane<kStepThreads>(c, 1);
        for (uint32_t i = rh; i < head; i += kStepThreads) scalar(i);
        for (uint32_t i = tail0 + rt; i < len; i += kStepThreads) scalar(i);

        const float4 *a4 = reinterpret_cast<const float4 *>(a + head);
        const uint2 *g4[KA];
#pragma unroll
        for (int j = 0; j < KA; ++j) g4[j] = reinterpret_cast<const uint2 *>(g[j] + head);
        float4 *p4 = reinterpret_cast<float4 *>(p + head);
        float4 *m4 = reinterpret_cast<float4 *>(m + head);
        float4 *v4 = reinterpret_cast<float4 *>(v + head);
        uint2 *b4 = reinterpret_cast<uint2 *>(bf + head);
        for (uint32_t base = threadIdx.x; base < nq; base += kStepThreads * U) {
            float4 av[U], pv[U], mv[U], vv[U];
            uint2 gv[U][KA];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t q = base + u * kStepThreads;
                if (q < nq) {
                    if (HAS_ACC) av[u] = __ldcs(a4 + q);
#pragma unroll
                    for (int j = 0; j < KMAX; ++j)
                        if (j < K) gv[u][j] = __ldcs(g4[j] + q);
                    pv[u] = __ldcs(p4 + q);
                    mv[u] = __ldcs(m4 + q);
                    vv[u] = __ldcs(v4 + q);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t q = base + u * kStepThreads;
                if (q < nq) {
                    const float4 e = fold_quad<HAS_ACC, KMAX>(av[u], gv[u], K);
                    const AdamOut o0 = adam_elem(__fmul_rn(e.x, gscale), pv[u].x, mv[u].x, vv[u].x, c_hi, c_lo, G);
                    const AdamOut o1 = adam_elem(__fmul_rn(e.y, gscale), pv[u].y, mv[u].y, vv[u].y, c_hi, c_lo, G);
                    const AdamOut o2 = adam_elem(__fmul_rn(e.z, gscale), pv[u].z, mv[u].z, vv[u].z, c_hi, c_lo, G);
                    const AdamOut o3 = adam_elem(__fmul_rn(e.w, gscale), pv[u].w, mv[u].w, vv[u].w, c_hi, c_lo, G);
                    __stcs(p4 + q, make_float4(o0.p, o1.p, o2.p, o3.p));
                    __stcs(m4 + q, make_float4(o0.m, o1.m, o2.m, o3.m));
                    __stcs(v4 + q, make_float4(o0.v, o1.v, o2.v, o3.v));
                    __stcs(b4 + q, make_uint2(pack_bf16x2(o0.p, o1.p), pack_bf16x2(o2.p, o3.p)));
                }
            }
        }
    }
    sch.release(c);
}


// ------------------------------------------------------ bulk-copy pipeline
// The traffic of the fused step and of the later accumulate passes moved by
// the SM's bulk asynchronous copy unit instead of per-thread vector loads and
// stores: cp.async.bulk copies whole runs of a stream between global and
// shared memory, loads completing on an mbarrier by transaction count, stores
// retired through bulk groups.  One thread of the CTA issues every copy; the
// other warps compute in shared memory.  Measured on the step's 18:14
// read:write mix over 2^30 elements: 7.20 TB/s against 7.00 TB/s for the best
// shape of 16-byte vector loads.

// Waits that gave up (see mbar_wait); read and cleared by
// bf16opt_pipeline_timeouts.
__device__ uint32_t g_pipe_timeouts;

constexpr uint64_t kPipeWaitNs = 2000000000ull;   // a stage wait normally takes microseconds
constexpr uint64_t kPipeDrainNs = 200000000ull;   // copies still in flight after a timeout

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}
// Makes the initialised barriers visible to the asynchronous proxy.
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// One arrival that also expects `bytes` of bulk-copy transactions this phase.
__device__ __forceinline__ void mbar_arrive_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase of parity `parity` of *b to complete, for at most
// limit_ns; a wait that gives up is counted in g_pipe_timeouts and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, uint64_t limit_ns) {
    if (mbar_test(b, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(b, parity)) return true;
        if ((i & 63u) == 0 && global_ns() - t0 > limit_ns) {
            atomicAdd(&g_pipe_timeouts, 1u);
            return false;
        }
    }
}
// L2 policy of the bulk copies: evict first, like the streaming loads and
// stores (ld/st .cs) of every other pass.  Without it the copies leave their
// lines at normal priority; the L2 then evicts the other passes' evict-first
// lines ahead of them, and every pass after the step ran 1.4 % slower (the
// step kernel of another handle too) until a kernel touched those lines again.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global -> shared, `bytes` (a multiple of 16, both addresses 16-byte aligned),
// completing as transactions on *bar.
__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar,
                                          uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}
// Shared -> global, in the current bulk group.
__device__ __forceinline__ void bulk_store(void *dst, const void *src_smem, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                 "r"(smem_addr(src_smem)), "r"(bytes), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until at most N of this thread's most recent bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's shared-memory writes before later asynchronous-proxy
// (bulk copy) reads of them.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

#ifndef BF16K_PIPE_WARPS
#define BF16K_PIPE_WARPS 8
#endif
#ifndef BF16K_PIPE_SMEM
#define BF16K_PIPE_SMEM (200u * 1024u)
#endif
constexpr int kPipeWarps = BF16K_PIPE_WARPS;            // compute warps (one more warp issues the copies)
constexpr int kPipeThreads = 32 * (kPipeWarps + 1);
constexpr int kPipeCompute = 32 * kPipeWarps;
constexpr uint32_t kPipeSmem = BF16K_PIPE_SMEM;         // stage buffers per CTA (one CTA per SM)
constexpr int kPipeMaxStages = 8;
constexpr int kPipeLag = 1;                             // stores still reading a stage when the next load is issued
static_assert(kPipeWarps >= 2, "the head and tail scalars go to compute warps 0 and 1");

// Bytes of one fused-step stage per 4-element quad: the accumulator, K
// gradient slots (one when K = 0: the bf16 output; otherwise slot 0 takes the
// bf16 output after the gradients are read), master, m, v.
__host__ __device__ constexpr uint32_t pipe_quad_bytes(bool has_acc, int K) {
    return (has_acc ? 16u : 0u) + 8u * (uint32_t)(K > 0 ? K : 1) + 48u;
}
// Quads per fused-step tile (a stage holds one tile): even, so that every
// bf16 run is a multiple of 16 bytes.
constexpr uint32_t kPipeTileQuads = 512;
// The pipeline takes fused steps whose stage is at most 80 bytes per quad (the
// accumulator with up to 2 deferred gradients, or up to 4 without it): five
// 40 KB stages.  Folding more gradients, a stage holds one 4 KB run per
// gradient; folding 8 of them through the pipeline made the whole step 7-13 %
// slower than with vector loads (the GAS-32 and 72-tensor shards).
constexpr uint32_t kPipeMaxQuadBytes = 80;
__host__ __device__ constexpr bool pipe_fits(bool has_acc, int K) {
    return pipe_quad_bytes(has_acc, K) <= kPipeMaxQuadBytes;
}
__host__ __device__ constexpr int pipe_stages(bool has_acc, int K) {
    return (int)(kPipeSmem / (pipe_quad_bytes(has_acc, K) * kPipeTileQuads)) < kPipeMaxStages
               ? (int)(kPipeSmem / (pipe_quad_bytes(has_acc, K) * kPipeTileQuads))
               : kPipeMaxStages;
}
static_assert(pipe_stages(false, 4) > kPipeLag && pipe_stages(false, 4) >= 4, "pipeline depth");

// An accumulate pass's stage: one tile of 2,048 quads (8,192 elements, one
// claimed unit), accumulator 32 KB + gradient 16 KB; four stages.  Probe on
// a later pass's traffic (6:4 bytes read:written) over 1.8e9 elements: 7.22
// TB/s against 7.15 with 16-byte vector loads; with 4,096-element tiles it
// was slower than vector loads (the copy thread's work per tile dominated).
constexpr uint32_t kAccTileQuads = 2048;
constexpr uint32_t kAccQuadBytes = 24;
constexpr int kAccStages = (int)(kPipeSmem / (kAccQuadBytes * kAccTileQuads)) < kPipeMaxStages
                               ? (int)(kPipeSmem / (kAccQuadBytes * kAccTileQuads))
                               : kPipeMaxStages;
static_assert(kAccStages > kPipeLag && kAccStages >= 4, "accumulate pipeline depth");

// Leading scalar elements of a chunk before its bulk body: up to the first
// element at which the bf16 parameter pointer is 16-byte aligned.  The host
// runs the pipeline only on segments whose FP32 pointers share their element
// index modulo 4 and whose bf16 pointers share it modulo 8 (the two agreeing
// modulo 4), so every stream is 16-byte aligned there.
__host__ __device__ __forceinline__ uint32_t pipe_head(const uint16_t *bf, uint32_t len) {
    const uint32_t h = (8u - (uint32_t)(((uintptr_t)bf >> 1) & 7u)) & 7u;
    return h < len ? h : len;
}

// The pipelined passes' unit of work, claimed one at a time: up to
// kPipeUnitQuads quads of one chunk's body (a chunk without body, only scalar
// elements, is one unit with nq = 0).  The host lists the units of every
// chunk in chunk order.  Measured on the 1.72B-element shard (step kernel):
// units of 2,048 / 8,192 / 16,384 / 32,768 elements took 8.19 / 7.74 / 7.78 /
// 7.82 ms (vector loads, chunk claims: 7.93).  Smaller claims keep the SMs
// streaming from nearby addresses, but one claim per stage tile cost more
// than that gained.
#ifndef BF16K_PIPE_UNIT_QUADS
#define BF16K_PIPE_UNIT_QUADS 2048
#endif
constexpr uint32_t kPipeUnitQuads = BF16K_PIPE_UNIT_QUADS;
static_assert(kPipeUnitQuads % kPipeTileQuads == 0 && kPipeUnitQuads % kAccTileQuads == 0, "a unit is whole tiles");
struct PipeUnit {
    uint64_t el;        // first body element, relative to the segment
    uint32_t seg;
    uint32_t chunk;
    uint32_t nq;        // body quads (even; at most kPipeUnitQuads)
    uint32_t scalars;   // the chunk's first unit, and the chunk has scalar head or tail elements
};

// What the copy thread tells the compute warps about the tile in a stage.
struct TileDesc {
    void *out[4];       // the tile's first body element in each stream the pass stores
    uint32_t group;
    uint32_t nq;        // body quads in the tile (even; 0 for a chunk without body)
    uint32_t chunk;     // its chunk; kTileEnd: no more tiles for this CTA
    uint32_t scalars;   // this tile also does the chunk's scalar head and tail
};
constexpr uint32_t kTileEnd = 0xffffffffu;

// The barriers and descriptors of a pipelined pass (static shared memory).
struct PipeShared {
    uint64_t full[kPipeMaxStages];   // a stage's loads landed (or a tile without body, or the end)
    uint64_t done[kPipeMaxStages];   // the compute warps finished a stage
    TileDesc desc[kPipeMaxStages];
};

// A pipelined pass over units [u0, u1): the same ring of shared-memory stages
// for every pass, and an `Ops` type for what a pass moves and computes:
//   kTileQuads                 quads per tile (even; divides kPipeUnitQuads)
//   stages, stage_bytes        ring depth, bytes of one stage
//   tile_bytes(nq)             bytes the loads of a tile of nq quads bring in
//   set_seg(sg)                the copy thread's per-segment set-up
//   misaligned(sg, e)          a stream not 16-byte aligned at element e (checked build)
//   load(sg, e, nq, stage, bar, pol)   the tile's bulk loads, completing on bar
//   outputs(sg, e, out)        where the tile's results go
//   store(d, stage, pol)       the tile's bulk stores
//   compute(d, stage, ct)      compute thread ct's quads of a stage, in place
//   scalar(ch, sg, i, group)   element i of a chunk, from and to global memory
//
// Warp 0, lane 0, is the copy thread.  It claims units (from `queue`, or the
// fixed stride when it is null), the next unit and its table entry one unit
// ahead.  It cuts each unit into tiles and streams each tile through the
// ring.  A stage is refilled once the tile that used it was stored and its
// stores have read it; D = stages - kPipeLag tiles stay loaded ahead of the
// oldest one not yet stored.  The compute warps take the stages in order,
// update them in place, and release them to the copy thread; warps 0 and 1
// also do a chunk's scalar head and tail elements with its first tile.
//
// Every wait is bounded (kPipeWaitNs).  A copy thread that gives up lets its
// loads in flight land, keeps the counter's reset rule and returns; compute
// warps that give up return.  g_pipe_timeouts counts every wait that gave up.
template <class Ops>
__device__ __forceinline__ void pipe_copy_thread(Ops &ops, const Seg *__restrict__ segs,
                                                 const PipeUnit *__restrict__ units, uint32_t u0, uint32_t u1,
                                                 unsigned *queue, unsigned char *smem, PipeShared &sh) {
    constexpr int L = kPipeLag;
    constexpr uint32_t tq = Ops::kTileQuads;
    const int nst = ops.stages;
    const int D = nst - L;
    const uint64_t pol = l2_evict_first();
    int issued = 0, stored = 0;
    bool ok = true;
    // The oldest computed tile's results go out.
    auto retire = [&]() -> bool {
        const int s = stored % nst;
        if (!mbar_wait(&sh.done[s], (uint32_t)(stored / nst) & 1u, kPipeWaitNs)) return false;
        if (sh.desc[s].nq) ops.store(sh.desc[s], smem + (size_t)s * ops.stage_bytes, pol);
        bulk_commit();
        ++stored;
        return true;
    };
    // Stage for tile `issued`: free once the tile that used it was stored
    // and its stores have read it.
    auto acquire = [&]() -> int {
        while (stored <= issued - D) {
            if (!retire()) return -1;
            bulk_wait_read<L>();
        }
        return issued % nst;
    };
    const bool claims = queue != nullptr;
    uint32_t u = claims ? u0 + atomicAdd(queue, 1u) : u0 + blockIdx.x;
    uint32_t last = u;                  // the most recent claim
    uint32_t un = u;
    if (u < u1) last = un = claims ? u0 + atomicAdd(queue, 1u) : u + gridDim.x;
    PipeUnit rec{};
    if (u < u1) rec = units[u];
    uint32_t cur_seg = 0xffffffffu;
    Seg sg{};
    while (ok && u < u1) {
        const bool more = un < u1;
        PipeUnit recn{};
        if (more) recn = units[un];
        const uint32_t unn = more ? (claims ? u0 + atomicAdd(queue, 1u) : un + gridDim.x) : un;
        if (more) last = unn;
        if (rec.seg != cur_seg) {
            cur_seg = rec.seg;
            sg = segs[cur_seg];
            ops.set_seg(sg);
        }
        const uint64_t e0 = rec.el;
        bool bad = check_fails(e0 + 4ull * rec.nq > sg.numel, kFaultChunkRange);
        if (rec.nq) bad = bad || check_fails(ops.misaligned(sg, e0), kFaultAlign);
        if (!bad) {
            for (uint32_t q = 0; q < rec.nq || q == 0; q += tq) {
                const uint32_t nq = rec.nq - q < tq ? rec.nq - q : tq;
                const int s = acquire();
                if (s < 0) {
                    ok = false;
                    break;
                }
                const uint64_t e = e0 + 4ull * q;
                TileDesc &d = sh.desc[s];
                ops.outputs(sg, e, d.out);
                d.group = sg.group;
                d.nq = nq;
                d.chunk = rec.chunk;
                d.scalars = q == 0 ? rec.scalars : 0u;
                if (nq) {
                    mbar_arrive_tx(&sh.full[s], ops.tile_bytes(nq));
                    ops.load(sg, e, nq, smem + (size_t)s * ops.stage_bytes, &sh.full[s], pol);
                } else {
                    mbar_arrive(&sh.full[s]);
                }
                ++issued;
            }
        }
        u = un;
        un = unn;
        rec = recn;
    }
    if (ok) {
        const int s = acquire();
        if (s >= 0) {
            sh.desc[s].chunk = kTileEnd;
            mbar_arrive(&sh.full[s]);
            while (stored < issued)
                if (!retire()) break;
        }
    }
    if (stored < issued) {
        // gave up: let the loads still in flight land before leaving
        for (int i = stored; i < issued; ++i)
            mbar_wait(&sh.full[i % nst], (uint32_t)(i / nst) & 1u, kPipeDrainNs);
        // and keep the counter's reset rule: claim (without work) up to the first claim past the end
        if (claims)
            while (last < u1) last = u0 + atomicAdd(queue, 1u);
    }
    bulk_wait_all();
    // every CTA's claims ended on exactly one past the end; the last such claim resets the counter
    if (claims && last - u0 == (u1 - u0) + gridDim.x - 1) atomicExch(queue, 0u);
}

template <class Ops>
__device__ __forceinline__ void pipe_compute_warps(const Ops &ops, const Seg *__restrict__ segs,
                                                   const Chunk *__restrict__ chunks, unsigned char *smem,
                                                   PipeShared &sh) {
    const uint32_t ct = threadIdx.x - 32;
    const int nst = ops.stages;
    for (int i = 0;; ++i) {
        const int s = i % nst;
        if (!mbar_wait(&sh.full[s], (uint32_t)(i / nst) & 1u, kPipeWaitNs)) return;
        const TileDesc d = sh.desc[s];
        if (d.chunk == kTileEnd) return;
        unsigned char *stg = smem + (size_t)s * ops.stage_bytes;
        ops.compute(d, stg, ct);
        if (d.scalars) {
            // the chunk's head (warp 0) and tail (warp 1) elements, straight from global memory
            const Chunk ch = chunks[d.chunk];
            const Seg sg = segs[ch.seg];
            const uint32_t len = ch.len;
            const uint32_t hb = pipe_head(sg.bf + ch.start, len);
            const uint32_t tail0 = hb + ((((len - hb) >> 3) << 1) << 2);
            const uint32_t w = ct >> 5, lane = ct & 31u;
            const uint32_t i0 = w == 0 ? lane : (w == 1 ? tail0 + lane : len);
            if (i0 < (w == 0 ? hb : len) && !check_fails(ch.start + len > sg.numel, kFaultChunkRange))
                ops.scalar(ch, sg, i0, d.group);
        }
        fence_async_smem();
        mbar_arrive(&sh.done[s]);
    }
}

// Sets up the barriers (thread 0), then runs the copy thread (warp 0, lane 0;
// the rest of warp 0 leaves) or the compute warps.
template <class Ops>
__device__ __forceinline__ void pipe_run(Ops &ops, const Seg *__restrict__ segs, const Chunk *__restrict__ chunks,
                                         const PipeUnit *__restrict__ units, uint32_t u0, uint32_t u1,
                                         unsigned *queue, unsigned char *smem, PipeShared &sh) {
    if (threadIdx.x == 0) {
        for (int i = 0; i < ops.stages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.done[i], kPipeCompute);
        }
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) pipe_copy_thread(ops, segs, units, u0, u1, queue, smem, sh);
        return;
    }
    pipe_compute_warps(ops, segs, chunks, smem, sh);
}

// The fused step's traffic and arithmetic per tile (see k_step_pipe).
template <bool HAS_ACC, int KMAX, class GT>
struct StepOps {
    static constexpr uint32_t kTileQuads = kPipeTileQuads;
    static constexpr int KA = KMAX > 0 ? KMAX : 1;
    const GT *gt;
    const GroupK *gtab;                 // the groups' scalars (shared memory)
    int K;
    float gscale, c_hi, c_lo;
    int stages;
    uint32_t stage_bytes, off_g, off_p, off_m, off_v;
    const uint16_t *gb[KA];             // copy thread: the current segment's gradient bases

    __device__ StepOps(const GT *g, const GroupK *tab, int k, float gs, float hi, float lo)
        : gt(g), gtab(tab), K(k), gscale(gs), c_hi(hi), c_lo(lo) {
        stages = pipe_stages(HAS_ACC, K);
        off_g = HAS_ACC ? 16u * kTileQuads : 0u;
        off_p = off_g + 8u * kTileQuads * (uint32_t)(K > 0 ? K : 1);
        off_m = off_p + 16u * kTileQuads;
        off_v = off_m + 16u * kTileQuads;
        stage_bytes = off_v + 16u * kTileQuads;
    }
    __device__ uint32_t tile_bytes(uint32_t nq) const {
        return nq * (pipe_quad_bytes(HAS_ACC, K) - (K == 0 ? 8u : 0u));   // no gradient slot is loaded when K = 0
    }
    __device__ void set_seg(const Seg &sg) {
#pragma unroll
        for (int j = 0; j < KA; ++j) gb[j] = (j < K) ? gt->get(sg.grad_slot, j) + sg.grad_off : nullptr;
    }
    __device__ bool misaligned(const Seg &sg, uint64_t e) const {
        bool mis = mis16(sg.p + e) || mis16(sg.m + e) || mis16(sg.v + e) || mis16(sg.bf + e) ||
                   (HAS_ACC && mis16(sg.acc + e));
#pragma unroll
        for (int j = 0; j < KA; ++j)
            if (j < K) mis = mis || mis16(gb[j] + e);
        return mis;
    }
    __device__ void load(const Seg &sg, uint64_t e, uint32_t nq, unsigned char *stg, uint64_t *bar,
                         uint64_t pol) const {
        if (HAS_ACC) bulk_load(stg, sg.acc + e, 16u * nq, bar, pol);
#pragma unroll
        for (int j = 0; j < KA; ++j)
            if (j < K) bulk_load(stg + off_g + 8u * kTileQuads * j, gb[j] + e, 8u * nq, bar, pol);
        bulk_load(stg + off_p, sg.p + e, 16u * nq, bar, pol);
        bulk_load(stg + off_m, sg.m + e, 16u * nq, bar, pol);
        bulk_load(stg + off_v, sg.v + e, 16u * nq, bar, pol);
    }
    __device__ void outputs(const Seg &sg, uint64_t e, void **out) const {
        out[0] = sg.p + e;
        out[1] = sg.m + e;
        out[2] = sg.v + e;
        out[3] = sg.bf + e;
    }
    __device__ void store(const TileDesc &d, unsigned char *stg, uint64_t pol) const {
        bulk_store(d.out[0], stg + off_p, 16u * d.nq, pol);
        bulk_store(d.out[1], stg + off_m, 16u * d.nq, pol);
        bulk_store(d.out[2], stg + off_v, 16u * d.nq, pol);
        bulk_store(d.out[3], stg + off_g, 8u * d.nq, pol);
    }
    __device__ void compute(const TileDesc &d, unsigned char *stg, uint32_t ct) const {
        const GroupK G = gtab[d.group];
        const float4 *a4 = reinterpret_cast<const float4 *>(stg);
        uint2 *g4 = reinterpret_cast<uint2 *>(stg + off_g);
        float4 *p4 = reinterpret_cast<float4 *>(stg + off_p);
        float4 *m4 = reinterpret_cast<float4 *>(stg + off_m);
        float4 *v4 = reinterpret_cast<float4 *>(stg + off_v);
        for (uint32_t q = ct; q < d.nq; q += kPipeCompute) {
            float4 av = make_float4(0.f, 0.f, 0.f, 0.f);
            uint2 gv[KA];
            if (HAS_ACC) av = a4[q];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < K) gv[j] = g4[(size_t)kTileQuads * j + q];
            const float4 pv = p4[q], mv = m4[q], vv = v4[q];
            const float4 e = fold_quad<HAS_ACC, KMAX>(av, gv, K);
            const AdamOut o0 = adam_elem(__fmul_rn(e.x, gscale), pv.x, mv.x, vv.x, c_hi, c_lo, G);
            const AdamOut o1 = adam_elem(__fmul_rn(e.y, gscale), pv.y, mv.y, vv.y, c_hi, c_lo, G);
            const AdamOut o2 = adam_elem(__fmul_rn(e.z, gscale), pv.z, mv.z, vv.z, c_hi, c_lo, G);
            const AdamOut o3 = adam_elem(__fmul_rn(e.w, gscale), pv.w, mv.w, vv.w, c_hi, c_lo, G);
            p4[q] = make_float4(o0.p, o1.p, o2.p, o3.p);
            m4[q] = make_float4(o0.m, o1.m, o2.m, o3.m);
            v4[q] = make_float4(o0.v, o1.v, o2.v, o3.v);
            g4[q] = make_uint2(pack_bf16x2(o0.p, o1.p), pack_bf16x2(o2.p, o3.p));
        }
    }
    __device__ void scalar(const Chunk &ch, const Seg &sg, uint32_t i, uint32_t group) const {
        const uint16_t *g[KA];
#pragma unroll
        for (int j = 0; j < KA; ++j) g[j] = (j < K) ? gt->get(sg.grad_slot, j) + sg.grad_off + ch.start : nullptr;
        float *p = sg.p + ch.start;
        float *m = sg.m + ch.start;
        float *v = sg.v + ch.start;
        const float ev = __fmul_rn(fold_scalar<HAS_ACC, KMAX>(sg.acc + ch.start, g, K, i), gscale);
        const AdamOut o = adam_elem(ev, p[i], m[i], v[i], c_hi, c_lo, gtab[group]);
        p[i] = o.p;
        m[i] = o.m;
        v[i] = o.v;
        sg.bf[ch.start + i] = __bfloat16_as_ushort(__float2bfloat16_rn(o.p));
    }
};

// Fused clip + AdamW + master update + bf16 cast over units [u0, u1), the
// same arithmetic per element as k_step (bit-identical results), with the
// traffic moved by bulk copies (pipe_run): acc, the deferred gradients,
// master, m and v in; master, m, v and the bf16 parameters out, in place.
// One CTA per SM.  The host launches it only when pipe_fits(HAS_ACC, K).
template <bool HAS_ACC, int KMAX, class GT>
__global__ void __launch_bounds__(kPipeThreads, 1)
k_step_pipe(const Seg *__restrict__ segs, const Chunk *__restrict__ chunks, const PipeUnit *__restrict__ units,
            uint32_t u0, uint32_t u1, const __grid_constant__ GT gt, StepState *st,
            const NormState *__restrict__ ns, float gscale, int commit_t, unsigned *queue) {
    extern __shared__ __align__(128) unsigned char pipe_smem[];
    __shared__ PipeShared sh;
    __shared__ GroupK sh_g[kMaxGroups];
    pdl_enter();
    if (st->skip) return;                   // non-finite norm, skipping enabled (no CTA claims a unit)
    if (commit_t && blockIdx.x == 0 && threadIdx.x == 0) st->t += 1;
    for (int i = threadIdx.x; i < kMaxGroups; i += kPipeThreads) sh_g[i] = st->gtab.g[i];
    StepOps<HAS_ACC, KMAX, GT> ops(&gt, sh_g, KMAX <= 1 ? KMAX : (int)gt.k, gscale, ns->c_hi, ns->c_lo);
    pipe_run(ops, segs, chunks, units, u0, u1, queue, pipe_smem, sh);
}

// One gradient added to the accumulator per tile (acc = acc + g), stored back
// (see k_accum_pipe).
template <class GT>
struct AccumOps {
    static constexpr uint32_t kTileQuads = kAccTileQuads;
    static constexpr int stages = kAccStages;
    static constexpr uint32_t stage_bytes = kAccQuadBytes * kAccTileQuads;
    static constexpr uint32_t off_g = 16u * kAccTileQuads;
    const GT *gt;
    const uint16_t *gb;                 // copy thread: the current segment's gradient base

    __device__ explicit AccumOps(const GT *g) : gt(g), gb(nullptr) {}
    __device__ uint32_t tile_bytes(uint32_t nq) const { return nq * kAccQuadBytes; }
    __device__ void set_seg(const Seg &sg) { gb = gt->get(sg.grad_slot, 0) + sg.grad_off; }
    __device__ bool misaligned(const Seg &sg, uint64_t e) const { return mis16(sg.acc + e) || mis16(gb + e); }
    __device__ void load(const Seg &sg, uint64_t e, uint32_t nq, unsigned char *stg, uint64_t *bar,
                         uint64_t pol) const {
        bulk_load(stg, sg.acc + e, 16u * nq, bar, pol);
        bulk_load(stg + off_g, gb + e, 8u * nq, bar, pol);
    }
    __device__ void outputs(const Seg &sg, uint64_t e, void **out) const {
        out[0] = sg.acc + e;
        out[1] = out[2] = out[3] = nullptr;
    }
    __device__ void store(const TileDesc &d, unsigned char *stg, uint64_t pol) const {
        bulk_store(d.out[0], stg, 16u * d.nq, pol);
    }
    __device__ void compute(const TileDesc &d, unsigned char *stg, uint32_t ct) const {
        float4 *a4 = reinterpret_cast<float4 *>(stg);
        const uint2 *g4 = reinterpret_cast<const uint2 *>(stg + off_g);
        for (uint32_t q = ct; q < d.nq; q += kPipeCompute) {
            const uint2 gv = g4[q];
            a4[q] = fold_quad<true, 1>(a4[q], &gv, 1);
        }
    }
    __device__ void scalar(const Chunk &ch, const Seg &sg, uint32_t i, uint32_t) const {
        const uint16_t *g = gt->get(sg.grad_slot, 0) + sg.grad_off + ch.start;
        float *a = sg.acc + ch.start;
        a[i] = fold_scalar<true, 1>(a, &g, 1, i);
    }
};

// An accumulate pass after FIRST that adds one gradient to the accumulator
// and stores it (no norm): the same FP32 add per element as k_accum
// (bit-identical), with the traffic moved by bulk copies (pipe_run).  One CTA
// per SM.
template <class GT>
__global__ void __launch_bounds__(kPipeThreads, 1)
k_accum_pipe(const Seg *__restrict__ segs, const Chunk *__restrict__ chunks, const PipeUnit *__restrict__ units,
             uint32_t u0, uint32_t u1, const __grid_constant__ GT gt, unsigned *queue) {
    extern __shared__ __align__(128) unsigned char pipe_smem[];
    __shared__ PipeShared sh;
    pdl_enter();
    AccumOps<GT> ops(&gt);
    pipe_run(ops, segs, chunks, units, u0, u1, queue, pipe_smem, sh);
}

}  // namespace bf16k

// bf16opt.cu -- host side of the C ABI declared in include/bf16opt.h.
//
// Validates descriptors, builds the segment and chunk tables once on the
// device, keeps the accumulate -> grad_norm -> step sequence on the host and
// launches the kernels of kernels.cuh on the caller's stream (the per-step
// AdamW scalars are computed on the device, from a device step counter).  No
// CPU fallback: every element of the path is computed by those kernels.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <algorithm>
#include <type_traits>
#include <utility>
#include <vector>
#include <mutex>
#include <unordered_set>

#include <cuda.h>   // driver types only (CUcontext, CUresult); no libcuda link
#include <nvtx3/nvToolsExt.h>

#include "../../include/bf16opt.h"
#include "host_adam.h"
#include "kernels.cuh"

using namespace bf16k;

namespace {

enum State { S_IDLE = 0, S_ACC, S_ACC_DONE, S_ACC_DEFERRED, S_LOCAL_NORMED, S_NORMED };

thread_local std::string g_create_error;

// Live handles: every entry point rejects a pointer that bf16opt_create did not
// return or that bf16opt_destroy already freed, instead of dereferencing it.
std::mutex g_live_mu;
std::unordered_set<const void *> g_live;

}  // namespace

struct bf16opt {
    int device = 0;
    int mode = BF16OPT_FLAT;
    uint64_t n = 0;
    uint32_t n_tensors = 0;
    std::vector<Seg> segs;
    uint32_t n_chunks = 0;
    Seg *segs_d = nullptr;
    Chunk *chunks_d = nullptr;
    PipeUnit *units_d = nullptr;         // units of the pipelined step, in chunk order
    std::vector<uint32_t> chunk_unit0;   // first unit of chunk c (n_chunks + 1 entries)
    double *partials_d = nullptr;
    NormState *norm_d = nullptr;
    unsigned *queue_d = nullptr;         // chunk counter of the pass in flight (0 between passes)
    StepParams *params_d = nullptr;      // hyper-parameters + schedule (device)
    StepState *step_d = nullptr;         // device step counter + this step's scalars
    std::vector<bf16opt_group_t> groups;
    float max_norm = 1.0f;
    float gscale = 1.0f;
    State state = S_IDLE;
    bool acc_valid = false;              // acc holds the fold of the micro-batches folded so far
    double local_sumsq = 0.0;            // this partition's sum of squares, as grad_norm_local returned it
    // Deferred micro-batches not yet folded into acc, in micro-batch order:
    // FLAT one pointer each, LIST one pointer per tensor each.
    std::vector<const uint16_t *> pend_flat;
    std::vector<std::vector<const uint16_t *>> pend_list;
    std::vector<uint32_t> slot_chunk0;   // LIST: first chunk of tensor s (n_tensors + 1 entries)
    int sm_count = 0;
    int max_grid = 0;                    // optional cap on CTAs per launch (BF16OPT_MAX_GRID), 0 = none
    std::vector<std::pair<const void *, int>> occ;  // resident CTAs per SM, per kernel (queried once)
    bool has_sched = false;
    bool skip_nonfinite = false;
    bool pdl = true;                     // launch with programmatic stream serialization (BF16OPT_PDL=0: off)
    bool claim = true;                   // CTAs claim chunks from queue_d (BF16OPT_SCHEDULE=static: fixed stride)
    bool pipe = true;                    // step and later accumulates through the bulk-copy pipeline (BF16OPT_PIPE)
    int step_path = BF16OPT_PATH_NONE;   // data path of the last step (bf16opt_step_path)
    bool scalars_ready = false;          // the norm kernel prepared this step's scalars (groups' own lr)
    bf16opt_lr_schedule_t sched{};
    std::string last_error;
    // ZeRO-Offload handle (bf16opt_create_offload): master and moments in host
    // memory, updated by the host cores; the accumulator and the bf16
    // parameters stay on the device.
    bool offload = false;
    float *host_p = nullptr, *host_m = nullptr, *host_v = nullptr;
    float *dev_acc = nullptr;
    uint16_t *dev_bf = nullptr;
    float *stage_acc[2] = {nullptr, nullptr};        // page-locked, one block each
    uint16_t *stage_bf[2] = {nullptr, nullptr};
    StepState *stage_step = nullptr;                 // page-locked copies of the step's scalars
    NormState *stage_norm = nullptr;
    cudaEvent_t ev_d2h[2] = {nullptr, nullptr}, ev_h2d[2] = {nullptr, nullptr};
    bf16host::Pool *pool = nullptr;
};

namespace {

bool live(const bf16opt_t *h) {
    if (!h) return false;
    std::lock_guard<std::mutex> lock(g_live_mu);
    return g_live.count(h) != 0;
}

int fail(bf16opt_t *h, int code, const std::string &msg) {
    if (h) h->last_error = msg;
    else g_create_error = msg;
    return code;
}

int cuda_fail(bf16opt_t *h, cudaError_t e, const char *what) {
    return fail(h, BF16OPT_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Named host range around each API call, seen by profilers that attach through
// NVTX (no-op otherwise).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool finite_f(float x) { return std::isfinite(x); }

int check_group(const bf16opt_group_t &g, uint32_t i, std::string &msg) {
    char buf[160];
    if (!finite_f(g.lr) || g.lr < 0.f) { snprintf(buf, sizeof buf, "group %u: lr must be finite and >= 0", i); msg = buf; return -1; }
    if (!(g.beta1 >= 0.f && g.beta1 < 1.f) || !(g.beta2 >= 0.f && g.beta2 < 1.f)) {
        snprintf(buf, sizeof buf, "group %u: betas must lie in [0, 1)", i); msg = buf; return -1;
    }
    if (!finite_f(g.eps) || !(g.eps > 0.f)) { snprintf(buf, sizeof buf, "group %u: eps must be finite and > 0", i); msg = buf; return -1; }
    if (!finite_f(g.weight_decay) || g.weight_decay < 0.f) {
        snprintf(buf, sizeof buf, "group %u: weight_decay must be finite and >= 0", i); msg = buf; return -1;
    }
    return 0;
}

struct Interval {
    uintptr_t lo, hi;
};

bool overlaps(std::vector<Interval> &iv) {
    std::sort(iv.begin(), iv.end(), [](const Interval &a, const Interval &b) { return a.lo < b.lo; });
    for (size_t i = 1; i < iv.size(); ++i)
        if (iv[i].lo < iv[i - 1].hi) return true;
    return false;
}

// Elements per chunk of a shard of `total` elements: kChunk from 2^25
// elements up; smaller shards get proportionally smaller chunks (a power of
// two, at least kMinChunk) so that they still spread over every SM -- about
// kChunkTarget chunks (a 1M-element shard in 32,768-element chunks kept 32 of
// 152 SMs busy), or about kSmallChunkTarget on shards of at most
// kSmallShard elements, where a pass is one wave of CTAs and a CTA that walks
// several short chunks pays their descriptor loads one after another.
// Depends only on the shard's size, never on the GPU.
#ifndef BF16K_CHUNK_TARGET
#define BF16K_CHUNK_TARGET 1024
#endif
#ifndef BF16K_SMALL_CHUNK_TARGET
#define BF16K_SMALL_CHUNK_TARGET 128
#endif
#ifndef BF16K_SMALL_SHARD
#define BF16K_SMALL_SHARD (uint64_t(1) << 22)
#endif
constexpr uint32_t kMinChunk = 2048;
static_assert(kMinChunk % kHeadAlign == 0 && kMinChunk <= kChunk, "chunk sizes are multiples of kHeadAlign");
uint32_t chunk_elems(uint64_t total) {
    const uint64_t target = total <= BF16K_SMALL_SHARD ? BF16K_SMALL_CHUNK_TARGET : BF16K_CHUNK_TARGET;
    uint64_t c = kMinChunk;
    while (c < kChunk && c * target < total) c <<= 1;
    return (uint32_t)c;
}

// Elements by which the first chunk over an FP32 buffer starting at `p` is
// shorter than the others: p's element index modulo kHeadAlign.
uint32_t first_chunk_cut(const void *p) { return (uint32_t)(((uintptr_t)p >> 2) & (kHeadAlign - 1)); }

bool mis4(const void *p) { return ((uintptr_t)p & 3u) != 0; }
bool mis2(const void *p) { return ((uintptr_t)p & 1u) != 0; }

unsigned long long current_ctx_id();   // below, with the allocation-free norm

// A function attribute set once per kernel, device and context (kernels of
// one template share a function type, so the kernel's address is the key; a
// context that replaced a reset one has the module loaded afresh, without
// the attribute, and a new id).  Set on every call when the context's id
// cannot be read.
template <class K>
cudaError_t kernel_attr_once(K kernel, int dev, cudaFuncAttribute attr, int value) {
    struct Done {
        const void *kernel;
        int dev, attr;
        unsigned long long ctx;
    };
    static std::mutex mu;
    static std::vector<Done> done;
    const void *key = reinterpret_cast<const void *>(kernel);
    const unsigned long long ctx = current_ctx_id();
    std::lock_guard<std::mutex> lock(mu);
    if (ctx != 0)
        for (const Done &d : done)
            if (d.kernel == key && d.dev == dev && d.attr == (int)attr && d.ctx == ctx) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, attr, value);
    if (e == cudaSuccess && ctx != 0) done.push_back({key, dev, (int)attr, ctx});
    return e;
}

// Shared-memory carveout of the streaming kernels: the least shared memory,
// the most L1.  Without the preference a kernel that fits the shared-memory
// configuration the step's copy pipeline left behind runs in it, with a small
// L1 -- where its loads in flight are staged -- and the accumulate passes ran
// 1.4 % slower.
#ifndef BF16K_STREAM_CARVEOUT
#define BF16K_STREAM_CARVEOUT 0
#endif

template <class K>
int grid_for(bf16opt_t *h, K kernel, uint32_t nchunks, int threads = kThreads) {
    int per_sm = 0;
    const void *key = reinterpret_cast<const void *>(kernel);
    for (const auto &e : h->occ)
        if (e.first == key) per_sm = e.second;
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm < 1) {
            cudaGetLastError();
            per_sm = 1;
        }
        h->occ.emplace_back(key, per_sm);
    }
    if (per_sm > BF16K_MAX_CTAS_PER_SM) per_sm = BF16K_MAX_CTAS_PER_SM;
    uint64_t g = (uint64_t)h->sm_count * (uint64_t)per_sm;
    if (h->max_grid > 0 && g > (uint64_t)h->max_grid) g = (uint64_t)h->max_grid;
    return (int)std::max<uint64_t>(1, std::min<uint64_t>(g, nchunks));
}

// Launches `kernel` on `st`, with programmatic stream serialization unless
// the handle has it switched off: the kernel may then be scheduled while its
// predecessor drains, and waits on the device (griddepcontrol.wait) before
// its first memory access -- see pdl_enter in kernels.cuh.
template <class... KArgs, class... Args>
cudaError_t launch_smem(const bf16opt_t *h, void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                        cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = h->pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
template <class... KArgs, class... Args>
cudaError_t launch(const bf16opt_t *h, void (*kernel)(KArgs...), unsigned grid, unsigned block, cudaStream_t st,
                   Args &&...args) {
    return launch_smem(h, kernel, grid, block, 0, st, std::forward<Args>(args)...);
}

// Gradients a pass folds: K micro-batches (FLAT: one pointer each; LIST: one
// per tensor each), in micro-batch order.
struct FoldSet {
    std::vector<const uint16_t *> flat;
    std::vector<const std::vector<const uint16_t *> *> list;
    size_t count() const { return flat.size() > list.size() ? flat.size() : list.size(); }
};

inline int kmax_for(size_t K) { return K <= 1 ? (int)K : (K <= 4 ? 4 : 8); }

// Visit every launch of a pass: FLAT one launch over all chunks; LIST launches
// of consecutive tensors such that K gradient pointers per tensor fit the
// kernel parameter table.
template <class F>
int for_each_launch(bf16opt_t *h, const FoldSet &fs, F &&launch) {
    const size_t K = fs.count();
    if (K > (size_t)kMaxFold) return fail(h, BF16OPT_ERR_INVALID_ARG, "internal: more gradients than one pass folds");
    if (h->n_chunks == 0) return 0;
    if (h->mode == BF16OPT_FLAT) {
        FlatGrads gt;
        memset(&gt, 0, sizeof gt);
        gt.k = (uint32_t)K;
        for (size_t j = 0; j < K; ++j) gt.base[j] = fs.flat[j];
        launch(gt, 0u, h->n_chunks);
    } else {
        const uint32_t per = (uint32_t)(kListSlots / (K ? K : 1));
        for (uint32_t s0 = 0; s0 < h->n_tensors; s0 += per) {
            const uint32_t s1 = std::min<uint32_t>(h->n_tensors, s0 + per);
            const uint32_t c0 = h->slot_chunk0[s0], c1 = h->slot_chunk0[s1];
            if (c1 == c0) continue;
            ListGrads gt;
            gt.slot_base = s0;
            gt.nslots = s1 - s0;
            gt.k = (uint32_t)K;
            gt.pad = 0;
            for (size_t j = 0; j < K; ++j)
                for (uint32_t i = 0; i < s1 - s0; ++i) gt.ptr[j * (s1 - s0) + i] = (*fs.list[j])[s0 + i];
            launch(gt, c0, c1);
        }
    }
    return 0;
}

// Grid of a pipelined pass: one CTA per SM (its stages fill the SM's shared
// memory), no more CTAs than units, within the BF16OPT_MAX_GRID cap.
unsigned pipe_grid(const bf16opt_t *h, uint64_t units) {
    uint64_t g = std::min<uint64_t>((uint64_t)h->sm_count, units);
    if (h->max_grid > 0 && g > (uint64_t)h->max_grid) g = (uint64_t)h->max_grid;
    return (unsigned)std::max<uint64_t>(1, g);
}

// The bulk-copy passes need every stream of a chunk's body 16-byte aligned at
// one element: per segment, the FP32 pointers (master, m, v, the accumulator
// if used) share their element index modulo 4, the bf16 ones (parameters,
// folded gradients) share theirs modulo 8, and the two agree modulo 4.  (The
// units' bodies start where the bf16 parameters are 16-byte aligned.)
bool pipe_aligned(const bf16opt_t *h, const FoldSet &fs, bool has_acc) {
    const size_t K = fs.count();
    for (const Seg &s : h->segs) {
        if (s.numel == 0) continue;
        const uint32_t f = (uint32_t)(((uintptr_t)s.p >> 2) & 3u);
        const uint32_t b = (uint32_t)(((uintptr_t)s.bf >> 1) & 7u);
        if ((b & 3u) != f) return false;
        for (const float *x : {s.m, s.v})
            if ((uint32_t)(((uintptr_t)x >> 2) & 3u) != f) return false;
        if (has_acc && (uint32_t)(((uintptr_t)s.acc >> 2) & 3u) != f) return false;
        for (size_t j = 0; j < K; ++j) {
            const uint16_t *g = (h->mode == BF16OPT_FLAT ? fs.flat[j] : (*fs.list[j])[s.grad_slot]) + s.grad_off;
            if ((uint32_t)(((uintptr_t)g >> 1) & 7u) != b) return false;
        }
    }
    return true;
}

template <bool HAS_ACC, int KMAX, bool WRITE, bool NORM>
int launch_accum_k(bf16opt_t *h, const FoldSet &fs, cudaStream_t st) {
    constexpr int U = KMAX <= 1 ? BF16K_ACC_U : (KMAX <= 4 ? BF16K_FOLD4_ACC_U : BF16K_FOLD8_ACC_U);
    cudaError_t e = cudaSuccess;
    // A pass that adds one gradient to the stored accumulator and stores it
    // takes the bulk-copy pipeline where the fused step does (the pipeline's
    // size rule, buffers aligned alike): on the 1.72B shard 2.398 against
    // 2.443 ms.  The FIRST pass (no accumulator read) was slower through it
    // (1.560 against 1.499 ms); passes with the norm or several gradients keep
    // vector loads too.
    const bool pipe = HAS_ACC && KMAX == 1 && WRITE && !NORM && h->pipe && pipe_aligned(h, fs, true);
    int rc = for_each_launch(h, fs, [&](const auto &gt, uint32_t c0, uint32_t c1) {
        using GT = std::decay_t<decltype(gt)>;
        if constexpr (HAS_ACC && KMAX == 1 && WRITE && !NORM) {
            if (pipe) {
                auto kp = k_accum_pipe<GT>;
                constexpr size_t smem = (size_t)kAccStages * kAccQuadBytes * kAccTileQuads;
                cudaError_t e1 = kernel_attr_once(kp, h->device, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  (int)smem);
                const uint32_t u0 = h->chunk_unit0[c0], u1 = h->chunk_unit0[c1];
                if (e1 == cudaSuccess)
                    e1 = launch_smem(h, kp, pipe_grid(h, u1 - u0), kPipeThreads, smem, st,
                                     (const Seg *)h->segs_d, (const Chunk *)h->chunks_d,
                                     (const PipeUnit *)h->units_d, u0, u1, gt, h->claim ? h->queue_d : nullptr);
                if (e == cudaSuccess) e = e1;
                return;
            }
        }
        auto k = k_accum<HAS_ACC, KMAX, WRITE, NORM, GT, U>;
#if BF16K_STREAM_CARVEOUT >= 0
        if (kernel_attr_once(k, h->device, cudaFuncAttributePreferredSharedMemoryCarveout, BF16K_STREAM_CARVEOUT) !=
            cudaSuccess)
            cudaGetLastError();   // a hint: the pass runs without it
#endif
        const cudaError_t e1 = launch(h, k, grid_for(h, k, c1 - c0), kThreads, st, (const Seg *)h->segs_d,
                                      (const Chunk *)h->chunks_d, c0, c1, gt, h->partials_d, h->gscale,
                                      h->claim ? h->queue_d : nullptr);
        if (e == cudaSuccess) e = e1;
    });
    if (rc) return rc;
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? 0 : cuda_fail(h, e, "accumulate kernel launch");
}

// fold(acc?, fs) -> (acc if WRITE) and (norm partials if NORM).
template <bool WRITE, bool NORM>
int launch_accum(bf16opt_t *h, bool has_acc, const FoldSet &fs, cudaStream_t st) {
    switch (kmax_for(fs.count())) {
    case 0: return fail(h, BF16OPT_ERR_INVALID_ARG, "internal: an accumulate pass without a gradient");
    case 1: return has_acc ? launch_accum_k<true, 1, WRITE, NORM>(h, fs, st) : launch_accum_k<false, 1, WRITE, NORM>(h, fs, st);
    case 4: return has_acc ? launch_accum_k<true, 4, WRITE, NORM>(h, fs, st) : launch_accum_k<false, 4, WRITE, NORM>(h, fs, st);
    default: return has_acc ? launch_accum_k<true, 8, WRITE, NORM>(h, fs, st) : launch_accum_k<false, 8, WRITE, NORM>(h, fs, st);
    }
}

constexpr uint64_t kStepClaimChunksPerCta = 64;



// commit_t: the first launch advances the device step counter (the step's
// scalars were prepared by the norm kernel; otherwise k_step_scalars did both).
template <bool HAS_ACC, int KMAX>
int launch_step_k(bf16opt_t *h, const FoldSet &fs, cudaStream_t st, bool commit_t) {
    constexpr int U = KMAX <= 1 ? BF16K_STEP_U : (KMAX <= 4 ? BF16K_FOLD4_STEP_U : BF16K_FOLD8_STEP_U);
    cudaError_t e = cudaSuccess;
    bool first = true;
    const int K = (int)fs.count();
    const bool pipe = KMAX <= 4 && h->pipe && pipe_fits(HAS_ACC, K) && pipe_aligned(h, fs, HAS_ACC);
    h->step_path = h->n_chunks == 0 ? BF16OPT_PATH_NONE : (pipe ? BF16OPT_PATH_PIPELINE : BF16OPT_PATH_VECTOR);
    int rc = for_each_launch(h, fs, [&](const auto &gt, uint32_t c0, uint32_t c1) {
        using GT = std::decay_t<decltype(gt)>;
        if constexpr (KMAX <= 4) {
          if (pipe) {
            auto kp = k_step_pipe<HAS_ACC, KMAX, GT>;
            const size_t smem = (size_t)pipe_stages(HAS_ACC, K) * pipe_quad_bytes(HAS_ACC, K) * kPipeTileQuads;
            cudaError_t e1 = kernel_attr_once(kp, h->device, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)kPipeSmem);   // the most any K of the variant takes
            const uint32_t u0 = h->chunk_unit0[c0], u1 = h->chunk_unit0[c1];
            if (e1 == cudaSuccess)
                e1 = launch_smem(h, kp, pipe_grid(h, u1 - u0), kPipeThreads, smem, st,
                                 (const Seg *)h->segs_d, (const Chunk *)h->chunks_d, (const PipeUnit *)h->units_d,
                                 u0, u1, gt, h->step_d, (const NormState *)h->norm_d, h->gscale,
                                 (commit_t && first) ? 1 : 0, h->claim ? h->queue_d : nullptr);
            first = false;
            if (e == cudaSuccess) e = e1;
            return;
          }
        }
        auto k = k_step<HAS_ACC, KMAX, GT, U>;
        const int grid = grid_for(h, k, c1 - c0, kStepThreads);
        // one CTA per SM: claiming pays once every CTA has many chunks to go
        // through (on a 134M-element shard, 27 per CTA, it cost 3 %)
        const bool claim = h->claim && (uint64_t)(c1 - c0) >= kStepClaimChunksPerCta * (uint64_t)grid;
        const cudaError_t e1 = launch(h, k, grid, kStepThreads, st, (const Seg *)h->segs_d,
                                      (const Chunk *)h->chunks_d, c0, c1, gt, h->step_d,
                                      (const NormState *)h->norm_d, h->gscale, (commit_t && first) ? 1 : 0,
                                      claim ? h->queue_d : nullptr);
        first = false;
        if (e == cudaSuccess) e = e1;
    });
    if (rc) return rc;
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? 0 : cuda_fail(h, e, "step kernel launch");
}

int launch_step(bf16opt_t *h, bool has_acc, const FoldSet &fs, cudaStream_t st, bool commit_t) {
    switch (kmax_for(fs.count())) {
    case 0: return launch_step_k<true, 0>(h, fs, st, commit_t);
    case 1: return has_acc ? launch_step_k<true, 1>(h, fs, st, commit_t) : launch_step_k<false, 1>(h, fs, st, commit_t);
    case 4: return has_acc ? launch_step_k<true, 4>(h, fs, st, commit_t) : launch_step_k<false, 4>(h, fs, st, commit_t);
    default: return has_acc ? launch_step_k<true, 8>(h, fs, st, commit_t) : launch_step_k<false, 8>(h, fs, st, commit_t);
    }
}

FoldSet pending_set(const bf16opt_t *h) {
    FoldSet fs;
    fs.flat = h->pend_flat;
    for (const auto &v : h->pend_list) fs.list.push_back(&v);
    return fs;
}

void free_offload(bf16opt_t *h) {
    for (int i = 0; i < 2; ++i) {
        if (h->stage_acc[i]) cudaFreeHost(h->stage_acc[i]);
        if (h->stage_bf[i]) cudaFreeHost(h->stage_bf[i]);
        if (h->ev_d2h[i]) cudaEventDestroy(h->ev_d2h[i]);
        if (h->ev_h2d[i]) cudaEventDestroy(h->ev_h2d[i]);
        h->stage_acc[i] = nullptr;
        h->stage_bf[i] = nullptr;
        h->ev_d2h[i] = h->ev_h2d[i] = nullptr;
    }
    if (h->stage_step) cudaFreeHost(h->stage_step);
    if (h->stage_norm) cudaFreeHost(h->stage_norm);
    h->stage_step = nullptr;
    h->stage_norm = nullptr;
    delete h->pool;
    h->pool = nullptr;
}

void free_scratch(bf16opt_t *h) {
    free_offload(h);
    if (h->segs_d) cudaFree(h->segs_d);
    if (h->chunks_d) cudaFree(h->chunks_d);
    if (h->units_d) cudaFree(h->units_d);
    h->units_d = nullptr;
    if (h->partials_d) cudaFree(h->partials_d);
    if (h->norm_d) cudaFree(h->norm_d);
    if (h->queue_d) cudaFree(h->queue_d);
    h->queue_d = nullptr;
    if (h->params_d) cudaFree(h->params_d);
    if (h->step_d) cudaFree(h->step_d);
    h->params_d = nullptr;
    h->step_d = nullptr;
    h->segs_d = nullptr;
    h->chunks_d = nullptr;
    h->partials_d = nullptr;
    h->norm_d = nullptr;
}

// The calls that read or write the device step state or hyper-parameters with
// a plain copy first wait for all work on the handle's device: a step still in
// flight on a non-blocking stream (which the legacy stream of cudaMemcpy does
// not wait for) is then ordered before them.  Not allowed during a capture.
cudaError_t quiesce() { return cudaDeviceSynchronize(); }

// Hyper-parameters and schedule -> device (synchronous; not during a capture).
cudaError_t upload_params(bf16opt_t *h) {
    StepParams p;
    memset(&p, 0, sizeof p);
    p.n_groups = (int32_t)h->groups.size();
    for (size_t i = 0; i < h->groups.size(); ++i) {
        p.lr[i] = h->groups[i].lr;
        p.beta1[i] = h->groups[i].beta1;
        p.beta2[i] = h->groups[i].beta2;
        p.eps[i] = h->groups[i].eps;
        p.wd[i] = h->groups[i].weight_decay;
    }
    p.has_sched = h->has_sched ? 1 : 0;
    p.warmup = h->sched.warmup_steps;
    p.decay = h->sched.decay_steps;
    p.min_ratio = h->sched.min_lr_ratio;
    p.skip_nonfinite = h->skip_nonfinite ? 1 : 0;
    return cudaMemcpy(h->params_d, &p, sizeof p, cudaMemcpyHostToDevice);
}

// Elements per block of the offloaded step's pipeline: the accumulator of
// block k + 1 is copied to the host while the host cores update block k, and
// the bf16 parameters of block k go back to the device while block k + 1 is
// updated.  2^24 elements: 64 MiB + 32 MiB of page-locked staging per buffer.
constexpr uint64_t kOffloadBlock = uint64_t(1) << 24;

// The step of an offload handle: the scalars, the step counter and the skip
// decision come from the same device kernel as the device step; the update
// itself runs on the host over the host-resident master and moments.
int offload_step(bf16opt_t *h, const LrOverride &ov, cudaStream_t st) {
    if (!h->pend_flat.empty()) {      // fold micro-batches still deferred: the host reads a complete accumulator
        int rc = launch_accum<true, false>(h, h->acc_valid, pending_set(h), st);
        if (rc) return rc;
        h->acc_valid = true;
        h->pend_flat.clear();
    }
    cudaError_t e = launch(h, k_step_scalars, 1, 32, st, (const StepParams *)h->params_d, h->step_d, ov,
                           (const NormState *)h->norm_d);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->stage_step, h->step_d, sizeof(StepState), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->stage_norm, h->norm_d, sizeof(NormState), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(h, e, "offloaded step: step scalars");
    if (h->stage_step->skip) return BF16OPT_OK;        // non-finite norm, skipping enabled
    const float c_hi = h->stage_norm->c_hi, c_lo = h->stage_norm->c_lo;
    bf16host::HostGroup G[kMaxGroups];
    for (size_t g = 0; g < h->groups.size(); ++g) {
        const GroupK &k = h->stage_step->gtab.g[g];
        G[g] = {k.b1, k.omb1, k.b2, k.omb2, k.eps, k.decay, k.step_size, k.inv_sqrt_bc2};
    }
    const uint64_t n = h->n, nb = (n + kOffloadBlock - 1) / kOffloadBlock;
    auto fetch = [&](uint64_t k) {
        const uint64_t lo = k * kOffloadBlock, len = std::min(kOffloadBlock, n - lo);
        cudaError_t r = cudaMemcpyAsync(h->stage_acc[k & 1], h->dev_acc + lo, len * sizeof(float),
                                        cudaMemcpyDeviceToHost, st);
        return r == cudaSuccess ? cudaEventRecord(h->ev_d2h[k & 1], st) : r;
    };
    if (nb > 0 && (e = fetch(0)) != cudaSuccess) return cuda_fail(h, e, "offloaded step: copy to host");
    for (uint64_t k = 0; k < nb; ++k) {
        const uint64_t lo = k * kOffloadBlock, len = std::min(kOffloadBlock, n - lo);
        if (k + 1 < nb && (e = fetch(k + 1)) != cudaSuccess) return cuda_fail(h, e, "offloaded step: copy to host");
        // this block's gradient has arrived; its bf16 staging buffer (two blocks
        // ago, or the previous step) has been copied out
        if ((e = cudaEventSynchronize(h->ev_d2h[k & 1])) != cudaSuccess ||
            (e = cudaEventSynchronize(h->ev_h2d[k & 1])) != cudaSuccess)
            return cuda_fail(h, e, "offloaded step: waiting for a copy");
        const float *acc = h->stage_acc[k & 1];
        uint16_t *bf = h->stage_bf[k & 1];
        h->pool->run([&](int w, int nw) {
            const uint64_t a = lo + len * (uint64_t)w / (uint64_t)nw, b = lo + len * (uint64_t)(w + 1) / (uint64_t)nw;
            for (const Seg &sg : h->segs) {
                const uint64_t s0 = std::max(a, sg.grad_off), s1 = std::min(b, sg.grad_off + sg.numel);
                if (s0 < s1)
                    bf16host::adam_range(acc + (s0 - lo), h->host_p + s0, h->host_m + s0, h->host_v + s0,
                                         bf + (s0 - lo), s1 - s0, h->gscale, c_hi, c_lo, G[sg.group]);
            }
        });
        if ((e = cudaMemcpyAsync(h->dev_bf + lo, bf, len * sizeof(uint16_t), cudaMemcpyHostToDevice, st)) != cudaSuccess ||
            (e = cudaEventRecord(h->ev_h2d[k & 1], st)) != cudaSuccess)
            return cuda_fail(h, e, "offloaded step: copy to device");
    }
    return BF16OPT_OK;
}

// cudaPointerGetAttributes' kind of p; cudaMemoryTypeUnregistered when it fails.
cudaMemoryType memory_kind(const void *p, int *device) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return cudaMemoryTypeUnregistered;
    }
    if (device) *device = a.device;
    return a.type;
}

}  // namespace

extern "C" {

int bf16opt_abi_version(void) { return BF16OPT_ABI_VERSION; }

const char *bf16opt_error_string(int code) {
    switch (code) {
    case BF16OPT_OK: return "ok";
    case BF16OPT_WARN_NONFINITE: return "gradient norm is not finite";
    case BF16OPT_ERR_INVALID_ARG: return "invalid argument";
    case BF16OPT_ERR_ALIGNMENT: return "misaligned pointer";
    case BF16OPT_ERR_SEQUENCE: return "call out of sequence (accumulate FIRST..LAST -> grad_norm -> step)";
    case BF16OPT_ERR_OOM: return "out of device memory";
    case BF16OPT_ERR_CUDA: return "CUDA error";
    case BF16OPT_ERR_UNSUPPORTED: return "unsupported (no usable CUDA device)";
    default: return "unknown status";
    }
}

const char *bf16opt_last_error(const bf16opt_t *h) {
    if (!h) return g_create_error.c_str();
    return live(h) ? h->last_error.c_str() : "not a live bf16opt handle (never created, or destroyed)";
}

int bf16opt_create(const bf16opt_desc_t *d, bf16opt_t **out) {
    NvtxRange nvtx("bf16opt_create");
    if (out) *out = nullptr;
    if (!d || !out) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "desc and out must be non-NULL");
    if (d->mode != BF16OPT_FLAT && d->mode != BF16OPT_LIST)
        return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "mode must be BF16OPT_FLAT or BF16OPT_LIST");
    if (d->n_groups < 1 || d->n_groups > (uint32_t)kMaxGroups || !d->groups)
        return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "n_groups must be in [1, 16] with a groups array");
    std::string msg;
    for (uint32_t i = 0; i < d->n_groups; ++i)
        if (check_group(d->groups[i], i, msg)) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, msg);
    if (!finite_f(d->max_grad_norm)) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "max_grad_norm must be finite");
    if (!finite_f(d->grad_scale) || d->grad_scale == 0.f)
        return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "grad_scale must be finite and non-zero");

    std::vector<Seg> segs;
    std::vector<Interval> iv;
    if (d->mode == BF16OPT_FLAT) {
        const uint64_t n = d->n;
        if (n > 0) {
            if (!d->master || !d->exp_avg || !d->exp_avg_sq || !d->grad_accum || !d->param_bf16)
                return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "FLAT: all five buffers must be non-NULL");
            if (mis4(d->master) || mis4(d->exp_avg) || mis4(d->exp_avg_sq) || mis4(d->grad_accum) || mis2(d->param_bf16))
                return fail(nullptr, BF16OPT_ERR_ALIGNMENT, "FLAT: FP32 buffers need 4-B and bf16 2-B alignment");
            if (n > (UINT64_MAX / 8)) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "FLAT: n too large");
            iv.push_back({(uintptr_t)d->master, (uintptr_t)d->master + 4 * n});
            iv.push_back({(uintptr_t)d->exp_avg, (uintptr_t)d->exp_avg + 4 * n});
            iv.push_back({(uintptr_t)d->exp_avg_sq, (uintptr_t)d->exp_avg_sq + 4 * n});
            iv.push_back({(uintptr_t)d->grad_accum, (uintptr_t)d->grad_accum + 4 * n});
            iv.push_back({(uintptr_t)d->param_bf16, (uintptr_t)d->param_bf16 + 2 * n});
        }
        std::vector<bf16opt_range_t> ranges;
        if (d->n_ranges == 0 || !d->ranges) {
            if (d->n_ranges != 0) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "FLAT: n_ranges > 0 with NULL ranges");
            ranges.push_back({0, n, 0, 0});
        } else {
            ranges.assign(d->ranges, d->ranges + d->n_ranges);
        }
        uint64_t expect = 0;
        for (size_t i = 0; i < ranges.size(); ++i) {
            const bf16opt_range_t &r = ranges[i];
            if (r.begin != expect || r.end < r.begin || r.end > n || r.group >= d->n_groups || r.reserved != 0)
                return fail(nullptr, BF16OPT_ERR_INVALID_ARG,
                            "FLAT: ranges must tile [0, n) in order with valid groups (range " + std::to_string(i) + ")");
            expect = r.end;
            if (r.end > r.begin) {
                Seg s;
                s.acc = d->grad_accum + r.begin;
                s.p = d->master + r.begin;
                s.m = d->exp_avg + r.begin;
                s.v = d->exp_avg_sq + r.begin;
                s.bf = d->param_bf16 + r.begin;
                s.numel = r.end - r.begin;
                s.grad_off = r.begin;
                s.grad_slot = 0;
                s.group = r.group;
                segs.push_back(s);
            }
        }
        if (expect != n) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "FLAT: ranges do not cover [0, n)");
    } else {
        if (d->n_tensors > 0 && !d->tensors) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "LIST: tensors is NULL");
        for (uint32_t i = 0; i < d->n_tensors; ++i) {
            const bf16opt_tensor_t &t = d->tensors[i];
            const std::string at = "LIST: tensor " + std::to_string(i);
            if (t.group >= d->n_groups || t.reserved != 0) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, at + ": bad group");
            if (t.numel == 0) continue;
            if (t.numel > (UINT64_MAX / 8)) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, at + ": numel too large");
            if (!t.master || !t.exp_avg || !t.exp_avg_sq || !t.grad_accum || !t.param_bf16)
                return fail(nullptr, BF16OPT_ERR_INVALID_ARG, at + ": NULL buffer");
            if (mis4(t.master) || mis4(t.exp_avg) || mis4(t.exp_avg_sq) || mis4(t.grad_accum) || mis2(t.param_bf16))
                return fail(nullptr, BF16OPT_ERR_ALIGNMENT, at + ": FP32 buffers need 4-B and bf16 2-B alignment");
            iv.push_back({(uintptr_t)t.master, (uintptr_t)t.master + 4 * t.numel});
            iv.push_back({(uintptr_t)t.exp_avg, (uintptr_t)t.exp_avg + 4 * t.numel});
            iv.push_back({(uintptr_t)t.exp_avg_sq, (uintptr_t)t.exp_avg_sq + 4 * t.numel});
            iv.push_back({(uintptr_t)t.grad_accum, (uintptr_t)t.grad_accum + 4 * t.numel});
            iv.push_back({(uintptr_t)t.param_bf16, (uintptr_t)t.param_bf16 + 2 * t.numel});
            Seg s;
            s.acc = t.grad_accum;
            s.p = t.master;
            s.m = t.exp_avg;
            s.v = t.exp_avg_sq;
            s.bf = t.param_bf16;
            s.numel = t.numel;
            s.grad_off = 0;
            s.grad_slot = i;
            s.group = t.group;
            segs.push_back(s);
        }
    }
    if (overlaps(iv)) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "state buffers overlap");

    // Chunk table: every segment cut into chunks of at most `chunk` elements, in
    // segment order.  The first chunk of a segment is shortened by the
    // accumulator's element offset from a kHeadAlign boundary, so that every
    // later chunk starts on such a boundary: those chunks need no scalar head,
    // and no 128-byte line of the (equally offset) buffers is split between two
    // chunks.  The accumulator is the buffer every norm pass streams, so the
    // norm's chunking -- and its bits -- depend on it alone: an offload handle
    // (master in host memory) and a device handle over accumulators with the
    // same offset reduce the same chunks, as does bf16opt_grad_norm_static.
    uint64_t total = 0;
    for (const Seg &s : segs) total += s.numel;
    const uint32_t chunk = chunk_elems(total);
    std::vector<Chunk> chunks;
    for (uint32_t si = 0; si < segs.size(); ++si) {
        const Seg &s = segs[si];
        const uint64_t first = chunk - first_chunk_cut(s.acc);
        for (uint64_t off = 0; off < s.numel;) {
            if (chunks.size() >= 0xffffffffull) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "too many chunks");
            const uint64_t len = std::min<uint64_t>(off == 0 ? first : chunk, s.numel - off);
            chunks.push_back({off, si, (uint32_t)len});
            off += len;
        }
    }
    // LIST: first chunk of every tensor (empty tensors point at the next one's).
    std::vector<uint32_t> slot_chunk0;
    if (d->mode == BF16OPT_LIST) {
        slot_chunk0.assign(d->n_tensors + 1, (uint32_t)chunks.size());
        for (uint32_t c = (uint32_t)chunks.size(); c-- > 0;) slot_chunk0[segs[chunks[c].seg].grad_slot] = c;
        for (uint32_t s = d->n_tensors; s-- > 0;)
            if (slot_chunk0[s] > slot_chunk0[s + 1]) slot_chunk0[s] = slot_chunk0[s + 1];
    }

    // Units of the pipelined step: each chunk's body -- from its first element
    // at which the bf16 parameters are 16-byte aligned, a multiple of 8
    // elements -- cut into runs of kPipeUnitQuads quads, in chunk order.
    std::vector<PipeUnit> units;
    std::vector<uint32_t> chunk_unit0(chunks.size() + 1, 0);
    for (uint32_t c = 0; c < chunks.size(); ++c) {
        if (units.size() >= 0xffffffffull) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "too many step units");
        chunk_unit0[c] = (uint32_t)units.size();
        const Chunk &ch = chunks[c];
        const Seg &sg = segs[ch.seg];
        const uint32_t hb = pipe_head(sg.bf + ch.start, ch.len);
        const uint32_t nqb = ((ch.len - hb) >> 3) << 1;
        const uint32_t scal = (hb != 0 || hb + 4u * nqb != ch.len) ? 1u : 0u;
        uint32_t q = 0;
        do {
            const uint32_t nq = std::min(kPipeUnitQuads, nqb - q);
            units.push_back({ch.start + hb + 4ull * q, ch.seg, c, nq, q == 0 ? scal : 0u});
            q += kPipeUnitQuads;
        } while (q < nqb);
    }
    chunk_unit0[chunks.size()] = (uint32_t)units.size();

    // Device and scratch.
    int dev = 0, ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev < 1) {
        cudaGetLastError();
        return fail(nullptr, BF16OPT_ERR_UNSUPPORTED, "no CUDA device");
    }
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(nullptr, BF16OPT_ERR_UNSUPPORTED, "cudaGetDevice failed");

    bf16opt_t *h = new (std::nothrow) bf16opt_t();
    if (!h) return fail(nullptr, BF16OPT_ERR_OOM, "host allocation failed");
    h->device = dev;
    h->mode = d->mode;
    h->n = d->mode == BF16OPT_FLAT ? d->n : 0;
    h->n_tensors = d->mode == BF16OPT_LIST ? d->n_tensors : 0;
    h->segs = segs;
    h->slot_chunk0 = slot_chunk0;
    h->chunk_unit0 = chunk_unit0;
    h->n_chunks = (uint32_t)chunks.size();
    h->groups.assign(d->groups, d->groups + d->n_groups);
    h->max_norm = d->max_grad_norm;
    h->gscale = d->grad_scale;
    if (cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || h->sm_count < 1)
        h->sm_count = 1;
    // Optional cap on the CTAs of every launch (testing that results do not
    // depend on the grid: the norm's partials are per chunk, not per CTA).
    if (const char *mg = std::getenv("BF16OPT_MAX_GRID")) h->max_grid = std::max(0, std::atoi(mg));
    // Programmatic dependent launch is on unless BF16OPT_PDL=0 (to compare).
    if (const char *pd = std::getenv("BF16OPT_PDL")) h->pdl = std::atoi(pd) != 0;
    // Chunks are claimed from a counter on shards of full-size chunks (from 2^25
    // elements): there a CTA works through tens to hundreds of chunks and the
    // balance pays; a smaller shard gives each CTA one to a few short chunks,
    // where the claim's round trip would cost more than it balances.
    // BF16OPT_SCHEDULE=static / claim overrides (to compare).
    h->claim = total >= (uint64_t(1) << 25);
    if (const char *sc = std::getenv("BF16OPT_SCHEDULE")) h->claim = std::strcmp(sc, "static") != 0;
    // The fused step and the accumulate passes after FIRST move their traffic
    // with bulk copies on shards of 2^25 elements and more (they also need
    // buffers aligned alike, see pipe_aligned); on a 1M-element shard the
    // pipeline's fill cost more than it gained (step 12.4 vs 10.4 us).
    // BF16OPT_PIPE=1 / 0 overrides (to test and compare).
    h->pipe = total >= (uint64_t(1) << 25);
    if (const char *sp = std::getenv("BF16OPT_PIPE")) h->pipe = std::atoi(sp) != 0;

    cudaError_t e = cudaSuccess;
    const size_t nseg = std::max<size_t>(1, segs.size()), nch = std::max<size_t>(1, chunks.size());
    if ((e = cudaMalloc(&h->segs_d, nseg * sizeof(Seg))) != cudaSuccess ||
        (e = cudaMalloc(&h->chunks_d, nch * sizeof(Chunk))) != cudaSuccess ||
        (e = cudaMalloc(&h->units_d, std::max<size_t>(1, units.size()) * sizeof(PipeUnit))) != cudaSuccess ||
        (e = cudaMalloc(&h->partials_d, nch * sizeof(double))) != cudaSuccess ||
        (e = cudaMalloc(&h->norm_d, sizeof(NormState))) != cudaSuccess ||
        (e = cudaMalloc(&h->queue_d, sizeof(unsigned))) != cudaSuccess ||
        (e = cudaMalloc(&h->params_d, sizeof(StepParams))) != cudaSuccess ||
        (e = cudaMalloc(&h->step_d, sizeof(StepState))) != cudaSuccess) {
        free_scratch(h);
        delete h;
        cudaGetLastError();
        return fail(nullptr, e == cudaErrorMemoryAllocation ? BF16OPT_ERR_OOM : BF16OPT_ERR_CUDA,
                    std::string("scratch allocation: ") + cudaGetErrorString(e));
    }
    if ((!segs.empty() && (e = cudaMemcpy(h->segs_d, segs.data(), segs.size() * sizeof(Seg), cudaMemcpyHostToDevice)) != cudaSuccess) ||
        (!chunks.empty() && (e = cudaMemcpy(h->chunks_d, chunks.data(), chunks.size() * sizeof(Chunk), cudaMemcpyHostToDevice)) != cudaSuccess) ||
        (!units.empty() && (e = cudaMemcpy(h->units_d, units.data(), units.size() * sizeof(PipeUnit), cudaMemcpyHostToDevice)) != cudaSuccess) ||
        (e = cudaMemset(h->norm_d, 0, sizeof(NormState))) != cudaSuccess ||
        (e = cudaMemset(h->queue_d, 0, sizeof(unsigned))) != cudaSuccess ||
        (e = cudaMemset(h->step_d, 0, sizeof(StepState))) != cudaSuccess ||
        (e = upload_params(h)) != cudaSuccess) {
        free_scratch(h);
        delete h;
        return fail(nullptr, BF16OPT_ERR_CUDA, std::string("table upload: ") + cudaGetErrorString(e));
    }
    {
        std::lock_guard<std::mutex> lock(g_live_mu);
        g_live.insert(h);
    }
    g_create_error.clear();
    *out = h;
    return BF16OPT_OK;
}

int bf16opt_create_offload(const bf16opt_desc_t *d, int n_threads, bf16opt_t **out) {
    NvtxRange nvtx("bf16opt_create_offload");
    if (out) *out = nullptr;
    if (!d || !out) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "desc and out must be non-NULL");
    if (d->mode != BF16OPT_FLAT) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "offload: FLAT mode only");
    bf16opt_t *h = nullptr;
    int rc = bf16opt_create(d, &h);      // validates the descriptor, builds the tables and the device scratch
    if (rc) return rc;
    auto bail = [&](int code, const std::string &msg) {
        bf16opt_destroy(h);
        return fail(nullptr, code, msg);
    };
    if (d->n > 0) {
        // master and moments: host memory the host threads read and write;
        // accumulator and bf16 parameters: memory of the handle's device
        for (const void *p : {(const void *)d->master, (const void *)d->exp_avg, (const void *)d->exp_avg_sq}) {
            const cudaMemoryType k = memory_kind(p, nullptr);
            if (k != cudaMemoryTypeUnregistered && k != cudaMemoryTypeHost)
                return bail(BF16OPT_ERR_INVALID_ARG, "offload: master, exp_avg and exp_avg_sq must be host memory");
        }
        for (const void *p : {(const void *)d->grad_accum, (const void *)d->param_bf16}) {
            int dev = -1;
            if (memory_kind(p, &dev) != cudaMemoryTypeDevice || dev != h->device)
                return bail(BF16OPT_ERR_INVALID_ARG, "offload: grad_accum and param_bf16 must be memory of the current device");
        }
    }
    h->offload = true;
    h->host_p = d->master;
    h->host_m = d->exp_avg;
    h->host_v = d->exp_avg_sq;
    h->dev_acc = d->grad_accum;
    h->dev_bf = d->param_bf16;
    const uint64_t blk = std::max<uint64_t>(1, std::min<uint64_t>(kOffloadBlock, d->n));
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
        if ((e = cudaMallocHost(&h->stage_acc[i], blk * sizeof(float))) == cudaSuccess &&
            (e = cudaMallocHost(&h->stage_bf[i], blk * sizeof(uint16_t))) == cudaSuccess &&
            (e = cudaEventCreateWithFlags(&h->ev_d2h[i], cudaEventDisableTiming)) == cudaSuccess)
            e = cudaEventCreateWithFlags(&h->ev_h2d[i], cudaEventDisableTiming);
    }
    if (e == cudaSuccess && (e = cudaMallocHost(&h->stage_step, sizeof(StepState))) == cudaSuccess)
        e = cudaMallocHost(&h->stage_norm, sizeof(NormState));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return bail(e == cudaErrorMemoryAllocation ? BF16OPT_ERR_OOM : BF16OPT_ERR_CUDA,
                    std::string("offload staging: ") + cudaGetErrorString(e));
    }
    int nt = n_threads;
    if (nt <= 0) nt = (int)std::max(1u, std::thread::hardware_concurrency());
    try {
        h->pool = new bf16host::Pool(std::min(nt, 256));
    } catch (...) {
        return bail(BF16OPT_ERR_OOM, "offload: cannot start the host threads");
    }
    *out = h;
    return BF16OPT_OK;
}

int bf16opt_destroy(bf16opt_t *h) {
    NvtxRange nvtx("bf16opt_destroy");
    if (!h) return BF16OPT_OK;
    {
        std::lock_guard<std::mutex> lock(g_live_mu);
        if (g_live.erase(h) == 0) return BF16OPT_ERR_INVALID_ARG;   // never created, or destroyed twice
    }
    DeviceGuard dg(h->device);
    cudaDeviceSynchronize();
    free_scratch(h);
    // Everything the handle owns is released, but the small struct itself is
    // kept (a tombstone): were its address handed out again by a later create,
    // a stale copy of this handle would pass the registry check.
    std::vector<Seg>().swap(h->segs);
    std::vector<const uint16_t *>().swap(h->pend_flat);
    std::vector<std::vector<const uint16_t *>>().swap(h->pend_list);
    std::vector<uint32_t>().swap(h->slot_chunk0);
    std::vector<std::pair<const void *, int>>().swap(h->occ);
    std::vector<bf16opt_group_t>().swap(h->groups);
    std::string().swap(h->last_error);
    return BF16OPT_OK;
}

int bf16opt_get_step(const bf16opt_t *h, int64_t *t) {
    if (!live(h) || !t) return BF16OPT_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    int64_t v = 0;
    if (quiesce() != cudaSuccess || cudaMemcpy(&v, &h->step_d->t, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return BF16OPT_ERR_CUDA;
    }
    *t = v;
    return BF16OPT_OK;
}

int bf16opt_set_step(bf16opt_t *h, int64_t t) {
    NvtxRange nvtx("bf16opt_set_step");
    if (!live(h)) return BF16OPT_ERR_INVALID_ARG;
    if (t < 0) return fail(h, BF16OPT_ERR_INVALID_ARG, "step must be >= 0");
    DeviceGuard dg(h->device);
    cudaError_t e = quiesce();
    if (e != cudaSuccess) return cuda_fail(h, e, "waiting for the device");
    e = cudaMemcpy(&h->step_d->t, &t, sizeof t, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(h, e, "writing the step counter");
    h->scalars_ready = false;   // prepared for the old counter
    return BF16OPT_OK;
}

int bf16opt_accumulate(bf16opt_t *h, const uint16_t *grad_flat, const uint16_t *const *grad_list, unsigned flags,
                       void *stream) {
    NvtxRange nvtx("bf16opt_accumulate");
    if (!live(h)) return BF16OPT_ERR_INVALID_ARG;
    const bool first = flags & BF16OPT_FIRST, last = flags & BF16OPT_LAST, defer = flags & BF16OPT_DEFER;
    if (flags & ~(BF16OPT_FIRST | BF16OPT_LAST | BF16OPT_DEFER)) return fail(h, BF16OPT_ERR_INVALID_ARG, "unknown flag");
    if (!first && h->state != S_ACC) return fail(h, BF16OPT_ERR_SEQUENCE, "accumulate without FIRST outside an accumulation");
    if (h->mode == BF16OPT_FLAT) {
        if (grad_list) return fail(h, BF16OPT_ERR_INVALID_ARG, "FLAT: grad_list must be NULL");
        if (h->n > 0 && !grad_flat) return fail(h, BF16OPT_ERR_INVALID_ARG, "FLAT: grad_flat is NULL");
        if (mis2(grad_flat)) return fail(h, BF16OPT_ERR_ALIGNMENT, "grad_flat must be 2-B aligned");
    } else {
        if (grad_flat) return fail(h, BF16OPT_ERR_INVALID_ARG, "LIST: grad_flat must be NULL");
        if (h->n_tensors > 0 && !grad_list) return fail(h, BF16OPT_ERR_INVALID_ARG, "LIST: grad_list is NULL");
        for (const Seg &s : h->segs) {
            const uint16_t *g = grad_list[s.grad_slot];
            if (!g) return fail(h, BF16OPT_ERR_INVALID_ARG, "LIST: NULL gradient pointer for tensor " + std::to_string(s.grad_slot));
            if (mis2(g)) return fail(h, BF16OPT_ERR_ALIGNMENT, "LIST: gradient pointers must be 2-B aligned");
        }
    }
    const size_t pending_before = first ? 0 : h->pend_flat.size() + h->pend_list.size();
    if (defer && pending_before + 1 > (size_t)kMaxFold)
        return fail(h, BF16OPT_ERR_INVALID_ARG, "at most 8 deferred micro-batches may be pending");
    DeviceGuard dg(h->device);
    if (!dg.ok) return fail(h, BF16OPT_ERR_CUDA, "cannot select the handle's device");
    cudaStream_t st = (cudaStream_t)stream;

    // A stored call with a full pending set: fold the pending set into acc first
    // (same adds, same order), so no pass folds more than kMaxFold gradients.
    if (!first && !defer && pending_before == (size_t)kMaxFold) {
        int rc0 = launch_accum<true, false>(h, h->acc_valid, pending_set(h), st);
        if (rc0) return rc0;
        h->acc_valid = true;
        h->pend_flat.clear();
        h->pend_list.clear();
    }
    // The gradients this call folds (or keeps): the pending ones, then this one.
    const bool has_acc = first ? false : h->acc_valid;
    std::vector<const uint16_t *> pf = first ? std::vector<const uint16_t *>() : h->pend_flat;
    std::vector<std::vector<const uint16_t *>> pl = first ? std::vector<std::vector<const uint16_t *>>() : h->pend_list;
    if (h->mode == BF16OPT_FLAT) pf.push_back(grad_flat);
    else pl.emplace_back(grad_list, grad_list + h->n_tensors);
    FoldSet fs;
    fs.flat = pf;
    for (const auto &v : pl) fs.list.push_back(&v);

    int rc = 0;
    if (!defer) rc = last ? launch_accum<true, true>(h, has_acc, fs, st) : launch_accum<true, false>(h, has_acc, fs, st);
    else if (last) rc = launch_accum<false, true>(h, has_acc, fs, st);
    if (rc) return rc;

    h->acc_valid = has_acc;
    if (!defer) {
        h->acc_valid = true;
        h->pend_flat.clear();
        h->pend_list.clear();
    } else {
        h->pend_flat = std::move(pf);
        h->pend_list = std::move(pl);
    }
    h->state = !last ? S_ACC : (defer ? S_ACC_DEFERRED : S_ACC_DONE);
    return BF16OPT_OK;
}

int bf16opt_grad_norm(bf16opt_t *h, void *stream, double *host_norm) {
    NvtxRange nvtx("bf16opt_grad_norm");
    if (!live(h)) return BF16OPT_ERR_INVALID_ARG;
    if (h->state != S_ACC_DONE && h->state != S_ACC_DEFERRED)
        return fail(h, BF16OPT_ERR_SEQUENCE, "grad_norm needs a completed accumulation (FIRST ... LAST)");
    DeviceGuard dg(h->device);
    if (!dg.ok) return fail(h, BF16OPT_ERR_CUDA, "cannot select the handle's device");
    cudaStream_t st = (cudaStream_t)stream;
    // the chunk partials were written by the LAST pass
    cudaError_t e = launch(h, k_norm_final, 1, kFinalThreads, st, (const double *)h->partials_d, h->n_chunks,
                           h->max_norm, h->norm_d, (const StepParams *)h->params_d, h->step_d);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(h, e, "norm kernel launch");
    h->state = S_NORMED;
    h->scalars_ready = true;
    if (host_norm) {
        double nrm = 0.0;
        if ((e = cudaMemcpyAsync(&nrm, &h->norm_d->norm, sizeof(double), cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
            (e = cudaStreamSynchronize(st)) != cudaSuccess)
            return cuda_fail(h, e, "reading the norm");
        *host_norm = nrm;
        if (!std::isfinite(nrm)) {
            h->last_error = "gradient norm is not finite";
            return BF16OPT_WARN_NONFINITE;
        }
    }
    return BF16OPT_OK;
}

int bf16opt_grad_norm_local(bf16opt_t *h, void *stream, double *local_sumsq) {
    NvtxRange nvtx("bf16opt_grad_norm_local");
    if (!live(h)) return BF16OPT_ERR_INVALID_ARG;
    if (!local_sumsq) return fail(h, BF16OPT_ERR_INVALID_ARG, "grad_norm_local: local_sumsq is NULL");
    if (h->state != S_ACC_DONE && h->state != S_ACC_DEFERRED)
        return fail(h, BF16OPT_ERR_SEQUENCE, "grad_norm_local needs a completed accumulation (FIRST ... LAST)");
    double nrm = 0.0;
    int rc = bf16opt_grad_norm(h, stream, &nrm);
    if (rc < 0) return rc;
    DeviceGuard dg(h->device);
    double S = 0.0;
    cudaError_t e;
    if ((e = cudaMemcpy(&S, &h->norm_d->sumsq, sizeof(double), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(h, e, "reading the local sum of squares");
    *local_sumsq = S;
    h->local_sumsq = S;
    h->state = S_LOCAL_NORMED;
    return BF16OPT_OK;
}

int bf16opt_set_global_sumsq(bf16opt_t *h, double global_sumsq, void *stream) {
    NvtxRange nvtx("bf16opt_set_global_sumsq");
    if (!live(h)) return BF16OPT_ERR_INVALID_ARG;
    if (h->state != S_LOCAL_NORMED) return fail(h, BF16OPT_ERR_SEQUENCE, "set_global_sumsq needs grad_norm_local first");
    DeviceGuard dg(h->device);
    if (!dg.ok) return fail(h, BF16OPT_ERR_CUDA, "cannot select the handle's device");
    cudaError_t e = launch(h, k_norm_from_sumsq, 1, 64, (cudaStream_t)stream, global_sumsq, h->max_norm, h->norm_d,
                           (const StepParams *)h->params_d, h->step_d);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(h, e, "norm kernel launch");
    h->state = S_NORMED;
    h->scalars_ready = true;
    if (!std::isfinite(global_sumsq)) {
        h->last_error = "global gradient norm is not finite";
        return BF16OPT_WARN_NONFINITE;
    }
    return BF16OPT_OK;
}

int bf16opt_sum_rank_sumsqs(const double *per_rank, uint32_t n_ranks, double *global_sumsq) {
    if (!per_rank || !global_sumsq || n_ranks == 0) return BF16OPT_ERR_INVALID_ARG;
    // one FP64 add per rank, rank 0 first: every rank that sums the same
    // gathered values gets the same bits
    double S = 0.0;
    for (uint32_t r = 0; r < n_ranks; ++r) S += per_rank[r];
    *global_sumsq = S;
    return BF16OPT_OK;
}

int bf16opt_set_rank_sumsqs(bf16opt_t *h, const double *per_rank, uint32_t n_ranks, uint32_t rank, void *stream,
                            double *global_norm) {
    NvtxRange nvtx("bf16opt_set_rank_sumsqs");
    if (!live(h)) return BF16OPT_ERR_INVALID_ARG;
    if (!per_rank || n_ranks == 0 || rank >= n_ranks)
        return fail(h, BF16OPT_ERR_INVALID_ARG, "set_rank_sumsqs: need per_rank[n_ranks], n_ranks >= 1, rank < n_ranks");
    if (h->state != S_LOCAL_NORMED) return fail(h, BF16OPT_ERR_SEQUENCE, "set_rank_sumsqs needs grad_norm_local first");
    // this rank's entry must be the value grad_norm_local handed out: a gather
    // that placed the values out of rank order is caught here
    if (std::memcmp(&per_rank[rank], &h->local_sumsq, sizeof(double)) != 0)
        return fail(h, BF16OPT_ERR_INVALID_ARG,
                    "set_rank_sumsqs: per_rank[rank] is not this partition's sum of squares (gathered out of order?)");
    double S = 0.0;
    bf16opt_sum_rank_sumsqs(per_rank, n_ranks, &S);
    int rc = bf16opt_set_global_sumsq(h, S, stream);
    if (rc < 0) return rc;
    if (global_norm) *global_norm = std::sqrt(S);
    return rc;
}

int bf16opt_lr_factor(const bf16opt_lr_schedule_t *s, int64_t t, double *factor) {
    if (!s || !factor || t < 1) return BF16OPT_ERR_INVALID_ARG;
    if (s->warmup_steps < 0 || s->decay_steps < s->warmup_steps || !(s->min_lr_ratio >= 0.f && s->min_lr_ratio <= 1.f) ||
        s->reserved != 0)
        return BF16OPT_ERR_INVALID_ARG;
    const double r = (double)s->min_lr_ratio;
    const int64_t w = s->warmup_steps, d = s->decay_steps;
    if (t <= w) {
        *factor = (double)t / (double)w;
    } else if (t <= d) {
        const double x = (double)(t - w) / (double)(d - w);
        *factor = r + (1.0 - r) * 0.5 * (1.0 + std::cos(M_PI * x));
    } else {
        *factor = r;
    }
    return BF16OPT_OK;
}

int bf16opt_set_skip_nonfinite(bf16opt_t *h, int enable) {
    NvtxRange nvtx("bf16opt_set_skip_nonfinite");
    if (!live(h)) return BF16OPT_ERR_INVALID_ARG;
    DeviceGuard dg(h->device);
    cudaError_t e = quiesce();
    if (e != cudaSuccess) return cuda_fail(h, e, "waiting for the device");
    h->skip_nonfinite = enable != 0;
    h->scalars_ready = false;   // the skip decision was prepared with the old setting
    e = upload_params(h);
    if (e != cudaSuccess) return cuda_fail(h, e, "uploading the skip setting");
    return BF16OPT_OK;
}

int bf16opt_set_lr_schedule(bf16opt_t *h, const bf16opt_lr_schedule_t *s) {
    NvtxRange nvtx("bf16opt_set_lr_schedule");
    if (!live(h)) return BF16OPT_ERR_INVALID_ARG;
    double f = 0.0;
    if (s && bf16opt_lr_factor(s, 1, &f) != BF16OPT_OK)
        return fail(h, BF16OPT_ERR_INVALID_ARG, "lr schedule: need 0 <= warmup_steps <= decay_steps, min_lr_ratio in [0, 1]");
    DeviceGuard dg(h->device);
    cudaError_t e = quiesce();
    if (e != cudaSuccess) return cuda_fail(h, e, "waiting for the device");
    h->has_sched = s != nullptr;
    if (s) h->sched = *s;
    h->scalars_ready = false;   // prepared with the old schedule
    e = upload_params(h);
    if (e != cudaSuccess) return cuda_fail(h, e, "uploading the schedule");
    return BF16OPT_OK;
}

int bf16opt_step(bf16opt_t *h, const float *lr_override, void *stream) {
    NvtxRange nvtx("bf16opt_step");
    if (!live(h)) return BF16OPT_ERR_INVALID_ARG;
    if (h->state != S_NORMED) return fail(h, BF16OPT_ERR_SEQUENCE, "step needs grad_norm first");
    LrOverride ov;
    memset(&ov, 0, sizeof ov);
    if (lr_override) {
        ov.use = 1;
        for (size_t i = 0; i < h->groups.size(); ++i) {
            if (!std::isfinite(lr_override[i]) || lr_override[i] < 0.f)
                return fail(h, BF16OPT_ERR_INVALID_ARG, "lr_override must be finite and >= 0");
            ov.lr[i] = lr_override[i];
        }
    }
    DeviceGuard dg(h->device);
    if (!dg.ok) return fail(h, BF16OPT_ERR_CUDA, "cannot select the handle's device");
    cudaStream_t st = (cudaStream_t)stream;
    if (h->offload) {
        int rc = offload_step(h, ov, st);
        if (rc) return rc;
        h->state = S_IDLE;
        h->acc_valid = false;
        h->pend_flat.clear();
        h->scalars_ready = false;
        return BF16OPT_OK;
    }
    // The norm kernel prepared the scalars of step t + 1 with the groups' own
    // learning rates; the step kernel then advances t itself.  A learning-rate
    // override, a setting changed since the norm, or an empty shard take one
    // more one-warp kernel that computes them (and advances t).  Either way
    // everything is computed on the device, so a captured step replays right.
    const bool prepared = !lr_override && h->scalars_ready && h->n_chunks > 0;
    if (!prepared) {
        cudaError_t e = launch(h, k_step_scalars, 1, 32, st, (const StepParams *)h->params_d, h->step_d, ov,
                               (const NormState *)h->norm_d);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(h, e, "step scalars launch");
    }
    int rc = launch_step(h, h->acc_valid, pending_set(h), st, prepared);
    if (rc) return rc;
    h->scalars_ready = false;
    h->state = S_IDLE;
    h->acc_valid = false;
    h->pend_flat.clear();
    h->pend_list.clear();
    return BF16OPT_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free one-shot norm (bf16opt_grad_norm_static).
//
// Some callers cannot call cudaMalloc: code running inside another
// framework's launch path that is handed only a stream and a pre-planned
// workspace (plugins, custom-op launchers), processes whose device memory is
// already held by a caching allocator (a raw cudaMalloc can then fail), and
// latency-sensitive loops that cannot take the device synchronisation that
// cudaMalloc/cudaFree imply.  For them this entry point keeps its scratch --
// one FP64 partial per 32,768-element chunk -- in a file-scope device array
// of fixed size, so it never allocates.  The array exists once per GPU that
// loads this library and stays allocated until the process exits.
// ---------------------------------------------------------------------------

namespace {

constexpr uint32_t kStaticMaxChunks = 65536;  // 512 KiB of FP64 partials
constexpr int kStaticMaxDevices = 64;
static_assert((BF16OPT_STATIC_NORM_MAX_ELEMS + kHeadAlign - 1 + kChunk - 1) / kChunk <= kStaticMaxChunks,
              "the static norm scratch must hold one partial per chunk of the largest accepted n");

static __device__ __align__(256) double g_static_partials[kStaticMaxChunks];

// The array's device address depends on the context that loaded this module:
// after cudaDeviceReset (or a reset of the primary context) the next context
// loads it again, possibly elsewhere.  The address is therefore cached per
// device together with the id of the context it was looked up in (context ids
// are never reused within a process, unlike context handles) and looked up
// again when the current context's id differs.  The two driver calls are
// fetched through the runtime, so the library does not link libcuda.
struct DriverCtx {
    CUresult (*get_current)(CUcontext *) = nullptr;
    CUresult (*get_id)(CUcontext, unsigned long long *) = nullptr;
};

const DriverCtx &driver_ctx() {
    static const DriverCtx d = [] {
        DriverCtx r;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            r.get_current = reinterpret_cast<CUresult (*)(CUcontext *)>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            r.get_id = reinterpret_cast<CUresult (*)(CUcontext, unsigned long long *)>(p);
        cudaGetLastError();
        return r;
    }();
    return d;
}

// Id of the current context; 0 when there is none yet or it cannot be read.
unsigned long long current_ctx_id() {
    const DriverCtx &d = driver_ctx();
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!d.get_current || !d.get_id || d.get_current(&c) != CUDA_SUCCESS || !c || d.get_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

struct StaticSlot {
    unsigned long long ctx_id;
    double *ptr;
};
std::mutex g_static_mu;
StaticSlot g_static_slot[kStaticMaxDevices] = {};

// Device address of g_static_partials in the current context of device `dev`
// (the current device).  In host code the array's name is only a host-side
// stand-in, so the kernels must be given this address.
int static_scratch(int dev, double **out, std::string &msg) {
    const unsigned long long id = current_ctx_id();
    std::lock_guard<std::mutex> lock(g_static_mu);
    StaticSlot &sl = g_static_slot[dev];
    if (!sl.ptr || id == 0 || sl.ctx_id != id) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_partials);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            msg = std::string("cudaGetSymbolAddress of the static norm scratch failed: ") + cudaGetErrorString(e);
            return BF16OPT_ERR_CUDA;
        }
        sl.ptr = static_cast<double *>(p);
        sl.ctx_id = current_ctx_id();   // the lookup makes the primary context current if it was not
    }
    *out = sl.ptr;
    return BF16OPT_OK;
}

// Address under which the kernels on device `dev` may use `p`: device memory
// of that device or managed memory as is, page-locked host memory through its
// mapped device address.  Anything else -- pageable host memory, another
// device's memory, an unknown pointer -- gives nullptr.
void *device_view(const void *p, int dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    switch (a.type) {
    case cudaMemoryTypeDevice: return a.device == dev ? const_cast<void *>(p) : nullptr;
    case cudaMemoryTypeManaged: return const_cast<void *>(p);
    case cudaMemoryTypeHost: return a.devicePointer;
    default: return nullptr;
    }
}

// Partial sums of squares of implicit chunks (sized and cut as in the handle's chunk table) of
// a flat FP32 buffer: the same thread->element map, compensated sum and CTA tree
// as the handle's norm pass over a one-range FLAT shard.
template <int U>
__global__ void __launch_bounds__(kThreads)
k_static_partials(const float *__restrict__ acc, uint64_t n, uint32_t nchunks, uint32_t chunk, uint32_t cut,
                  float gscale, double *__restrict__ partials) {
    __shared__ double sh[kThreads / 32];
    for (uint32_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        // chunk c = [c chunk - cut, (c + 1) chunk - cut) clipped to [0, n): the
        // handle's chunking of a one-range FLAT shard over the same buffer
        const uint64_t start = c == 0 ? 0 : (uint64_t)c * chunk - cut;
        const uint64_t lim = (uint64_t)(c + 1) * chunk - cut;
        const uint64_t end = lim < n ? lim : n;
        const uint32_t len = (uint32_t)(end - start);
        const float *a = acc + start;
        uint32_t head = (kHeadAlign - phaseA_f32(a)) & (kHeadAlign - 1);
        if (head > len) head = len;
        const uint32_t nq = (len - head) >> 2;
        const uint32_t tail0 = head + (nq << 2);
        if (check_fails(end > n, kFaultChunkRange) || check_fails(tail0 > len, kFaultBody) ||
            check_fails(nq != 0 && mis16(a + head), kFaultAlign))
            continue;
        Comp cs = {0.f, 0.f};
        const uint32_t rh = scalar_lane<kThreads>(c, 0), rt = scalar_lane<kThreads>(c, 1);
        for (uint32_t i = rh; i < head; i += kThreads) comp_add_sq(cs, __fmul_rn(a[i], gscale));
        for (uint32_t i = tail0 + rt; i < len; i += kThreads) comp_add_sq(cs, __fmul_rn(a[i], gscale));
        const float4 *a4 = reinterpret_cast<const float4 *>(a + head);
        for (uint32_t base = threadIdx.x; base < nq; base += kThreads * U) {
            float4 av[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t j = base + u * kThreads;
                if (j < nq) av[u] = __ldcs(a4 + j);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t j = base + u * kThreads;
                if (j < nq) {
                    comp_add_sq(cs, __fmul_rn(av[u].x, gscale));
                    comp_add_sq(cs, __fmul_rn(av[u].y, gscale));
                    comp_add_sq(cs, __fmul_rn(av[u].z, gscale));
                    comp_add_sq(cs, __fmul_rn(av[u].w, gscale));
                }
            }
        }
        double mine = (double)cs.s + (double)cs.c;
        if (!isfinite(mine)) {                          // rare: a square overflowed FP32
            GradPtrs<1> gp;
            gp.p[0] = nullptr;
            mine = sumsq_rescaled<false, true, 0, 1, kThreads>(a, gp, 0, head, nq, len, gscale, rh, rt);
        }
        const double tot = cta_sum(mine, sh);
        if (threadIdx.x == 0) partials[c] = tot;
    }
}

// Fixed-order sum of the partials, norm and clip coefficient into the
// caller's result: the same helpers as the handle's k_norm_final.
__global__ void __launch_bounds__(kFinalThreads)
k_static_final(const double *__restrict__ partials, uint32_t n, float max_norm, bf16opt_norm_result_t *out) {
    __shared__ double sh[kFinalThreads];
    const double S = final_sum(partials, n, sh);
    if (threadIdx.x == 0) {
        const NormClip r = norm_and_clip(S, max_norm);
        out->sumsq = r.sumsq;
        out->norm = r.norm;
        out->clip_coef = r.c;
    }
}

}  // namespace

extern "C" int bf16opt_grad_norm_static(const float *grad_accum, uint64_t n, float grad_scale, float max_grad_norm,
                                        bf16opt_norm_result_t *out, void *stream) {
    g_create_error.clear();
    if (!out) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "grad_norm_static: out is NULL");
    if (((uintptr_t)out & 7u) != 0) return fail(nullptr, BF16OPT_ERR_ALIGNMENT, "grad_norm_static: out must be 8-B aligned");
    if (n > BF16OPT_STATIC_NORM_MAX_ELEMS)
        return fail(nullptr, BF16OPT_ERR_INVALID_ARG,
                    "grad_norm_static: n = " + std::to_string(n) + " exceeds the static scratch limit of " +
                        std::to_string((unsigned long long)BF16OPT_STATIC_NORM_MAX_ELEMS) + " elements");
    if (n > 0 && !grad_accum) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "grad_norm_static: grad_accum is NULL");
    if (mis4(grad_accum)) return fail(nullptr, BF16OPT_ERR_ALIGNMENT, "grad_norm_static: grad_accum must be 4-B aligned");
    if (!finite_f(grad_scale) || grad_scale == 0.f || !finite_f(max_grad_norm))
        return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "grad_norm_static: grad_scale and max_grad_norm must be finite, grad_scale != 0");
    int dev = 0, ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev < 1 || cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return fail(nullptr, BF16OPT_ERR_UNSUPPORTED, "grad_norm_static: no CUDA device");
    }
    if (dev < 0 || dev >= kStaticMaxDevices) return fail(nullptr, BF16OPT_ERR_UNSUPPORTED, "grad_norm_static: device ordinal too large");
    // The kernels write `out` and read `grad_accum` directly: both must be
    // memory the device can use (checked here; a pageable host pointer would
    // otherwise fault inside the kernel instead of returning an error).
    auto *out_d = static_cast<bf16opt_norm_result_t *>(device_view(out, dev));
    if (!out_d) return fail(nullptr, BF16OPT_ERR_INVALID_ARG,
                            "grad_norm_static: out must be device, managed or page-locked host memory of the current device");
    const float *acc_d = nullptr;
    if (n > 0 && !(acc_d = static_cast<const float *>(device_view(grad_accum, dev))))
        return fail(nullptr, BF16OPT_ERR_INVALID_ARG,
                    "grad_norm_static: grad_accum must be device, managed or page-locked host memory of the current device");
    double *partials = nullptr;
    std::string msg;
    int rc = static_scratch(dev, &partials, msg);
    if (rc) return fail(nullptr, rc, msg);
    int sms = 1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
    const uint32_t chunk = chunk_elems(n), cut = first_chunk_cut(acc_d);
    const uint32_t nchunks = n == 0 ? 0u : (uint32_t)((n + cut + chunk - 1) / chunk);
    cudaStream_t st = (cudaStream_t)stream;
    if (nchunks > 0) {
        const uint32_t grid = std::min<uint32_t>(nchunks, (uint32_t)sms * 8u);
        k_static_partials<BF16K_ACC_U><<<grid, kThreads, 0, st>>>(acc_d, n, nchunks, chunk, cut, grad_scale, partials);
    }
    k_static_final<<<1, kFinalThreads, 0, st>>>(partials, nchunks, max_grad_norm, out_d);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "grad_norm_static kernel launch");
    return BF16OPT_OK;
}

int bf16opt_step_path(const bf16opt_t *h, int *path) {
    if (path) *path = BF16OPT_PATH_NONE;
    if (!live(h)) return fail(nullptr, BF16OPT_ERR_INVALID_ARG, "not a live handle");
    if (!path) return fail(const_cast<bf16opt_t *>(h), BF16OPT_ERR_INVALID_ARG, "path must be non-NULL");
    *path = h->offload ? BF16OPT_PATH_HOST : h->step_path;
    return BF16OPT_OK;
}

// ---------------------------------------------------------------------------
// Waits of the fused step's copy pipeline that gave up (see kernels.cuh).
// ---------------------------------------------------------------------------
extern "C" int bf16opt_pipeline_timeouts(uint32_t *count) {
    if (!count) return BF16OPT_ERR_INVALID_ARG;
    *count = 0;
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return fail(nullptr, BF16OPT_ERR_UNSUPPORTED, "no CUDA device");
    }
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_pipe_timeouts, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_pipe_timeouts, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "reading the pipeline's timeout count");
    *count = v;
    return BF16OPT_OK;
}

// ---------------------------------------------------------------------------
// Fault word of the checked build (see kernels.cuh).
// ---------------------------------------------------------------------------
extern "C" int bf16opt_debug_faults(uint32_t *bits) {
    if (!bits) return BF16OPT_ERR_INVALID_ARG;
    *bits = 0;
#ifdef BF16K_CHECKS
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_check_faults, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_check_faults, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "reading the fault word");
    *bits = v;
    return BF16OPT_OK;
#else
    return fail(nullptr, BF16OPT_ERR_UNSUPPORTED, "not a checked build (compile with -DBF16K_CHECKS)");
#endif
}

// hbm_probe.cu -- the HBM bandwidth probe declared in include/hbm_probe.h.
//
// A measurement tool beside the optimizer: streaming kernels over
// caller-owned buffers, 16-byte vectors, 64 KiB chunks taken from a counter
// (the optimizer's passes take theirs the same way).  The counter resets
// itself: every CTA makes exactly one claim past the last chunk, and the CTA
// holding the last such claim stores 0, after which no CTA of the grid
// touches it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/hbm_probe.h"

namespace {

constexpr int kT = 256;                 // threads per CTA
constexpr uint32_t kVecPerChunk = 4096; // 16-byte vectors (or quads) per chunk

struct Claim {
    unsigned *ctr;
    uint32_t nch;
    uint32_t *sh;
    __device__ __forceinline__ uint32_t next() {
        __syncthreads();
        if (threadIdx.x == 0) *sh = atomicAdd(ctr, 1u);
        __syncthreads();
        return *sh;
    }
    __device__ __forceinline__ void done(uint32_t last) {
        if (threadIdx.x == 0 && last == nch + gridDim.x - 1) atomicExch(ctr, 0u);
    }
};

template <int U>
__global__ void __launch_bounds__(kT) k_copy(const float4 *__restrict__ src, float4 *__restrict__ dst, uint32_t nch,
                                            unsigned *ctr) {
    __shared__ uint32_t sh;
    Claim cl{ctr, nch, &sh};
    uint32_t c = cl.next();
    for (; c < nch; c = cl.next()) {
        const uint64_t v0 = (uint64_t)c * kVecPerChunk;
        for (uint32_t b = threadIdx.x; b < kVecPerChunk; b += kT * U) {
            float4 x[U];
#pragma unroll
            for (int u = 0; u < U; ++u) x[u] = __ldcs(src + v0 + b + u * kT);
#pragma unroll
            for (int u = 0; u < U; ++u) __stcs(dst + v0 + b + u * kT, x[u]);
        }
    }
    cl.done(c);
}

template <int U>
__global__ void __launch_bounds__(kT) k_write(float4 *__restrict__ dst, uint32_t nch, unsigned *ctr) {
    __shared__ uint32_t sh;
    Claim cl{ctr, nch, &sh};
    uint32_t c = cl.next();
    for (; c < nch; c = cl.next()) {
        const uint64_t v0 = (uint64_t)c * kVecPerChunk;
        const float f = (float)c;
        for (uint32_t b = threadIdx.x; b < kVecPerChunk; b += kT * U) {
#pragma unroll
            for (int u = 0; u < U; ++u) __stcs(dst + v0 + b + u * kT, make_float4(f, f, f, f));
        }
    }
    cl.done(c);
}

template <int U>
__global__ void __launch_bounds__(kT) k_read(const uint4 *__restrict__ src, uint32_t *__restrict__ sink,
                                            uint32_t nch, unsigned *ctr) {
    __shared__ uint32_t sh;
    Claim cl{ctr, nch, &sh};
    uint32_t acc = 0;
    uint32_t c = cl.next();
    for (; c < nch; c = cl.next()) {
        const uint64_t v0 = (uint64_t)c * kVecPerChunk;
        for (uint32_t b = threadIdx.x; b < kVecPerChunk; b += kT * U) {
            uint4 x[U];
#pragma unroll
            for (int u = 0; u < U; ++u) x[u] = __ldcs(src + v0 + b + u * kT);
#pragma unroll
            for (int u = 0; u < U; ++u) acc ^= x[u].x ^ x[u].y ^ x[u].z ^ x[u].w;
        }
    }
    cl.done(c);
    atomicXor(&sink[blockIdx.x], acc);   // keeps the loads
}

// The fused step's traffic: 5 streams read, 4 written, little arithmetic.
template <int U>
__global__ void __launch_bounds__(kT) k_mix(const float4 *__restrict__ a, const uint2 *__restrict__ g,
                                           float4 *__restrict__ p, float4 *__restrict__ m, float4 *__restrict__ v,
                                           uint2 *__restrict__ bf, uint32_t nch, unsigned *ctr) {
    __shared__ uint32_t sh;
    Claim cl{ctr, nch, &sh};
    uint32_t c = cl.next();
    for (; c < nch; c = cl.next()) {
        const uint64_t q0 = (uint64_t)c * kVecPerChunk;
        for (uint32_t b = threadIdx.x; b < kVecPerChunk; b += kT * U) {
            float4 av[U], pv[U], mv[U], vv[U];
            uint2 gv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint64_t q = q0 + b + u * kT;
                av[u] = __ldcs(a + q);
                gv[u] = __ldcs(g + q);
                pv[u] = __ldcs(p + q);
                mv[u] = __ldcs(m + q);
                vv[u] = __ldcs(v + q);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint64_t q = q0 + b + u * kT;
                const float4 np = make_float4(pv[u].x + av[u].x, pv[u].y + av[u].y, pv[u].z + av[u].z,
                                              pv[u].w + av[u].w);
                __stcs(p + q, np);
                __stcs(m + q, make_float4(mv[u].x + av[u].x, mv[u].y, mv[u].z, mv[u].w + __uint_as_float(gv[u].x)));
                __stcs(v + q, make_float4(vv[u].x, vv[u].y + av[u].y, vv[u].z, vv[u].w + __uint_as_float(gv[u].y)));
                __stcs(bf + q, make_uint2((__float_as_uint(np.x) >> 16) | (__float_as_uint(np.y) & 0xffff0000u),
                                          (__float_as_uint(np.z) >> 16) | (__float_as_uint(np.w) & 0xffff0000u)));
            }
        }
    }
    cl.done(c);
}

// The accumulate passes' traffic: bf16 quads read (8 B), FP32 quads written
// (16 B), and with HAS_ACC the FP32 quads read first (16 B).
template <bool HAS_ACC, int U>
__global__ void __launch_bounds__(kT) k_acc_mix(const uint2 *__restrict__ g, float4 *__restrict__ a, uint32_t nch,
                                               unsigned *ctr) {
    __shared__ uint32_t sh;
    Claim cl{ctr, nch, &sh};
    uint32_t c = cl.next();
    for (; c < nch; c = cl.next()) {
        const uint64_t q0 = (uint64_t)c * kVecPerChunk;
        for (uint32_t b = threadIdx.x; b < kVecPerChunk; b += kT * U) {
            uint2 gv[U];
            float4 av[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                gv[u] = __ldcs(g + q0 + b + u * kT);
                if (HAS_ACC) av[u] = __ldcs(a + q0 + b + u * kT);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float4 x = make_float4(__uint_as_float(gv[u].x << 16), __uint_as_float(gv[u].x & 0xffff0000u),
                                             __uint_as_float(gv[u].y << 16), __uint_as_float(gv[u].y & 0xffff0000u));
                __stcs(a + q0 + b + u * kT,
                       HAS_ACC ? make_float4(av[u].x + x.x, av[u].y + x.y, av[u].z + x.z, av[u].w + x.w) : x);
            }
        }
    }
    cl.done(c);
}

// ---------------------------------------------------------------- bulk copies
// The pipelined passes' traffic moved the way they move it: one thread per
// CTA issues cp.async.bulk loads into a ring of shared-memory stages
// (completing on an mbarrier by transaction count) and bulk stores out of it;
// eight compute warps touch every stage (the same few adds as k_mix /
// k_acc_mix) and release it.  Every mbarrier wait gives up after 2 s and
// counts the timeout; the run then reports a CUDA error.
__device__ uint32_t g_bulk_timeouts;
constexpr int kBulkWarps = 8;
constexpr int kBulkThreads = 32 * (kBulkWarps + 1);
constexpr int kBulkMaxStages = 8;
constexpr uint32_t kBulkEnd = 0xffffffffu;

__device__ __forceinline__ uint32_t sa(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool bar_test(uint64_t *b, uint32_t par) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok)
                 : "r"(sa(b)), "r"(par)
                 : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool bar_wait(uint64_t *b, uint32_t par) {
    if (bar_test(b, par)) return true;
    const uint64_t t0 = now_ns();
    for (uint32_t i = 1;; ++i) {
        if (bar_test(b, par)) return true;
        if ((i & 63u) == 0 && now_ns() - t0 > 2000000000ull) {
            atomicAdd(&g_bulk_timeouts, 1u);
            return false;
        }
    }
}
__device__ __forceinline__ void bar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ void bar_arrive_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void ld_bulk(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            sa(dst)),
        "l"(src), "r"(bytes), "r"(sa(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void st_bulk(void *dst, const void *src, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                 "r"(sa(src)), "r"(bytes), "l"(pol)
                 : "memory");
}

// MIX 0: the fused step's 18:14 (a, g, p, m, v in; p, m, v, bf out), tiles of
// 512 quads, five stages, four tiles per claim (the library's units);
// MIX 1: a later accumulate's 6:4 (g, acc in; acc out), tiles of 2,048 quads,
// four stages, one tile per claim.
template <int MIX>
struct BulkMix {
    static constexpr uint32_t Q = MIX == 0 ? 512u : 2048u;
    static constexpr uint32_t quad_bytes = MIX == 0 ? 72u : 24u;
    static constexpr uint32_t stage_bytes = Q * quad_bytes;
    static constexpr int stages = MIX == 0 ? 5 : 4;
    static constexpr uint32_t tiles_per_claim = MIX == 0 ? 4u : 1u;
};

template <int MIX>
__global__ void __launch_bounds__(kBulkThreads, 1)
k_bulk_mix(void *const *__restrict__ bufs, uint32_t nt, unsigned *ctr) {
    using C = BulkMix<MIX>;
    constexpr uint32_t Q = C::Q;
    constexpr int S = C::stages;
    extern __shared__ __align__(128) unsigned char smb[];
    __shared__ uint64_t full[kBulkMaxStages], done[kBulkMaxStages];
    __shared__ uint32_t tile[kBulkMaxStages];
    float4 *a = (float4 *)bufs[MIX == 0 ? 0 : 1];   // step: the accumulator (read); accumulate: acc (read, written)
    uint2 *g = (uint2 *)bufs[MIX == 0 ? 1 : 0];
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&full[i])), "r"(1) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&done[i])), "r"(32 * kBulkWarps) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        if (threadIdx.x != 0) return;
        uint64_t pol;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
        const uint32_t ncl = (nt + C::tiles_per_claim - 1) / C::tiles_per_claim;
        int issued = 0, stored = 0;
        bool ok = true;
        auto retire = [&]() -> bool {
            const int s = stored % S;
            if (!bar_wait(&done[s], (uint32_t)(stored / S) & 1u)) return false;
            unsigned char *st = smb + (size_t)s * C::stage_bytes;
            const uint64_t q0 = (uint64_t)tile[s] * Q;
            if (MIX == 0) {
                st_bulk((float4 *)bufs[2] + q0, st + 24 * Q, 16 * Q, pol);
                st_bulk((float4 *)bufs[3] + q0, st + 40 * Q, 16 * Q, pol);
                st_bulk((float4 *)bufs[4] + q0, st + 56 * Q, 16 * Q, pol);
                st_bulk((uint2 *)bufs[5] + q0, st + 16 * Q, 8 * Q, pol);
            } else {
                st_bulk(a + q0, st, 16 * Q, pol);
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            ++stored;
            return true;
        };
        auto acquire = [&]() -> int {
            while (stored <= issued - (S - 1)) {
                if (!retire()) return -1;
                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            }
            return issued % S;
        };
        uint32_t k = atomicAdd(ctr, 1u);
        while (ok && k < ncl) {
            const uint32_t t1 = (k + 1) * C::tiles_per_claim < nt ? (k + 1) * C::tiles_per_claim : nt;
            for (uint32_t t = k * C::tiles_per_claim; t < t1; ++t) {
                const int s = acquire();
                if (s < 0) {
                    ok = false;
                    break;
                }
                tile[s] = t;
                unsigned char *st = smb + (size_t)s * C::stage_bytes;
                const uint64_t q0 = (uint64_t)t * Q;
                bar_arrive_tx(&full[s], C::stage_bytes);
                ld_bulk(st, a + q0, 16 * Q, &full[s], pol);
                ld_bulk(st + 16 * Q, g + q0, 8 * Q, &full[s], pol);
                if (MIX == 0) {
                    ld_bulk(st + 24 * Q, (const float4 *)bufs[2] + q0, 16 * Q, &full[s], pol);
                    ld_bulk(st + 40 * Q, (const float4 *)bufs[3] + q0, 16 * Q, &full[s], pol);
                    ld_bulk(st + 56 * Q, (const float4 *)bufs[4] + q0, 16 * Q, &full[s], pol);
                }
                ++issued;
            }
            if (ok) k = atomicAdd(ctr, 1u);
        }
        if (ok) {
            const int s = acquire();
            if (s >= 0) {
                tile[s] = kBulkEnd;
                bar_arrive(&full[s]);
                while (stored < issued)
                    if (!retire()) break;
            }
        }
        for (int i = stored; i < issued; ++i) bar_wait(&full[i % S], (uint32_t)(i / S) & 1u);   // after a timeout
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        while (k < ncl) k = atomicAdd(ctr, 1u);                 // one claim past the end, as always
        if (k == ncl + gridDim.x - 1) atomicExch(ctr, 0u);
        return;
    }
    const uint32_t ct = threadIdx.x - 32;
    for (int i = 0;; ++i) {
        const int s = i % S;
        if (!bar_wait(&full[s], (uint32_t)(i / S) & 1u)) return;
        if (tile[s] == kBulkEnd) return;
        unsigned char *st = smb + (size_t)s * C::stage_bytes;
        float4 *a4 = (float4 *)st;
        uint2 *g4 = (uint2 *)(st + 16 * Q);
        for (uint32_t q = ct; q < Q; q += 32 * kBulkWarps) {
            const float4 av = a4[q];
            const uint2 gv = g4[q];
            if (MIX == 0) {
                float4 *p4 = (float4 *)(st + 24 * Q), *m4 = (float4 *)(st + 40 * Q), *v4 = (float4 *)(st + 56 * Q);
                const float4 pv = p4[q], mv = m4[q], vv = v4[q];
                const float4 np = make_float4(pv.x + av.x, pv.y + av.y, pv.z + av.z, pv.w + av.w);
                p4[q] = np;
                m4[q] = make_float4(mv.x + av.x, mv.y, mv.z, mv.w + __uint_as_float(gv.x));
                v4[q] = make_float4(vv.x, vv.y + av.y, vv.z, vv.w + __uint_as_float(gv.y));
                g4[q] = make_uint2((__float_as_uint(np.x) >> 16) | (__float_as_uint(np.y) & 0xffff0000u),
                                   (__float_as_uint(np.z) >> 16) | (__float_as_uint(np.w) & 0xffff0000u));
            } else {
                a4[q] = make_float4(av.x + __uint_as_float(gv.x << 16), av.y + __uint_as_float(gv.x & 0xffff0000u),
                                    av.z + __uint_as_float(gv.y << 16), av.w + __uint_as_float(gv.y & 0xffff0000u));
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        bar_arrive(&done[s]);
    }
}

std::mutex g_mu;
unsigned *g_ctr[64] = {};

int counter(int dev, unsigned **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev < 0 || dev >= 64) return -1;
    if (!g_ctr[dev]) {
        if (cudaMalloc(&g_ctr[dev], sizeof(unsigned)) != cudaSuccess ||
            cudaMemset(g_ctr[dev], 0, sizeof(unsigned)) != cudaSuccess) {
            cudaGetLastError();
            g_ctr[dev] = nullptr;
            return -5;
        }
    }
    *out = g_ctr[dev];
    return 0;
}

template <class K>
int grid_of(K kernel, int *grid) {
    int dev = 0, sms = 0, per = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, kT, 0) != cudaSuccess || per < 1) {
        cudaGetLastError();
        return -5;
    }
    *grid = sms * per;
    return 0;
}

// The bulk kernels' shared memory opt-in (set on every run: a run is long,
// and a context that replaced a reset one would not have it) and grid (one CTA
// per SM).
int bulk_setup(int dev, bool step, int *grid) {
    cudaError_t e = step ? cudaFuncSetAttribute(k_bulk_mix<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)(BulkMix<0>::stages * BulkMix<0>::stage_bytes))
                         : cudaFuncSetAttribute(k_bulk_mix<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)(BulkMix<1>::stages * BulkMix<1>::stage_bytes));
    int sms = 0;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms < 1) {
        cudaGetLastError();
        return -5;
    }
    *grid = sms;
    return 0;
}

bool mis16(const void *p) { return ((uintptr_t)p & 15u) != 0; }

}  // namespace

extern "C" int hbm_probe_sink_bytes(uint64_t *bytes) {
    if (!bytes) return -1;
    int grid = 0;
    int rc = grid_of(k_read<8>, &grid);
    if (rc) return rc;
    *bytes = (uint64_t)grid * 4u;
    return 0;
}

extern "C" int hbm_probe_run(int kind, void *const *buf, uint64_t n, int warmup, int reps, void *stream, float *ms,
                             double *bytes) {
    if (!buf || !ms || !bytes || n == 0 || n % kVecPerChunk != 0 || reps < 1 || warmup < 0) return -1;
    const int nbuf = kind == HBM_PROBE_COPY ? 2 : kind == HBM_PROBE_WRITE ? 1 : kind == HBM_PROBE_READ ? 2
                   : (kind == HBM_PROBE_STEP_MIX || kind == HBM_PROBE_BULK_STEP_MIX) ? 6
                   : (kind == HBM_PROBE_FIRST_MIX || kind == HBM_PROBE_ACC_MIX || kind == HBM_PROBE_BULK_ACC_MIX) ? 2
                   : 0;
    if (nbuf == 0) return -1;
    for (int i = 0; i < nbuf; ++i)
        if (!buf[i] || mis16(buf[i])) return -1;
    if (n / kVecPerChunk > 0xffffffffull) return -1;
    const uint32_t nch = (uint32_t)(n / kVecPerChunk);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -5;
    }
    unsigned *ctr = nullptr;
    int rc = counter(dev, &ctr);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    int grid = 0;
    double b = 0.0;
    void **dbufs = nullptr;     // the bulk kernels read the buffer table from device memory
    if (kind == HBM_PROBE_BULK_STEP_MIX || kind == HBM_PROBE_BULK_ACC_MIX) {
        const bool step = kind == HBM_PROBE_BULK_STEP_MIX;
        rc = bulk_setup(dev, step, &grid);
        if (rc) return rc;
        if (cudaMalloc(&dbufs, 6 * sizeof(void *)) != cudaSuccess ||
            cudaMemcpy(dbufs, buf, nbuf * sizeof(void *), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            if (dbufs) cudaFree(dbufs);
            return -5;
        }
    }
    const uint32_t ntiles_step = (uint32_t)(n / BulkMix<0>::Q), ntiles_acc = (uint32_t)(n / BulkMix<1>::Q);
    auto launch = [&]() {
        switch (kind) {
        case HBM_PROBE_COPY: k_copy<8><<<grid, kT, 0, st>>>((const float4 *)buf[0], (float4 *)buf[1], nch, ctr); break;
        case HBM_PROBE_WRITE: k_write<8><<<grid, kT, 0, st>>>((float4 *)buf[0], nch, ctr); break;
        case HBM_PROBE_READ: k_read<8><<<grid, kT, 0, st>>>((const uint4 *)buf[0], (uint32_t *)buf[1], nch, ctr); break;
        case HBM_PROBE_FIRST_MIX: k_acc_mix<false, 8><<<grid, kT, 0, st>>>((const uint2 *)buf[0], (float4 *)buf[1], nch, ctr); break;
        case HBM_PROBE_ACC_MIX: k_acc_mix<true, 8><<<grid, kT, 0, st>>>((const uint2 *)buf[0], (float4 *)buf[1], nch, ctr); break;
        case HBM_PROBE_BULK_STEP_MIX:
            k_bulk_mix<0><<<grid, kBulkThreads, BulkMix<0>::stages * BulkMix<0>::stage_bytes, st>>>(dbufs, ntiles_step, ctr);
            break;
        case HBM_PROBE_BULK_ACC_MIX:
            k_bulk_mix<1><<<grid, kBulkThreads, BulkMix<1>::stages * BulkMix<1>::stage_bytes, st>>>(dbufs, ntiles_acc, ctr);
            break;
        default:
            k_mix<4><<<grid, kT, 0, st>>>((const float4 *)buf[0], (const uint2 *)buf[1], (float4 *)buf[2],
                                         (float4 *)buf[3], (float4 *)buf[4], (uint2 *)buf[5], nch, ctr);
        }
    };
    switch (kind) {
    case HBM_PROBE_COPY: rc = grid_of(k_copy<8>, &grid); b = 32.0 * (double)n; break;
    case HBM_PROBE_WRITE: rc = grid_of(k_write<8>, &grid); b = 16.0 * (double)n; break;
    case HBM_PROBE_READ: rc = grid_of(k_read<8>, &grid); b = 16.0 * (double)n; break;
    case HBM_PROBE_FIRST_MIX: rc = grid_of(k_acc_mix<false, 8>, &grid); b = 24.0 * (double)n; break;   // 6 B x 4
    case HBM_PROBE_ACC_MIX: rc = grid_of(k_acc_mix<true, 8>, &grid); b = 40.0 * (double)n; break;      // 10 B x 4
    case HBM_PROBE_BULK_STEP_MIX: b = 128.0 * (double)n; break;     // grid: one CTA per SM (bulk_setup)
    case HBM_PROBE_BULK_ACC_MIX: b = 40.0 * (double)n; break;
    default: rc = grid_of(k_mix<4>, &grid); b = 128.0 * (double)n; break;   // 4 elements x 32 B per quad
    }
    if (rc) return rc;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e == cudaSuccess) {
        for (int i = 0; i < warmup; ++i) launch();
        e = cudaEventRecord(e0, st);
    }
    if (e == cudaSuccess) {
        for (int i = 0; i < reps; ++i) launch();
        e = cudaEventRecord(e1, st);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float t = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, e0, e1);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (dbufs) {
        // a wait that gave up makes the run an error (and is cleared)
        uint32_t to = 0, zero = 0;
        if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&to, g_bulk_timeouts, sizeof to);
        if (e == cudaSuccess && to) {
            cudaMemcpyToSymbol(g_bulk_timeouts, &zero, sizeof zero);
            e = cudaErrorLaunchTimeout;
        }
        cudaFree(dbufs);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return -5;
    }
    *ms = t / (float)reps;
    *bytes = b;
    return 0;
}

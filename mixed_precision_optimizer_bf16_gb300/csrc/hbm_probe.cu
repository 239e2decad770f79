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
                   : kind == HBM_PROBE_STEP_MIX ? 6 : (kind == HBM_PROBE_FIRST_MIX || kind == HBM_PROBE_ACC_MIX) ? 2 : 0;
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
    auto launch = [&]() {
        switch (kind) {
        case HBM_PROBE_COPY: k_copy<8><<<grid, kT, 0, st>>>((const float4 *)buf[0], (float4 *)buf[1], nch, ctr); break;
        case HBM_PROBE_WRITE: k_write<8><<<grid, kT, 0, st>>>((float4 *)buf[0], nch, ctr); break;
        case HBM_PROBE_READ: k_read<8><<<grid, kT, 0, st>>>((const uint4 *)buf[0], (uint32_t *)buf[1], nch, ctr); break;
        case HBM_PROBE_FIRST_MIX: k_acc_mix<false, 8><<<grid, kT, 0, st>>>((const uint2 *)buf[0], (float4 *)buf[1], nch, ctr); break;
        case HBM_PROBE_ACC_MIX: k_acc_mix<true, 8><<<grid, kT, 0, st>>>((const uint2 *)buf[0], (float4 *)buf[1], nch, ctr); break;
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
    if (e != cudaSuccess) {
        cudaGetLastError();
        return -5;
    }
    *ms = t / (float)reps;
    *bytes = b;
    return 0;
}

// synth_gpu.cu -- device fill kernels over synth.h (harness only).
//
// Builds libsynth_gpu.so, which the tests and the benchmark use to write a
// workload's seeded gradients and initial masters straight into device
// memory.  Same functions as the host library (integer hashing, one IEEE
// double multiply, one double->float conversion), so the values are the
// same bits the host generator -- and hence the CPU oracle -- produces.
// None of the optimizer's arithmetic is here.
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth.h"

namespace {

constexpr int kT = 256;

__global__ void fill_grad_kernel(uint16_t *out, uint64_t n, uint64_t first, uint64_t key, double scale,
                                 uint64_t zero_key, uint64_t zero_thresh) {
    for (uint64_t j = blockIdx.x * (uint64_t)kT + threadIdx.x; j < n; j += (uint64_t)gridDim.x * kT)
        out[j] = synth_grad_bf16(key, first + j, scale, zero_key, zero_thresh);
}

__global__ void fill_normal_kernel(float *out, uint64_t n, uint64_t first, uint64_t key, double scale) {
    for (uint64_t j = blockIdx.x * (uint64_t)kT + threadIdx.x; j < n; j += (uint64_t)gridDim.x * kT)
        out[j] = synth_normal_f32(key, first + j, scale);
}

__global__ void fill_loguniform_kernel(float *out, uint64_t n, uint64_t first, uint64_t key, int e_lo, int e_hi) {
    for (uint64_t j = blockIdx.x * (uint64_t)kT + threadIdx.x; j < n; j += (uint64_t)gridDim.x * kT)
        out[j] = synth_loguniform_f32(key, first + j, e_lo, e_hi);
}

int grid(uint64_t n) {
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    uint64_t g = (n + kT - 1) / kT, cap = (uint64_t)sms * 8;
    return (int)(g < cap ? (g ? g : 1) : cap);
}

int status() { return cudaGetLastError() == cudaSuccess ? 0 : -1; }

}  // namespace

extern "C" {

int synth_gpu_fill_grad_bf16(uint16_t *out, uint64_t n, uint64_t first, uint64_t key, double scale,
                             uint64_t zero_key, uint64_t zero_thresh, void *stream) {
    if (n == 0) return 0;
    fill_grad_kernel<<<grid(n), kT, 0, (cudaStream_t)stream>>>(out, n, first, key, scale, zero_key, zero_thresh);
    return status();
}

int synth_gpu_fill_normal_f32(float *out, uint64_t n, uint64_t first, uint64_t key, double scale, void *stream) {
    if (n == 0) return 0;
    fill_normal_kernel<<<grid(n), kT, 0, (cudaStream_t)stream>>>(out, n, first, key, scale);
    return status();
}

int synth_gpu_fill_loguniform_f32(float *out, uint64_t n, uint64_t first, uint64_t key, int e_lo, int e_hi,
                                  void *stream) {
    if (n == 0) return 0;
    fill_loguniform_kernel<<<grid(n), kT, 0, (cudaStream_t)stream>>>(out, n, first, key, e_lo, e_hi);
    return status();
}

}  // extern "C"

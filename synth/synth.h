/*
 * synth.h -- seeded, counter-based synthetic inputs for the BF16 optimizer step.
 *
 * Harness code, not part of the optimizer: it turns (stream key, element index)
 * into the bit patterns of micro-batch gradients and initial master weights.
 * It holds none of the optimizer's arithmetic (no accumulation, no norm, no
 * AdamW, no round-to-nearest bf16 cast): every value is built from integers,
 * one IEEE double multiply and one double->float conversion, so the host and
 * any other consumer get bit-identical inputs.
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  Output i of the stream
 * keyed by K is mix64(K + (i+1)*gamma), so any element can be produced on its
 * own, in any order, by any thread.
 *
 * "~N(0, sigma)" values are Irwin-Hall sums of four 16-bit uniforms, centred
 * and scaled to standard deviation sigma (support +-3.46 sigma).
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stdint.h>
#include <string.h>

#ifdef __CUDACC__
#define SYNTH_HD __host__ __device__
#else
#define SYNTH_HD
#endif

#define SYNTH_GAMMA 0x9e3779b97f4a7c15ULL

/* Buffer kinds of a stream key. */
enum { SYNTH_KIND_GRAD = 1, SYNTH_KIND_MASTER = 2, SYNTH_KIND_ZERO_MASK = 3 };

static inline SYNTH_HD uint64_t synth_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

/* The i-th 64-bit output of the stream keyed by `key`. */
static inline SYNTH_HD uint64_t synth_bits(uint64_t key, uint64_t i) {
    return synth_mix64(key + (i + 1) * SYNTH_GAMMA);
}

/* Stream key of one buffer: (seed, workload id, kind, step, micro-batch). */
static inline SYNTH_HD uint64_t synth_key(uint64_t seed, uint32_t workload, uint32_t kind,
                                 uint32_t step, uint32_t micro) {
    uint64_t k = synth_mix64(seed + SYNTH_GAMMA);
    k = synth_mix64(k ^ ((uint64_t)workload << 32 | kind));
    k = synth_mix64(k ^ ((uint64_t)step << 32 | micro));
    return k;
}

/* Irwin-Hall(4) integer in [-131070, 131070], mean 0. */
static inline SYNTH_HD int32_t synth_ih4(uint64_t h) {
    int32_t s = (int32_t)(h & 0xffff) + (int32_t)((h >> 16) & 0xffff) +
                (int32_t)((h >> 32) & 0xffff) + (int32_t)(h >> 48);
    return s - 131070;
}

/* Standard deviation of synth_ih4: sqrt(4 * (65536^2 - 1) / 12). */
#define SYNTH_IH4_STD 37837.227237206484

/* Multiplier that maps synth_ih4 to standard deviation sigma. */
static inline double synth_scale_for_sigma(double sigma) { return sigma / SYNTH_IH4_STD; }

static inline SYNTH_HD uint32_t synth_f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static inline SYNTH_HD float synth_bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* ~N(0, sigma) FP32 value: (float)(ih4 * scale), scale = synth_scale_for_sigma(sigma). */
static inline SYNTH_HD float synth_normal_f32(uint64_t key, uint64_t i, double scale) {
    return (float)((double)synth_ih4(synth_bits(key, i)) * scale);
}

/* ~N(0, sigma) bf16 bit pattern: the FP32 value above with its low 16 bits
 * dropped (truncation toward zero, a property of this generator only).
 * If zero_thresh != 0, element i is exactly +0 whenever
 * synth_bits(zero_key, i) < zero_thresh (zero_thresh = frac * 2^64), i.e. the
 * same positions are zero in every stream that shares zero_key. */
static inline SYNTH_HD uint16_t synth_grad_bf16(uint64_t key, uint64_t i, double scale,
                                       uint64_t zero_key, uint64_t zero_thresh) {
    if (zero_thresh != 0 && synth_bits(zero_key, i) < zero_thresh) return 0;
    return (uint16_t)(synth_f32_bits(synth_normal_f32(key, i, scale)) >> 16);
}

/* Log-uniform over binary octaves with random sign: |x| = (1 + f) * 2^e with
 * e uniform in [e_lo, e_hi] and f a uniform 23-bit fraction, built directly
 * as an FP32 bit pattern.  e in [-26, 9] spans [1.49e-8, 1024). */
static inline SYNTH_HD float synth_loguniform_f32(uint64_t key, uint64_t i, int e_lo, int e_hi) {
    uint64_t h = synth_bits(key, i);
    uint32_t n_oct = (uint32_t)(e_hi - e_lo + 1);
    uint32_t e = (uint32_t)((((h >> 32) & 0xffffffffULL) * n_oct) >> 32);   /* [0, n_oct) */
    uint32_t sign = (uint32_t)(h >> 31) & 1u;
    uint32_t frac = (uint32_t)h & 0x7fffffu;
    uint32_t bits = (sign << 31) | ((uint32_t)(e_lo + 127 + (int)e) << 23) | frac;
    return synth_bits_f32(bits);
}

#endif /* SYNTH_H */

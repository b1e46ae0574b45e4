/*
 * synth.h -- seeded, counter-based synthetic input generator.
 *
 * This module produces the inputs (activations, history K/V, positions,
 * slot choices) that both the CPU oracle and the CUDA path consume.  It holds
 * none of the attention method's arithmetic: only hashing and the mapping of
 * hash bits to numbers.
 *
 * Every value is a pure function of (seed, stream, index), so any element of
 * any tensor can be regenerated on its own, on the host or on the device,
 * with bit-identical results:
 *
 *   key(seed, stream)  = mix64(seed XOR mix64(stream + GOLDEN))
 *   bits(key, index)   = mix64(key + (index + 1) * GOLDEN)
 *
 * mix64 is the SplitMix64 output finaliser (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014; the
 * constants are the ones Vigna published for splitmix64.c).
 *
 * Standard-normal stand-in: the Irwin-Hall sum of the four 16-bit fields of
 * one 64-bit draw, centred and scaled to unit variance.  The centred sum is an
 * integer of magnitude <= 131070 (exact in f32) and the scale is one
 * correctly rounded f32 multiply, so host and device agree bit for bit.
 * Its support is [-3.464, 3.464]; mean 0, variance 1.
 *
 * Integer draws (positions, permutations, subsets) take the top 32 bits and
 * map them to [0, n) by a 32x32->64 multiply-high (Lemire's method without
 * the rejection step; the bias is below n / 2^32).
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stdint.h>

#ifdef __CUDACC__
#define SYNTH_FN __host__ __device__ static inline
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL
/* 1 / sqrt((65536^2 - 1) / 3) rounded to f32 */
#define SYNTH_NORMAL_SCALE 0x1.bb67aep-16f

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

SYNTH_FN uint64_t synth_key(uint64_t seed, uint64_t stream) {
    return synth_mix64(seed ^ synth_mix64(stream + SYNTH_GOLDEN));
}

SYNTH_FN uint64_t synth_bits(uint64_t key, uint64_t index) {
    return synth_mix64(key + (index + 1ULL) * SYNTH_GOLDEN);
}

SYNTH_FN float synth_normal_from_bits(uint64_t h) {
    int32_t s = (int32_t)(h & 0xFFFFu) + (int32_t)((h >> 16) & 0xFFFFu) +
                (int32_t)((h >> 32) & 0xFFFFu) + (int32_t)((h >> 48) & 0xFFFFu) -
                131070;
#ifdef __CUDA_ARCH__
    return __fmul_rn((float)s, SYNTH_NORMAL_SCALE);
#else
    return (float)s * SYNTH_NORMAL_SCALE;
#endif
}

SYNTH_FN float synth_normal(uint64_t key, uint64_t index) {
    return synth_normal_from_bits(synth_bits(key, index));
}

/* uniform integer in [0, n), n >= 1 */
SYNTH_FN uint32_t synth_below(uint64_t key, uint64_t index, uint32_t n) {
    uint64_t hi = synth_bits(key, index) >> 32;
    return (uint32_t)((hi * (uint64_t)n) >> 32);
}

/* Stream ids of the tensors a workload draws.  A multi-step workload offsets
 * the per-step activations by SYNTH_STEP_STRIDE * step. */
enum {
    SYNTH_S_HIST_K = 1,
    SYNTH_S_HIST_V = 2,
    SYNTH_S_Q = 3,
    SYNTH_S_KNEW = 4,
    SYNTH_S_VNEW = 5,
    SYNTH_S_QNORM_W = 6,
    SYNTH_S_KNORM_W = 7,
    SYNTH_S_SINKS = 8,
    SYNTH_S_POS = 9,
    SYNTH_S_SLOTS = 10,
    SYNTH_STEP_STRIDE = 16
};

#endif /* SYNTH_H */

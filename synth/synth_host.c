/*
 * synth_host.c -- host side of the synthetic input generator (see synth.h).
 *
 * Exports plain C functions that fill caller-owned host arrays.  Built with
 * -ffp-contract=off so that the affine map mean + sd * x is two separately
 * rounded f32 operations on every host architecture.
 */
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>

#include "synth.h"

typedef struct {
    float* dst;
    uint64_t begin, end, key, index0;
    float mean, sd;
    int affine;
} fill_job;

static void* fill_worker(void* arg) {
    fill_job* j = (fill_job*)arg;
    for (uint64_t i = j->begin; i < j->end; ++i) {
        float x = synth_normal(j->key, j->index0 + i);
        if (j->affine) {
            float t = x * j->sd;
            x = t + j->mean;
        }
        j->dst[i] = x;
    }
    return NULL;
}

static int fill_any(float* dst, uint64_t count, uint64_t seed, uint64_t stream,
                    uint64_t index0, float mean, float sd, int affine, int n_threads) {
    if (!dst && count) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 64) n_threads = 64;
    if (count < (1u << 20)) n_threads = 1;
    uint64_t key = synth_key(seed, stream);
    fill_job jobs[64];
    pthread_t tids[64];
    int started[64] = {0};
    uint64_t per = (count + (uint64_t)n_threads - 1) / (uint64_t)n_threads;
    for (int t = 0; t < n_threads; ++t) {
        uint64_t b = per * (uint64_t)t, e = b + per;
        if (b > count) b = count;
        if (e > count) e = count;
        fill_job j = {dst, b, e, key, index0, mean, sd, affine};
        jobs[t] = j;
    }
    for (int t = 1; t < n_threads; ++t)
        started[t] = pthread_create(&tids[t], NULL, fill_worker, &jobs[t]) == 0;
    fill_worker(&jobs[0]);
    for (int t = 1; t < n_threads; ++t) {
        if (started[t])
            pthread_join(tids[t], NULL);
        else
            fill_worker(&jobs[t]);
    }
    return 0;
}

/* dst[i] = N01(seed, stream, index0 + i) for i in [0, count) */
int synth_fill_normal(float* dst, uint64_t count, uint64_t seed, uint64_t stream,
                      uint64_t index0, int n_threads) {
    return fill_any(dst, count, seed, stream, index0, 0.f, 1.f, 0, n_threads);
}

/* dst[i] = mean + sd * N01(seed, stream, index0 + i), two rounded f32 ops */
int synth_fill_normal_affine(float* dst, uint64_t count, uint64_t seed,
                             uint64_t stream, uint64_t index0, float mean, float sd,
                             int n_threads) {
    return fill_any(dst, count, seed, stream, index0, mean, sd, 1, n_threads);
}

/* dst[i] = uniform integer in [0, n) drawn at index i */
int synth_fill_below(uint32_t* dst, uint64_t count, uint64_t seed, uint64_t stream,
                     uint32_t n) {
    if (n == 0 || (!dst && count)) return -1;
    uint64_t key = synth_key(seed, stream);
    for (uint64_t i = 0; i < count; ++i) dst[i] = synth_below(key, i, n);
    return 0;
}

/* First k entries of a Fisher-Yates shuffle of 0..n-1 (k <= n).  Draw i of
 * the shuffle (swap position n-1-i) uses index i. */
int synth_subset(uint32_t* dst, uint32_t n, uint32_t k, uint64_t seed, uint64_t stream,
                 uint32_t* scratch_n) {
    if (k > n || !scratch_n || (!dst && k)) return -1;
    uint64_t key = synth_key(seed, stream);
    for (uint32_t i = 0; i < n; ++i) scratch_n[i] = i;
    for (uint32_t i = 0; n > 1 && i < n - 1; ++i) {
        uint32_t top = n - 1 - i;
        uint32_t j = synth_below(key, i, top + 1);
        uint32_t t = scratch_n[top];
        scratch_n[top] = scratch_n[j];
        scratch_n[j] = t;
    }
    for (uint32_t i = 0; i < k; ++i) dst[i] = scratch_n[i];
    return 0;
}

uint64_t synth_key_of(uint64_t seed, uint64_t stream) { return synth_key(seed, stream); }

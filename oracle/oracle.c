/*
 * oracle.c -- CPU oracle for batched slot-KV decode attention.
 *
 * TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's
 * CPU-baseline arm use it.  It is a plain, slow, direct statement of what one
 * batched decode step computes, written from the zinc engine's API pages:
 *
 *   "Forward Cuda Gemma", decodeBatch: B independent sequences each advance
 *   by one token; per row, per-head Q/K norm, RoPE, KV write, then a causal
 *   softmax over slot slots[b]'s history [0..positions[b]] only.  The slot
 *   must already hold [0..pos-1]; the step writes the row's new K/V at pos.
 *
 *   "Forward Cuda Gemma", slotKvOffsetBytes (and "Forward Cuda", the slot KV
 *   offset): byte offset (slot*slot_ctx + pos)*kv_dim*sizeof(f32).
 *
 *   "Forward Cuda", init: inv_freq and the attention sinks are uploaded to the
 *   device, so both are inputs here.
 *
 * Readings where the pages are silent (each listed with its reason in the
 * design notes): RMS norm is x / sqrt(mean(x^2) + eps) * w with one weight
 * vector per head dimension; RoPE rotates the half-split pairs (i, i + hd/2)
 * by the f32 angle fl32((float)pos * inv_freq[i]); the cache holds the normed
 * and rotated K and the raw V; the history range is inclusive of pos; a sink
 * is one unscaled logit per query head that joins the max and the
 * denominator and carries no value; query head h reads kv head h / (n_head /
 * n_kv_head).
 *
 * Options (oracle_decode_batch_opts), from the per-head "V/Q/K norm" of the
 * Gemma path on the same page: ORACLE_VNORM caches and attends the
 * weightless RMS norm of v_new instead of v_new; ORACLE_NORM_PLUS_ONE applies
 * the Q and K norm weights as (1 + w).
 *
 * Build with -ffp-contract=off: the one f32 product (the RoPE angle) must be
 * a single rounded multiply.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

uint64_t oracle_slot_kv_offset_bytes(uint32_t slot, uint32_t pos, uint32_t slot_ctx,
                                     uint32_t kv_dim) {
    return ((uint64_t)slot * slot_ctx + pos) * (uint64_t)kv_dim * sizeof(float);
}

/* y = x / sqrt(mean(x^2) + eps) * w, in f64 */
static void rms_norm(const float* x, const float* w, uint32_t n, double eps, double* y) {
    double sum_sq = 0.0;
    for (uint32_t i = 0; i < n; ++i) sum_sq += (double)x[i] * (double)x[i];
    double inv_rms = 1.0 / sqrt(sum_sq / (double)n + eps);
    for (uint32_t i = 0; i < n; ++i) y[i] = (double)x[i] * inv_rms * (double)w[i];
}

/* Gemma's forms: the weight applied as (1 + w), or no weight at all (w NULL) */
static void rms_norm_gemma(const float* x, const float* w, uint32_t n, double eps, double* y) {
    double sum_sq = 0.0;
    for (uint32_t i = 0; i < n; ++i) sum_sq += (double)x[i] * (double)x[i];
    double inv_rms = 1.0 / sqrt(sum_sq / (double)n + eps);
    for (uint32_t i = 0; i < n; ++i)
        y[i] = (double)x[i] * inv_rms * (w ? 1.0 + (double)w[i] : 1.0);
}

/* Rotate pairs (i, i + hd/2) by angle fl32(pos * inv_freq[i]). */
static void rope(double* y, uint32_t hd, uint32_t pos, const float* inv_freq) {
    uint32_t half = hd / 2;
    for (uint32_t i = 0; i < half; ++i) {
        float angle_f32 = (float)pos * inv_freq[i];
        double c = cos((double)angle_f32);
        double s = sin((double)angle_f32);
        double x0 = y[i];
        double x1 = y[i + half];
        y[i] = x0 * c - x1 * s;
        y[i + half] = x1 * c + x0 * s;
    }
}

void oracle_norm_rope_head(const float* x, const float* w, uint32_t hd, float eps,
                           uint32_t pos, const float* inv_freq, double* y) {
    rms_norm(x, w, hd, (double)eps, y);
    rope(y, hd, pos, inv_freq);
}

typedef struct {
    uint32_t n_slots, slot_ctx, n_head, n_kv_head, hd, B;
    const float *q, *k_new, *v_new;
    const uint32_t *positions, *slots;
    const float *q_norm_w, *k_norm_w, *inv_freq, *sinks;
    float eps, scale;
    uint32_t flags;
    float *K, *V, *out;
    double* out64;
    uint32_t row_begin, row_end;
    int skipped;
} batch_job;

/* One row of the step: write its new K/V, then attend for every query head. */
static void decode_row(batch_job* j, uint32_t b, double* qv, double* kv, double* score,
                       double* acc) {
    const uint32_t hd = j->hd;
    const uint32_t kv_dim = j->n_kv_head * hd;
    const uint32_t group = j->n_head / j->n_kv_head;
    const uint32_t p = j->positions[b];
    const uint32_t slot = j->slots[b];
    if (slot >= j->n_slots || p >= j->slot_ctx) {
        j->skipped += 1;
        return;
    }
    /* element offset of (slot, pos) in the slot buffers */
    const uint64_t row0 = (uint64_t)slot * j->slot_ctx * kv_dim;
    const uint64_t at_p = row0 + (uint64_t)p * kv_dim;

    /* KV write: the cache holds the normed, rotated K (rounded to f32) and the raw V */
    for (uint32_t g = 0; g < j->n_kv_head; ++g) {
        const float* k_in = j->k_new + ((uint64_t)b * j->n_kv_head + g) * hd;
        const float* v_in = j->v_new + ((uint64_t)b * j->n_kv_head + g) * hd;
        if (j->flags & ORACLE_NORM_PLUS_ONE) {
            rms_norm_gemma(k_in, j->k_norm_w, hd, (double)j->eps, kv);
            rope(kv, hd, p, j->inv_freq);
        } else {
            oracle_norm_rope_head(k_in, j->k_norm_w, hd, j->eps, p, j->inv_freq, kv);
        }
        for (uint32_t i = 0; i < hd; ++i) j->K[at_p + (uint64_t)g * hd + i] = (float)kv[i];
        if (j->flags & ORACLE_VNORM) {
            /* the cached V is the weightless RMS norm of v_new */
            rms_norm_gemma(v_in, NULL, hd, (double)j->eps, kv);
            for (uint32_t i = 0; i < hd; ++i) j->V[at_p + (uint64_t)g * hd + i] = (float)kv[i];
        } else {
            for (uint32_t i = 0; i < hd; ++i) j->V[at_p + (uint64_t)g * hd + i] = v_in[i];
        }
    }

    /* causal softmax over keys 0..p of this slot, one query head at a time */
    for (uint32_t h = 0; h < j->n_head; ++h) {
        const uint32_t g = h / group;
        const float* q_in = j->q + ((uint64_t)b * j->n_head + h) * hd;
        if (j->flags & ORACLE_NORM_PLUS_ONE) {
            rms_norm_gemma(q_in, j->q_norm_w, hd, (double)j->eps, qv);
            rope(qv, hd, p, j->inv_freq);
        } else {
            oracle_norm_rope_head(q_in, j->q_norm_w, hd, j->eps, p, j->inv_freq, qv);
        }

        double m = -INFINITY;
        for (uint32_t t = 0; t <= p; ++t) {
            const float* k_row = j->K + row0 + (uint64_t)t * kv_dim + (uint64_t)g * hd;
            double dot = 0.0;
            for (uint32_t i = 0; i < hd; ++i) dot += qv[i] * (double)k_row[i];
            score[t] = (double)j->scale * dot;
            if (score[t] > m) m = score[t];
        }
        double sink = 0.0;
        if (j->sinks) {
            sink = (double)j->sinks[h];
            if (sink > m) m = sink;
        }
        /* weights e^(s_t - m) and their sum, plus the sink's share of the denominator */
        double denom = 0.0;
        for (uint32_t t = 0; t <= p; ++t) {
            score[t] = exp(score[t] - m);
            denom += score[t];
        }
        if (j->sinks) denom += exp(sink - m);

        for (uint32_t i = 0; i < hd; ++i) acc[i] = 0.0;
        for (uint32_t t = 0; t <= p; ++t) {
            const float* v_row = j->V + row0 + (uint64_t)t * kv_dim + (uint64_t)g * hd;
            for (uint32_t i = 0; i < hd; ++i) acc[i] += score[t] * (double)v_row[i];
        }
        for (uint32_t i = 0; i < hd; ++i) {
            double o = acc[i] / denom;
            uint64_t oi = ((uint64_t)b * j->n_head + h) * hd + i;
            j->out[oi] = (float)o;
            if (j->out64) j->out64[oi] = o;
        }
    }
}

static void* batch_worker(void* arg) {
    batch_job* j = (batch_job*)arg;
    double* qv = (double*)malloc(sizeof(double) * j->hd);
    double* kv = (double*)malloc(sizeof(double) * j->hd);
    double* score = (double*)malloc(sizeof(double) * j->slot_ctx);
    double* acc = (double*)malloc(sizeof(double) * j->hd);
    if (!qv || !kv || !score || !acc) {
        j->skipped = -1;
    } else {
        for (uint32_t b = j->row_begin; b < j->row_end; ++b)
            decode_row(j, b, qv, kv, score, acc);
    }
    free(acc);
    free(qv);
    free(kv);
    free(score);
    return NULL;
}

int oracle_decode_batch(uint32_t n_slots, uint32_t slot_ctx, uint32_t n_head,
                        uint32_t n_kv_head, uint32_t head_dim, uint32_t B,
                        const float* q, const float* k_new, const float* v_new,
                        const uint32_t* positions, const uint32_t* slots,
                        const float* q_norm_w, const float* k_norm_w,
                        const float* inv_freq, const float* sinks, float eps,
                        float scale, float* K, float* V, float* out, double* out64,
                        int n_threads) {
    return oracle_decode_batch_opts(n_slots, slot_ctx, n_head, n_kv_head, head_dim, B, q,
                                    k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                                    inv_freq, sinks, eps, scale, 0u, K, V, out, out64,
                                    n_threads);
}

int oracle_decode_batch_opts(uint32_t n_slots, uint32_t slot_ctx, uint32_t n_head,
                             uint32_t n_kv_head, uint32_t head_dim, uint32_t B,
                             const float* q, const float* k_new, const float* v_new,
                             const uint32_t* positions, const uint32_t* slots,
                             const float* q_norm_w, const float* k_norm_w,
                             const float* inv_freq, const float* sinks, float eps,
                             float scale, uint32_t flags, float* K, float* V, float* out,
                             double* out64, int n_threads) {
    if (B == 0) return 0;
    if (!q || !k_new || !v_new || !positions || !slots || !q_norm_w || !k_norm_w ||
        !inv_freq || !K || !V || !out)
        return -1;
    if (n_kv_head == 0 || n_head % n_kv_head != 0 || head_dim == 0 || head_dim % 2 != 0)
        return -1;
    if (n_threads < 1) n_threads = 1;
    if ((uint32_t)n_threads > B) n_threads = (int)B;
    if (n_threads > 256) n_threads = 256;

    batch_job* jobs = (batch_job*)calloc((size_t)n_threads, sizeof(batch_job));
    pthread_t* tids = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
    int* started = (int*)calloc((size_t)n_threads, sizeof(int));
    if (!jobs || !tids || !started) {
        free(jobs);
        free(tids);
        free(started);
        return -1;
    }
    uint32_t per = (B + (uint32_t)n_threads - 1) / (uint32_t)n_threads;
    for (int t = 0; t < n_threads; ++t) {
        batch_job* j = &jobs[t];
        j->n_slots = n_slots;
        j->slot_ctx = slot_ctx;
        j->n_head = n_head;
        j->n_kv_head = n_kv_head;
        j->hd = head_dim;
        j->B = B;
        j->q = q;
        j->k_new = k_new;
        j->v_new = v_new;
        j->positions = positions;
        j->slots = slots;
        j->q_norm_w = q_norm_w;
        j->k_norm_w = k_norm_w;
        j->inv_freq = inv_freq;
        j->sinks = sinks;
        j->eps = eps;
        j->scale = scale;
        j->flags = flags;
        j->K = K;
        j->V = V;
        j->out = out;
        j->out64 = out64;
        j->row_begin = per * (uint32_t)t < B ? per * (uint32_t)t : B;
        j->row_end = per * (uint32_t)(t + 1) < B ? per * (uint32_t)(t + 1) : B;
    }
    for (int t = 1; t < n_threads; ++t)
        started[t] = pthread_create(&tids[t], NULL, batch_worker, &jobs[t]) == 0;
    batch_worker(&jobs[0]);
    int skipped = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (t > 0) {
            if (started[t])
                pthread_join(tids[t], NULL);
            else
                batch_worker(&jobs[t]);
        }
        if (jobs[t].skipped < 0) skipped = -1;
        if (skipped >= 0) skipped += jobs[t].skipped;
    }
    free(jobs);
    free(tids);
    free(started);
    return skipped;
}

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
 * Paged mode (oracle_decode_batch_paged): the buffers are a pool of n_slots
 * blocks of slot_ctx positions, and row b's key t lives in block
 * block_tables[b][t / slot_ctx] at offset t % slot_ctx (the paged KV cache
 * with per-sequence block tables of the Qwen3SsmLayer page,
 * decode_multi_seq).
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
    const uint32_t* block_tables; /* paged mode: [B][bt_stride] block ids, else NULL */
    uint32_t bt_stride;
    float *K, *V, *out;
    double* out64;
    uint32_t row_begin, row_end;
    int skipped;
} batch_job;

/* Element offset of key (position) t of row b in the K/V buffers.  Slot
 * mode: (slot * slot_ctx + t) * kv_dim.  Paged mode, where the buffers are
 * n_slots blocks of slot_ctx positions: block block_tables[b][t / slot_ctx],
 * offset t % slot_ctx within it. */
static uint64_t key_offset(const batch_job* j, uint32_t b, uint32_t t) {
    const uint64_t kv_dim = (uint64_t)j->n_kv_head * j->hd;
    if (j->block_tables) {
        const uint32_t blk = j->block_tables[(uint64_t)b * j->bt_stride + t / j->slot_ctx];
        return ((uint64_t)blk * j->slot_ctx + t % j->slot_ctx) * kv_dim;
    }
    return ((uint64_t)j->slots[b] * j->slot_ctx + t) * kv_dim;
}

/* Does row b satisfy the precondition (its keys 0..p all addressable)? */
static int row_in_range(const batch_job* j, uint32_t b) {
    const uint32_t p = j->positions[b];
    if (!j->block_tables) return j->slots[b] < j->n_slots && p < j->slot_ctx;
    if ((uint64_t)p >= (uint64_t)j->bt_stride * j->slot_ctx) return 0;
    for (uint32_t i = 0; i <= p / j->slot_ctx; ++i)
        if (j->block_tables[(uint64_t)b * j->bt_stride + i] >= j->n_slots) return 0;
    return 1;
}

/* One row of the step: write its new K/V, then attend for every query head. */
static void decode_row(batch_job* j, uint32_t b, double* qv, double* kv, double* score,
                       double* acc) {
    const uint32_t hd = j->hd;
    const uint32_t group = j->n_head / j->n_kv_head;
    const uint32_t p = j->positions[b];
    if (!row_in_range(j, b)) {
        j->skipped += 1;
        return;
    }
    const uint64_t at_p = key_offset(j, b, p);

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
            const float* k_row = j->K + key_offset(j, b, t) + (uint64_t)g * hd;
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
            const float* v_row = j->V + key_offset(j, b, t) + (uint64_t)g * hd;
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
    /* a row attends over at most slot_ctx keys (slot mode) or the span of
     * its block table (paged mode) */
    const uint64_t max_keys =
        j->block_tables ? (uint64_t)j->bt_stride * j->slot_ctx : (uint64_t)j->slot_ctx;
    double* score = (double*)malloc(sizeof(double) * max_keys);
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

static int run_batch(batch_job* proto, int n_threads);

int oracle_decode_batch_paged(uint32_t n_blocks, uint32_t block_size, uint32_t n_head,
                              uint32_t n_kv_head, uint32_t head_dim, uint32_t B,
                              const float* q, const float* k_new, const float* v_new,
                              const uint32_t* positions, const uint32_t* block_tables,
                              uint32_t bt_stride, const float* q_norm_w,
                              const float* k_norm_w, const float* inv_freq,
                              const float* sinks, float eps, float scale, uint32_t flags,
                              float* K, float* V, float* out, double* out64, int n_threads) {
    if (B == 0) return 0;
    if (!block_tables || bt_stride == 0 || block_size == 0) return -1;
    batch_job proto;
    memset(&proto, 0, sizeof(proto));
    proto.n_slots = n_blocks;
    proto.slot_ctx = block_size;
    proto.n_head = n_head;
    proto.n_kv_head = n_kv_head;
    proto.hd = head_dim;
    proto.B = B;
    proto.q = q;
    proto.k_new = k_new;
    proto.v_new = v_new;
    proto.positions = positions;
    proto.slots = NULL;
    proto.block_tables = block_tables;
    proto.bt_stride = bt_stride;
    proto.q_norm_w = q_norm_w;
    proto.k_norm_w = k_norm_w;
    proto.inv_freq = inv_freq;
    proto.sinks = sinks;
    proto.eps = eps;
    proto.scale = scale;
    proto.flags = flags;
    proto.K = K;
    proto.V = V;
    proto.out = out;
    proto.out64 = out64;
    return run_batch(&proto, n_threads);
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
    if (!slots) return -1;
    batch_job proto;
    memset(&proto, 0, sizeof(proto));
    proto.n_slots = n_slots;
    proto.slot_ctx = slot_ctx;
    proto.n_head = n_head;
    proto.n_kv_head = n_kv_head;
    proto.hd = head_dim;
    proto.B = B;
    proto.q = q;
    proto.k_new = k_new;
    proto.v_new = v_new;
    proto.positions = positions;
    proto.slots = slots;
    proto.block_tables = NULL;
    proto.q_norm_w = q_norm_w;
    proto.k_norm_w = k_norm_w;
    proto.inv_freq = inv_freq;
    proto.sinks = sinks;
    proto.eps = eps;
    proto.scale = scale;
    proto.flags = flags;
    proto.K = K;
    proto.V = V;
    proto.out = out;
    proto.out64 = out64;
    return run_batch(&proto, n_threads);
}

/* Rows split over threads (rows touch disjoint slots or blocks). */
static int run_batch(batch_job* proto, int n_threads) {
    const uint32_t B = proto->B;
    if (!proto->q || !proto->k_new || !proto->v_new || !proto->positions ||
        !proto->q_norm_w || !proto->k_norm_w || !proto->inv_freq || !proto->K || !proto->V ||
        !proto->out)
        return -1;
    if (proto->n_kv_head == 0 || proto->n_head % proto->n_kv_head != 0 || proto->hd == 0 ||
        proto->hd % 2 != 0)
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
        jobs[t] = *proto;
        jobs[t].row_begin = per * (uint32_t)t < B ? per * (uint32_t)t : B;
        jobs[t].row_end = per * (uint32_t)(t + 1) < B ? per * (uint32_t)(t + 1) : B;
        jobs[t].skipped = 0;
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

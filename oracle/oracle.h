/*
 * oracle.h -- CPU oracle for batched slot-KV decode attention.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline arm may load this.  It shares no code with the
 * CUDA library: it includes nothing from it and it is built separately.
 *
 * Everything is computed in f64 from f32 inputs; results that the method
 * stores in f32 (the written K, the output) are rounded once at the end.
 *
 * Parity status: every function below is pinned by the not-gpu tests
 * (closed forms, invariants, brute force on tiny cases, planted mutants).
 */
#ifndef SLOTKV_ORACLE_H
#define SLOTKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Byte offset of (slot, pos) in one layer's slot K (or V) buffer. */
uint64_t oracle_slot_kv_offset_bytes(uint32_t slot, uint32_t pos, uint32_t slot_ctx,
                                     uint32_t kv_dim);

/* Per-head RMS norm followed by RoPE at `pos`, for one head vector x[hd].
 * y[hd] receives the f64 result (not rounded). */
void oracle_norm_rope_head(const float* x, const float* w, uint32_t hd, float eps,
                           uint32_t pos, const float* inv_freq, double* y);

/* One batched decode step over slot KV (see oracle.c for the definition).
 * K and V are the host copies of the slot buffers, f32[n_slots][slot_ctx][kv_dim],
 * and are updated in place.  out is f32[B][n_head][hd]; out64 (may be NULL)
 * receives the unrounded f64 output.  sinks may be NULL.
 * Returns the number of rows skipped for an out-of-range slot or position,
 * or -1 on an argument error. */
int oracle_decode_batch(uint32_t n_slots, uint32_t slot_ctx, uint32_t n_head,
                        uint32_t n_kv_head, uint32_t head_dim, uint32_t B,
                        const float* q, const float* k_new, const float* v_new,
                        const uint32_t* positions, const uint32_t* slots,
                        const float* q_norm_w, const float* k_norm_w,
                        const float* inv_freq, const float* sinks, float eps,
                        float scale, float* K, float* V, float* out, double* out64,
                        int n_threads);

/* The same step with options (bit flags):
 *   ORACLE_VNORM          the cached and attended V is the weightless RMS norm
 *                         of v_new (rounded to f32);
 *   ORACLE_NORM_PLUS_ONE  the Q and K norm weights apply as (1 + w). */
#define ORACLE_VNORM 1u
#define ORACLE_NORM_PLUS_ONE 2u
int oracle_decode_batch_opts(uint32_t n_slots, uint32_t slot_ctx, uint32_t n_head,
                             uint32_t n_kv_head, uint32_t head_dim, uint32_t B,
                             const float* q, const float* k_new, const float* v_new,
                             const uint32_t* positions, const uint32_t* slots,
                             const float* q_norm_w, const float* k_norm_w,
                             const float* inv_freq, const float* sinks, float eps,
                             float scale, uint32_t flags, float* K, float* V, float* out,
                             double* out64, int n_threads);

/* The same step over a paged pool: K, V are f32[n_blocks][block_size][kv_dim];
 * row b's key t is at block block_tables[b * bt_stride + t / block_size],
 * offset t % block_size.  A row whose position is >= bt_stride * block_size
 * or whose blocks 0..pos/block_size include an id >= n_blocks is skipped. */
int oracle_decode_batch_paged(uint32_t n_blocks, uint32_t block_size, uint32_t n_head,
                              uint32_t n_kv_head, uint32_t head_dim, uint32_t B,
                              const float* q, const float* k_new, const float* v_new,
                              const uint32_t* positions, const uint32_t* block_tables,
                              uint32_t bt_stride, const float* q_norm_w,
                              const float* k_norm_w, const float* inv_freq,
                              const float* sinks, float eps, float scale, uint32_t flags,
                              float* K, float* V, float* out, double* out64, int n_threads);

#ifdef __cplusplus
}
#endif
#endif

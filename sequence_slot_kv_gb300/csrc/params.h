// params.h -- launch parameters shared by the host side and the kernels of
// libslotkv.  Plain data only.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace slotkv {

struct DecodeParams {
    const float* q;          // [B][n_head][hd]
    const float* k_new;      // [B][n_kv_head][hd]
    const float* v_new;      // [B][n_kv_head][hd]
    const uint32_t* positions;
    const uint32_t* slots;
    const float* q_norm_w;   // [hd]
    const float* k_norm_w;   // [hd]
    const float* inv_freq;   // [hd/2]
    const float* sinks;      // [n_head] or null
    float* out;              // [B][n_head][hd]
    float* K;                // slot buffers [n_slots][slot_ctx][n_kv_head][hd]
    float* V;
    float* ws_ml;            // split partials (m, l): [rows][n_head][max_splits][2]
    float* ws_acc;           // split partials acc:    [rows][n_head][max_splits][hd]
    uint32_t* counters;      // finished-split counters: [rows][n_kv_head]
    uint32_t* items;         // work list: [rows * n_kv_head * max_splits][4] records
                             // (packed item, position, tensor row of key p, 0)
    uint32_t* plan;          // [0] items in the list, [1] next item to hand out
    uint32_t* status;        // sticky SLOTKV_DEV_* flags
    uint32_t n_slots, slot_ctx, n_head, n_kv_head, B;
    uint32_t chunk_min;      // split policy, see split_chunk()
    uint32_t max_splits;
    float eps;
    float scale_log2;        // softmax scale * log2(e): scores live in base 2
    uint32_t flags;          // SLOTKV_OPT_* norm options
    uint32_t prefill;        // 1: rows are prefill tokens (keys all read from the slot)
    // Paged mode (block_tables non-null): K and V are a pool of n_slots blocks
    // of slot_ctx positions and row b's key t lives in block
    // block_tables[b * bt_stride + t / slot_ctx] at offset t % slot_ctx;
    // slot_ctx is then a multiple of the tile height.  slots is unused.
    const uint32_t* block_tables = nullptr;
    uint32_t bt_stride = 0;
    // Static first items: decode CTA c < static_items starts with
    // split 0 of (row c / n_kv_head, kv head c % n_kv_head) without waiting for
    // the plan, which leaves those items out of its list.  0: none.
    uint32_t static_items = 0;
    // Static second items (only when static_items covers every pair): decode
    // CTA static_items + q, q < static_second, starts with split 1 of pair q
    // if that row has a second split, and the plan leaves those items out of
    // its list too.  0: none.
    uint32_t static_second = 0;
    // 1: every item is a static first item (no more (row, kv head) pairs than
    // CTAs, one split each): no plan kernel runs, its list is empty, and the
    // decode kernel is launched in plain stream order.
    uint32_t no_plan = 0;
};

// The tensor-core prefill (head dims 64 and 128): prep, plan and attention
// kernels over tiles of consecutive same-slot tokens (see prefill_tc.cuh).
struct PrefillParams {
    const float* q;          // [n_tok][n_head][hd]
    const float* k_new;      // [n_tok][n_kv_head][hd]
    const float* v_new;      // [n_tok][n_kv_head][hd]
    const uint32_t* positions;
    const uint32_t* slots;
    const float* q_norm_w;
    const float* k_norm_w;
    const float* inv_freq;
    const float* sinks;      // [n_head] or null
    float* out;              // [n_tok][n_head][hd]
    float* K;                // slot buffers [n_slots][slot_ctx][n_kv_head][hd]
    float* V;
    float* q_rot;            // workspace [n_tok][n_head][hd]: normed, rotated, scaled q
    uint32_t* tiles;         // workspace [n_tok][4]: first token, tokens, slot, largest position
    uint32_t* tile_of;       // workspace [n_tok]: each token's tile, then the tiles' hand-out order
    uint32_t* plan;          // [0] items (tiles * n_kv_head), [1] next item to hand out
    uint32_t* status;        // sticky SLOTKV_DEV_* flags
    uint32_t n_slots, slot_ctx, n_head, n_kv_head, n_tok;
    float eps;
    float scale_log2;        // softmax scale * log2(e)
    uint32_t flags;          // SLOTKV_OPT_* norm options
};

// Keys per split chunk for a row with n_keys keys (p + 1).  Depends only on
// n_keys and the geometry so that a row's result never depends on the batch.
__host__ __device__ inline uint32_t split_chunk(uint32_t n_keys, uint32_t chunk_min,
                                                uint32_t max_splits, uint32_t tile) {
    uint32_t per = (n_keys + max_splits - 1) / max_splits;
    per = (per + tile - 1) / tile * tile;
    return per > chunk_min ? per : chunk_min;
}

// Tile height (keys per pipeline stage) for a head dim: 16 KiB of K + 16 KiB of V.
__host__ __device__ constexpr int tile_keys(int hd) { return 4096 / hd; }

// A work item is one (row, split, kv head), packed as row << 16 | split << 8 |
// kv head; rows <= 65535, splits and kv heads <= 256.
__host__ __device__ inline uint32_t pack_item(uint32_t b, uint32_t split, uint32_t kvh) {
    return (b << 16) | (split << 8) | kvh;
}

// Work-list records the workspace must hold: one per (row, kv head, split);
// each record is 4 u32 (16 bytes).
inline size_t plan_capacity(uint32_t rows, uint32_t n_kv_head, uint32_t max_splits) {
    return (size_t)rows * n_kv_head * max_splits;
}
constexpr int kItemWords = 4;

// Sets the calling thread's slot_kv_last_error() message.
void set_last_error(const char* msg);

// Launchers, one translation unit per head dim.  Each enqueues the plan kernel
// and then the persistent decode kernel on `stream` with `ctas` CTAs.  Return a
// cudaError_t value.
int launch_decode_hd64(int G, const DecodeParams& p, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, unsigned ctas, cudaStream_t stream);
int launch_decode_hd128(int G, const DecodeParams& p, const CUtensorMap& tmK,
                        const CUtensorMap& tmV, unsigned ctas, cudaStream_t stream);
int launch_decode_hd256(int G, const DecodeParams& p, const CUtensorMap& tmK,
                        const CUtensorMap& tmV, unsigned ctas, cudaStream_t stream);

// The small-call decode kernel (one CTA per (row, kv head), see
// decode_small.cuh): taken when a decode call has at most two CTAs' worth
// of (row, kv head) pairs per SM and slots of at most small_max_keys keys.
int launch_small_hd64(int G, const DecodeParams& p, cudaStream_t stream);
int launch_small_hd128(int G, const DecodeParams& p, cudaStream_t stream);
int launch_small_hd256(int G, const DecodeParams& p, cudaStream_t stream);
__host__ __device__ constexpr int small_max_keys(int hd) { return 8 * tile_keys(hd); }

// Tensor-core prefill launchers (prep, plan, attention on `stream`); tmK and
// tmV are the 128-byte-swizzled views of the slot buffers with a box of 32
// floats x prefill_tile_keys(hd) rows.  Return a cudaError_t value.
int launch_prefill_tc_hd64(int G, const PrefillParams& p, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, unsigned ctas, cudaStream_t stream);
int launch_prefill_tc_hd128(int G, const PrefillParams& p, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, unsigned ctas, cudaStream_t stream);

// Keys per pipeline stage of the tensor-core prefill.
__host__ __device__ constexpr int prefill_tile_keys(int) { return 64; }

}  // namespace slotkv

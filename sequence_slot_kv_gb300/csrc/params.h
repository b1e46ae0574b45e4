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
    uint32_t* status;        // sticky SLOTKV_DEV_* flags
    uint32_t n_slots, slot_ctx, n_head, n_kv_head, B;
    uint32_t chunk_min;      // split policy, see split_chunk()
    uint32_t max_splits;
    float eps;
    float scale_log2;        // softmax scale * log2(e): scores live in base 2
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

// Sets the calling thread's slot_kv_last_error() message.
void set_last_error(const char* msg);

// Launchers, one translation unit per head dim.  Return a cudaError_t value.
int launch_decode_hd64(int G, const DecodeParams& p, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, dim3 grid, cudaStream_t stream);
int launch_decode_hd128(int G, const DecodeParams& p, const CUtensorMap& tmK,
                        const CUtensorMap& tmV, dim3 grid, cudaStream_t stream);
int launch_decode_hd256(int G, const DecodeParams& p, const CUtensorMap& tmK,
                        const CUtensorMap& tmV, dim3 grid, cudaStream_t stream);

}  // namespace slotkv

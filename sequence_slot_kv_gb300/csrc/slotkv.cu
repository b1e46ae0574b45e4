// slotkv.cu -- host side of the libslotkv C ABI (declared in include/slotkv.h):
// handle life cycle, slot offsets, argument checks, the split-K workspace,
// TMA descriptors for the slot buffers, and kernel dispatch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/slotkv.h"
#include "params.h"

using slotkv::DecodeParams;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(SLOTKV_ERR_CUDA, "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
}

typedef CUresult (*encode_tiled_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

// Looked up on first use; an atomic, so handles may be allocated from
// several threads at once (a failed lookup is retried on the next call).
encode_tiled_fn get_encoder() {
    static std::atomic<encode_tiled_fn> fn{nullptr};
    encode_tiled_fn f = fn.load(std::memory_order_acquire);
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<encode_tiled_fn>(p);
            fn.store(f, std::memory_order_release);
        }
    }
    return f;
}

}  // namespace

struct slotkv_s {
    int device = 0;
    uint32_t n_slots = 0, slot_ctx = 0, n_kv_head = 0, head_dim = 0, kv_dim = 0;
    float* K = nullptr;
    float* V = nullptr;
    bool owns_kv = false;
    uint32_t max_rows = 0, max_n_head = 0;
    uint32_t chunk_min = 0, max_splits = 0;
    bool auto_split = true;  // chunk size from the batch's shape until slot_kv_set_split
    uint32_t options = 0;
    float* ws_ml = nullptr;
    float* ws_acc = nullptr;
    uint32_t* counters = nullptr;
    uint32_t* items = nullptr;  // work list built by the plan kernel
    uint32_t* plan = nullptr;   // [0] list length, [1] hand-out counter
    uint32_t* status = nullptr;
    int sm_count = 0;
    // device staging for decode_batch_attn_host
    float* st_q = nullptr;
    float* st_k = nullptr;
    float* st_v = nullptr;
    float* st_out = nullptr;
    uint32_t* st_pos = nullptr;
    uint32_t* st_slots = nullptr;
    uint32_t* st_tab = nullptr;  // block tables for decode_batch_attn_paged_host
    size_t st_tab_bytes = 0;     // (grown on demand)
    CUtensorMap tmK, tmV;
    // tensor-core prefill (head dims 64, 128): 128-byte-swizzled views of the
    // slot buffers, and a workspace grown on demand by prefill calls
    bool tc_prefill = false;
    CUtensorMap tmKs, tmVs;
    float* pf_q = nullptr;           // [tokens][n_head][hd] rotated q
    uint32_t* pf_tiles = nullptr;    // [tokens][4] tile records
    uint32_t* pf_tile_of = nullptr;  // [tokens]
    uint32_t* pf_plan = nullptr;     // item count, hand-out counter
    size_t pf_q_elems = 0, pf_tok = 0;
    std::vector<slotkv_host_call_s*> calls;  // prepared host calls on this handle
    cudaStream_t copy_stream = nullptr;      // their enqueued input copies (created on demand)
    // prefill_batch_attn_host in parts: its outputs' copies, the second
    // stream its parts alternate on, and the order of copies and kernels
    // (created on demand)
    cudaStream_t out_stream = nullptr, pf_stream2 = nullptr;
    cudaEvent_t pf_ev[2 * SLOTKV_PREFILL_HOST_MAX_PARTS + 2] = {};
};

// A prepared host call (slot_kv_host_call_create): the arguments of
// decode_batch_attn_host or decode_batch_attn_paged_host, checked once, and
// the device aliases of its host buffers resolved once.  h is cleared when
// the handle is freed first.
struct slotkv_host_call_s {
    slotkv_s* h = nullptr;
    uint32_t B = 0, n_head = 0, bt_stride = 0;  // bt_stride 0: slots
    const float *q = nullptr, *k_new = nullptr, *v_new = nullptr;
    const uint32_t *positions = nullptr, *idx = nullptr;
    const float *q_norm_w = nullptr, *k_norm_w = nullptr, *inv_freq = nullptr, *sinks = nullptr;
    float* out = nullptr;
    float eps = 0.f, scale = 0.f;
    bool mapped = false;
    void* dp[6] = {};
    // the enqueue path: the call's own device staging (allocated by its first
    // enqueue), filled by the copy engines on the handle's copy stream;
    // in_ready orders the step after its copies, done the next copies after
    // the step that read the staging
    int device = 0;
    float *st_q = nullptr, *st_k = nullptr, *st_v = nullptr, *st_out = nullptr;
    uint32_t *st_pos = nullptr, *st_idx = nullptr;
    cudaEvent_t in_ready = nullptr, done = nullptr;
    bool used = false;
};

namespace {

void free_workspace(slotkv_s* h) {
    cudaFree(h->ws_ml);
    cudaFree(h->ws_acc);
    cudaFree(h->counters);
    cudaFree(h->items);
    cudaFree(h->plan);
    h->ws_ml = h->ws_acc = nullptr;
    h->counters = h->items = h->plan = nullptr;
}

void release(slotkv_s* h) {
    if (!h) return;
    for (slotkv_host_call_s* c : h->calls) c->h = nullptr;  // they refuse to run from now on
    // the handle's memory and work live on its own device
    int cur = 0;
    const bool switched = cudaGetDevice(&cur) == cudaSuccess && cur != h->device &&
                          cudaSetDevice(h->device) == cudaSuccess;
    cudaDeviceSynchronize();
    if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
    if (h->out_stream) cudaStreamDestroy(h->out_stream);
    if (h->pf_stream2) cudaStreamDestroy(h->pf_stream2);
    for (cudaEvent_t ev : h->pf_ev)
        if (ev) cudaEventDestroy(ev);
    free_workspace(h);
    cudaFree(h->status);
    cudaFree(h->st_q);
    cudaFree(h->st_k);
    cudaFree(h->st_v);
    cudaFree(h->st_out);
    cudaFree(h->st_pos);
    cudaFree(h->st_slots);
    cudaFree(h->st_tab);
    cudaFree(h->pf_q);
    cudaFree(h->pf_tiles);
    cudaFree(h->pf_tile_of);
    cudaFree(h->pf_plan);
    if (h->owns_kv) {
        cudaFree(h->K);
        cudaFree(h->V);
    }
    if (switched) cudaSetDevice(cur);
    delete h;
}

// Split-K workspace: partial (m, l) and acc per (row, query head, split),
// one finished-split counter per (row, kv head) (zeroed), and the work list
// with its two counters (rebuilt by every call).
int alloc_workspace(slotkv_s* h) {
    free_workspace(h);
    const size_t units = (size_t)h->max_rows * h->max_n_head * h->max_splits;
    cudaError_t e;
    if ((e = cudaMalloc(&h->ws_ml, units * 2 * sizeof(float))) != cudaSuccess)
        return cuda_fail(e, "workspace (m, l)");
    if ((e = cudaMalloc(&h->ws_acc, units * h->head_dim * sizeof(float))) != cudaSuccess)
        return cuda_fail(e, "workspace (acc)");
    const size_t nc = (size_t)h->max_rows * h->n_kv_head;
    if ((e = cudaMalloc(&h->counters, nc * sizeof(uint32_t))) != cudaSuccess)
        return cuda_fail(e, "workspace (counters)");
    if ((e = cudaMemset(h->counters, 0, nc * sizeof(uint32_t))) != cudaSuccess)
        return cuda_fail(e, "workspace clear");
    const size_t ni = slotkv::plan_capacity(h->max_rows, h->n_kv_head, h->max_splits);
    if ((e = cudaMalloc(&h->items, ni * slotkv::kItemWords * sizeof(uint32_t))) != cudaSuccess)
        return cuda_fail(e, "workspace (work list)");
    if ((e = cudaMalloc(&h->plan, 2 * sizeof(uint32_t))) != cudaSuccess)
        return cuda_fail(e, "workspace (plan counters)");
    return SLOTKV_OK;
}

int encode_maps(slotkv_s* h) {
    encode_tiled_fn enc = get_encoder();
    if (!enc) return fail(SLOTKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {h->kv_dim, (cuuint64_t)h->n_slots * h->slot_ctx};
    const cuuint64_t strides[1] = {(cuuint64_t)h->kv_dim * sizeof(float)};
    const cuuint32_t box[2] = {h->head_dim, (cuuint32_t)slotkv::tile_keys((int)h->head_dim)};
    const cuuint32_t estr[2] = {1, 1};
    float* bufs[2] = {h->K, h->V};
    CUtensorMap* maps[2] = {&h->tmK, &h->tmV};
    for (int i = 0; i < 2; ++i) {
        CUresult r = enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, bufs[i], dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(SLOTKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    // the tensor-core prefill reads [keys][32 floats] boxes, 128-byte swizzled
    h->tc_prefill = h->head_dim == 64 || h->head_dim == 128;
    if (h->tc_prefill) {
        const cuuint32_t sbox[2] = {32, (cuuint32_t)slotkv::prefill_tile_keys((int)h->head_dim)};
        CUtensorMap* smaps[2] = {&h->tmKs, &h->tmVs};
        for (int i = 0; i < 2; ++i) {
            CUresult r = enc(smaps[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, bufs[i], dims, strides,
                             sbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS)
                return fail(SLOTKV_ERR_CUDA, "cuTensorMapEncodeTiled (swizzled) failed (%d)",
                            (int)r);
        }
    }
    return SLOTKV_OK;
}

// The tensor-core prefill's workspace, grown to n_tok tokens of n_head heads
// (cudaMalloc synchronises the device the first time it grows).
int prefill_workspace(slotkv_s* h, uint32_t n_tok, uint32_t n_head) {
    const size_t qe = (size_t)n_tok * n_head * h->head_dim;
    cudaError_t e;
    if (qe > h->pf_q_elems) {
        cudaFree(h->pf_q);
        h->pf_q = nullptr;
        h->pf_q_elems = 0;
        if ((e = cudaMalloc(&h->pf_q, qe * sizeof(float))) != cudaSuccess)
            return cuda_fail(e, "prefill workspace (q)");
        h->pf_q_elems = qe;
    }
    if (n_tok > h->pf_tok) {
        cudaFree(h->pf_tiles);
        cudaFree(h->pf_tile_of);
        h->pf_tiles = h->pf_tile_of = nullptr;
        h->pf_tok = 0;
        if ((e = cudaMalloc(&h->pf_tiles, (size_t)n_tok * 16)) != cudaSuccess ||
            (e = cudaMalloc(&h->pf_tile_of, (size_t)n_tok * 4)) != cudaSuccess)
            return cuda_fail(e, "prefill workspace (tiles)");
        h->pf_tok = n_tok;
    }
    // one (items, hand-out counter) pair per part of a host call in parts
    if (!h->pf_plan && (e = cudaMalloc(&h->pf_plan, 2 * SLOTKV_PREFILL_HOST_MAX_PARTS *
                                                        sizeof(uint32_t))) != cudaSuccess)
        return cuda_fail(e, "prefill workspace (plan)");
    return SLOTKV_OK;
}

bool valid_handle(slotkv_t h) { return h && h->K && h->V && h->status; }

// A handle's buffers, workspace and tensor maps belong to the device it was
// allocated on; work is only enqueued with that device current.
int check_device(slotkv_t h) {
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device)
        return fail(SLOTKV_ERR_STATE, "the handle belongs to device %d but device %d is current",
                    h->device, cur);
    return SLOTKV_OK;
}

// The most splits any row of this slot_ctx can need: nsplit(n) <= ceil(n /
// chunk_min) because chunks are >= chunk_min keys, and <= max_splits.
uint32_t grid_splits(const slotkv_s* h, uint64_t max_keys, uint32_t chunk_min) {
    const uint64_t bound = (max_keys + chunk_min - 1) / chunk_min;
    return (uint32_t)(bound < h->max_splits ? bound : h->max_splits);
}

// The default policy's chunk size, from the batch's shape alone (rows, kv
// heads, the context capacity max_keys, the SM count): about three items per
// persistent CTA if contexts were half full, between chunk_min (512 KiB of
// K+V per kv head) and four times that.  Fewer, larger items mean fewer item
// boundaries and split merges; a small batch still gets the splits it needs
// to fill the GPU.
uint32_t auto_chunk(const slotkv_s* h, uint32_t B, uint64_t max_keys) {
    const uint32_t T = (uint32_t)slotkv::tile_keys((int)h->head_dim);
    const uint64_t lo = h->chunk_min, hi = 4ull * h->chunk_min;
    const uint64_t ctas = 2ull * (uint64_t)(h->sm_count > 0 ? h->sm_count : 1);
    uint64_t c = (uint64_t)B * h->n_kv_head * (max_keys / 2) / (3 * ctas);
    c = c / T * T;
    return (uint32_t)(c < lo ? lo : (c > hi ? hi : c));
}

// How a call of B rows runs: the split chunk, the persistent CTAs, the
// static items (split 0 of the first pairs, then split 1 for CTAs to spare),
// whether the plan kernel runs, and the kernels launched.
struct CallShape {
    uint32_t chunk, ctas, static_items, static_second, no_plan, kernels;
    uint32_t small;  // the small-call kernel (one CTA per (row, kv head))
};

CallShape call_shape(const slotkv_s* h, uint32_t B, uint64_t max_keys, bool prefill) {
    CallShape c;
    c.small = 0;
    // a few rows over short slots: one CTA per (row, kv head), no persistent
    // pipeline to set up.  Only under the default policy, whose bits may
    // already depend on the batch's shape (a fixed policy promises a row the
    // same bits in any batch); the stall test option needs the pipeline's
    // waits.  Slot and paged calls of the same capacity take the same path.
    const uint64_t sms = (uint64_t)(h->sm_count > 0 ? h->sm_count : 1);
    if (!prefill && h->auto_split && !(h->options & SLOTKV_OPT_TEST_STALL) &&
        (uint64_t)B * h->n_kv_head <= 2 * sms &&
        max_keys <= (uint64_t)slotkv::small_max_keys((int)h->head_dim)) {
        c.small = 1;
        c.chunk = (uint32_t)slotkv::tile_keys((int)h->head_dim);
        c.ctas = B * h->n_kv_head;
        c.static_items = c.static_second = 0;
        c.no_plan = 1;
        c.kernels = 1;
        return c;
    }
    if (prefill && h->tc_prefill) {
        // prep, plan and the persistent tensor-core kernel (one CTA per SM)
        c.chunk = (uint32_t)slotkv::prefill_tile_keys((int)h->head_dim);
        c.ctas = (uint32_t)(h->sm_count > 0 ? h->sm_count : 1);
        c.static_items = c.static_second = 0;
        c.no_plan = 0;
        c.kernels = 3;
        return c;
    }
    c.chunk = h->auto_split ? auto_chunk(h, B, max_keys) : h->chunk_min;
    // persistent CTAs: two per SM, never more than there can be work items
    const uint32_t gsplits = grid_splits(h, max_keys, c.chunk);
    const uint64_t most = (uint64_t)B * h->n_kv_head * gsplits;
    const uint64_t want = 2ull * (uint64_t)(h->sm_count > 0 ? h->sm_count : 1);
    c.ctas = (uint32_t)(most < want ? most : want);
    // CTA c < pairs starts on split 0 of pair c; when that covers every item
    // (one split per row, a CTA per pair) no plan is needed
    const uint64_t pairs = (uint64_t)B * h->n_kv_head;
    c.static_items = (uint32_t)(pairs < c.ctas ? pairs : c.ctas);
    // CTAs left over once every pair has one start on split 1 of a pair
    const uint64_t spare = c.ctas - c.static_items;
    c.static_second = (gsplits >= 2 && spare) ? (uint32_t)(spare < pairs ? spare : pairs) : 0u;
    c.no_plan = (gsplits == 1 && pairs <= c.ctas) ? 1u : 0u;
    c.kernels = (prefill ? 1u : 0u) + (c.no_plan ? 0u : 1u) + 1u;
    return c;
}

int launch(slotkv_s* h, uint32_t B, uint32_t n_head, const float* q, const float* k_new,
           const float* v_new, const uint32_t* positions, const uint32_t* slots,
           const float* q_norm_w, const float* k_norm_w, const float* inv_freq,
           const float* sinks, float* out, float eps, float scale, cudaStream_t stream,
           bool prefill = false, const uint32_t* block_tables = nullptr,
           uint32_t bt_stride = 0) {
    DecodeParams P;
    P.prefill = prefill ? 1u : 0u;
    P.block_tables = block_tables;
    P.bt_stride = bt_stride;
    P.q = q;
    P.k_new = k_new;
    P.v_new = v_new;
    P.positions = positions;
    P.slots = slots;
    P.q_norm_w = q_norm_w;
    P.k_norm_w = k_norm_w;
    P.inv_freq = inv_freq;
    P.sinks = sinks;
    P.out = out;
    P.K = h->K;
    P.V = h->V;
    P.ws_ml = h->ws_ml;
    P.ws_acc = h->ws_acc;
    P.counters = h->counters;
    P.items = h->items;
    P.plan = h->plan;
    P.status = h->status;
    P.n_slots = h->n_slots;
    P.slot_ctx = h->slot_ctx;
    P.n_head = n_head;
    P.n_kv_head = h->n_kv_head;
    P.B = B;
    const uint64_t max_keys = block_tables ? (uint64_t)bt_stride * h->slot_ctx : h->slot_ctx;
    const CallShape cs = call_shape(h, B, max_keys, prefill);
    P.chunk_min = cs.chunk;
    P.max_splits = h->max_splits;
    P.eps = eps;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.flags = h->options;
    const int G = (int)(n_head / h->n_kv_head);
    const unsigned ctas = cs.ctas;
    P.static_items = cs.static_items;
    P.static_second = cs.static_second;
    P.no_plan = cs.no_plan;
    int rc;
    if (cs.small) {
        switch (h->head_dim) {
            case 64: rc = slotkv::launch_small_hd64(G, P, stream); break;
            case 128: rc = slotkv::launch_small_hd128(G, P, stream); break;
            default: rc = slotkv::launch_small_hd256(G, P, stream); break;
        }
        if (rc != 0) return cuda_fail((cudaError_t)rc, "small decode kernel launch");
        return SLOTKV_OK;
    }
    switch (h->head_dim) {
        case 64: rc = slotkv::launch_decode_hd64(G, P, h->tmK, h->tmV, ctas, stream); break;
        case 128: rc = slotkv::launch_decode_hd128(G, P, h->tmK, h->tmV, ctas, stream); break;
        case 256: rc = slotkv::launch_decode_hd256(G, P, h->tmK, h->tmV, ctas, stream); break;
        default: return fail(SLOTKV_ERR_UNSUPPORTED, "head_dim %u", h->head_dim);
    }
    if (rc != 0) return cuda_fail((cudaError_t)rc, "decode kernel launch");
    return SLOTKV_OK;
}

int check_decode_args(slotkv_t h, uint32_t B, uint32_t n_head, const void* q,
                      const void* k_new, const void* v_new, const void* positions,
                      const void* slots, const void* q_norm_w, const void* k_norm_w,
                      const void* inv_freq, const void* out, bool device_ptrs = true) {
    if (!valid_handle(h)) return fail(SLOTKV_ERR_STATE, "handle is not allocated");
    if (check_device(h) != SLOTKV_OK) return SLOTKV_ERR_STATE;
    if (B > h->max_rows) return fail(SLOTKV_ERR_ARG, "B=%u exceeds max_rows=%u", B, h->max_rows);
    if (n_head == 0 || n_head % h->n_kv_head != 0)
        return fail(SLOTKV_ERR_ARG, "n_head=%u is not a multiple of n_kv_head=%u", n_head,
                    h->n_kv_head);
    if (n_head > h->max_n_head)
        return fail(SLOTKV_ERR_ARG, "n_head=%u exceeds max_n_head=%u", n_head, h->max_n_head);
    const uint32_t G = n_head / h->n_kv_head;
    if (G < 1 || G > 8) return fail(SLOTKV_ERR_UNSUPPORTED, "G=%u outside 1..8", G);
    if (B == 0) return SLOTKV_OK;
    if (!q || !k_new || !v_new || !positions || !slots || !q_norm_w || !k_norm_w || !inv_freq ||
        !out)
        return fail(SLOTKV_ERR_ARG, "null tensor pointer");
    if (((uintptr_t)q | (uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)positions |
         (uintptr_t)slots | (uintptr_t)q_norm_w | (uintptr_t)k_norm_w | (uintptr_t)inv_freq |
         (uintptr_t)out) & 3)
        return fail(SLOTKV_ERR_ARG, "tensor pointers must be 4-byte aligned");
    // the kernel stages q, k_new and v_new with bulk copies and writes out in
    // 16-byte stores
    if (device_ptrs && (((uintptr_t)q | (uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)out) & 15))
        return fail(SLOTKV_ERR_ARG, "q, k_new, v_new and out must be 16-byte aligned");
    return SLOTKV_OK;
}

}  // namespace

namespace slotkv {
void set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

// Copies up to kMaxSegs byte ranges (each a multiple of 4 bytes) with one
// grid: the host entry's inputs from pinned host memory (mapped into the
// device's address space) to device staging, or its output back.  16-byte
// accesses where a segment allows them.
constexpr int kMaxSegs = 6;
struct CopySegs {
    const uint8_t* src[kMaxSegs];
    uint8_t* dst[kMaxSegs];
    size_t bytes[kMaxSegs];
    int n;
};

__global__ void copy_segments_kernel(const CopySegs c) {
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t nth = (size_t)gridDim.x * blockDim.x;
    for (int k = 0; k < c.n; ++k) {
        const uint8_t* src = c.src[k];
        uint8_t* dst = c.dst[k];
        const size_t bytes = c.bytes[k];
        if ((((uintptr_t)src | (uintptr_t)dst | bytes) & 15) == 0) {
            const uint4* s4 = reinterpret_cast<const uint4*>(src);
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            for (size_t i = tid; i < bytes / 16; i += nth) d4[i] = s4[i];
        } else {
            const uint32_t* s1 = reinterpret_cast<const uint32_t*>(src);
            uint32_t* d1 = reinterpret_cast<uint32_t*>(dst);
            for (size_t i = tid; i < bytes / 4; i += nth) d1[i] = s1[i];
        }
    }
}

__global__ void advance_positions_kernel(uint32_t* __restrict__ pos, uint32_t B,
                                         uint32_t delta) {
    const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) pos[b] += delta;
}
}  // namespace slotkv

namespace {

// The host entries' per-step buffers: q, k_new, v_new, positions and the row
// index (slots, or block tables of idx_bytes) in host memory, and out.
struct HostStep {
    const float* q;
    const float* k_new;
    const float* v_new;
    const uint32_t* positions;
    const uint32_t* idx;
    size_t idx_bytes;
    uint32_t* idx_stage;  // device staging for idx
    float* out;
};

// Move a step's host inputs into the handle's device staging on `s`, run the
// step (`run(q, k_new, v_new, positions, idx, out)` with device pointers),
// move out back and synchronise `s`.  When every host buffer is page-locked
// (pinned, hence mapped into the device's address space), one copy kernel
// gathers the inputs over the host link and the step writes out straight
// into host memory (through a second copy kernel if out is not 16-byte
// aligned), instead of separate copy-engine transfers; otherwise each buffer
// is copied with cudaMemcpyAsync.
// The device aliases dp of the step's six host buffers (q, k_new, v_new,
// positions, idx, out) when every one is page-locked (mapped into the
// device's address space); false when any is not.
bool resolve_mapped(const HostStep& hs, void* dp[6]) {
    const void* hp[6] = {hs.q, hs.k_new, hs.v_new, hs.positions, hs.idx, hs.out};
    bool mapped = true;
    for (int i = 0; i < 6 && mapped; ++i) {
        cudaPointerAttributes at;
        mapped = cudaPointerGetAttributes(&at, hp[i]) == cudaSuccess &&
                 at.type == cudaMemoryTypeHost && at.devicePointer != nullptr;
        dp[i] = mapped ? at.devicePointer : nullptr;
    }
    cudaGetLastError();  // a failed attribute query leaves an error behind
    return mapped;
}

// host_step with the buffers already resolved (mapped, dp from resolve_mapped);
// sync false leaves the final synchronisation of s to the caller.
template <typename Run>
int host_step_resolved(slotkv_s* h, uint32_t B, uint32_t n_head, const HostStep& hs,
                       bool mapped, void* const dp[6], cudaStream_t s, Run run,
                       bool sync = true) {
    const size_t nq = (size_t)B * n_head * h->head_dim * sizeof(float);
    const size_t nk = (size_t)B * h->kv_dim * sizeof(float);
    const size_t ni = (size_t)B * sizeof(uint32_t);
    cudaError_t e;
    int rc;
    if (mapped) {
        const int threads = 256;
        const unsigned grid = (unsigned)(h->sm_count > 0 ? h->sm_count : 1);
        slotkv::CopySegs in{};
        void* st[5] = {h->st_q, h->st_k, h->st_v, h->st_pos, hs.idx_stage};
        const size_t nb[5] = {nq, nk, nk, ni, hs.idx_bytes};
        for (int i = 0; i < 5; ++i) {
            in.src[i] = static_cast<const uint8_t*>(dp[i]);
            in.dst[i] = static_cast<uint8_t*>(st[i]);
            in.bytes[i] = nb[i];
        }
        in.n = 5;
        slotkv::copy_segments_kernel<<<grid, threads, 0, s>>>(in);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "input gather launch");
        // an aligned out is written by the decode kernel itself, over the link
        const bool direct_out = ((uintptr_t)dp[5] & 15) == 0;
        rc = run(h->st_q, h->st_k, h->st_v, h->st_pos, hs.idx_stage,
                 direct_out ? static_cast<float*>(dp[5]) : h->st_out);
        if (rc != SLOTKV_OK) return rc;
        if (!direct_out) {
            slotkv::CopySegs outc{};
            outc.src[0] = reinterpret_cast<const uint8_t*>(h->st_out);
            outc.dst[0] = static_cast<uint8_t*>(dp[5]);
            outc.bytes[0] = nq;
            outc.n = 1;
            slotkv::copy_segments_kernel<<<grid, threads, 0, s>>>(outc);
            if ((e = cudaGetLastError()) != cudaSuccess)
                return cuda_fail(e, "output scatter launch");
        }
        if (sync && (e = cudaStreamSynchronize(s)) != cudaSuccess)
            return cuda_fail(e, "stream sync");
        return SLOTKV_OK;
    }
    if ((e = cudaMemcpyAsync(h->st_q, hs.q, nq, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(h->st_k, hs.k_new, nk, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(h->st_v, hs.v_new, nk, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(h->st_pos, hs.positions, ni, cudaMemcpyHostToDevice, s)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(hs.idx_stage, hs.idx, hs.idx_bytes, cudaMemcpyHostToDevice, s)) !=
            cudaSuccess)
        return cuda_fail(e, "host-to-device input copy");
    rc = run(h->st_q, h->st_k, h->st_v, h->st_pos, hs.idx_stage, h->st_out);
    if (rc != SLOTKV_OK) return rc;
    if ((e = cudaMemcpyAsync(hs.out, h->st_out, nq, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e, "device-to-host output copy");
    if (sync && (e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "stream sync");
    return SLOTKV_OK;
}

template <typename Run>
int host_step(slotkv_s* h, uint32_t B, uint32_t n_head, const HostStep& hs, cudaStream_t s,
              Run run) {
    void* dp[6];
    const bool mapped = resolve_mapped(hs, dp);
    return host_step_resolved(h, B, n_head, hs, mapped, dp, s, run);
}

}  // namespace

extern "C" {

const char* slot_kv_last_error(void) { return g_err; }

int slot_kv_alloc(slotkv_t* handle, uint32_t n_slots, uint32_t slot_ctx, uint32_t n_kv_head,
                  uint32_t head_dim, float* k_buf, float* v_buf, uint32_t max_rows,
                  uint32_t max_n_head) {
    g_err[0] = 0;
    if (!handle) return fail(SLOTKV_ERR_ARG, "handle pointer is null");
    if (*handle) {
        release(*handle);
        *handle = nullptr;
    }
    if (n_slots == 0 || slot_ctx == 0 || n_kv_head == 0)
        return fail(SLOTKV_ERR_ARG, "n_slots, slot_ctx and n_kv_head must be >= 1");
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(SLOTKV_ERR_UNSUPPORTED, "head_dim=%u (64, 128 or 256)", head_dim);
    // TMA row coordinates are int32: keep every tile start (row + tile) below 2^31
    if ((uint64_t)n_slots * slot_ctx + 256 >= (1ull << 31))
        return fail(SLOTKV_ERR_ARG, "n_slots*slot_ctx must be < 2^31 - 256");
    if (n_kv_head > 256) return fail(SLOTKV_ERR_ARG, "n_kv_head must be <= 256");
    if ((k_buf == nullptr) != (v_buf == nullptr))
        return fail(SLOTKV_ERR_ARG, "give both k_buf and v_buf, or neither");
    if ((k_buf && ((uintptr_t)k_buf & 15)) || (v_buf && ((uintptr_t)v_buf & 15)))
        return fail(SLOTKV_ERR_ARG, "k_buf and v_buf must be 16-byte aligned");
    if (max_rows == 0 || max_rows > 65535)
        return fail(SLOTKV_ERR_ARG, "max_rows must be 1..65535");
    if (max_n_head < n_kv_head || max_n_head > 8 * n_kv_head)
        return fail(SLOTKV_ERR_ARG, "max_n_head must be n_kv_head..8*n_kv_head");

    slotkv_s* h = new (std::nothrow) slotkv_s();
    if (!h) return fail(SLOTKV_ERR_ARG, "out of host memory");
    cudaGetDevice(&h->device);
    cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device);
    h->n_slots = n_slots;
    h->slot_ctx = slot_ctx;
    h->n_kv_head = n_kv_head;
    h->head_dim = head_dim;
    h->kv_dim = n_kv_head * head_dim;
    h->max_rows = max_rows;
    h->max_n_head = max_n_head;
    // default split policy: chunks of >= 512 KiB of K+V per kv head, <= 64 splits
    h->chunk_min = (512u * 1024u) / (8u * head_dim);
    h->max_splits = 64;

    const size_t elems = (size_t)n_slots * slot_ctx * h->kv_dim;
    cudaError_t e;
    int rc = SLOTKV_OK;
    if (k_buf) {
        h->K = k_buf;
        h->V = v_buf;
        h->owns_kv = false;
    } else {
        h->owns_kv = true;
        if ((e = cudaMalloc(&h->K, elems * sizeof(float))) != cudaSuccess ||
            (e = cudaMalloc(&h->V, elems * sizeof(float))) != cudaSuccess) {
            rc = cuda_fail(e, "slot KV allocation");
        } else if ((e = cudaMemset(h->K, 0, elems * sizeof(float))) != cudaSuccess ||
                   (e = cudaMemset(h->V, 0, elems * sizeof(float))) != cudaSuccess) {
            rc = cuda_fail(e, "slot KV clear");
        }
    }
    if (rc == SLOTKV_OK) {
        if ((e = cudaMalloc(&h->status, sizeof(uint32_t))) != cudaSuccess ||
            (e = cudaMemset(h->status, 0, sizeof(uint32_t))) != cudaSuccess)
            rc = cuda_fail(e, "status word");
    }
    if (rc == SLOTKV_OK) {
        const size_t nq = (size_t)max_rows * max_n_head * head_dim;
        const size_t nk = (size_t)max_rows * h->kv_dim;
        if ((e = cudaMalloc(&h->st_q, nq * 4)) != cudaSuccess ||
            (e = cudaMalloc(&h->st_out, nq * 4)) != cudaSuccess ||
            (e = cudaMalloc(&h->st_k, nk * 4)) != cudaSuccess ||
            (e = cudaMalloc(&h->st_v, nk * 4)) != cudaSuccess ||
            (e = cudaMalloc(&h->st_pos, (size_t)max_rows * 4)) != cudaSuccess ||
            (e = cudaMalloc(&h->st_slots, (size_t)max_rows * 4)) != cudaSuccess)
            rc = cuda_fail(e, "host-call staging");
    }
    if (rc == SLOTKV_OK) rc = alloc_workspace(h);
    if (rc == SLOTKV_OK) rc = encode_maps(h);
    if (rc != SLOTKV_OK) {
        char keep[sizeof(g_err)];
        memcpy(keep, g_err, sizeof(keep));
        release(h);
        memcpy(g_err, keep, sizeof(keep));
        return rc;
    }
    *handle = h;
    return SLOTKV_OK;
}

int slot_kv_free(slotkv_t handle) {
    g_err[0] = 0;
    release(handle);
    return SLOTKV_OK;
}

size_t slot_kv_offset_bytes(slotkv_t h, uint32_t slot, uint32_t pos) {
    if (!h || slot >= h->n_slots || pos >= h->slot_ctx) return SIZE_MAX;
    return ((size_t)slot * h->slot_ctx + pos) * h->kv_dim * sizeof(float);
}

int slot_kv_reset(slotkv_t h, uint32_t slot, slotkv_stream_t stream) {
    g_err[0] = 0;
    if (!valid_handle(h)) return fail(SLOTKV_ERR_STATE, "handle is not allocated");
    if (check_device(h) != SLOTKV_OK) return SLOTKV_ERR_STATE;
    if (slot >= h->n_slots) return fail(SLOTKV_ERR_ARG, "slot=%u >= n_slots=%u", slot, h->n_slots);
    const size_t off = slot_kv_offset_bytes(h, slot, 0);
    const size_t bytes = (size_t)h->slot_ctx * h->kv_dim * sizeof(float);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    if ((e = cudaMemsetAsync((char*)h->K + off, 0, bytes, s)) != cudaSuccess ||
        (e = cudaMemsetAsync((char*)h->V + off, 0, bytes, s)) != cudaSuccess)
        return cuda_fail(e, "slot reset");
    return SLOTKV_OK;
}

int slot_kv_k_ptr(slotkv_t h, float** k) {
    if (!valid_handle(h) || !k) return fail(SLOTKV_ERR_ARG, "bad handle or output pointer");
    *k = h->K;
    return SLOTKV_OK;
}

int slot_kv_v_ptr(slotkv_t h, float** v) {
    if (!valid_handle(h) || !v) return fail(SLOTKV_ERR_ARG, "bad handle or output pointer");
    *v = h->V;
    return SLOTKV_OK;
}

int slot_kv_geometry(slotkv_t h, uint32_t* n_slots, uint32_t* slot_ctx, uint32_t* n_kv_head,
                     uint32_t* head_dim, uint32_t* max_rows, uint32_t* max_n_head) {
    if (!valid_handle(h)) return fail(SLOTKV_ERR_STATE, "handle is not allocated");
    if (n_slots) *n_slots = h->n_slots;
    if (slot_ctx) *slot_ctx = h->slot_ctx;
    if (n_kv_head) *n_kv_head = h->n_kv_head;
    if (head_dim) *head_dim = h->head_dim;
    if (max_rows) *max_rows = h->max_rows;
    if (max_n_head) *max_n_head = h->max_n_head;
    return SLOTKV_OK;
}

int decode_batch_attn(slotkv_t h, uint32_t B, uint32_t n_head, const float* q,
                      const float* k_new, const float* v_new, const uint32_t* positions,
                      const uint32_t* slots, const float* q_norm_w, const float* k_norm_w,
                      const float* inv_freq, const float* sinks, float* out, float eps,
                      float scale, slotkv_stream_t stream) {
    g_err[0] = 0;
    int rc = check_decode_args(h, B, n_head, q, k_new, v_new, positions, slots, q_norm_w,
                               k_norm_w, inv_freq, out);
    if (rc != SLOTKV_OK || B == 0) return rc;
    return launch(h, B, n_head, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w, inv_freq,
                  sinks, out, eps, scale, (cudaStream_t)stream);
}

}  // extern "C"

namespace {
// prefill_batch_attn_host cuts a call into parts whose tokens share no slot
// (one part's host-link copies then overlap another part's kernels): one
// part per kPfPartTok tokens, at most SLOTKV_PREFILL_HOST_MAX_PARTS, none
// under kPfPartMin, each cut the allowed one nearest its target.  The
// targets make the first and the last part half the size of the others:
// the first part's inputs and the last part's output overlap nothing.
constexpr uint32_t kPfPartTok = 512, kPfPartMin = 256;

uint32_t prefill_parts(uint32_t n, const uint32_t* slots, uint32_t* cut) {
    const uint32_t want = std::min<uint32_t>(SLOTKV_PREFILL_HOST_MAX_PARTS, n / kPfPartTok);
    cut[0] = 0;
    uint32_t np = 0;
    // (host memory for the search; should it run out, the call stays whole)
    if (want >= 2) try {
        // a cut before token m is allowed when tokens [0, m) hold every
        // occurrence of their slots
        std::unordered_map<uint32_t, uint32_t> last;
        last.reserve(n);
        for (uint32_t i = 0; i < n; ++i) last[slots[i]] = i;
        std::vector<uint32_t> allowed;
        uint32_t reach = 0;
        for (uint32_t i = 0; i + 1 < n; ++i) {
            reach = std::max(reach, last[slots[i]]);
            if (reach == i) allowed.push_back(i + 1);
        }
        for (uint32_t j = 1; j < want; ++j) {
            const uint64_t target = (uint64_t)n * (2 * j - 1) / (2 * (want - 1));
            uint32_t best = 0;
            uint64_t best_d = UINT64_MAX;
            for (uint32_t m : allowed) {
                if (m < cut[np] + kPfPartMin || (uint64_t)m + kPfPartMin > n) continue;
                const uint64_t d = m > target ? m - target : target - m;
                if (d < best_d) {
                    best_d = d;
                    best = m;
                }
            }
            if (best == 0) break;
            cut[++np] = best;
        }
    } catch (const std::bad_alloc&) {
        np = 0;
    }
    cut[++np] = n;
    return np;
}

// The prefill step on device pointers (arguments already checked).  A part
// of a host call in parts uses the workspace rows from token ws_tok on and
// its own plan counters (plan_slot), so parts can run concurrently.
int run_prefill(slotkv_t h, uint32_t n_tok, uint32_t n_head, const float* q,
                const float* k_new, const float* v_new, const uint32_t* positions,
                const uint32_t* slots, const float* q_norm_w, const float* k_norm_w,
                const float* inv_freq, const float* sinks, float* out, float eps, float scale,
                cudaStream_t stream, size_t ws_tok = 0, uint32_t plan_slot = 0) {
    if (!h->tc_prefill)  // head dim 256: the decode kernel in prefill mode
        return launch(h, n_tok, n_head, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                      inv_freq, sinks, out, eps, scale, stream, true);
    int rc = prefill_workspace(h, n_tok, n_head);
    if (rc != SLOTKV_OK) return rc;
    slotkv::PrefillParams P;
    P.q = q;
    P.k_new = k_new;
    P.v_new = v_new;
    P.positions = positions;
    P.slots = slots;
    P.q_norm_w = q_norm_w;
    P.k_norm_w = k_norm_w;
    P.inv_freq = inv_freq;
    P.sinks = sinks;
    P.out = out;
    P.K = h->K;
    P.V = h->V;
    P.q_rot = h->pf_q + ws_tok * n_head * h->head_dim;
    P.tiles = h->pf_tiles + 4 * ws_tok;
    P.tile_of = h->pf_tile_of + ws_tok;
    P.plan = h->pf_plan + 2 * plan_slot;
    P.status = h->status;
    P.n_slots = h->n_slots;
    P.slot_ctx = h->slot_ctx;
    P.n_head = n_head;
    P.n_kv_head = h->n_kv_head;
    P.n_tok = n_tok;
    P.eps = eps;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.flags = h->options;
    const int G = (int)(n_head / h->n_kv_head);
    const unsigned ctas = (unsigned)(h->sm_count > 0 ? h->sm_count : 1);
    rc = h->head_dim == 64
             ? slotkv::launch_prefill_tc_hd64(G, P, h->tmKs, h->tmVs, ctas, stream)
             : slotkv::launch_prefill_tc_hd128(G, P, h->tmKs, h->tmVs, ctas, stream);
    if (rc != 0) return cuda_fail((cudaError_t)rc, "prefill kernel launch");
    return SLOTKV_OK;
}

// prefill_batch_attn_host in parts [cut[i], cut[i+1]) (slot-disjoint, so each
// part is a prefill of its own with the same tiles and bits): inputs in on
// the handle's copy stream part by part; each part's kernels, once its
// inputs have landed, on `s` or the handle's second stream by turns, with
// its own workspace rows and plan counters, so that a part's kernels start
// on the SMs the previous part's attention kernel leaves in its tail; each
// part's out back on the out stream as soon as it is done.  `s` waits for
// the second stream and the last copy and is synchronised.
int prefill_host_in_parts(slotkv_t h, uint32_t n_tok, uint32_t n_head, const float* q,
                          const float* k_new, const float* v_new, const uint32_t* positions,
                          const uint32_t* slots, const float* q_norm_w, const float* k_norm_w,
                          const float* inv_freq, const float* sinks, float* out, float eps,
                          float scale, cudaStream_t s, const uint32_t* cut, uint32_t parts) {
    // the workspace at its full size first: a later part must not regrow
    // (free) it while an earlier part's kernels still use it
    int rc = prefill_workspace(h, n_tok, n_head);
    if (rc != SLOTKV_OK) return rc;
    cudaError_t e = cudaSuccess;
    if (!h->copy_stream)
        e = cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess && !h->out_stream)
        e = cudaStreamCreateWithFlags(&h->out_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess && !h->pf_stream2)
        e = cudaStreamCreateWithFlags(&h->pf_stream2, cudaStreamNonBlocking);
    for (cudaEvent_t& ev : h->pf_ev)
        if (e == cudaSuccess && !ev) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "prefill copy streams");
    const cudaStream_t cin = h->copy_stream, cout = h->out_stream, s2 = h->pf_stream2;
    cudaEvent_t* in_ready = h->pf_ev;                                // [parts]
    cudaEvent_t* done = h->pf_ev + SLOTKV_PREFILL_HOST_MAX_PARTS;    // [parts]
    cudaEvent_t entry = h->pf_ev[2 * SLOTKV_PREFILL_HOST_MAX_PARTS];  // then: outputs back
    cudaEvent_t joined = h->pf_ev[2 * SLOTKV_PREFILL_HOST_MAX_PARTS + 1];  // s2's parts done
    // whatever fails, nothing of this call is left running on return
    auto bail = [&](cudaError_t err, const char* what) {
        cudaStreamSynchronize(cin);
        cudaStreamSynchronize(s2);
        cudaStreamSynchronize(cout);
        cudaStreamSynchronize(s);
        return err == cudaSuccess ? rc : cuda_fail(err, what);
    };
    const size_t qrow = (size_t)n_head * h->head_dim, krow = h->kv_dim;
    // the staging and the workspace may still be in use by work enqueued on
    // s before this call
    if ((e = cudaEventRecord(entry, s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(cin, entry, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s2, entry, 0)) != cudaSuccess)
        return bail(e, "prefill copy order");
    for (uint32_t i = 0; i < parts; ++i) {
        const size_t t0 = cut[i], nt = cut[i + 1] - cut[i];
        if ((e = cudaMemcpyAsync(h->st_q + t0 * qrow, q + t0 * qrow, nt * qrow * sizeof(float),
                                 cudaMemcpyHostToDevice, cin)) != cudaSuccess ||
            (e = cudaMemcpyAsync(h->st_k + t0 * krow, k_new + t0 * krow,
                                 nt * krow * sizeof(float), cudaMemcpyHostToDevice, cin)) !=
                cudaSuccess ||
            (e = cudaMemcpyAsync(h->st_v + t0 * krow, v_new + t0 * krow,
                                 nt * krow * sizeof(float), cudaMemcpyHostToDevice, cin)) !=
                cudaSuccess ||
            (e = cudaMemcpyAsync(h->st_pos + t0, positions + t0, nt * sizeof(uint32_t),
                                 cudaMemcpyHostToDevice, cin)) != cudaSuccess ||
            (e = cudaMemcpyAsync(h->st_slots + t0, slots + t0, nt * sizeof(uint32_t),
                                 cudaMemcpyHostToDevice, cin)) != cudaSuccess ||
            (e = cudaEventRecord(in_ready[i], cin)) != cudaSuccess)
            return bail(e, "host-to-device input copy");
    }
    for (uint32_t i = 0; i < parts; ++i) {
        const size_t t0 = cut[i];
        const cudaStream_t cs = (i & 1) ? s2 : s;
        if ((e = cudaStreamWaitEvent(cs, in_ready[i], 0)) != cudaSuccess)
            return bail(e, "prefill copy order");
        rc = run_prefill(h, cut[i + 1] - cut[i], n_head, h->st_q + t0 * qrow, h->st_k + t0 * krow,
                         h->st_v + t0 * krow, h->st_pos + t0, h->st_slots + t0, q_norm_w,
                         k_norm_w, inv_freq, sinks, h->st_out + t0 * qrow, eps, scale, cs, t0, i);
        if (rc != SLOTKV_OK) return bail(cudaSuccess, nullptr);
        if ((e = cudaEventRecord(done[i], cs)) != cudaSuccess)
            return bail(e, "prefill copy order");
    }
    for (uint32_t i = 0; i < parts; ++i) {
        const size_t t0 = cut[i], nt = cut[i + 1] - cut[i];
        if ((e = cudaStreamWaitEvent(cout, done[i], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(out + t0 * qrow, h->st_out + t0 * qrow,
                                 nt * qrow * sizeof(float), cudaMemcpyDeviceToHost, cout)) !=
                cudaSuccess)
            return bail(e, "device-to-host output copy");
    }
    if ((e = cudaEventRecord(entry, cout)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, entry, 0)) != cudaSuccess ||
        (e = cudaEventRecord(joined, s2)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, joined, 0)) != cudaSuccess)
        return bail(e, "prefill copy order");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "stream sync");
    return SLOTKV_OK;
}
}  // namespace

extern "C" {

int slot_kv_prefill_host_parts(uint32_t n_tok, const uint32_t* slots, uint32_t* cuts,
                               uint32_t cuts_len, uint32_t* n_parts) {
    g_err[0] = 0;
    if (!cuts || !n_parts || (n_tok && !slots))
        return fail(SLOTKV_ERR_ARG, "slots, cuts and n_parts must not be null");
    if (cuts_len < SLOTKV_PREFILL_HOST_MAX_PARTS + 1)
        return fail(SLOTKV_ERR_ARG, "cuts holds %u entries, fewer than %u", cuts_len,
                    SLOTKV_PREFILL_HOST_MAX_PARTS + 1);
    *n_parts = prefill_parts(n_tok, slots, cuts);
    return SLOTKV_OK;
}

int prefill_batch_attn(slotkv_t h, uint32_t n_tok, uint32_t n_head, const float* q,
                       const float* k_new, const float* v_new, const uint32_t* positions,
                       const uint32_t* slots, const float* q_norm_w, const float* k_norm_w,
                       const float* inv_freq, const float* sinks, float* out, float eps,
                       float scale, slotkv_stream_t stream) {
    g_err[0] = 0;
    int rc = check_decode_args(h, n_tok, n_head, q, k_new, v_new, positions, slots, q_norm_w,
                               k_norm_w, inv_freq, out);
    if (rc != SLOTKV_OK || n_tok == 0) return rc;
    return run_prefill(h, n_tok, n_head, q, k_new, v_new, positions, slots, q_norm_w, k_norm_w,
                       inv_freq, sinks, out, eps, scale, (cudaStream_t)stream);
}

int prefill_batch_attn_host(slotkv_t h, uint32_t n_tok, uint32_t n_head, const float* q,
                            const float* k_new, const float* v_new, const uint32_t* positions,
                            const uint32_t* slots, const float* q_norm_w,
                            const float* k_norm_w, const float* inv_freq, const float* sinks,
                            float* out, float eps, float scale, slotkv_stream_t stream) {
    g_err[0] = 0;
    int rc = check_decode_args(h, n_tok, n_head, q, k_new, v_new, positions, slots, q_norm_w,
                               k_norm_w, inv_freq, out, false);
    if (rc != SLOTKV_OK || n_tok == 0) return rc;
    // A prefill moves tens of MB each way: the copy engines move them faster
    // than a gather kernel, and an out written into host memory by the
    // attention kernel itself would stall its epilogue on the host link, so
    // every buffer goes through cudaMemcpyAsync and device staging.
    uint32_t cut[SLOTKV_PREFILL_HOST_MAX_PARTS + 1];
    const uint32_t parts = h->tc_prefill ? prefill_parts(n_tok, slots, cut) : 1u;
    if (parts > 1)
        return prefill_host_in_parts(h, n_tok, n_head, q, k_new, v_new, positions, slots,
                                     q_norm_w, k_norm_w, inv_freq, sinks, out, eps, scale,
                                     (cudaStream_t)stream, cut, parts);
    const HostStep hs{q, k_new, v_new, positions, slots, (size_t)n_tok * sizeof(uint32_t),
                      h->st_slots, out};
    void* const none[6] = {};
    return host_step_resolved(
        h, n_tok, n_head, hs, false, none, (cudaStream_t)stream,
        [&](const float* dq, const float* dk, const float* dv, const uint32_t* dpos,
            const uint32_t* didx, float* dout) {
            return run_prefill(h, n_tok, n_head, dq, dk, dv, dpos, didx, q_norm_w, k_norm_w,
                               inv_freq, sinks, dout, eps, scale, (cudaStream_t)stream);
        });
}

int decode_batch_attn_paged(slotkv_t h, uint32_t B, uint32_t n_head, const float* q,
                            const float* k_new, const float* v_new, const uint32_t* positions,
                            const uint32_t* block_tables, uint32_t bt_stride,
                            const float* q_norm_w, const float* k_norm_w,
                            const float* inv_freq, const float* sinks, float* out, float eps,
                            float scale, slotkv_stream_t stream) {
    g_err[0] = 0;
    int rc = check_decode_args(h, B, n_head, q, k_new, v_new, positions, block_tables,
                               q_norm_w, k_norm_w, inv_freq, out);
    if (rc != SLOTKV_OK) return rc;
    const uint32_t T = (uint32_t)slotkv::tile_keys((int)h->head_dim);
    if (h->slot_ctx % T != 0)
        return fail(SLOTKV_ERR_UNSUPPORTED, "block size %u is not a multiple of %u keys",
                    h->slot_ctx, T);
    if (bt_stride == 0) return fail(SLOTKV_ERR_ARG, "bt_stride must be >= 1");
    if (B == 0) return SLOTKV_OK;
    return launch(h, B, n_head, q, k_new, v_new, positions, nullptr, q_norm_w, k_norm_w,
                  inv_freq, sinks, out, eps, scale, (cudaStream_t)stream, false, block_tables,
                  bt_stride);
}

int decode_batch_attn_host(slotkv_t h, uint32_t B, uint32_t n_head, const float* q,
                           const float* k_new, const float* v_new, const uint32_t* positions,
                           const uint32_t* slots, const float* q_norm_w,
                           const float* k_norm_w, const float* inv_freq, const float* sinks,
                           float* out, float eps, float scale, slotkv_stream_t stream) {
    g_err[0] = 0;
    int rc = check_decode_args(h, B, n_head, q, k_new, v_new, positions, slots, q_norm_w,
                               k_norm_w, inv_freq, out, false);
    if (rc != SLOTKV_OK || B == 0) return rc;
    const HostStep hs{q, k_new, v_new, positions, slots, (size_t)B * sizeof(uint32_t),
                      h->st_slots, out};
    return host_step(h, B, n_head, hs, (cudaStream_t)stream,
                     [&](const float* dq, const float* dk, const float* dv, const uint32_t* dpos,
                         const uint32_t* didx, float* dout) {
                         return launch(h, B, n_head, dq, dk, dv, dpos, didx, q_norm_w, k_norm_w,
                                       inv_freq, sinks, dout, eps, scale, (cudaStream_t)stream);
                     });
}

int decode_batch_attn_paged_host(slotkv_t h, uint32_t B, uint32_t n_head, const float* q,
                                 const float* k_new, const float* v_new,
                                 const uint32_t* positions, const uint32_t* block_tables,
                                 uint32_t bt_stride, const float* q_norm_w,
                                 const float* k_norm_w, const float* inv_freq,
                                 const float* sinks, float* out, float eps, float scale,
                                 slotkv_stream_t stream) {
    g_err[0] = 0;
    int rc = check_decode_args(h, B, n_head, q, k_new, v_new, positions, block_tables,
                               q_norm_w, k_norm_w, inv_freq, out, false);
    if (rc != SLOTKV_OK) return rc;
    const uint32_t T = (uint32_t)slotkv::tile_keys((int)h->head_dim);
    if (h->slot_ctx % T != 0)
        return fail(SLOTKV_ERR_UNSUPPORTED, "block size %u is not a multiple of %u keys",
                    h->slot_ctx, T);
    if (bt_stride == 0) return fail(SLOTKV_ERR_ARG, "bt_stride must be >= 1");
    if (B == 0) return SLOTKV_OK;
    // the tables' device staging grows to the largest B * bt_stride seen
    const size_t tab_bytes = (size_t)B * bt_stride * sizeof(uint32_t);
    if (tab_bytes > h->st_tab_bytes) {
        cudaError_t e = cudaFree(h->st_tab);
        h->st_tab = nullptr;
        h->st_tab_bytes = 0;
        if (e == cudaSuccess) e = cudaMalloc(&h->st_tab, tab_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "block-table staging");
        h->st_tab_bytes = tab_bytes;
    }
    const HostStep hs{q, k_new, v_new, positions, block_tables, tab_bytes, h->st_tab, out};
    return host_step(h, B, n_head, hs, (cudaStream_t)stream,
                     [&](const float* dq, const float* dk, const float* dv, const uint32_t* dpos,
                         const uint32_t* didx, float* dout) {
                         return launch(h, B, n_head, dq, dk, dv, dpos, nullptr, q_norm_w,
                                       k_norm_w, inv_freq, sinks, dout, eps, scale,
                                       (cudaStream_t)stream, false, didx, bt_stride);
                     });
}

int slot_kv_host_call_create(slotkv_t h, slotkv_host_call_t* call, uint32_t B,
                             uint32_t n_head, const float* q, const float* k_new,
                             const float* v_new, const uint32_t* positions,
                             const uint32_t* idx, uint32_t bt_stride, const float* q_norm_w,
                             const float* k_norm_w, const float* inv_freq, const float* sinks,
                             float* out, float eps, float scale) {
    g_err[0] = 0;
    if (!call) return fail(SLOTKV_ERR_ARG, "call pointer is null");
    *call = nullptr;
    int rc = check_decode_args(h, B, n_head, q, k_new, v_new, positions, idx, q_norm_w,
                               k_norm_w, inv_freq, out, false);
    if (rc != SLOTKV_OK) return rc;
    if (B == 0) return fail(SLOTKV_ERR_ARG, "a prepared call needs B >= 1");
    size_t idx_bytes = (size_t)B * sizeof(uint32_t);
    if (bt_stride) {
        const uint32_t T = (uint32_t)slotkv::tile_keys((int)h->head_dim);
        if (h->slot_ctx % T != 0)
            return fail(SLOTKV_ERR_UNSUPPORTED, "block size %u is not a multiple of %u keys",
                        h->slot_ctx, T);
        idx_bytes = (size_t)B * bt_stride * sizeof(uint32_t);
        if (idx_bytes > h->st_tab_bytes) {  // the tables' staging, grown once here
            cudaError_t e = cudaFree(h->st_tab);
            h->st_tab = nullptr;
            h->st_tab_bytes = 0;
            if (e == cudaSuccess) e = cudaMalloc(&h->st_tab, idx_bytes);
            if (e != cudaSuccess) return cuda_fail(e, "block-table staging");
            h->st_tab_bytes = idx_bytes;
        }
    }
    slotkv_host_call_s* c = new (std::nothrow) slotkv_host_call_s();
    if (!c) return fail(SLOTKV_ERR_ARG, "out of host memory");
    c->h = h;
    c->B = B;
    c->n_head = n_head;
    c->bt_stride = bt_stride;
    c->q = q;
    c->k_new = k_new;
    c->v_new = v_new;
    c->positions = positions;
    c->idx = idx;
    c->q_norm_w = q_norm_w;
    c->k_norm_w = k_norm_w;
    c->inv_freq = inv_freq;
    c->sinks = sinks;
    c->out = out;
    c->eps = eps;
    c->scale = scale;
    const HostStep hs{q, k_new, v_new, positions, idx, idx_bytes, nullptr, out};
    c->mapped = resolve_mapped(hs, c->dp);
    try {
        h->calls.push_back(c);
    } catch (const std::bad_alloc&) {
        delete c;
        return fail(SLOTKV_ERR_ARG, "out of host memory");
    }
    *call = c;
    return SLOTKV_OK;
}

namespace {
int host_call_step(slotkv_host_call_t c, slotkv_stream_t stream, bool sync) {
    if (!c) return fail(SLOTKV_ERR_ARG, "call is null");
    slotkv_s* h = c->h;
    if (!h) return fail(SLOTKV_ERR_STATE, "the call's handle has been freed");
    if (check_device(h) != SLOTKV_OK) return SLOTKV_ERR_STATE;
    const uint32_t B = c->B, n_head = c->n_head, bt_stride = c->bt_stride;
    const cudaStream_t s = (cudaStream_t)stream;
    const size_t idx_bytes = (size_t)B * (bt_stride ? bt_stride : 1u) * sizeof(uint32_t);
    const HostStep hs{c->q, c->k_new, c->v_new, c->positions, c->idx, idx_bytes,
                      bt_stride ? h->st_tab : h->st_slots, c->out};
    return host_step_resolved(
        h, B, n_head, hs, c->mapped, c->dp, s,
        [&](const float* dq, const float* dk, const float* dv, const uint32_t* dpos,
            const uint32_t* didx, float* dout) {
            return bt_stride
                       ? launch(h, B, n_head, dq, dk, dv, dpos, nullptr, c->q_norm_w,
                                c->k_norm_w, c->inv_freq, c->sinks, dout, c->eps, c->scale, s,
                                false, didx, bt_stride)
                       : launch(h, B, n_head, dq, dk, dv, dpos, didx, c->q_norm_w, c->k_norm_w,
                                c->inv_freq, c->sinks, dout, c->eps, c->scale, s);
        },
        sync);
}
}  // namespace

namespace {
void free_call_staging(slotkv_host_call_s* c) {
    cudaFree(c->st_q);
    cudaFree(c->st_k);
    cudaFree(c->st_v);
    cudaFree(c->st_out);
    cudaFree(c->st_pos);
    cudaFree(c->st_idx);
    if (c->in_ready) cudaEventDestroy(c->in_ready);
    if (c->done) cudaEventDestroy(c->done);
    c->st_q = c->st_k = c->st_v = c->st_out = nullptr;
    c->st_pos = c->st_idx = nullptr;
    c->in_ready = c->done = nullptr;
    c->used = false;
}

// The enqueued step.  With work still in flight on `stream`, the inputs go
// to the call's own staging by the copy engines on the handle's copy stream
// (so they overlap that work), the step waits for them, and the next copies
// into this staging wait for the step.  On an idle stream nothing would
// overlap, and the lower-latency path of run (one gather kernel over the host
// link) is taken, without its final synchronisation.  Both run the same
// kernels on the same values.
int host_call_enqueue(slotkv_host_call_t c, slotkv_stream_t stream) {
    if (!c) return fail(SLOTKV_ERR_ARG, "call is null");
    slotkv_s* h = c->h;
    if (!h) return fail(SLOTKV_ERR_STATE, "the call's handle has been freed");
    if (check_device(h) != SLOTKV_OK) return SLOTKV_ERR_STATE;
    {
        const cudaError_t q = cudaStreamQuery((cudaStream_t)stream);
        if (q == cudaSuccess) return host_call_step(c, stream, false);
        if (q != cudaErrorNotReady) return cuda_fail(q, "stream query");
    }
    const uint32_t B = c->B, n_head = c->n_head, bt_stride = c->bt_stride;
    const cudaStream_t s = (cudaStream_t)stream;
    const size_t nq = (size_t)B * n_head * h->head_dim * sizeof(float);
    const size_t nk = (size_t)B * h->kv_dim * sizeof(float);
    const size_t ni = (size_t)B * sizeof(uint32_t);
    const size_t nidx = (size_t)B * (bt_stride ? bt_stride : 1u) * sizeof(uint32_t);
    cudaError_t e;
    if (!c->st_q) {
        c->device = h->device;
        if ((e = cudaMalloc(&c->st_q, nq)) != cudaSuccess ||
            (e = cudaMalloc(&c->st_k, nk)) != cudaSuccess ||
            (e = cudaMalloc(&c->st_v, nk)) != cudaSuccess ||
            (e = cudaMalloc(&c->st_out, nq)) != cudaSuccess ||
            (e = cudaMalloc(&c->st_pos, ni)) != cudaSuccess ||
            (e = cudaMalloc(&c->st_idx, nidx)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&c->in_ready, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&c->done, cudaEventDisableTiming)) != cudaSuccess) {
            free_call_staging(c);
            return cuda_fail(e, "prepared call staging");
        }
    }
    if (!h->copy_stream &&
        (e = cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail(e, "copy stream");
    const cudaStream_t cs = h->copy_stream;
    if (c->used && (e = cudaStreamWaitEvent(cs, c->done, 0)) != cudaSuccess)
        return cuda_fail(e, "staging reuse order");
    if ((e = cudaMemcpyAsync(c->st_q, c->q, nq, cudaMemcpyHostToDevice, cs)) != cudaSuccess ||
        (e = cudaMemcpyAsync(c->st_k, c->k_new, nk, cudaMemcpyHostToDevice, cs)) != cudaSuccess ||
        (e = cudaMemcpyAsync(c->st_v, c->v_new, nk, cudaMemcpyHostToDevice, cs)) != cudaSuccess ||
        (e = cudaMemcpyAsync(c->st_pos, c->positions, ni, cudaMemcpyHostToDevice, cs)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(c->st_idx, c->idx, nidx, cudaMemcpyHostToDevice, cs)) != cudaSuccess ||
        (e = cudaEventRecord(c->in_ready, cs)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, c->in_ready, 0)) != cudaSuccess)
        return cuda_fail(e, "enqueued input copies");
    // out straight into host memory when it is page-locked and 16-byte aligned
    const bool direct_out = c->mapped && ((uintptr_t)c->dp[5] & 15) == 0;
    float* dout = direct_out ? static_cast<float*>(c->dp[5]) : c->st_out;
    const int rc = bt_stride
                       ? launch(h, B, n_head, c->st_q, c->st_k, c->st_v, c->st_pos, nullptr,
                                c->q_norm_w, c->k_norm_w, c->inv_freq, c->sinks, dout, c->eps,
                                c->scale, s, false, c->st_idx, bt_stride)
                       : launch(h, B, n_head, c->st_q, c->st_k, c->st_v, c->st_pos, c->st_idx,
                                c->q_norm_w, c->k_norm_w, c->inv_freq, c->sinks, dout, c->eps,
                                c->scale, s);
    if (rc != SLOTKV_OK) return rc;
    if (!direct_out &&
        (e = cudaMemcpyAsync(c->out, c->st_out, nq, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e, "enqueued output copy");
    if ((e = cudaEventRecord(c->done, s)) != cudaSuccess) return cuda_fail(e, "step order");
    c->used = true;
    return SLOTKV_OK;
}
}  // namespace

int slot_kv_host_call_run(slotkv_host_call_t c, slotkv_stream_t stream) {
    g_err[0] = 0;
    return host_call_step(c, stream, true);
}

int slot_kv_host_call_enqueue(slotkv_host_call_t c, slotkv_stream_t stream) {
    g_err[0] = 0;
    return host_call_enqueue(c, stream);
}

int slot_kv_host_call_free(slotkv_host_call_t c) {
    g_err[0] = 0;
    if (!c) return SLOTKV_OK;
    if (c->h) {
        std::vector<slotkv_host_call_s*>& v = c->h->calls;
        v.erase(std::remove(v.begin(), v.end(), c), v.end());
    }
    if (c->st_q || c->in_ready) {
        // the call's staging belongs to its device; its last step must be done
        int cur = 0;
        const bool switched = cudaGetDevice(&cur) == cudaSuccess && cur != c->device &&
                              cudaSetDevice(c->device) == cudaSuccess;
        if (c->done && c->used) cudaEventSynchronize(c->done);
        free_call_staging(c);
        if (switched) cudaSetDevice(cur);
    }
    delete c;
    return SLOTKV_OK;
}

// Slot ownership: rank r of n_ranks owns the global slots
// [floor(r*n/N), floor((r+1)*n/N)); every rank owns at least one when
// n_slots >= n_ranks.  The owner of slot s < n is the largest r whose range
// starts at or below s: r = floor((s*N + N - 1) / n).
static uint32_t shard_first(uint32_t n_ranks, uint32_t n_slots, uint32_t r) {
    return (uint32_t)(((uint64_t)r * n_slots) / n_ranks);
}

int slot_kv_shard_range(uint32_t n_ranks, uint32_t n_slots, uint32_t rank, uint32_t* first,
                        uint32_t* count) {
    g_err[0] = 0;
    if (n_ranks == 0 || n_slots < n_ranks)
        return fail(SLOTKV_ERR_ARG, "need 1 <= n_ranks <= n_slots (n_ranks=%u, n_slots=%u)",
                    n_ranks, n_slots);
    if (rank >= n_ranks) return fail(SLOTKV_ERR_ARG, "rank=%u >= n_ranks=%u", rank, n_ranks);
    const uint32_t a = shard_first(n_ranks, n_slots, rank);
    const uint32_t b = shard_first(n_ranks, n_slots, rank + 1);
    if (first) *first = a;
    if (count) *count = b - a;
    return SLOTKV_OK;
}

int slot_kv_shard_route(uint32_t n_ranks, uint32_t n_slots, uint32_t B, const uint32_t* slots,
                        uint32_t* order, uint32_t* offsets, uint32_t* local_slots) {
    g_err[0] = 0;
    if (n_ranks == 0 || n_slots < n_ranks)
        return fail(SLOTKV_ERR_ARG, "need 1 <= n_ranks <= n_slots (n_ranks=%u, n_slots=%u)",
                    n_ranks, n_slots);
    if (!offsets || (B > 0 && (!slots || !order || !local_slots)))
        return fail(SLOTKV_ERR_ARG, "null pointer");
    auto owner = [&](uint32_t s) -> uint32_t {
        if (s >= n_slots) return n_ranks - 1;  // out of range: the last rank skips it
        return (uint32_t)(((uint64_t)s * n_ranks + n_ranks - 1) / n_slots);
    };
    // counting sort by owner: stable, so rows keep their order within a rank
    for (uint32_t r = 0; r <= n_ranks; ++r) offsets[r] = 0;
    for (uint32_t b = 0; b < B; ++b) ++offsets[owner(slots[b]) + 1];
    for (uint32_t r = 0; r < n_ranks; ++r) offsets[r + 1] += offsets[r];
    for (uint32_t b = 0; b < B; ++b) {
        const uint32_t r = owner(slots[b]);
        // offsets[r] is used as rank r's cursor, then restored below
        const uint32_t at = offsets[r]++;
        order[at] = b;
        local_slots[at] = slots[b] - shard_first(n_ranks, n_slots, r);
    }
    for (uint32_t r = n_ranks; r > 0; --r) offsets[r] = offsets[r - 1];
    offsets[0] = 0;
    return SLOTKV_OK;
}

int slot_kv_advance_positions(uint32_t* positions, uint32_t B, uint32_t delta,
                              slotkv_stream_t stream) {
    g_err[0] = 0;
    if (B == 0) return SLOTKV_OK;
    if (!positions) return fail(SLOTKV_ERR_ARG, "positions is null");
    slotkv::advance_positions_kernel<<<(B + 255) / 256, 256, 0, (cudaStream_t)stream>>>(
        positions, B, delta);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "advance kernel launch");
    return SLOTKV_OK;
}

int slot_kv_get_status(slotkv_t h, slotkv_stream_t stream, uint32_t* flags) {
    g_err[0] = 0;
    if (!valid_handle(h) || !flags) return fail(SLOTKV_ERR_ARG, "bad handle or flags pointer");
    if (check_device(h) != SLOTKV_OK) return SLOTKV_ERR_STATE;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t v = 0;
    cudaError_t e;
    if ((e = cudaMemcpyAsync(&v, h->status, sizeof(v), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return cuda_fail(e, "status read");
    if (v) {
        if ((e = cudaMemsetAsync(h->status, 0, sizeof(uint32_t), s)) != cudaSuccess)
            return cuda_fail(e, "status clear");
        if (v & SLOTKV_DEV_TIMEOUT) {
            const size_t nc = (size_t)h->max_rows * h->n_kv_head * sizeof(uint32_t);
            if ((e = cudaMemsetAsync(h->counters, 0, nc, s)) != cudaSuccess)
                return cuda_fail(e, "workspace clear");
        }
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "stream sync");
    }
    *flags = v;
    return SLOTKV_OK;
}

int slot_kv_set_options(slotkv_t h, uint32_t flags) {
    g_err[0] = 0;
    if (!valid_handle(h)) return fail(SLOTKV_ERR_STATE, "handle is not allocated");
    if (flags & ~(SLOTKV_OPT_VNORM | SLOTKV_OPT_NORM_PLUS_ONE | SLOTKV_OPT_TEST_STALL))
        return fail(SLOTKV_ERR_ARG, "unknown option bits 0x%x", flags);
    h->options = flags;
    return SLOTKV_OK;
}

int slot_kv_call_shape(slotkv_t h, uint32_t B, uint32_t bt_stride, uint32_t prefill,
                       uint32_t* chunk_keys, uint32_t* ctas, uint32_t* kernels) {
    g_err[0] = 0;
    if (!valid_handle(h)) return fail(SLOTKV_ERR_STATE, "handle is not allocated");
    if (B == 0 || B > h->max_rows) return fail(SLOTKV_ERR_ARG, "B=%u outside 1..max_rows", B);
    const uint64_t max_keys = bt_stride ? (uint64_t)bt_stride * h->slot_ctx : h->slot_ctx;
    const CallShape cs = call_shape(h, B, max_keys, prefill != 0);
    if (chunk_keys) *chunk_keys = cs.chunk;
    if (ctas) *ctas = cs.ctas;
    if (kernels) *kernels = cs.kernels;
    return SLOTKV_OK;
}

int slot_kv_set_split(slotkv_t h, uint32_t min_chunk_keys, uint32_t max_splits) {
    g_err[0] = 0;
    if (!valid_handle(h)) return fail(SLOTKV_ERR_STATE, "handle is not allocated");
    const uint32_t T = (uint32_t)slotkv::tile_keys((int)h->head_dim);
    if (check_device(h) != SLOTKV_OK) return SLOTKV_ERR_STATE;
    if (min_chunk_keys == 0 || min_chunk_keys % T != 0)
        return fail(SLOTKV_ERR_ARG, "min_chunk_keys must be a positive multiple of %u", T);
    if (max_splits == 0 || max_splits > 256) return fail(SLOTKV_ERR_ARG, "max_splits 1..256");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "synchronize");
    h->chunk_min = min_chunk_keys;
    h->max_splits = max_splits;
    h->auto_split = false;
    return alloc_workspace(h);
}

}  // extern "C"

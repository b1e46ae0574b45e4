// noalloc.cu -- decode_batch_attn_noalloc: the batched decode attention step
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a host framework may own every byte of
// device memory through its own pool or budget, or the calling code path may
// not tolerate the device synchronisation that cudaMalloc/cudaFree can imply.
// The regular entry point needs a handle from slot_kv_alloc, which allocates
// the split-K workspace.  This entry point takes the slot K/V buffers and
// every input and output from the caller and allocates nothing: the split-K
// partials, the merge counters and a status word live in one file-scope
// device array of fixed size (kNoAllocScratchBytes), which every GPU that
// loads the library holds until the process exits.
//
// It launches the same fused kernel as decode_batch_attn.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "../../include/slotkv.h"
#include "params.h"

namespace {

constexpr size_t kNoAllocScratchBytes = SLOTKV_NOALLOC_SCRATCH_BYTES;
// split policy of this entry point: at most 16 splits per row keeps the
// partials of typical batches inside the fixed scratch
constexpr uint32_t kNoAllocMaxSplits = 16;
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the symbol; the
// device address comes from cudaGetSymbolAddress, once per device and CUDA
// context.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// A __device__ symbol's address belongs to the context that loaded the
// module: after cudaDeviceReset, or with another (driver-API) context
// current, the address must be looked up again.  The cache is keyed on the
// current context's unique id (cuCtxGetId), which no later context reuses.
struct ScratchAddr {
    unsigned long long ctx_id;
    void* ptr;
};
std::mutex g_setup_mutex;
ScratchAddr g_scratch_addr[kMaxDevices] = {};

typedef CUresult (*ctx_get_current_fn)(CUcontext*);
typedef CUresult (*ctx_get_id_fn)(CUcontext, unsigned long long*);

// The unique id of the calling thread's current context; false when no
// context is current yet or the CUDA driver API cannot say.  Call with
// g_setup_mutex held.
bool current_context_id(unsigned long long* id) {
    static ctx_get_current_fn get_current = nullptr;
    static ctx_get_id_fn get_id = nullptr;
    if (!get_current || !get_id) {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault,
                                             &qa) != cudaSuccess ||
            qa != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
                cudaSuccess ||
            qb != cudaDriverEntryPointSuccess || !a || !b)
            return false;
        get_current = reinterpret_cast<ctx_get_current_fn>(a);
        get_id = reinterpret_cast<ctx_get_id_fn>(b);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Failures are reported like every other call: a status code, and a message
// for slot_kv_last_error().
int noalloc_fail(int code, const char* fmt, ...) {
    char msg[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof(msg), fmt, ap);
    va_end(ap);
    slotkv::set_last_error(msg);
    return code;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

typedef CUresult (*encode_tiled_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

}  // namespace

extern "C" int decode_batch_attn_noalloc(
    float* K, float* V, uint32_t n_slots, uint32_t slot_ctx, uint32_t n_kv_head,
    uint32_t head_dim, uint32_t B, uint32_t n_head, const float* q, const float* k_new,
    const float* v_new, const uint32_t* positions, const uint32_t* slots,
    const float* q_norm_w, const float* k_norm_w, const float* inv_freq, const float* sinks,
    float* out, uint32_t* dev_flags, float eps, float scale, slotkv_stream_t stream) {
    slotkv::set_last_error("");
    if (B == 0) return SLOTKV_OK;
    if (!K || !V || !q || !k_new || !v_new || !positions || !slots || !q_norm_w || !k_norm_w ||
        !inv_freq || !out)
        return noalloc_fail(SLOTKV_ERR_ARG, "null tensor pointer");
    if (((uintptr_t)K & 15) || ((uintptr_t)V & 15))
        return noalloc_fail(SLOTKV_ERR_ARG, "K and V must be 16-byte aligned");
    if (((uintptr_t)q | (uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)out) & 15)
        return noalloc_fail(SLOTKV_ERR_ARG, "q, k_new, v_new and out must be 16-byte aligned");
    if (((uintptr_t)positions | (uintptr_t)slots | (uintptr_t)q_norm_w | (uintptr_t)k_norm_w |
         (uintptr_t)inv_freq | (uintptr_t)sinks) & 3)
        return noalloc_fail(SLOTKV_ERR_ARG, "tensor pointers must be 4-byte aligned");
    if (n_slots == 0 || slot_ctx == 0 || n_kv_head == 0)
        return noalloc_fail(SLOTKV_ERR_ARG, "n_slots, slot_ctx and n_kv_head must be >= 1");
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return noalloc_fail(SLOTKV_ERR_UNSUPPORTED, "head_dim=%u (64, 128 or 256)", head_dim);
    if ((uint64_t)n_slots * slot_ctx + 256 >= (1ull << 31))
        return noalloc_fail(SLOTKV_ERR_ARG, "n_slots*slot_ctx must be < 2^31 - 256");
    if (n_kv_head > 256) return noalloc_fail(SLOTKV_ERR_ARG, "n_kv_head must be <= 256");
    if (n_head == 0 || n_head % n_kv_head != 0 || n_head / n_kv_head > 8)
        return noalloc_fail(SLOTKV_ERR_UNSUPPORTED, "n_head/n_kv_head must be 1..8");
    if (B > 65535) return noalloc_fail(SLOTKV_ERR_ARG, "B must be <= 65535");

    // scratch layout: status word | plan counters | merge counters [B][n_kv_head]
    //                 | work list | (m, l) | acc
    const uint32_t chunk_min = (512u * 1024u) / (8u * head_dim);
    const size_t units = (size_t)B * n_head * kNoAllocMaxSplits;
    const size_t off_plan = 128;
    const size_t off_cnt = 256;
    const size_t off_items = off_cnt + align256((size_t)B * n_kv_head * sizeof(uint32_t));
    const size_t off_ml =
        off_items + align256(slotkv::plan_capacity(B, n_kv_head, kNoAllocMaxSplits) * 4 *
                             slotkv::kItemWords);
    const size_t off_acc = off_ml + align256(units * 2 * sizeof(float));
    const size_t need = off_acc + units * head_dim * sizeof(float);
    if (need > kNoAllocScratchBytes)
        return noalloc_fail(SLOTKV_ERR_ARG,
                            "batch needs %zu bytes of scratch; decode_batch_attn_noalloc holds "
                            "%zu (use decode_batch_attn with a handle for larger batches)",
                            need, kNoAllocScratchBytes);

    // once per device and context, with that device current: the scratch's
    // device address
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return noalloc_fail(SLOTKV_ERR_CUDA, "cudaGetDevice failed");
    unsigned char* scratch;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        unsigned long long ctx_id = 0;
        const bool known = current_context_id(&ctx_id);
        ScratchAddr& c = g_scratch_addr[dev];
        if (!known || !c.ptr || c.ctx_id != ctx_id) {
            // (the lookup also creates the device's primary context if no
            // context is current yet)
            void* ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || !ptr)
                return noalloc_fail(SLOTKV_ERR_CUDA, "cudaGetSymbolAddress: %s",
                                    cudaGetErrorString(e));
            if (!current_context_id(&ctx_id))
                return noalloc_fail(SLOTKV_ERR_CUDA, "no current CUDA context after set-up");
            c.ctx_id = ctx_id;
            c.ptr = ptr;
        }
        scratch = static_cast<unsigned char*>(c.ptr);
    }

    // the status word and the merge counters must start at zero
    cudaStream_t s = (cudaStream_t)stream;
    e = cudaMemsetAsync(scratch, 0, off_items, s);
    if (e != cudaSuccess)
        return noalloc_fail(SLOTKV_ERR_CUDA, "scratch clear: %s", cudaGetErrorString(e));

    // TMA descriptors for the caller's K and V (host-side encoding only)
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qres;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &qres) != cudaSuccess ||
        qres != cudaDriverEntryPointSuccess || !fn)
        return noalloc_fail(SLOTKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    encode_tiled_fn enc = reinterpret_cast<encode_tiled_fn>(fn);
    const uint32_t kv_dim = n_kv_head * head_dim;
    const cuuint64_t dims[2] = {kv_dim, (cuuint64_t)n_slots * slot_ctx};
    const cuuint64_t strides[1] = {(cuuint64_t)kv_dim * sizeof(float)};
    const cuuint32_t box[2] = {head_dim, (cuuint32_t)slotkv::tile_keys((int)head_dim)};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap tmK, tmV;
    if (enc(&tmK, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, K, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&tmV, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, V, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return noalloc_fail(SLOTKV_ERR_CUDA, "cuTensorMapEncodeTiled failed");

    slotkv::DecodeParams P;
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
    P.K = K;
    P.V = V;
    P.status = dev_flags ? dev_flags : reinterpret_cast<uint32_t*>(scratch);
    P.counters = reinterpret_cast<uint32_t*>(scratch + off_cnt);
    P.items = reinterpret_cast<uint32_t*>(scratch + off_items);
    P.plan = reinterpret_cast<uint32_t*>(scratch + off_plan);
    P.ws_ml = reinterpret_cast<float*>(scratch + off_ml);
    P.ws_acc = reinterpret_cast<float*>(scratch + off_acc);
    P.n_slots = n_slots;
    P.slot_ctx = slot_ctx;
    P.n_head = n_head;
    P.n_kv_head = n_kv_head;
    P.B = B;
    P.chunk_min = chunk_min;
    P.max_splits = kNoAllocMaxSplits;
    P.eps = eps;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.flags = 0;
    P.prefill = 0;
    const uint64_t bound = ((uint64_t)slot_ctx + chunk_min - 1) / chunk_min;
    const uint64_t splits = bound < kNoAllocMaxSplits ? bound : kNoAllocMaxSplits;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const uint64_t most = (uint64_t)B * n_kv_head * splits;
    const uint64_t want = 2ull * (uint64_t)(sms > 0 ? sms : 1);
    const unsigned ctas = (unsigned)(most < want ? most : want);
    const int G = (int)(n_head / n_kv_head);
    int rc;
    switch (head_dim) {
        case 64: rc = slotkv::launch_decode_hd64(G, P, tmK, tmV, ctas, s); break;
        case 128: rc = slotkv::launch_decode_hd128(G, P, tmK, tmV, ctas, s); break;
        default: rc = slotkv::launch_decode_hd256(G, P, tmK, tmV, ctas, s); break;
    }
    if (rc != 0)
        return noalloc_fail(SLOTKV_ERR_CUDA, "decode kernel launch: %s",
                            cudaGetErrorString((cudaError_t)rc));
    return SLOTKV_OK;
}

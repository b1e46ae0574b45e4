// decode_small.cuh -- the decode step for small calls: a few rows over short
// slots ("Forward Cuda Gemma", decodeBatch; the same step as
// slotkv_decode_attn_kernel, for calls whose work is too small to amortise
// the persistent kernel's set-up: mbarriers, register hand-over, TMA
// descriptor fetch and the producer / prep / consumer hand-offs).
//
// One CTA of four warps per (row b, kv head g), all keys of the row.  A
// call this small is bound by the latency of its dependent memory round
// trips, so the kernel has two on its critical path (p and the slot, then the
// history), with everything else fetched alongside:
//   1. at entry every thread loads positions[b] and slots[b] and issues
//      cp.async copies of the row's q (G heads), k_new, v_new, the norm
//      weights, inv_freq and the G sink logits into shared memory;
//   2. an out-of-range row (in paged mode: p past the table or a used entry
//      outside the pool, checked by every warp) raises SLOTKV_DEV_RANGE and
//      the CTA leaves with nothing written;
//   3. the history keys [0, p) are copied chunk by chunk (T keys of K and V,
//      16 KiB each) into shared memory with cp.async, two chunks in flight (a
//      paged block holds whole chunks: its size is a multiple of T);
//   4. meanwhile warp 0 forms k' = RoPE(RMSnorm(k_new) w) (and the weightless
//      norm of v_new under SLOTKV_OPT_VNORM) and writes K and V row p; warps
//      1-3 form the G query vectors q' = RoPE(RMSnorm(q) w) * scale * log2 e
//      (the decode kernel's vector routines, so the bits are the same);
//   5. the chunks are attended with the persistent kernel's consumer scheme
//      and routines (attend_rows / attend_rows_tr): groups of L lanes take one
//      key each, RC keys per softmax update, a base-2 online softmax whose
//      max is raised lazily; warp 0 then adds key p from shared memory;
//   6. each warp merges its key groups by halving (merge_warp_groups), the
//      four warps' (m, l, acc) merge through shared memory, the sink joins
//      the max and the denominator, and out is written.
// No spin-waits: only __syncthreads and cp.async groups.
#pragma once

#include "decode_attn.cuh"

namespace slotkv {

template <int HD, int G>
struct SCfg {
    static constexpr int T = tile_keys(HD);      // keys per chunk (the persistent kernel's tile)
    static constexpr int W = 4;                  // warps
    static constexpr int CHUNK = T * HD;         // floats per chunk of K (or V)
    // shared memory: K chunks [2] | V chunks [2] | q [G][HD] | k [HD] | v [HD]
    // | q norm weights [HD] | k norm weights [HD] | inv_freq [HD/2] | sinks [8]
    // | probabilities [NG][NV] of the transposed reduction; the merge reuses
    // the chunk space: acc [W][G][HD], m, l [W][G]
    static constexpr int OFF_V = 2 * CHUNK * 4;
    static constexpr int OFF_Q = 4 * CHUNK * 4;
    static constexpr int OFF_K1 = OFF_Q + G * HD * 4;
    static constexpr int OFF_V1 = OFF_K1 + HD * 4;
    static constexpr int OFF_QW = OFF_V1 + HD * 4;
    static constexpr int OFF_KW = OFF_QW + HD * 4;
    static constexpr int OFF_IF = OFF_KW + HD * 4;
    static constexpr int OFF_SK = OFF_IF + HD / 2 * 4;
    static constexpr int OFF_PG = OFF_SK + 8 * 4;
    static constexpr int SMEM = OFF_PG + KCfg<HD, G>::NG * KCfg<HD, G>::NV * 4;
    static_assert(KCfg<HD, G>::CONS == W * 32, "the consumer shapes assume four warps");
    static_assert(W * G * HD * 4 + 2 * W * G * 4 <= OFF_Q, "the merge fits in the chunk space");
    static_assert(CHUNK % (128 * 4) == 0, "whole 16-byte copies per thread");
    static_assert(OFF_PG % 16 == 0, "probabilities are read as float4");
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int HD, int G>
__global__ void __launch_bounds__(128) slotkv_decode_small_kernel(const DecodeParams P) {
    using C = SCfg<HD, G>;
    using KC = KCfg<HD, G>;
    constexpr int T = C::T, W = C::W, E = KC::E, L = KC::L;
    constexpr float kLog2e = 1.4426950408889634f;
    extern __shared__ __align__(1024) uint8_t smem[];
    float* kc = reinterpret_cast<float*>(smem);                // [2][T][HD]
    float* vc = reinterpret_cast<float*>(smem + C::OFF_V);     // [2][T][HD]
    float* qs = reinterpret_cast<float*>(smem + C::OFF_Q);     // [G][HD]
    float* k1 = reinterpret_cast<float*>(smem + C::OFF_K1);    // [HD]
    float* v1 = reinterpret_cast<float*>(smem + C::OFF_V1);    // [HD]
    float* qw = reinterpret_cast<float*>(smem + C::OFF_QW);    // [HD]
    float* kw = reinterpret_cast<float*>(smem + C::OFF_KW);    // [HD]
    float* ifr = reinterpret_cast<float*>(smem + C::OFF_IF);   // [HD / 2]
    float* sks = reinterpret_cast<float*>(smem + C::OFF_SK);   // [G]
    float* pgs = reinterpret_cast<float*>(smem + C::OFF_PG);   // [NG][NV] probabilities

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t b = blockIdx.x / P.n_kv_head, g = blockIdx.x % P.n_kv_head;
    const uint32_t p = __ldg(P.positions + b);
    const uint32_t* tab = P.block_tables ? P.block_tables + static_cast<size_t>(b) * P.bt_stride
                                         : nullptr;
    const uint32_t slot = tab ? 0u : __ldg(P.slots + b);
    // the row's vectors and the call's weights (none depends on p): q, k_new
    // and v_new are 16-byte aligned, the others 4-byte aligned
    {
        const size_t qat = (static_cast<size_t>(b) * P.n_head + g * G) * HD;
        const size_t kat = (static_cast<size_t>(b) * P.n_kv_head + g) * HD;
        for (int i = tid; i < G * HD / 4; i += 128) cp_async16(qs + 4 * i, P.q + qat + 4 * i);
        for (int i = tid; i < HD / 4; i += 128) {
            cp_async16(k1 + 4 * i, P.k_new + kat + 4 * i);
            cp_async16(v1 + 4 * i, P.v_new + kat + 4 * i);
        }
        for (int i = tid; i < HD; i += 128) {
            cp_async4(qw + i, P.q_norm_w + i);
            cp_async4(kw + i, P.k_norm_w + i);
        }
        for (int i = tid; i < HD / 2; i += 128) cp_async4(ifr + i, P.inv_freq + i);
        if (P.sinks && tid < G) cp_async4(sks + tid, P.sinks + g * G + tid);
        cp_async_commit();
    }
    bool ok;
    if (tab) {  // p within the table, every used entry (blocks 0 .. p / block) in the pool
        bool bad = static_cast<uint64_t>(p) >= static_cast<uint64_t>(P.bt_stride) * P.slot_ctx;
        const uint32_t used = bad ? 0u : p / P.slot_ctx + 1;
        for (uint32_t i = lane; i < used; i += 32) bad |= __ldg(tab + i) >= P.n_slots;
        ok = !__any_sync(0xffffffffu, bad);
    } else {
        ok = slot < P.n_slots && p < P.slot_ctx;
    }
    if (!ok) {
        cp_async_wait<0>();  // no copy outlives the CTA
        if (tid == 0) atomicOr(P.status, kDevRange);
        return;
    }
    // row of key t in the [rows][n_kv_head * HD] view of K and V; keys t .. t + T - 1
    // of a chunk start (t a multiple of T) are consecutive rows
    auto row_of = [&](uint32_t t) -> size_t {
        return tab ? static_cast<size_t>(__ldg(tab + t / P.slot_ctx)) * P.slot_ctx +
                         t % P.slot_ctx
                   : static_cast<size_t>(slot) * P.slot_ctx + t;
    };
    const size_t kvd = static_cast<size_t>(P.n_kv_head) * HD;
    const uint32_t nchunks = (p + T - 1) / T;  // chunks of keys [0, p)
    // history chunk c into buffer c & 1: keys [c T, min((c + 1) T, p))
    auto issue = [&](uint32_t c) {
        const uint32_t k0 = c * T;
        const uint32_t nk = p - k0 < static_cast<uint32_t>(T) ? p - k0 : T;
        const size_t r0 = row_of(k0);
        float* kd = kc + (c & 1) * C::CHUNK;
        float* vd = vc + (c & 1) * C::CHUNK;
        for (uint32_t i = tid; i < nk * (HD / 4); i += 128) {
            const uint32_t r = i / (HD / 4), c4 = i % (HD / 4);
            const size_t src = (r0 + r) * kvd + static_cast<size_t>(g) * HD + 4 * c4;
            cp_async16(kd + r * HD + 4 * c4, P.K + src);
            cp_async16(vd + r * HD + 4 * c4, P.V + src);
        }
        cp_async_commit();
    };
    if (nchunks > 0) issue(0);
    if (nchunks > 1) issue(1);
    // the vectors' group is the oldest: wait until at most the chunks' groups
    // are in flight
    if (nchunks > 1) cp_async_wait<2>();
    else if (nchunks == 1) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncthreads();

    // the row's vectors (bit for bit as the decode kernel's prep warp forms them)
    {
        float cs[HD / 64], sn[HD / 64];
        warp_rope_angles<HD>(p, ifr, cs, sn, lane);
        const float w1 = (P.flags & kOptNormPlusOne) ? 1.0f : 0.0f;
        if (warp == 0) {
            warp_norm_rope<HD>(k1, k1, kw, w1, 1.0f, P.eps, cs, sn, lane);
            if (P.flags & kOptVNorm) warp_rms_norm_plain<HD>(v1, v1, P.eps, lane);
            __syncwarp();
            // key p's K and V rows into the slot
            const size_t dst = row_of(p) * kvd + static_cast<size_t>(g) * HD;
#pragma unroll
            for (int j = 0; j < HD / 32; ++j) {
                P.K[dst + lane + 32 * j] = k1[lane + 32 * j];
                P.V[dst + lane + 32 * j] = v1[lane + 32 * j];
            }
        } else {
            for (int h = warp - 1; h < G; h += W - 1)
                warp_norm_rope<HD>(qs + h * HD, qs + h * HD, qw, w1, P.scale_log2, P.eps, cs, sn,
                                   lane);
        }
    }
    __syncthreads();
    // The persistent kernel's consumer scheme over the chunks: groups of L
    // lanes each take one key at a time, lane li of a group holding E
    // elements of the G queries and accumulators; RC keys per softmax update.
    float q[G][E], m[G], l[G], acc[G][E];
    float m_t[KC::CNT], l_t[KC::CNT];
    const int gid = tid / L, li = tid % L;
#pragma unroll
    for (int j = 0; j < KC::CNT; ++j) {
        m_t[j] = -CUDART_INF_F;
        l_t[j] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int c = 0; c < E / 4; ++c) {
            const float4 v = *reinterpret_cast<const float4*>(qs + h * HD + c * 4 * L + li * 4);
            q[h][4 * c + 0] = v.x;
            q[h][4 * c + 1] = v.y;
            q[h][4 * c + 2] = v.z;
            q[h][4 * c + 3] = v.w;
        }
        m[h] = -CUDART_INF_F;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[h][e] = 0.f;
    }
    for (uint32_t c = 0; c < nchunks; ++c) {
        if (c + 1 < nchunks) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();  // chunk c is in shared memory for every thread
        const uint32_t nk = p - c * T < static_cast<uint32_t>(T) ? p - c * T : T;
        const float* Kt = kc + (c & 1) * C::CHUNK;
        const float* Vt = vc + (c & 1) * C::CHUNK;
#pragma unroll
        for (int r0 = 0; r0 < KC::R; r0 += KC::RC) {
            int row[KC::RC];
            bool valid[KC::RC];
#pragma unroll
            for (int r = 0; r < KC::RC; ++r) {
                row[r] = gid + KC::NG * (r0 + r);
                valid[r] = static_cast<uint32_t>(row[r]) < nk;
            }
            if constexpr (KC::TR)
                attend_rows_tr<HD, G, E, L, KC::RC, KC::GP, KC::CNT>(Kt, Vt, row, valid, li, lane,
                                                                     q, m_t, l_t, acc,
                                                                     pgs + gid * KC::NV);
            else
                attend_rows<HD, G, E, L, KC::RC>(Kt, Vt, row, valid, li, q, m, l, acc);
        }
        __syncthreads();  // buffer c & 1 is free again
        if (c + 2 < nchunks) issue(c + 2);
    }
    if constexpr (KC::TR) tr_state_to_heads<G, L, KC::RC, KC::GP, KC::CNT>(li, lane, m_t, l_t, m, l);
    if (warp == 0) {  // key p: the row's own k' and v
        const int row1[1] = {0};
        const bool valid1[1] = {gid == 0};
        attend_rows<HD, G, E, L, 1>(k1, v1, row1, valid1, li, q, m, l, acc);
    }
    // merge the key groups of each warp, then the four warps through shared
    // memory (the chunk space): acc [W][G][HD], m, l [W][G]
    constexpr int EF = HD / 32;
    const int e0 = merge_warp_groups<G, E, L>(lane, m, l, acc);
    float* macc = reinterpret_cast<float*>(smem);
    float* mm = macc + W * G * HD;
    float* ml = mm + W * G;
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int t = 0; t < EF; t += 2) {
            const int d = ((e0 + t) >> 2) * 4 * L + 4 * li + ((e0 + t) & 3);
            *reinterpret_cast<float2*>(macc + (warp * G + h) * HD + d) =
                make_float2(acc[h][t], acc[h][t + 1]);
        }
        if (lane == 0) {
            mm[warp * G + h] = m[h];
            ml[warp * G + h] = l[h];
        }
    }
    __syncthreads();
    for (int i = tid; i < G * HD / 4; i += 128) {
        const int h = i / (HD / 4), d4 = i % (HD / 4);
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w2 = 0; w2 < W; ++w2) M = fmaxf(M, mm[w2 * G + h]);
        float Ls = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w2 = 0; w2 < W; ++w2) {
            const float wt = partial_weight(mm[w2 * G + h], M);
            const float4 a = reinterpret_cast<const float4*>(macc + (w2 * G + h) * HD)[d4];
            Ls = __fmaf_rn(ml[w2 * G + h], wt, Ls);
            o.x = __fmaf_rn(a.x, wt, o.x);
            o.y = __fmaf_rn(a.y, wt, o.y);
            o.z = __fmaf_rn(a.z, wt, o.z);
            o.w = __fmaf_rn(a.w, wt, o.w);
        }
        float cs = 1.f;
        if (P.sinks) {
            const float sk = sks[h] * kLog2e;
            const float M2 = fmaxf(M, sk);
            cs = exp2f(M - M2);
            Ls = __fmaf_rn(Ls, cs, exp2f(sk - M2));
        }
        const float f = __fmul_rn(cs, __frcp_rn(Ls));
        reinterpret_cast<float4*>(P.out + (static_cast<size_t>(b) * P.n_head + g * G + h) * HD)[d4] =
            make_float4(__fmul_rn(o.x, f), __fmul_rn(o.y, f), __fmul_rn(o.z, f),
                        __fmul_rn(o.w, f));
    }
}

template <int HD, int G>
int launch_small_one(const DecodeParams& p, cudaStream_t stream) {
    using C = SCfg<HD, G>;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!(configured.load(std::memory_order_acquire) & bit) || bit == 0) {
        cudaError_t e = cudaFuncSetAttribute(slotkv_decode_small_kernel<HD, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return static_cast<int>(e);
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    slotkv_decode_small_kernel<HD, G><<<p.B * p.n_kv_head, 128, C::SMEM, stream>>>(p);
    return static_cast<int>(cudaGetLastError());
}

template <int HD>
int launch_small_hd(int G, const DecodeParams& p, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_small_one<HD, 1>(p, stream);
        case 2: return launch_small_one<HD, 2>(p, stream);
        case 3: return launch_small_one<HD, 3>(p, stream);
        case 4: return launch_small_one<HD, 4>(p, stream);
        case 5: return launch_small_one<HD, 5>(p, stream);
        case 6: return launch_small_one<HD, 6>(p, stream);
        case 7: return launch_small_one<HD, 7>(p, stream);
        case 8: return launch_small_one<HD, 8>(p, stream);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace slotkv

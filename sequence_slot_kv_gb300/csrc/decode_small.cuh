// decode_small.cuh -- the decode step for small calls: a few rows over short
// slots ("Forward Cuda Gemma", decodeBatch; the same step as
// slotkv_decode_attn_kernel, for calls whose work is too small to amortise
// the persistent kernel's set-up: mbarriers, register hand-over, TMA
// descriptor fetch and the producer / prep / consumer hand-offs).
//
// One CTA of four warps per (row b, kv head g), all keys of the row:
//   1. every thread loads positions[b] and slots[b]; an out-of-range row
//      raises SLOTKV_DEV_RANGE and the CTA leaves (nothing written);
//   2. the history keys [0, p) are copied chunk by chunk (T keys of K and V,
//      16 KiB each) into shared memory with cp.async, two chunks in flight;
//   3. meanwhile warp 0 forms k' = RoPE(RMSnorm(k_new) w) (and the weightless
//      norm of v_new under SLOTKV_OPT_VNORM) and writes K and V row p; warps
//      1-3 form the G query vectors q' = RoPE(RMSnorm(q) w) * scale * log2 e
//      (the decode kernel's vector routines, so the bits are the same);
//   4. warp w attends keys w, w + 4, ... of every chunk, four keys per
//      softmax update: per lane hd / 32 elements of each vector, dots summed
//      by a butterfly over the warp, a base-2 online softmax (max raised
//      lazily, by 2^8), acc += p v; warp 0 then adds key p from shared memory;
//   5. the four warps' (m, l, acc) merge through shared memory, the sink joins
//      the max and the denominator, and out is written.
// No spin-waits: only __syncthreads and cp.async groups.
#pragma once

#include "decode_attn.cuh"

namespace slotkv {

template <int HD, int G>
struct SCfg {
    static constexpr int T = tile_keys(HD);      // keys per chunk
    static constexpr int E = HD / 32;            // elements per lane per vector
    static constexpr int W = 4;                  // warps
    static constexpr int RC = 4;                 // keys per softmax update
    static constexpr int CHUNK = T * HD;         // floats per chunk of K (or V)
    // shared memory: K chunks [2] | V chunks [2] | q [G][HD] | k [HD] | v [HD]
    // | p, slot; the merge reuses the chunk space: acc [W][G][HD], m, l [W][G]
    static constexpr int OFF_V = 2 * CHUNK * 4;
    static constexpr int OFF_Q = 4 * CHUNK * 4;
    static constexpr int OFF_K1 = OFF_Q + G * HD * 4;
    static constexpr int OFF_V1 = OFF_K1 + HD * 4;
    static constexpr int SMEM = OFF_V1 + HD * 4;
    static_assert(W * G * HD * 4 + 2 * W * G * 4 <= OFF_Q, "the merge fits in the chunk space");
    static_assert(CHUNK % (128 * 4) == 0, "whole 16-byte copies per thread");
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)),
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
    constexpr int T = C::T, E = C::E, W = C::W, RC = C::RC;
    constexpr float kLog2e = 1.4426950408889634f;
    extern __shared__ __align__(16) uint8_t smem[];
    float* kc = reinterpret_cast<float*>(smem);                // [2][T][HD]
    float* vc = reinterpret_cast<float*>(smem + C::OFF_V);     // [2][T][HD]
    float* qs = reinterpret_cast<float*>(smem + C::OFF_Q);     // [G][HD]
    float* k1 = reinterpret_cast<float*>(smem + C::OFF_K1);    // [HD]
    float* v1 = reinterpret_cast<float*>(smem + C::OFF_V1);    // [HD]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t b = blockIdx.x / P.n_kv_head, g = blockIdx.x % P.n_kv_head;
    const uint32_t p = __ldg(P.positions + b), slot = __ldg(P.slots + b);
    if (slot >= P.n_slots || p >= P.slot_ctx) {
        if (tid == 0) atomicOr(P.status, kDevRange);
        return;
    }
    const size_t kvd = static_cast<size_t>(P.n_kv_head) * HD;
    const size_t row0 = static_cast<size_t>(slot) * P.slot_ctx;  // row of key 0
    const uint32_t nchunks = (p + T - 1) / T;                    // chunks of keys [0, p)
    // history chunk c into buffer c & 1: keys [c T, min((c + 1) T, p))
    auto issue = [&](uint32_t c) {
        const uint32_t k0 = c * T;
        const uint32_t nk = p - k0 < static_cast<uint32_t>(T) ? p - k0 : T;
        float* kd = kc + (c & 1) * C::CHUNK;
        float* vd = vc + (c & 1) * C::CHUNK;
        for (uint32_t i = tid; i < nk * (HD / 4); i += 128) {
            const uint32_t r = i / (HD / 4), c4 = i % (HD / 4);
            const size_t src = (row0 + k0 + r) * kvd + static_cast<size_t>(g) * HD + 4 * c4;
            cp_async16(kd + r * HD + 4 * c4, P.K + src);
            cp_async16(vd + r * HD + 4 * c4, P.V + src);
        }
        cp_async_commit();
    };
    if (nchunks > 0) issue(0);
    if (nchunks > 1) issue(1);

    // the row's vectors (bit for bit as the decode kernel's prep warp forms them)
    {
        float cs[HD / 64], sn[HD / 64];
        warp_rope_angles<HD>(p, P.inv_freq, cs, sn, lane);
        const float w1 = (P.flags & kOptNormPlusOne) ? 1.0f : 0.0f;
        if (warp == 0) {
            const size_t at = (static_cast<size_t>(b) * P.n_kv_head + g) * HD;
            warp_norm_rope<HD>(P.k_new + at, k1, P.k_norm_w, w1, 1.0f, P.eps, cs, sn, lane);
            if (P.flags & kOptVNorm) {
                warp_rms_norm_plain<HD>(P.v_new + at, v1, P.eps, lane);
            } else {
#pragma unroll
                for (int j = 0; j < HD / 32; ++j) v1[lane + 32 * j] = P.v_new[at + lane + 32 * j];
            }
            __syncwarp();
            // key p's K and V rows into the slot
            const size_t dst = (row0 + p) * kvd + static_cast<size_t>(g) * HD;
#pragma unroll
            for (int j = 0; j < HD / 32; ++j) {
                P.K[dst + lane + 32 * j] = k1[lane + 32 * j];
                P.V[dst + lane + 32 * j] = v1[lane + 32 * j];
            }
        } else {
            for (int h = warp - 1; h < G; h += W - 1) {
                const size_t at = (static_cast<size_t>(b) * P.n_head + g * G + h) * HD;
                warp_norm_rope<HD>(P.q + at, qs + h * HD, P.q_norm_w, w1, P.scale_log2, P.eps,
                                   cs, sn, lane);
            }
        }
    }
    __syncthreads();
    // lane's slice: elements lane * E .. lane * E + E - 1 of each vector
    float q[G][E], acc[G][E], m[G], l[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            q[h][e] = qs[h * HD + lane * E + e];
            acc[h][e] = 0.f;
        }
        m[h] = -CUDART_INF_F;
        l[h] = 0.f;
    }
    // attend up to RC keys (rows of kt / vt); valid[r] false: a key to skip
    auto attend = [&](const float* kt, const float* vt, const int (&rowi)[RC],
                      const bool (&valid)[RC]) {
        float s[RC][G];
#pragma unroll
        for (int r = 0; r < RC; ++r) {
            float kv[E];
#pragma unroll
            for (int e = 0; e < E; ++e) kv[e] = valid[r] ? kt[rowi[r] * HD + lane * E + e] : 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) d = fmaf(q[h][e], kv[e], d);
                s[r][h] = d;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int r = 0; r < RC; ++r) {
#pragma unroll
                for (int h = 0; h < G; ++h) s[r][h] += __shfl_xor_sync(0xffffffffu, s[r][h], off);
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int r = 0; r < RC; ++r) mx = valid[r] ? fmaxf(mx, s[r][h]) : mx;
            if (mx > m[h] + 8.f) {
                const float corr = m[h] == -CUDART_INF_F ? 0.f : exp2f(m[h] - mx);
                l[h] *= corr;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[h][e] *= corr;
                m[h] = mx;
            }
        }
#pragma unroll
        for (int r = 0; r < RC; ++r) {
            if (!valid[r]) continue;
            float vv[E];
#pragma unroll
            for (int e = 0; e < E; ++e) vv[e] = vt[rowi[r] * HD + lane * E + e];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pr = exp2f(s[r][h] - m[h]);
                l[h] += pr;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[h][e] = fmaf(pr, vv[e], acc[h][e]);
            }
        }
    };
    for (uint32_t c = 0; c < nchunks; ++c) {
        if (c + 1 < nchunks) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();  // chunk c is in shared memory for every thread
        const uint32_t k0 = c * T;
        const uint32_t nk = p - k0 < static_cast<uint32_t>(T) ? p - k0 : T;
        const float* kt = kc + (c & 1) * C::CHUNK;
        const float* vt = vc + (c & 1) * C::CHUNK;
        // warp w: keys w, w + W, ... of the chunk, RC at a time
        for (uint32_t r0 = warp; r0 < nk; r0 += W * RC) {
            int rowi[RC];
            bool valid[RC];
#pragma unroll
            for (int r = 0; r < RC; ++r) {
                rowi[r] = static_cast<int>(r0 + r * W);
                valid[r] = r0 + r * W < nk;
                rowi[r] = valid[r] ? rowi[r] : 0;
            }
            attend(kt, vt, rowi, valid);
        }
        __syncthreads();  // buffer c & 1 is free again
        if (c + 2 < nchunks) issue(c + 2);
    }
    if (warp == 0) {  // key p: the row's own k' and v
        const int rowi[RC] = {0, 0, 0, 0};
        const bool valid[RC] = {true, false, false, false};
        attend(k1, v1, rowi, valid);
    }
    // merge the four warps' partials through shared memory (the chunk space)
    float* macc = reinterpret_cast<float*>(smem);              // [W][G][HD]
    float* mm = macc + W * G * HD;                             // [W][G]
    float* ml = mm + W * G;                                    // [W][G]
    __syncthreads();  // the chunk space is no longer read
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int e = 0; e < E; ++e) macc[(warp * G + h) * HD + lane * E + e] = acc[h][e];
        if (lane == 0) {
            mm[warp * G + h] = m[h];
            ml[warp * G + h] = l[h];
        }
    }
    __syncthreads();
    for (int i = tid; i < G * HD; i += 128) {
        const int h = i / HD, d = i % HD;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w2 = 0; w2 < W; ++w2) M = fmaxf(M, mm[w2 * G + h]);
        float L = 0.f, o = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < W; ++w2) {
            const float wt = partial_weight(mm[w2 * G + h], M);
            L = fmaf(ml[w2 * G + h], wt, L);
            o = fmaf(macc[(w2 * G + h) * HD + d], wt, o);
        }
        if (P.sinks) {
            const float sk = __ldg(P.sinks + g * G + h) * kLog2e;
            const float M2 = fmaxf(M, sk);
            const float c = exp2f(M - M2);
            L = fmaf(L, c, exp2f(sk - M2));
            o *= c;
        }
        P.out[(static_cast<size_t>(b) * P.n_head + g * G + h) * HD + d] = o / L;
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

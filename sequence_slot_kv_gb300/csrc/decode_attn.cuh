// decode_attn.cuh -- the fused batched decode attention kernel over slot KV.
//
// One CTA handles one work item (row b, kv head g, split s): the keys
// [s*C, min((s+1)*C, p+1)) of slot slots[b] for the G query heads that share
// kv head g (GQA), so every history K/V byte is read from HBM exactly once.
//
// Per CTA (the steps of "Forward Cuda Gemma", decodeBatch, fused):
//   * warp 4 (producer): streams the history K and V tiles of the chunk into
//     a 3-stage shared-memory ring with 2-D TMA copies (cp.async.bulk.tensor,
//     one [T keys x hd] box per tensor per stage) signalled on mbarriers;
//   * warps 0-3 (consumers): meanwhile per-head RMS-norm + RoPE of the G query
//     vectors (pre-multiplied by scale*log2 e) and, in the split holding key p,
//     of k_new; then for each tile, groups of L lanes each own one key: every
//     lane holds E = hd/L elements of the G queries and of G output
//     accumulators in registers, forms partial dots, reduces them with
//     xor-shuffles, and runs a base-2 online softmax that rescales only when
//     its running max grows;
//   * the split holding key p adds that key from shared memory (its K is the
//     freshly normed+rotated k', its V the raw v_new) and writes both rows to
//     the slot buffers at (slot*slot_ctx + p)*kv_dim;
//   * the groups' (m, l, acc) are merged in shared memory; a single-split row
//     writes out directly, otherwise the partial goes to the workspace and the
//     last CTA of the (row, kv head) to finish merges the splits in split order.
//
// Every wait on an mbarrier is bounded; on expiry the CTA raises
// SLOTKV_DEV_TIMEOUT, drains its own copies in flight (bounded) and returns.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "params.h"

namespace slotkv {

constexpr uint32_t kDevRange = 1u;
constexpr uint32_t kDevTimeout = 2u;

__host__ __device__ constexpr int pow2_floor(int x) {
    int r = 1;
    while (r * 2 <= x) r *= 2;
    return r;
}
__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int HD, int G>
struct KCfg {
    static constexpr int W = 4;                   // consumer warps
    static constexpr int CONS = W * 32;           // consumer threads
    static constexpr int THREADS = CONS + 32;     // + one producer warp
    static constexpr int S = 3;                   // pipeline stages
    static constexpr int T = tile_keys(HD);       // keys per tile
    // elements per lane: keep G*E <= 64 (queries + accumulators in registers)
    static constexpr int E = cmax(4, cmax(HD / 32, cmin(32, pow2_floor(64 / G))));
    static constexpr int L = HD / E;              // lanes per key group
    static constexpr int NG = CONS / L;           // key groups per CTA
    static constexpr int R = T / NG;              // keys per group per tile
    // keys attended per softmax update: keeps the live scores (RC*G) <= 16
    static constexpr int RC = pow2_floor(cmax(1, cmin(R, 16 / G)));
    static constexpr int TILE_BYTES = T * HD * 4;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int OFF_QS = S * STAGE_BYTES;
    static constexpr int OFF_KS = OFF_QS + G * HD * 4;
    static constexpr int OFF_VS = OFF_KS + HD * 4;
    static constexpr int OFF_CS = OFF_VS + HD * 4;
    static constexpr int OFF_SN = OFF_CS + HD * 2;
    static constexpr int OFF_BAR = OFF_SN + HD * 2;
    static constexpr int OFF_MISC = OFF_BAR + 2 * S * 8;
    static constexpr int SMEM = OFF_MISC + 16;
    static_assert(L >= 1 && L <= 32 && (32 % L) == 0, "lane group must divide a warp");
    static_assert(E % 4 == 0 && E * L == HD, "lane slice must be whole float4s");
    static_assert(R >= 1 && R * NG == T, "tile must split evenly over the groups");
    static_assert(R % RC == 0, "row chunks must divide the rows per tile");
    static_assert(G * E <= 64, "register budget");
    // merge scratch (reuses the stage ring): acc [NG][G][HD], m, l [NG][G],
    // merged max/sum [G], weights [NG][G] or [G][max_splits]
    static_assert(NG * G * HD * 4 + 4 * NG * G * 4 + 2 * G * 4 + G * 256 * 4 <=
                      S * STAGE_BYTES,
                  "merge scratch must fit in the stage ring");
    static_assert(HD == 64 || HD == 128 || HD == 256, "head dim");
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with parity `parity` to complete.  Bounded by
// both an iteration count and about 2^31 SM clocks (~1 s); false on expiry.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          long long clock_limit = (1ll << 31)) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > clock_limit) break;
    }
    return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

template <int N>
__device__ __forceinline__ void named_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// Attend NR keys held in shared memory rows (row[r] of the K tile Kt and V
// tile Vt, hd floats each).  Lane `li` of its L-lane group owns elements
// c*4L + 4*li + {0..3}, c < E/4, of every vector.  All 32 lanes of the warp
// must call this together (the reductions shuffle across the whole warp).
template <int HD, int G, int E, int L, int NR>
__device__ __forceinline__ void attend_rows(const float* __restrict__ Kt,
                                            const float* __restrict__ Vt,
                                            const int (&row)[NR], const bool (&valid)[NR],
                                            const int li, const float (&q)[G][E],
                                            float (&m)[G], float (&l)[G],
                                            float (&acc)[G][E]) {
    float s[NR][G];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float* kp = Kt + row[r] * HD + li * 4;
        float kv[E];
#pragma unroll
        for (int c = 0; c < E / 4; ++c) {
            const float4 v = *reinterpret_cast<const float4*>(kp + c * 4 * L);
            kv[4 * c + 0] = v.x;
            kv[4 * c + 1] = v.y;
            kv[4 * c + 2] = v.z;
            kv[4 * c + 3] = v.w;
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) d = fmaf(q[h][e], kv[e], d);
            s[r][h] = d;
        }
    }
#pragma unroll
    for (int off = 1; off < L; off <<= 1) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
#pragma unroll
            for (int h = 0; h < G; ++h) s[r][h] += __shfl_xor_sync(0xffffffffu, s[r][h], off);
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
#pragma unroll
        for (int h = 0; h < G; ++h) s[r][h] = valid[r] ? s[r][h] : -CUDART_INF_F;
    }
    // online softmax in base 2: rescale only when the running max grows
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float mx = s[0][h];
#pragma unroll
        for (int r = 1; r < NR; ++r) mx = fmaxf(mx, s[r][h]);
        if (mx > m[h]) {
            const float corr = exp2f(m[h] - mx);
            l[h] *= corr;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[h][e] *= corr;
            m[h] = mx;
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        if (valid[r]) {
            const float* vp = Vt + row[r] * HD + li * 4;
            float vv[E];
#pragma unroll
            for (int c = 0; c < E / 4; ++c) {
                const float4 v = *reinterpret_cast<const float4*>(vp + c * 4 * L);
                vv[4 * c + 0] = v.x;
                vv[4 * c + 1] = v.y;
                vv[4 * c + 2] = v.z;
                vv[4 * c + 3] = v.w;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pr = exp2f(s[r][h] - m[h]);
                l[h] += pr;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[h][e] = fmaf(pr, vv[e], acc[h][e]);
            }
        }
    }
}

template <int HD, int G>
__global__ void __launch_bounds__(KCfg<HD, G>::THREADS, 2)
    slotkv_decode_attn_kernel(const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmV,
                              const DecodeParams P) {
    using C = KCfg<HD, G>;
    constexpr int E = C::E, L = C::L, NG = C::NG, R = C::R, T = C::T, S = C::S;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t split = blockIdx.x;
    const uint32_t kvh = blockIdx.y;
    const uint32_t b = blockIdx.z;

    const uint32_t p = P.positions[b];
    const uint32_t slot = P.slots[b];
    if (slot >= P.n_slots || p >= P.slot_ctx) {
        if (split == 0 && kvh == 0 && tid == 0) atomicOr(P.status, kDevRange);
        return;
    }
    const uint32_t n_keys = p + 1;
    const uint32_t chunk = split_chunk(n_keys, P.chunk_min, P.max_splits, T);
    const uint32_t nsplit = (n_keys + chunk - 1) / chunk;
    if (split >= nsplit) return;
    const uint32_t k0 = split * chunk;
    const bool is_last = split == nsplit - 1;
    // keys read from the slot buffers: [k0, hist_end); key p comes from k_new
    const uint32_t hist_end = is_last ? p : k0 + chunk;
    const uint32_t n_hist = hist_end > k0 ? hist_end - k0 : 0;
    const uint32_t ntiles = (n_hist + T - 1) / T;
    const int row_k0 = static_cast<int>(slot * P.slot_ctx + k0);

    float* qs = reinterpret_cast<float*>(smem + C::OFF_QS);
    float* ks = reinterpret_cast<float*>(smem + C::OFF_KS);
    float* vs = reinterpret_cast<float*>(smem + C::OFF_VS);
    float* cs = reinterpret_cast<float*>(smem + C::OFF_CS);
    float* sn = reinterpret_cast<float*>(smem + C::OFF_SN);
    const uint32_t full0 = smem_addr(smem + C::OFF_BAR);
    const uint32_t empty0 = full0 + 8 * S;
    volatile int* misc = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
    // misc[0]: abort, misc[1]: this CTA merges the splits, misc[2]: tiles issued

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, C::W);
        }
        misc[0] = 0;
        misc[1] = 0;
        misc[2] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    // ---------------------------------------------------------------- producer
    if (warp == C::W) {
        if (lane == 0) {
            for (uint32_t t = 0; t < ntiles; ++t) {
                const int st = t % S;
                if (t >= static_cast<uint32_t>(S)) {
                    if (!mbar_wait(empty0 + 8 * st, ((t / S) - 1) & 1)) {
                        atomicOr(P.status, kDevTimeout);
                        misc[0] = 1;
                        break;
                    }
                }
                if (misc[0]) break;
                const uint32_t full = full0 + 8 * st;
                const uint32_t dst = smem_addr(smem + st * C::STAGE_BYTES);
                mbar_expect_tx(full, C::STAGE_BYTES);
                tma_load_2d(dst, &tmK, static_cast<int>(kvh * HD), row_k0 + static_cast<int>(t * T),
                            full);
                tma_load_2d(dst + C::TILE_BYTES, &tmV, static_cast<int>(kvh * HD),
                            row_k0 + static_cast<int>(t * T), full);
                misc[2] = static_cast<int>(t + 1);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // cos/sin of the f32 RoPE angles fl32(p * inv_freq[i])
    const float fp = static_cast<float>(p);
    for (int i = tid; i < HD / 2; i += C::CONS) {
        float s_, c_;
        sincosf(__fmul_rn(fp, P.inv_freq[i]), &s_, &c_);
        sn[i] = s_;
        cs[i] = c_;
    }
    named_sync<C::CONS>();
    {
        // per-head RMS norm + RoPE: the G query heads of this kv head, and k_new
        // in the split that owns key p.  One warp per head vector.
        const int nvec = G + (is_last ? 1 : 0);
        constexpr int PPL = HD / 64;  // rotation pairs per lane
        for (int x = warp; x < nvec; x += C::W) {
            const bool isq = x < G;
            const float* src = isq ? P.q + (static_cast<size_t>(b) * P.n_head + kvh * G + x) * HD
                                   : P.k_new + (static_cast<size_t>(b) * P.n_kv_head + kvh) * HD;
            const float* w = isq ? P.q_norm_w : P.k_norm_w;
            float x0[PPL], x1[PPL];
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < PPL; ++j) {
                x0[j] = src[lane + 32 * j];
                x1[j] = src[lane + 32 * j + HD / 2];
                ss = fmaf(x0[j], x0[j], ss);
                ss = fmaf(x1[j], x1[j], ss);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = 1.0f / sqrtf(ss * (1.0f / HD) + P.eps);
            const float mul = isq ? P.scale_log2 : 1.0f;
            float* dst = isq ? qs + x * HD : ks;
#pragma unroll
            for (int j = 0; j < PPL; ++j) {
                const int i = lane + 32 * j;
                const float y0 = x0[j] * inv * w[i];
                const float y1 = x1[j] * inv * w[i + HD / 2];
                dst[i] = (y0 * cs[i] - y1 * sn[i]) * mul;
                dst[i + HD / 2] = (y1 * cs[i] + y0 * sn[i]) * mul;
            }
        }
        if (is_last) {
            const float* vsrc = P.v_new + (static_cast<size_t>(b) * P.n_kv_head + kvh) * HD;
            for (int d = tid; d < HD; d += C::CONS) vs[d] = vsrc[d];
        }
    }
    named_sync<C::CONS>();

    const int gid = warp * (32 / L) + lane / L;  // key group
    const int li = lane % L;                     // lane within the group
    float q[G][E], m[G], l[G], acc[G][E];
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

    for (uint32_t t = 0; t < ntiles; ++t) {
        const int st = t % S;
        if (misc[0] || !mbar_wait(full0 + 8 * st, (t / S) & 1)) {
            atomicOr(P.status, kDevTimeout);
            misc[0] = 1;
            break;
        }
        const float* Kt = reinterpret_cast<const float*>(smem + st * C::STAGE_BYTES);
        const float* Vt = Kt + T * HD;
        const uint32_t kbase = k0 + t * T;
#pragma unroll
        for (int r0 = 0; r0 < R; r0 += C::RC) {
            int row[C::RC];
            bool valid[C::RC];
#pragma unroll
            for (int r = 0; r < C::RC; ++r) {
                row[r] = gid + NG * (r0 + r);
                valid[r] = kbase + static_cast<uint32_t>(row[r]) < hist_end;
            }
            attend_rows<HD, G, E, L, C::RC>(Kt, Vt, row, valid, li, q, m, l, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
    }
    // every consumer warp is past the ring; an abort by any of them is visible
    named_sync<C::CONS>();
    if (misc[0]) {
        // drain this CTA's own copies that may still be in flight: the newest
        // issued tile of each stage (older phases have completed already)
        if (tid == 0) {
            const uint32_t issued = static_cast<uint32_t>(misc[2]);
            for (uint32_t u = issued > static_cast<uint32_t>(S) ? issued - S : 0; u < issued; ++u)
                mbar_wait(full0 + 8 * (u % S), (u / S) & 1, 1ll << 28);
        }
        named_sync<C::CONS>();
        return;
    }
    if (is_last && warp == 0) {
        const int row1[1] = {0};
        const bool valid1[1] = {gid == 0};
        attend_rows<HD, G, E, L, 1>(ks, vs, row1, valid1, li, q, m, l, acc);
    }

    // ---------------------------------------------- merge the groups' partials
    named_sync<C::CONS>();  // warp 0 is done with key p
    float* red_acc = reinterpret_cast<float*>(smem);  // [NG][G][HD]
    float* red_m = red_acc + NG * G * HD;             // [NG][G]
    float* red_l = red_m + NG * G;                    // [NG][G]
    float* wgt = red_l + NG * G;                      // [NG][G]
    float* hM = wgt + NG * G;                         // [G]
    float* hL = hM + G;                               // [G]
    float* sw = hL + G;                               // [G][<=256]
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int c = 0; c < E / 4; ++c) {
            *reinterpret_cast<float4*>(red_acc + (gid * G + h) * HD + c * 4 * L + li * 4) =
                make_float4(acc[h][4 * c], acc[h][4 * c + 1], acc[h][4 * c + 2], acc[h][4 * c + 3]);
        }
        if (li == 0) {
            red_m[gid * G + h] = m[h];
            red_l[gid * G + h] = l[h];
        }
    }
    named_sync<C::CONS>();
    if (tid < G) {
        float M = -CUDART_INF_F;
        for (int g = 0; g < NG; ++g) M = fmaxf(M, red_m[g * G + tid]);
        float Ls = 0.f;
        for (int g = 0; g < NG; ++g) Ls += red_l[g * G + tid] * exp2f(red_m[g * G + tid] - M);
        hM[tid] = M;
        hL[tid] = Ls;
    }
    named_sync<C::CONS>();
    for (int i = tid; i < NG * G; i += C::CONS) wgt[i] = exp2f(red_m[i] - hM[i % G]);
    named_sync<C::CONS>();

    const uint32_t hq0 = kvh * G;  // first query head of this kv head
    constexpr float kLog2e = 1.4426950408889634f;
    if (nsplit == 1) {
        for (int o = tid; o < G * HD; o += C::CONS) {
            const int h = o / HD, d = o % HD;
            float A = 0.f;
            for (int g = 0; g < NG; ++g) A = fmaf(red_acc[(g * G + h) * HD + d], wgt[g * G + h], A);
            float M = hM[h], Ls = hL[h], c = 1.f;
            if (P.sinks) {
                const float sk = P.sinks[hq0 + h] * kLog2e;
                const float M2 = fmaxf(M, sk);
                c = exp2f(M - M2);
                Ls = Ls * c + exp2f(sk - M2);
            }
            P.out[(static_cast<size_t>(b) * P.n_head + hq0 + h) * HD + d] = (A * c) / Ls;
        }
    } else {
        const size_t MS = P.max_splits;
        for (int o = tid; o < G * HD; o += C::CONS) {
            const int h = o / HD, d = o % HD;
            float A = 0.f;
            for (int g = 0; g < NG; ++g) A = fmaf(red_acc[(g * G + h) * HD + d], wgt[g * G + h], A);
            const size_t base = (static_cast<size_t>(b) * P.n_head + hq0 + h) * MS + split;
            P.ws_acc[base * HD + d] = A;
            if (d == 0) {
                P.ws_ml[base * 2 + 0] = hM[h];
                P.ws_ml[base * 2 + 1] = hL[h];
            }
        }
        __threadfence();
        named_sync<C::CONS>();
        uint32_t* counter = P.counters + static_cast<size_t>(b) * P.n_kv_head + kvh;
        if (tid == 0) misc[1] = atomicAdd(counter, 1u) == nsplit - 1 ? 1 : 0;
        named_sync<C::CONS>();
        if (misc[1]) {
            // the last CTA of (row, kv head) to finish merges the splits, in
            // split order, so the result does not depend on finishing order
            __threadfence();
            if (tid < G) {
                const size_t base = (static_cast<size_t>(b) * P.n_head + hq0 + tid) * MS;
                float M = -CUDART_INF_F;
                for (uint32_t s2 = 0; s2 < nsplit; ++s2) M = fmaxf(M, __ldcg(P.ws_ml + (base + s2) * 2));
                float Ls = 0.f;
                for (uint32_t s2 = 0; s2 < nsplit; ++s2)
                    Ls += __ldcg(P.ws_ml + (base + s2) * 2 + 1) *
                          exp2f(__ldcg(P.ws_ml + (base + s2) * 2) - M);
                if (P.sinks) {
                    const float sk = P.sinks[hq0 + tid] * kLog2e;
                    const float M2 = fmaxf(M, sk);
                    Ls = Ls * exp2f(M - M2) + exp2f(sk - M2);
                    M = M2;
                }
                hM[tid] = M;
                hL[tid] = Ls;
            }
            named_sync<C::CONS>();
            for (uint32_t i = tid; i < G * nsplit; i += C::CONS) {
                const uint32_t h = i / nsplit, s2 = i % nsplit;
                const size_t base = (static_cast<size_t>(b) * P.n_head + hq0 + h) * MS + s2;
                sw[h * nsplit + s2] = exp2f(__ldcg(P.ws_ml + base * 2) - hM[h]);
            }
            named_sync<C::CONS>();
            for (int o = tid; o < G * HD; o += C::CONS) {
                const int h = o / HD, d = o % HD;
                const size_t base = (static_cast<size_t>(b) * P.n_head + hq0 + h) * MS;
                float A = 0.f;
                for (uint32_t s2 = 0; s2 < nsplit; ++s2)
                    A = fmaf(__ldcg(P.ws_acc + (base + s2) * HD + d), sw[h * nsplit + s2], A);
                P.out[(static_cast<size_t>(b) * P.n_head + hq0 + h) * HD + d] = A / hL[h];
            }
            if (tid == 0) *counter = 0u;
        }
    }

    // ------------------------------------------------ write key p into the slot
    if (is_last) {
        const size_t at = (static_cast<size_t>(slot) * P.slot_ctx + p) * P.n_kv_head + kvh;
        float4* kd = reinterpret_cast<float4*>(P.K + at * HD);
        float4* vd = reinterpret_cast<float4*>(P.V + at * HD);
        for (int i = tid; i < HD / 4; i += C::CONS) {
            kd[i] = reinterpret_cast<const float4*>(ks)[i];
            vd[i] = reinterpret_cast<const float4*>(vs)[i];
        }
    }
}

template <int HD, int G>
int launch_one(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
               dim3 grid, cudaStream_t stream) {
    using C = KCfg<HD, G>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(slotkv_decode_attn_kernel<HD, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return static_cast<int>(e);
        configured = true;
    }
    slotkv_decode_attn_kernel<HD, G><<<grid, C::THREADS, C::SMEM, stream>>>(tmK, tmV, p);
    return static_cast<int>(cudaGetLastError());
}

template <int HD>
int launch_hd(int G, const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
              dim3 grid, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_one<HD, 1>(p, tmK, tmV, grid, stream);
        case 2: return launch_one<HD, 2>(p, tmK, tmV, grid, stream);
        case 3: return launch_one<HD, 3>(p, tmK, tmV, grid, stream);
        case 4: return launch_one<HD, 4>(p, tmK, tmV, grid, stream);
        case 5: return launch_one<HD, 5>(p, tmK, tmV, grid, stream);
        case 6: return launch_one<HD, 6>(p, tmK, tmV, grid, stream);
        case 7: return launch_one<HD, 7>(p, tmK, tmV, grid, stream);
        case 8: return launch_one<HD, 8>(p, tmK, tmV, grid, stream);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace slotkv

// decode_attn.cuh -- the fused batched decode attention over slot KV.
//
// Work item = (row b, kv head g, split s): the keys [s*C, min((s+1)*C, p+1))
// of slot slots[b] for the G query heads that share kv head g (GQA), so every
// history K/V byte is read from HBM exactly once.  C comes from the split
// policy (see split_chunk and the host's choice of chunk_min).
//
// Kernels per call, on one stream (a call of a few rows over short slots
// runs slotkv_decode_small_kernel instead, see decode_small.cuh):
//   * slotkv_plan_kernel (one CTA): checks every row's slot and position,
//     lists the valid work items, largest first (leaving out the CTAs'
//     static items), and resets the hand-out counter.  Skipped when the
//     static items are all the work.  Launched as a programmatic dependent
//     of whatever precedes it, it waits for that grid before reading
//     anything; the previous call's decode kernel lets it launch once every
//     CTA has run out of items, so its launch overlaps that call's tail;
//   * slotkv_decode_attn_kernel (persistent, 2 CTAs per SM, launched as a
//     programmatic dependent of the plan): each CTA starts on its static
//     item -- split 0 of (row, kv head) pair blockIdx.x, or, for CTAs beyond
//     the pairs, split 1 of a pair -- while the plan runs, then takes items
//     from the list, each claimed a few tiles before the current one ends,
//     until it is exhausted.  The
//     steps of "Forward Cuda Gemma", decodeBatch, fused:
//       - warp 4 (producer) streams the items' history K and V tiles into a
//         3-stage shared-memory ring (2 stages for hd 256 with G >= 4) with
//         2-D TMA copies (cp.async.bulk.tensor, one [T keys x hd] box per
//         tensor per stage) on mbarriers, running
//         ahead across item boundaries, and stages each item's q (and, in the
//         split holding key p, k_new and v_new) one item ahead;
//       - warp 5 (prep) applies per-head RMS norm + RoPE to the staged vectors
//         (q pre-scaled by scale*log2 e);
//       - warps 0-3 (consumers), per tile: groups of L lanes each take one
//         key; every lane keeps E = hd/L elements of the G queries and of G
//         output accumulators in registers, forms partial dots with packed
//         f32x2 FMAs, reduces them over the group and runs a base-2 online
//         softmax whose running max is raised lazily;
//       - the split holding key p adds that key from shared memory (its K is
//         the freshly normed+rotated k', its V the raw v_new) and writes both
//         rows into the slot buffers at (slot*slot_ctx + p)*kv_dim (in paged
//         mode, into key p's block);
//       - the groups' (m, l, acc) merge by halving within each warp, then
//         across the four warps in shared memory; a one-split row writes out,
//         otherwise the partial goes to the workspace and the last split of
//         the (row, kv head) to finish is merged, in split order, by warp 6
//         (merge) or, at the kernel's tail, by the consumers themselves.
//   * slotkv_write_kv_kernel (prefill only, first): every token's K and V
//     rows, before the attention reads them.
//
// Paged mode (DecodeParams::block_tables set): the buffers are a pool of
// blocks and row b's key t sits in block block_tables[b][t / block_size].
// Block sizes are multiples of T and tile starts are multiples of T, so each
// tile lies inside one block: the producer only swaps the tile's first row
// (looked up one tile ahead), and the plan (or, for a static item, the
// producer warp) checks every used table entry.
//
// Every wait on an mbarrier is bounded; on expiry the CTA raises
// SLOTKV_DEV_TIMEOUT, drains its own copies in flight (bounded) and returns.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <atomic>

#include "params.h"

namespace slotkv {

constexpr uint32_t kDevRange = 1u;
constexpr uint32_t kDevTimeout = 2u;
constexpr uint32_t kOptVNorm = 1u;        // SLOTKV_OPT_VNORM
constexpr uint32_t kOptNormPlusOne = 2u;  // SLOTKV_OPT_NORM_PLUS_ONE
constexpr uint32_t kOptTestStall = 0x80000000u;  // SLOTKV_OPT_TEST_STALL
constexpr int kPlanThreads = 1024;
constexpr uint32_t kClaimLead = 4;  // tiles left in an item when the next is claimed
// Dynamic shared memory a decode CTA may use for two to fit on an SM: 228 KB
// per SM, of which 1 KB is reserved for each resident CTA.
constexpr int kSmemPerCta = (228 * 1024) / 2 - 1024;

__host__ __device__ constexpr int pow2_floor(int x) {
    int r = 1;
    while (r * 2 <= x) r *= 2;
    return r;
}
__host__ __device__ constexpr int pow2_ceil(int x) {
    int r = 1;
    while (r < x) r *= 2;
    return r;
}
__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int HD, int G>
struct KCfg {
    static constexpr int W = 4;                   // consumer warps (warpgroup 0)
    static constexpr int CONS = W * 32;           // consumer threads
    // + warpgroup 1: warp 4 streams (TMA), warp 5 prepares the next item's
    // vectors, warp 6 merges splits, warp 7 only hands its registers over
    static constexpr int THREADS = CONS + 128;
    static constexpr int WARP_TMA = 4, WARP_PREP = 5, WARP_MERGE = 6;
    // registers per thread: launched at 128 (two CTAs per SM), then moved from
    // warpgroup 1 to warpgroup 0: 128 * REG_CONS + 128 * REG_HELP = 256 * 128.
    // (200 / 56 leaves the consumers of the eight-heads-per-kv-head shapes
    // almost spill-free; the merge warp keeps four loads in flight to live
    // in 56.)
    static constexpr int REG_CONS = 200;
    static constexpr int REG_HELP = 56;
    static constexpr int T = tile_keys(HD);       // keys per tile
    // elements per lane: keep G*E <= 64 (queries + accumulators in registers)
    static constexpr int E = cmax(4, cmax(HD / 32, cmin(32, pow2_floor(64 / G))));
    static constexpr int L = HD / E;              // lanes per key group
    static constexpr int NG = CONS / L;           // key groups per CTA
    static constexpr int R = T / NG;              // keys per group per tile
    // keys attended per softmax update: keeps the live scores (RC*G) <= 16,
    // or <= 32 where only that many give the transposed reduction (below)
    // one value per lane (hd 256 with G >= 5)
    static constexpr int RC_S = pow2_floor(cmax(1, cmin(R, 16 / G)));
    static constexpr int RC_L = pow2_floor(cmax(1, cmin(R, 32 / G)));
    static constexpr int RC =
        RC_S * pow2_ceil(G) < L && RC_L * pow2_ceil(G) >= L ? RC_L : RC_S;
    // transposed reduction (see attend_rows_tr): G padded to a power of two,
    // values per lane after the reduction (each held by L / NV lanes when
    // there are fewer values than lanes); used from four values up
    static constexpr int GP = pow2_ceil(G);
    static constexpr int NV = RC * GP;
    static constexpr bool TR = NV >= 4;
    static constexpr int CNT = NV >= L ? NV / L : 1;
    static constexpr int TILE_BYTES = T * HD * 4;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int NMS = 4;                 // split-merge hand-off slots
    // shared memory: ring [S] | chain scratch acc [G][HD], m, l [G] | per-item
    // slots [2] of (q [G][HD], k [HD], v [HD]) | norm weights, inv_freq |
    // item descriptors [2] | hand-offs [NMS] | mbarriers | flags.
    // Offsets after the ring first, from 0:
    static constexpr int CHAIN_FLOATS = (G * HD + 2 * G + 3) / 4 * 4;
    static constexpr int REL_QBUF = CHAIN_FLOATS * 4;
    static constexpr int REL_KBUF = REL_QBUF + 2 * G * HD * 4;
    static constexpr int REL_VBUF = REL_KBUF + 2 * HD * 4;
    static constexpr int REL_QW = REL_VBUF + 2 * HD * 4;
    static constexpr int REL_KW = REL_QW + HD * 4;
    static constexpr int REL_IF = REL_KW + HD * 4;
    static constexpr int REL_PBUF = REL_IF + HD * 2;   // [NG][NV] probabilities
    static constexpr int REL_DESC = REL_PBUF + (TR ? NG * NV * 4 : 0);
    static constexpr int REL_HAND = REL_DESC + 2 * 64;
    static constexpr int REL_BAR = REL_HAND + NMS * 16;
    // mbarriers: full[S], empty[S], staged[2], prepared[2], slot_free[2],
    // handed[NMS], hand_free[NMS] (room kept for S = 3)
    static constexpr int NBAR = 2 * 3 + 6 + 2 * NMS;
    static constexpr int REL_MISC = REL_BAR + NBAR * 8;
    static constexpr int REL_PEND = REL_MISC + 16;  // the consumers' unmerged partial
    static constexpr int REL_END = REL_PEND + 32;
    // pipeline stages: three, or two where three would leave no room for a
    // second CTA on the SM (hd 256 with G >= 4)
    static constexpr int S = 3 * STAGE_BYTES + REL_END <= kSmemPerCta ? 3 : 2;
    static constexpr int OFF_CHAIN = S * STAGE_BYTES;
    static constexpr int OFF_QBUF = OFF_CHAIN + REL_QBUF;
    static constexpr int OFF_KBUF = OFF_CHAIN + REL_KBUF;
    static constexpr int OFF_VBUF = OFF_CHAIN + REL_VBUF;
    static constexpr int OFF_QW = OFF_CHAIN + REL_QW;
    static constexpr int OFF_KW = OFF_CHAIN + REL_KW;
    static constexpr int OFF_IF = OFF_CHAIN + REL_IF;
    static constexpr int OFF_PBUF = OFF_CHAIN + REL_PBUF;
    static constexpr int OFF_DESC = OFF_CHAIN + REL_DESC;
    static constexpr int OFF_HAND = OFF_CHAIN + REL_HAND;
    static constexpr int OFF_BAR = OFF_CHAIN + REL_BAR;
    static constexpr int OFF_MISC = OFF_CHAIN + REL_MISC;
    static constexpr int OFF_PEND = OFF_CHAIN + REL_PEND;
    static constexpr int SMEM = OFF_CHAIN + REL_END;
    static_assert(SMEM <= kSmemPerCta, "two CTAs per SM");
    static_assert(L >= 1 && L <= 32 && (32 % L) == 0, "lane group must divide a warp");
    static_assert(E % 4 == 0 && E * L == HD, "lane slice must be whole float4s");
    static_assert(R >= 1 && R * NG == T, "tile must split evenly over the groups");
    static_assert(R % RC == 0, "row chunks must divide the rows per tile");
    static_assert(G * E <= 64, "register budget");
    static_assert(HD == 64 || HD == 128 || HD == 256, "head dim");
    static_assert(OFF_CHAIN % 16 == 0 && OFF_QBUF % 16 == 0 && OFF_KBUF % 16 == 0 &&
                      OFF_VBUF % 16 == 0 && OFF_BAR % 8 == 0,
                  "alignment");
    static_assert(CONS * REG_CONS + 128 * REG_HELP == THREADS * 128,
                  "register hand-over must add up to the launch's registers");
};

// What the producer tells the other warps about an item.
// prow: row of key p in the [rows][kv_dim] view of the K and V buffers.
struct ItemDesc {
    uint32_t b, kvh, split, nsplit, p, prow, k0, hist_end, ntiles, is_last, end, pad;
};

// A finished multi-split partial handed to the merge warp.
struct HandOff {
    uint32_t b, kvh, nsplit, end;
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

// Non-blocking test: has the phase of `bar` with parity `parity` completed?
// (try_wait may suspend the thread for a while; this never does.)
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
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

// Contiguous global -> shared copy on the async proxy, completing on `bar`.
// Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// atomicAdd with acquire-release semantics at GPU scope.
__device__ __forceinline__ uint32_t atomic_add_acq_rel(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

// Warpgroup register re-allocation (all four warps of a warpgroup execute it).
template <int N>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void named_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch: wait for the grids this one depends on.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Programmatic dependent launch: let the dependent grid start launching.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Attend NR keys held in shared memory rows (row[r] of the K tile Kt and V
// tile Vt, hd floats each).  Lane `li` of its L-lane group owns elements
// c*4L + 4*li + {0..3}, c < E/4, of every vector.  All 32 lanes of the warp
// must call this together (the reductions shuffle across the whole warp).
// Packed f32x2 helpers (one instruction for two lanes of arithmetic, each
// element rounded exactly as the scalar operation would be).
//   dot_e: <q, k> over E elements as two interleaved partial sums (even and
//          odd elements), added at the end;
//   axpy_e: acc[e] += p * v[e] for every e;
//   scale_e: acc[e] *= c for every e.
template <int E>
__device__ __forceinline__ float dot_e(const float (&q)[E], const float (&k)[E]) {
    float2 d = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < E / 2; ++i)
        d = __ffma2_rn(make_float2(q[2 * i], q[2 * i + 1]), make_float2(k[2 * i], k[2 * i + 1]), d);
    return d.x + d.y;
}
template <int E>
__device__ __forceinline__ void axpy_e(float p, const float (&v)[E], float (&acc)[E]) {
    const float2 pp = make_float2(p, p);
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
        const float2 a = __ffma2_rn(pp, make_float2(v[2 * i], v[2 * i + 1]),
                                    make_float2(acc[2 * i], acc[2 * i + 1]));
        acc[2 * i] = a.x;
        acc[2 * i + 1] = a.y;
    }
}
template <int E>
__device__ __forceinline__ void scale_e(float c, float (&acc)[E]) {
    const float2 cc = make_float2(c, c);
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
        const float2 a = __fmul2_rn(cc, make_float2(acc[2 * i], acc[2 * i + 1]));
        acc[2 * i] = a.x;
        acc[2 * i + 1] = a.y;
    }
}

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
        for (int h = 0; h < G; ++h) s[r][h] = dot_e<E>(q[h], kv);
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
            scale_e<E>(corr, acc[h]);
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
                axpy_e<E>(pr, vv, acc[h]);
            }
        }
    }
}

// Attend NR keys like attend_rows, with a transposed reduction: the NV =
// NR * GP partial dots of a lane (key r, head h at index r * GP + h; heads
// past G are zero) are summed over the L lanes of the group by halving, so
// after log2(L) levels lane li holds the complete scores of indices
// li * CNT + j, j < CNT: one key, CNT consecutive heads.  With fewer values
// than lanes (NV < L) the halving stops at one value per lane and the last
// log2(REP) levels sum by butterfly, so the REP = L / NV lanes li with the
// same li / REP all hold index li / REP.  Only those scores get
// exponentials; the probabilities go to the group's NV-float buffer `pg`
// and every lane reads all of them back for the value update.
// State: the running max m_t[j] and sum l_t[j] of this lane's heads (equal
// across the lanes holding the same heads for other keys), acc as usual.
// The running max is lazy: it is raised (and acc, l rescaled) only when a
// score exceeds it by more than 2^8, so every probability stays <= 2^8.
template <int HD, int G, int E, int L, int NR, int GP, int CNT>
__device__ __forceinline__ void attend_rows_tr(const float* __restrict__ Kt,
                                               const float* __restrict__ Vt,
                                               const int (&row)[NR], const bool (&valid)[NR],
                                               const int li, const int lane,
                                               const float (&q)[G][E], float (&m_t)[CNT],
                                               float (&l_t)[CNT], float (&acc)[G][E],
                                               float* __restrict__ pg) {
    constexpr int NV = NR * GP;
    constexpr int REP = NV >= L ? 1 : L / NV;  // lanes holding each score
    constexpr float kLazy = 8.0f;
    float s[NV];
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
        for (int h = 0; h < GP; ++h) s[r * GP + h] = h < G ? dot_e<E>(q[h < G ? h : 0], kv) : 0.f;
    }
    // halving reduction over the group's lanes, then (NV < L) a butterfly
    // over the REP lanes left holding partial sums of the same value
#pragma unroll
    for (int off = L / 2, cnt = NV; off >= REP; off >>= 1, cnt >>= 1) {
        const bool upper = (li & off) != 0;
#pragma unroll
        for (int i = 0; i < cnt / 2; ++i) {
            const float send = upper ? s[i] : s[i + cnt / 2];
            const float keep = upper ? s[i + cnt / 2] : s[i];
            s[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int off = REP / 2; off >= 1; off >>= 1) s[0] += __shfl_xor_sync(0xffffffffu, s[0], off);
    // this lane's key and first head
    const int v0 = li / REP * CNT;
    const int my_r = v0 / GP;
    bool my_valid = valid[0];
#pragma unroll
    for (int r = 1; r < NR; ++r)
        if (my_r == r) my_valid = valid[r];
    float mx[CNT];
#pragma unroll
    for (int j = 0; j < CNT; ++j) {
        s[j] = my_valid ? s[j] : -CUDART_INF_F;
        mx[j] = s[j];
    }
    // max over the keys, per head: lanes holding the same heads for other keys
#pragma unroll
    for (int off = GP / CNT * REP; off < L; off <<= 1) {
#pragma unroll
        for (int j = 0; j < CNT; ++j) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], off));
    }
    bool need = false;
#pragma unroll
    for (int j = 0; j < CNT; ++j) need |= mx[j] > m_t[j] + kLazy;
    if (__any_sync(0xffffffffu, need)) {
        float corr[CNT];
#pragma unroll
        for (int j = 0; j < CNT; ++j) {
            const float mn = mx[j] > m_t[j] + kLazy ? mx[j] : m_t[j];
            corr[j] = m_t[j] == -CUDART_INF_F ? 0.f : exp2f(m_t[j] - mn);
            l_t[j] *= corr[j];
            m_t[j] = mn;
        }
        // every lane rescales acc for every head: take head h's factor from
        // the (first) lane that holds it for key 0
        const int gbase = lane - li;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float c = __shfl_sync(0xffffffffu, corr[h % CNT], gbase + h / CNT * REP);
            scale_e<E>(c, acc[h]);
        }
    }
#pragma unroll
    for (int j = 0; j < CNT; ++j) {
        const float pj = s[j] == -CUDART_INF_F ? 0.f : exp2f(s[j] - m_t[j]);
        l_t[j] += pj;
        if (li % REP == 0) pg[v0 + j] = pj;
    }
    __syncwarp();
    float pr[NV];
#pragma unroll
    for (int i = 0; i < NV / 4; ++i) {
        const float4 v = *reinterpret_cast<const float4*>(pg + 4 * i);
        pr[4 * i + 0] = v.x;
        pr[4 * i + 1] = v.y;
        pr[4 * i + 2] = v.z;
        pr[4 * i + 3] = v.w;
    }
    __syncwarp();
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
            for (int h = 0; h < G; ++h) axpy_e<E>(pr[r * GP + h], vv, acc[h]);
        }
    }
}

// The per-lane state of attend_rows_tr turned into the replicated form of
// attend_rows (every lane holds m and l of every head): l summed over the
// lanes holding the same heads for the other keys, then each head's m and l
// taken from the lane that holds it.
template <int G, int L, int NR, int GP, int CNT>
__device__ __forceinline__ void tr_state_to_heads(const int li, const int lane, float (&m_t)[CNT],
                                                  float (&l_t)[CNT], float (&m)[G],
                                                  float (&l)[G]) {
    constexpr int REP = NR * GP >= L ? 1 : L / (NR * GP);  // as in attend_rows_tr
#pragma unroll
    for (int off = GP / CNT * REP; off < L; off <<= 1) {
#pragma unroll
        for (int j = 0; j < CNT; ++j) l_t[j] += __shfl_xor_sync(0xffffffffu, l_t[j], off);
    }
    const int gbase = lane - li;
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = __shfl_sync(0xffffffffu, m_t[h % CNT], gbase + h / CNT * REP);
        l[h] = __shfl_sync(0xffffffffu, l_t[h % CNT], gbase + h / CNT * REP);
    }
}

// Merge statistics of nsplit split partials for NH query heads (nh of them
// used), by one warp: per head the max M over the splits' running maxima and
// L = sum_s l_s * exp2(m_s - M), then the sink joins both.  Head h's pairs
// (m_s, l_s) sit at ml0 + h * hstride + 2 s.  Lanes take splits lane, lane +
// 32, ... and the sums meet in a fixed xor tree, so every caller gets the
// same bits for the same partials.
template <int NH>
__device__ __forceinline__ void merge_stats(const float* ml0, size_t hstride, int nh,
                                            uint32_t nsplit, const float* sinks, int lane,
                                            float (&M)[NH], float (&L)[NH]) {
    constexpr float kLog2e = 1.4426950408889634f;
    float2 c[NH];  // this lane's first split
#pragma unroll
    for (int h = 0; h < NH; ++h) {
        c[h] = make_float2(-CUDART_INF_F, 0.f);
        if (h < nh && static_cast<uint32_t>(lane) < nsplit)
            c[h] = __ldcg(reinterpret_cast<const float2*>(ml0 + h * hstride) + lane);
        M[h] = c[h].x;
    }
    for (uint32_t s = lane + 32; s < nsplit; s += 32) {
#pragma unroll
        for (int h = 0; h < NH; ++h)
            if (h < nh) M[h] = fmaxf(M[h], __ldcg(ml0 + h * hstride + 2 * s));
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            M[h] = fmaxf(M[h], __shfl_xor_sync(0xffffffffu, M[h], off));
        L[h] = static_cast<uint32_t>(lane) < nsplit && h < nh
                   ? __fmaf_rn(c[h].y, exp2f(c[h].x - M[h]), 0.f) : 0.f;
    }
    for (uint32_t s = lane + 32; s < nsplit; s += 32) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            if (h < nh) {
                const float2 e = __ldcg(reinterpret_cast<const float2*>(ml0 + h * hstride) + s);
                L[h] = __fmaf_rn(e.y, exp2f(e.x - M[h]), L[h]);
            }
        }
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            L[h] = __fadd_rn(L[h], __shfl_xor_sync(0xffffffffu, L[h], off));
        if (sinks && h < nh) {
            const float sk = __fmul_rn(sinks[h], kLog2e);
            const float M2 = fmaxf(M[h], sk);
            L[h] = __fmaf_rn(L[h], exp2f(M[h] - M2), exp2f(sk - M2));
            M[h] = M2;
        }
    }
}

// exp2(m - M) as the weight of a partial whose running max is m, with an
// empty partial (m = -inf) weighing 0 even when M is -inf too.
__device__ __forceinline__ float partial_weight(float m, float M) {
    return m == -CUDART_INF_F ? 0.f : exp2f(m - M);
}

// Merge the (m, l, acc) states of a warp's 32 / L key groups by halving: at
// each level a lane keeps half of its elements (the upper half if its group
// bit is set) and takes its partner group's share of that half, so afterwards
// lane (li, group bits) holds, for every head, the warp's merged elements
// e0 .. e0 + hd/32 - 1 of its slice in acc[h][0 .. hd/32); e0 is returned.
// m and l are merged in one fixed order (lower group first) and stay equal on
// all lanes.  All 32 lanes call it together.
template <int G, int E, int L>
__device__ __forceinline__ int merge_warp_groups(const int lane, float (&m)[G], float (&l)[G],
                                                 float (&acc)[G][E]) {
    int e0 = 0;
#pragma unroll
    for (int off = L, cnt = E; off < 32; off <<= 1, cnt >>= 1) {
        const bool upper = (lane & off) != 0;
        float c_lo[G], c_hi[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
            const float lo = __shfl_xor_sync(0xffffffffu, l[h], off);
            const float m_lo = upper ? mo : m[h], m_hi = upper ? m[h] : mo;
            const float l_lo = upper ? lo : l[h], l_hi = upper ? l[h] : lo;
            const float M = fmaxf(m_lo, m_hi);
            c_lo[h] = partial_weight(m_lo, M);
            c_hi[h] = partial_weight(m_hi, M);
            l[h] = __fmaf_rn(l_lo, c_lo[h], __fmul_rn(l_hi, c_hi[h]));
            m[h] = M;
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int i = 0; i < cnt / 2; ++i) {
                const float send = upper ? acc[h][i] : acc[h][i + cnt / 2];
                const float keep = upper ? acc[h][i + cnt / 2] : acc[h][i];
                const float recv = __shfl_xor_sync(0xffffffffu, send, off);
                const float v_lo = upper ? recv : keep, v_hi = upper ? keep : recv;
                acc[h][i] = __fmaf_rn(v_lo, c_lo[h], __fmul_rn(v_hi, c_hi[h]));
            }
        }
        e0 += upper ? cnt / 2 : 0;
    }
    return e0;
}

// ------------------------------------------------ per-warp vector routines
// Shared by the decode kernel's prep warp and the prefill KV-write kernel, so
// both produce bit-identical vectors.  A lane owns the rotation pairs
// (i, i + hd/2) for i = lane + 32 j, j < hd/64.

// cos/sin of the f32 RoPE angles fl32((float)p * inv_freq[i]) of this lane's pairs.
template <int HD>
__device__ __forceinline__ void warp_rope_angles(uint32_t p, const float* inv_freq,
                                                 float (&cs)[HD / 64], float (&sn)[HD / 64],
                                                 int lane) {
    const float fp = static_cast<float>(p);
#pragma unroll
    for (int j = 0; j < HD / 64; ++j) sincosf(__fmul_rn(fp, inv_freq[lane + 32 * j]), &sn[j], &cs[j]);
}

// dst = RoPE(src / sqrt(mean(src^2) + eps) * (w1 + w)) * mul, one head vector;
// w1 is 0 (plain weights) or 1 (Gemma's (1 + w)).  src may equal dst.
template <int HD>
__device__ __forceinline__ void warp_norm_rope(const float* src, float* dst, const float* w,
                                               float w1, float mul, float eps,
                                               const float (&cs)[HD / 64],
                                               const float (&sn)[HD / 64], int lane) {
    constexpr int PPL = HD / 64;
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
    const float inv = 1.0f / sqrtf(ss * (1.0f / HD) + eps);
#pragma unroll
    for (int j = 0; j < PPL; ++j) {
        const int i = lane + 32 * j;
        const float y0 = x0[j] * inv * (w1 + w[i]);
        const float y1 = x1[j] * inv * (w1 + w[i + HD / 2]);
        dst[i] = (y0 * cs[j] - y1 * sn[j]) * mul;
        dst[i + HD / 2] = (y1 * cs[j] + y0 * sn[j]) * mul;
    }
}

// dst = src / sqrt(mean(src^2) + eps), the weightless RMS norm.  src may equal dst.
template <int HD>
__device__ __forceinline__ void warp_rms_norm_plain(const float* src, float* dst, float eps,
                                                    int lane) {
    float x[HD / 32];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < HD / 32; ++j) {
        x[j] = src[lane + 32 * j];
        ss = fmaf(x[j], x[j], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = 1.0f / sqrtf(ss * (1.0f / HD) + eps);
#pragma unroll
    for (int j = 0; j < HD / 32; ++j) dst[lane + 32 * j] = x[j] * inv;
}

// ------------------------------------------------------------------ plan
// One CTA.  Lists every valid (row, split, kv head) as a 16-byte record
// (packed item, position, row of key p), largest first: items are binned by
// their tile count and the bins laid out in descending order, so the small
// ragged last splits come last and fill the end of the kernel (the order of
// work never changes a result; only the split sizes could, and they depend on
// the row alone).  Raises SLOTKV_DEV_RANGE for rows whose slot or position
// is out of range -- in paged mode, whose position is past its table or any
// of whose blocks 0..p/block_size is not in the pool -- (they get no items)
// and resets the hand-out counter.  The decode CTAs' static items (split 0 of
// the first static_items pairs, split 1 of the first static_second pairs)
// are left out of the list.
constexpr int kPlanBins = 64;
constexpr int kPlanMaxRows = 65536;

template <int T>
__global__ void __launch_bounds__(kPlanThreads, 1) slotkv_plan_kernel(const DecodeParams P) {
    __shared__ uint32_t bin_count[kPlanBins];
    __shared__ uint32_t bin_cursor[kPlanBins];
    __shared__ uint32_t total;
    __shared__ uint32_t row_bad[kPlanMaxRows / 32];  // paged mode: rows failing the check
    // one round of rows (one per thread) handed from reservation to writing
    __shared__ uint32_t sh_p[kPlanThreads], sh_prow[kPlanThreads], sh_meta[kPlanThreads];
    __shared__ uint32_t sh_fb[kPlanThreads], sh_lb[kPlanThreads];
    __shared__ uint32_t sh_nf[kPlanThreads], sh_nl[kPlanThreads];
    // The plan kernel is a programmatic dependent of whatever precedes it on
    // the stream (the previous call's decode kernel lets it launch once every
    // CTA of that grid has run out of items): nothing may be read before the
    // preceding grid has finished.  The decode kernel may launch from here on.
    grid_dependency_wait();
    grid_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t nkv = P.n_kv_head;
    const bool paged = P.block_tables != nullptr;
    for (int i = tid; i < kPlanBins; i += kPlanThreads) bin_count[i] = 0;
    if (paged) {
        for (uint32_t i = tid; i < (P.B + 31) / 32; i += kPlanThreads) row_bad[i] = 0;
        __syncthreads();
        // pass 0 (paged): each warp checks the used table entries of four rows
        // at a time, two loads per row and lane in flight
        constexpr int RW = 4;
        for (uint32_t b0 = warp * RW; b0 < P.B; b0 += (kPlanThreads / 32) * RW) {
            uint32_t used[RW];
            bool bad[RW];
            const uint32_t* tab[RW];
            uint32_t most = 0;
#pragma unroll
            for (int u = 0; u < RW; ++u) {
                const uint32_t b = b0 + u;
                const uint32_t p = b < P.B ? P.positions[b] : 0u;
                bad[u] = b < P.B && static_cast<uint64_t>(p) >=
                                        static_cast<uint64_t>(P.bt_stride) * P.slot_ctx;
                used[u] = (b < P.B && !bad[u]) ? p / P.slot_ctx + 1 : 0u;
                tab[u] = P.block_tables + static_cast<size_t>(b < P.B ? b : 0) * P.bt_stride;
                most = used[u] > most ? used[u] : most;
            }
            for (uint32_t i0 = 0; i0 < most; i0 += 64) {
                uint32_t id[RW][2];
#pragma unroll
                for (int u = 0; u < RW; ++u)
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        const uint32_t i = i0 + v * 32 + lane;
                        id[u][v] = i < used[u] ? __ldg(tab[u] + i) : 0u;
                    }
#pragma unroll
                for (int u = 0; u < RW; ++u) bad[u] |= id[u][0] >= P.n_slots || id[u][1] >= P.n_slots;
            }
#pragma unroll
            for (int u = 0; u < RW; ++u) {
                const bool any = __any_sync(0xffffffffu, bad[u]);
                if (any && lane == 0) atomicOr(&row_bad[(b0 + u) >> 5], 1u << ((b0 + u) & 31));
            }
        }
    }
    __syncthreads();
    // A row's shape: position, row of key p in the [rows][kv_dim] view of K
    // and V, split count, the tile counts of its full and last splits, how
    // many of its listed items are full / last splits, and how many of its kv
    // heads have split 0 (ns) and split 1 (ns1) held by decode CTAs as static
    // items (split 0 of the first static_items pairs, split 1 of the first
    // static_second pairs when the row has a second split).
    struct Shape {
        uint32_t p, prow, nsplit, ft, lt, nfull, nlast, ns, ns1;
    };
    auto row_shape = [&](uint32_t b, Shape& r) {
        r.p = P.positions[b];
        if (paged) {
            if (row_bad[b >> 5] & (1u << (b & 31))) return false;
            r.prow = __ldg(P.block_tables + static_cast<size_t>(b) * P.bt_stride +
                           r.p / P.slot_ctx) * P.slot_ctx + r.p % P.slot_ctx;
        } else {
            const uint32_t slot = P.slots[b];
            if (slot >= P.n_slots || r.p >= P.slot_ctx) return false;
            r.prow = slot * P.slot_ctx + r.p;
        }
        const uint32_t chunk = split_chunk(r.p + 1, P.chunk_min, P.max_splits, T);
        r.nsplit = (r.p + 1 + chunk - 1) / chunk;
        r.ft = chunk / T;
        r.lt = (r.p + (P.prefill ? 1u : 0u) - (r.nsplit - 1) * chunk + T - 1) / T;
        const uint32_t first = b * nkv;
        r.ns = P.static_items > first
                   ? (P.static_items - first < nkv ? P.static_items - first : nkv)
                   : 0u;
        r.ns1 = r.nsplit > 1 && P.static_second > first
                    ? (P.static_second - first < nkv ? P.static_second - first : nkv)
                    : 0u;
        // full splits 0 .. nsplit-2, less the static ones; the last split
        // nsplit-1 (0 or 1 may be static)
        r.nfull = r.nsplit > 1 ? (r.nsplit - 1) * nkv - r.ns - (r.nsplit > 2 ? r.ns1 : 0u) : 0u;
        r.nlast = nkv - (r.nsplit == 1 ? r.ns : (r.nsplit == 2 ? r.ns1 : 0u));
        return true;
    };
    auto bin_of = [](uint32_t tiles) { return tiles < kPlanBins ? tiles : kPlanBins - 1u; };
    // pass 1: one thread per row, histogram of item sizes.  A thread keeps its
    // first row's shape for pass 2 (all of them when B <= kPlanThreads).
    Shape mine{};
    bool mine_ok = false;
    for (uint32_t b = tid; b < P.B; b += kPlanThreads) {
        Shape r{};
        const bool ok = row_shape(b, r);
        if (!ok) {
            atomicOr(P.status, kDevRange);
        } else {
            if (r.nfull) atomicAdd(&bin_count[bin_of(r.ft)], r.nfull);
            if (r.nlast) atomicAdd(&bin_count[bin_of(r.lt)], r.nlast);
        }
        if (b == static_cast<uint32_t>(tid)) {
            mine = r;
            mine_ok = ok;
        }
    }
    __syncthreads();
    // bins in descending order: lane l holds bins 63-2l and 62-2l; an
    // exclusive scan over the lanes gives each bin's first record
    static_assert(kPlanBins == 64, "the scan covers 64 bins with one warp");
    if (warp == 0) {
        const uint32_t hi = bin_count[63 - 2 * lane], lo = bin_count[62 - 2 * lane];
        uint32_t incl = hi + lo;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const uint32_t excl = incl - hi - lo;
        bin_cursor[63 - 2 * lane] = excl;
        bin_cursor[62 - 2 * lane] = excl + hi;
        if (lane == 31) total = incl;
    }
    __syncthreads();
    // pass 2, by rounds of kPlanThreads rows: each thread reserves its row's
    // ranges in the bins, then warps write the rows' records
    uint4* recs = reinterpret_cast<uint4*>(P.items);
    for (uint32_t r0 = 0; r0 < P.B; r0 += kPlanThreads) {
        const uint32_t b = r0 + tid;
        uint32_t meta = 0;  // nsplit | ns << 9 | ns1 << 18 of a row with items, else 0
        if (b < P.B) {
            Shape r = mine;
            const bool ok = r0 == 0 ? mine_ok : row_shape(b, r);
            if (ok) {
                sh_p[tid] = r.p;
                sh_prow[tid] = r.prow;
                sh_nf[tid] = r.nfull;
                sh_nl[tid] = r.nlast;
                sh_fb[tid] = r.nfull ? atomicAdd(&bin_cursor[bin_of(r.ft)], r.nfull) : 0u;
                sh_lb[tid] = r.nlast ? atomicAdd(&bin_cursor[bin_of(r.lt)], r.nlast) : 0u;
                meta = r.nsplit | (r.ns << 9) | (r.ns1 << 18);
            }
        }
        sh_meta[tid] = meta;
        __syncthreads();
        const uint32_t nrows = P.B - r0 < static_cast<uint32_t>(kPlanThreads)
                                   ? P.B - r0 : static_cast<uint32_t>(kPlanThreads);
        for (uint32_t i = warp; i < nrows; i += kPlanThreads / 32) {
            const uint32_t m = sh_meta[i];
            if (!m) continue;
            const uint32_t row = r0 + i, nsplit = m & 511u, ns = (m >> 9) & 511u, ns1 = m >> 18;
            const uint32_t p = sh_p[i], prow = sh_prow[i];
            const uint32_t nfull = sh_nf[i], nlast = sh_nl[i], fb = sh_fb[i], lb = sh_lb[i];
            // listed full splits, in (split, kv head) order: split 0 from kv
            // head ns, split 1 from ns1 (when it is not the last split), the
            // rest whole; listed last splits: kv heads nkv - nlast .. nkv - 1
            for (uint32_t j = lane; j < nfull; j += 32) {
                uint32_t split, kvh = j;
                if (kvh < nkv - ns) {
                    split = 0;
                    kvh += ns;
                } else if ((kvh -= nkv - ns) < nkv - ns1) {
                    split = 1;
                    kvh += ns1;
                } else {
                    kvh -= nkv - ns1;
                    split = 2 + kvh / nkv;
                    kvh %= nkv;
                }
                recs[fb + j] = make_uint4(pack_item(row, split, kvh), p, prow, 0u);
            }
            for (uint32_t j = lane; j < nlast; j += 32)
                recs[lb + j] = make_uint4(pack_item(row, nsplit - 1, j + (nkv - nlast)), p, prow, 0u);
        }
        __syncthreads();
    }
    if (tid == 0) {
        P.plan[0] = total;
        P.plan[1] = 0;
    }
}

// ------------------------------------------------------------------ decode
template <int HD, int G>
__global__ void __launch_bounds__(KCfg<HD, G>::THREADS, 2)
    slotkv_decode_attn_kernel(const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmV,
                              const DecodeParams P) {
    using C = KCfg<HD, G>;
    constexpr int E = C::E, L = C::L, NG = C::NG, R = C::R, T = C::T, S = C::S, W = C::W;
    constexpr int NMS = C::NMS;
    constexpr float kLog2e = 1.4426950408889634f;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    float* chain = reinterpret_cast<float*>(smem + C::OFF_CHAIN);  // acc [G][HD], m [G], l [G]
    float* chain_m = chain + G * HD;
    float* chain_l = chain_m + G;
    float* qbuf = reinterpret_cast<float*>(smem + C::OFF_QBUF);  // [2][G][HD]
    float* kbuf = reinterpret_cast<float*>(smem + C::OFF_KBUF);  // [2][HD]
    float* vbuf = reinterpret_cast<float*>(smem + C::OFF_VBUF);  // [2][HD]
    float* qw_s = reinterpret_cast<float*>(smem + C::OFF_QW);
    float* kw_s = reinterpret_cast<float*>(smem + C::OFF_KW);
    float* if_s = reinterpret_cast<float*>(smem + C::OFF_IF);
    volatile ItemDesc* desc = reinterpret_cast<volatile ItemDesc*>(smem + C::OFF_DESC);
    volatile HandOff* hand = reinterpret_cast<volatile HandOff*>(smem + C::OFF_HAND);
    const uint32_t full0 = smem_addr(smem + C::OFF_BAR);  // tile landed
    const uint32_t empty0 = full0 + 8 * S;                 // tile consumed
    const uint32_t staged0 = empty0 + 8 * S;               // item vectors landed
    const uint32_t prepared0 = staged0 + 16;               // item vectors normed+rotated
    const uint32_t free0 = prepared0 + 16;                 // item slot released
    const uint32_t handed0 = free0 + 16;                   // partial handed to the merge warp
    const uint32_t hfree0 = handed0 + 8 * NMS;             // hand-off slot released
    volatile int* misc = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
    // pend[0..3]: the last item's partial awaits its merge (flag, row, kv
    // head, splits); pend[4]: the consumers' tail-merge decision
    volatile uint32_t* pend = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_PEND);
    // misc[0]: abort, misc[2]: tiles issued, misc[3]: items staged

    // The CTA's static item: split 0 of pair blockIdx.x, or, for the CTAs
    // past the pairs, split 1 of pair blockIdx.x - static_items.  The producer
    // needs its row's position and slot: issue those loads before anything
    // else so they land during set-up.
    const bool has_static = blockIdx.x < P.static_items + P.static_second;
    const uint32_t st_split = blockIdx.x < P.static_items ? 0u : 1u;
    const uint32_t st_row = (blockIdx.x - st_split * P.static_items) / P.n_kv_head;
    uint32_t pre_p = 0, pre_slot = 0;
    if (warp == C::WARP_TMA && has_static) {
        pre_p = __ldg(P.positions + st_row);
        if (!P.block_tables) pre_slot = __ldg(P.slots + st_row);
    }
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, W);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(staged0 + 8 * i, 1);
            mbar_init(prepared0 + 8 * i, 1);
            mbar_init(free0 + 8 * i, W);
        }
        for (int i = 0; i < NMS; ++i) {
            mbar_init(handed0 + 8 * i, 1);
            mbar_init(hfree0 + 8 * i, 1);
        }
        misc[0] = 0;
        misc[1] = 0;
        pend[0] = 0;
        misc[2] = 0;
        misc[3] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    if (warp >= W) {
        regs_decrease<C::REG_HELP>();
        // ------------------------------------------------------------ producer
        // Items are staged one ahead: item k+1 is claimed near the end of item
        // k's tiles, and its descriptor and vectors go into its slot (free once
        // the consumers have finished item k-1) while item k's last tiles are
        // still streaming, so the prep warp has item k+1 ready before the
        // consumers reach it.
        // Paged mode: the whole producer warp checks the static item's row the
        // way the plan does (p within the table, every used entry in the pool)
        // and finds the row of key p.
        uint32_t pg_ok = 0, pg_prow = 0;
        if (warp == C::WARP_TMA && P.block_tables != nullptr && has_static) {
            const uint32_t* tab = P.block_tables + static_cast<size_t>(st_row) * P.bt_stride;
            bool bad = static_cast<uint64_t>(pre_p) >=
                       static_cast<uint64_t>(P.bt_stride) * P.slot_ctx;
            const uint32_t used = bad ? 0u : pre_p / P.slot_ctx + 1;
            for (uint32_t i0 = 0; i0 < used; i0 += 128) {
                uint32_t id[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t i = i0 + u * 32 + lane;
                    id[u] = i < used ? __ldg(tab + i) : 0u;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) bad |= id[u] >= P.n_slots;
            }
            if (!__any_sync(0xffffffffu, bad)) {
                pg_ok = 1;
                pg_prow = __ldg(tab + pre_p / P.slot_ctx) * P.slot_ctx + pre_p % P.slot_ctx;
            }
        }
        if (warp == C::WARP_TMA && lane == 0) {
            const uint4* recs = reinterpret_cast<const uint4*>(P.items);
            const bool paged = P.block_tables != nullptr;
            // The plan's list, its length and the hand-out counter may be read
            // only once the plan kernel has finished.  A CTA with a static
            // item waits for that lazily, streaming the item meanwhile.
            bool planned = false;
            uint32_t n_items = 0;
            auto await_plan = [&]() {
                if (!P.no_plan) {
                    grid_dependency_wait();
                    n_items = __ldcg(P.plan);
                }
                planned = true;
            };
            // stage item k from record `rec` (or the end marker); in paged mode
            // row_o is the item's first key and blk_o the block holding it
            auto stage = [&](uint32_t k, bool valid, uint4 rec, uint32_t& kvh_o, int& row_o,
                             uint32_t& ntiles_o, const uint32_t*& tab_o, uint32_t& blk_o) {
                const uint32_t is = k & 1;
                volatile ItemDesc* d = desc + is;
                const uint32_t staged = staged0 + 8 * is;
                if (!valid) {
                    d->end = 1;
                    mbar_arrive(staged);
                    return false;
                }
                const uint32_t b = rec.x >> 16, split = (rec.x >> 8) & 255u, kvh = rec.x & 255u;
                const uint32_t p = rec.y, prow = rec.z;
                const uint32_t chunk = split_chunk(p + 1, P.chunk_min, P.max_splits, T);
                const uint32_t nsplit = (p + 1 + chunk - 1) / chunk;
                const uint32_t k0 = split * chunk;
                // in prefill mode every key, p included, is read from the slot
                // (the KV-write kernel has written the new rows already)
                const bool is_last = !P.prefill && split == nsplit - 1;
                const uint32_t hist_end = is_last ? p : (k0 + chunk < p + 1 ? k0 + chunk : p + 1);
                const uint32_t n_hist = hist_end > k0 ? hist_end - k0 : 0;
                const uint32_t ntiles = (n_hist + T - 1) / T;
                d->b = b;
                d->kvh = kvh;
                d->split = split;
                d->nsplit = nsplit;
                d->p = p;
                d->prow = prow;
                d->k0 = k0;
                d->hist_end = hist_end;
                d->ntiles = ntiles;
                d->is_last = is_last ? 1u : 0u;
                d->end = 0;
                mbar_expect_tx(staged, G * HD * 4 + (is_last ? 2 * HD * 4 : 0));
                bulk_load(smem_addr(qbuf + is * G * HD),
                          P.q + (static_cast<size_t>(b) * P.n_head + kvh * G) * HD, G * HD * 4,
                          staged);
                if (is_last) {
                    const size_t kv_off = (static_cast<size_t>(b) * P.n_kv_head + kvh) * HD;
                    bulk_load(smem_addr(kbuf + is * HD), P.k_new + kv_off, HD * 4, staged);
                    bulk_load(smem_addr(vbuf + is * HD), P.v_new + kv_off, HD * 4, staged);
                }
                misc[3] = static_cast<int>(k + 1);
                kvh_o = kvh;
                ntiles_o = ntiles;
                if (paged) {
                    // the first block id is used only when the item's tiles
                    // start, so its load completes while earlier tiles stream
                    tab_o = P.block_tables + static_cast<size_t>(b) * P.bt_stride;
                    row_o = static_cast<int>(k0);
                    if (ntiles) blk_o = __ldg(tab_o + k0 / P.slot_ctx);
                } else {
                    row_o = static_cast<int>(prow - p + k0);
                }
                return true;
            };
            // first item: the CTA's static item (split st_split of pair
            // blockIdx.x - st_split * static_items), if its row is in range
            // and, for split 1, has a second split.  Its inputs come from work
            // that precedes the plan kernel on the stream, so they are
            // complete; the plan checks the row the same way and leaves the
            // item out of its list.  (The loads of p and the slot were issued
            // at kernel entry.)
            uint4 rec = make_uint4(0, 0, 0, 0);
            bool first_ok = false;
            if (has_static) {
                const uint32_t kvh = (blockIdx.x - st_split * P.static_items) % P.n_kv_head;
                const uint32_t p = pre_p, slot = pre_slot;
                const bool in_range = paged ? pg_ok != 0u : (slot < P.n_slots && p < P.slot_ctx);
                const uint32_t prow = paged ? pg_prow : slot * P.slot_ctx + p;
                first_ok = in_range &&
                           (st_split == 0 || p + 1 > split_chunk(p + 1, P.chunk_min, P.max_splits, T));
                if (first_ok) rec = make_uint4(pack_item(st_row, st_split, kvh), p, prow, 0u);
                // without a plan kernel (split-0 items only), the range flag
                // is raised here
                if (!in_range && P.no_plan) atomicOr(P.status, kDevRange);
            }
            if (!first_ok) {
                await_plan();
                const uint32_t it = atomicAdd(P.plan + 1, 1u);
                first_ok = it < n_items;
                if (first_ok) rec = __ldcg(recs + it);
            }
            uint32_t cur_kvh = 0, cur_nt = 0, nxt_kvh = 0, nxt_nt = 0;
            int cur_row = 0, nxt_row = 0;
            const uint32_t* cur_tab = nullptr;
            const uint32_t* nxt_tab = nullptr;
            uint32_t cur_blk = 0, nxt_blk = 0;
            bool cur_ok = stage(0, first_ok, rec, cur_kvh, cur_row, cur_nt, cur_tab, cur_blk);
            // The next item is claimed late: when kClaimLead tiles of the
            // current one are left to issue (at once for shorter items).  The
            // claim, the record load and the staging then take one tile each,
            // with tiles to spare before the next item's tiles are needed, and
            // the hand-out follows the kernel's actual progress -- largest
            // items first, the small ones to whichever CTAs free up at the end.
            uint32_t it_n = 0;
            bool claimed = false;
            auto claim = [&]() {
                if (!planned) await_plan();
                it_n = atomicAdd(P.plan + 1, 1u);
                claimed = true;
                // nothing left for this CTA: the next call's plan kernel may
                // launch once every CTA is here (it waits for this grid to
                // finish before it reads anything)
                if (it_n >= n_items) grid_launch_dependents();
            };
            uint4 rec_n = make_uint4(0, 0, 0, 0);
            bool rec_n_loaded = false;
            uint32_t tile_g = 0;
            for (uint32_t k = 0; cur_ok; ++k) {
                bool nxt_staged = false, nxt_ok = false;
                // slot of item k+1 is free once the consumers release item k-1
                const uint32_t nfree = free0 + 8 * ((k + 1) & 1);
                const uint32_t nparity = k >= 1 ? (((k + 1) >> 1) - 1) & 1 : 0;
                for (uint32_t t = 0; t < cur_nt; ++t, ++tile_g) {
                    const int st = tile_g % S;
                    if (tile_g >= static_cast<uint32_t>(S) &&
                        !mbar_wait(empty0 + 8 * st, ((tile_g / S) - 1) & 1)) {
                        atomicOr(P.status, kDevTimeout);
                        misc[0] = 1;
                        break;
                    }
                    if (misc[0]) break;
                    const uint32_t full = full0 + 8 * st;
                    const uint32_t dst = smem_addr(smem + st * C::STAGE_BYTES);
                    // the tile's first row: contiguous in a slot; in paged mode
                    // the tile lies inside one block (block size and tile starts
                    // are multiples of T), whose id was loaded one tile ahead
                    const uint32_t key = static_cast<uint32_t>(cur_row) + t * T;
                    const int trow = paged ? static_cast<int>(cur_blk * P.slot_ctx + key % P.slot_ctx)
                                           : cur_row + static_cast<int>(t * T);
                    if (paged && t + 1 < cur_nt) cur_blk = __ldg(cur_tab + (key + T) / P.slot_ctx);
                    mbar_expect_tx(full, C::STAGE_BYTES);
                    tma_load_2d(dst, &tmK, static_cast<int>(cur_kvh * HD), trow, full);
                    tma_load_2d(dst + C::TILE_BYTES, &tmV, static_cast<int>(cur_kvh * HD), trow,
                                full);
                    misc[2] = static_cast<int>(tile_g + 1);
                    // (a static item waits for the plan here, by when the
                    // plan kernel has long finished)
                    if (!claimed) {
                        if (t + kClaimLead >= cur_nt) claim();
                    } else if (!rec_n_loaded) {
                        if (it_n < n_items) rec_n = __ldcg(recs + it_n);
                        rec_n_loaded = true;
                    } else if (!nxt_staged && (k == 0 || mbar_test(nfree, nparity))) {
                        nxt_ok = stage(k + 1, it_n < n_items, rec_n, nxt_kvh, nxt_row, nxt_nt,
                                       nxt_tab, nxt_blk);
                        nxt_staged = true;
                    }
                }
                if (misc[0]) break;
                if (!claimed) claim();  // an item without tiles
                if (!nxt_staged) {
                    if (!rec_n_loaded && it_n < n_items) rec_n = __ldcg(recs + it_n);
                    if (k >= 1 && !mbar_wait(nfree, nparity)) {
                        atomicOr(P.status, kDevTimeout);
                        misc[0] = 1;
                        break;
                    }
                    nxt_ok = stage(k + 1, it_n < n_items, rec_n, nxt_kvh, nxt_row, nxt_nt,
                                   nxt_tab, nxt_blk);
                }
                claimed = false;
                rec_n_loaded = false;
                cur_ok = nxt_ok;
                cur_kvh = nxt_kvh;
                cur_row = nxt_row;
                cur_nt = nxt_nt;
                cur_tab = nxt_tab;
                cur_blk = nxt_blk;
            }
        }
        // ------------------------------------------------------------ prep
        // Per item: RoPE cos/sin at p (each lane for its own rotation pairs),
        // then per-head RMS norm + RoPE in place on the staged G query vectors
        // (pre-scaled by scale*log2 e) and, in the split owning key p, k_new.
        if (warp == C::WARP_PREP) {
            constexpr int PPL = HD / 64;  // rotation pairs per lane
            // the norm weights and inverse frequencies, used by this warp only:
            // every load in flight at once, then the stores
            {
                float wq[HD / 32], wk[HD / 32], wf[HD / 64];
#pragma unroll
                for (int j = 0; j < HD / 32; ++j) {
                    wq[j] = __ldg(P.q_norm_w + lane + 32 * j);
                    wk[j] = __ldg(P.k_norm_w + lane + 32 * j);
                }
#pragma unroll
                for (int j = 0; j < HD / 64; ++j) wf[j] = __ldg(P.inv_freq + lane + 32 * j);
#pragma unroll
                for (int j = 0; j < HD / 32; ++j) {
                    qw_s[lane + 32 * j] = wq[j];
                    kw_s[lane + 32 * j] = wk[j];
                }
#pragma unroll
                for (int j = 0; j < HD / 64; ++j) if_s[lane + 32 * j] = wf[j];
            }
            __syncwarp();
            for (uint32_t k = 0;; ++k) {
                const uint32_t is = k & 1;
                if (!mbar_wait(staged0 + 8 * is, (k >> 1) & 1)) {
                    if (lane == 0) atomicOr(P.status, kDevTimeout);
                    misc[0] = 1;
                    break;
                }
                if (misc[0]) break;
                const bool end = desc[is].end != 0;
                const uint32_t p = desc[is].p;
                const bool is_last = desc[is].is_last != 0;
                if (!end) {
                    float cs[PPL], sn[PPL];
                    warp_rope_angles<HD>(p, if_s, cs, sn, lane);
                    const float w1 = (P.flags & kOptNormPlusOne) ? 1.0f : 0.0f;
                    const int nvec = G + (is_last ? 1 : 0);
                    for (int x = 0; x < nvec; ++x) {
                        const bool isq = x < G;
                        float* v = isq ? qbuf + (is * G + x) * HD : kbuf + is * HD;
                        warp_norm_rope<HD>(v, v, isq ? qw_s : kw_s, w1,
                                           isq ? P.scale_log2 : 1.0f, P.eps, cs, sn, lane);
                    }
                    if (is_last && (P.flags & kOptVNorm))
                        warp_rms_norm_plain<HD>(vbuf + is * HD, vbuf + is * HD, P.eps, lane);
                }
                __syncwarp();
                // (the failure-path test option withholds the first item, so
                // the consumers' bounded wait runs out)
                if (lane == 0 && !(k == 0 && (P.flags & kOptTestStall)))
                    mbar_arrive(prepared0 + 8 * is);
                if (end) break;
            }
        }
        // ------------------------------------------------------------ merge
        // The last CTA of a (row, kv head) to finish merges its splits, in
        // split order, so the result does not depend on timing.
        if (warp == C::WARP_MERGE) {
            const size_t MS = P.max_splits;
            for (uint32_t j = 0;; ++j) {
                const uint32_t hs = j % NMS;
                if (!mbar_wait(handed0 + 8 * hs, (j / NMS) & 1)) {
                    if (lane == 0) atomicOr(P.status, kDevTimeout);
                    misc[0] = 1;
                    break;
                }
                if (misc[0]) break;
                const uint32_t b = hand[hs].b, kvh = hand[hs].kvh, nsplit = hand[hs].nsplit;
                const bool end = hand[hs].end != 0;
                __syncwarp();
                if (lane == 0) mbar_arrive(hfree0 + 8 * hs);
                if (end) break;
                uint32_t* counter = P.counters + static_cast<size_t>(b) * P.n_kv_head + kvh;
                uint32_t old = 0;
                if (lane == 0) old = atomic_add_acq_rel(counter, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old != nsplit - 1) continue;
                // Merge, up to 4 heads at a time so each lane keeps several loads
                // in flight: per head h the max M_h and weighted sum L_h over the
                // splits (sink included), then out = sum_s w_hs acc_hs / L_h with
                // w_hs = exp2(m_hs - M_h), taking the splits 32 at a time.
                constexpr int HG = G < 4 ? G : 4;
                const uint32_t hq0 = kvh * G;
                for (int h0 = 0; h0 < G; h0 += HG) {
                    const int nh = G - h0 < HG ? G - h0 : HG;
                    const size_t base0 = (static_cast<size_t>(b) * P.n_head + hq0 + h0) * MS;
                    float Mh[HG], Lh[HG];
                    merge_stats<HG>(P.ws_ml + base0 * 2, MS * 2, nh, nsplit,
                                    P.sinks ? P.sinks + hq0 + h0 : nullptr, lane, Mh, Lh);
                    // outputs: lanes over the hd/4 float4 columns (every lane
                    // runs every iteration: the shuffles name the whole warp),
                    // one head at a time, 4 splits' loads in flight per round
#pragma unroll
                    for (int h = 0; h < HG; ++h) {
                        if (h >= nh) break;
                        float* orow =
                            P.out + (static_cast<size_t>(b) * P.n_head + hq0 + h0 + h) * HD;
                        const float inv = __frcp_rn(Lh[h]);
                        const float Mhh = Mh[h];
                        const float* wsa = P.ws_acc + (base0 + h * MS) * HD;
                        const float* wsm = P.ws_ml + (base0 + h * MS) * 2;
                        for (int d0 = 0; d0 < HD / 4; d0 += 32) {
                            const int d4 = d0 + lane;
                            const bool act = d4 < HD / 4;
                            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                            for (uint32_t r0 = 0; r0 < nsplit; r0 += 32) {
                                const uint32_t mine = r0 + lane;
                                // this lane's split's weight; lanes past the end weigh 0
                                const float wl = mine < nsplit ? exp2f(__ldcg(wsm + mine * 2) - Mhh) : 0.f;
                                const uint32_t n = nsplit - r0 < 32u ? nsplit - r0 : 32u;
                                for (uint32_t i0 = 0; i0 < n; i0 += 4) {
                                    float4 v[4];
#pragma unroll
                                    for (int u = 0; u < 4; ++u) {
                                        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                                        if (act && i0 + u < n)
                                            v[u] = __ldcg(reinterpret_cast<const float4*>(
                                                              wsa + (r0 + i0 + u) * HD) + d4);
                                    }
#pragma unroll
                                    for (int u = 0; u < 4; ++u) {
                                        const float w = __shfl_sync(0xffffffffu, wl, (i0 + u) & 31);
                                        a.x = __fmaf_rn(w, v[u].x, a.x);
                                        a.y = __fmaf_rn(w, v[u].y, a.y);
                                        a.z = __fmaf_rn(w, v[u].z, a.z);
                                        a.w = __fmaf_rn(w, v[u].w, a.w);
                                    }
                                }
                            }
                            if (act)
                                reinterpret_cast<float4*>(orow)[d4] =
                                    make_float4(__fmul_rn(a.x, inv), __fmul_rn(a.y, inv),
                                                __fmul_rn(a.z, inv), __fmul_rn(a.w, inv));
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) *counter = 0u;
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    regs_increase<C::REG_CONS>();
    const int gid = warp * (32 / L) + lane / L;  // key group
    const int li = lane % L;                     // lane within the group
    uint32_t tile_g = 0, handed = 0;
    for (uint32_t k = 0;; ++k) {
        const uint32_t is = k & 1;
        if (!misc[0] && !mbar_wait(prepared0 + 8 * is, (k >> 1) & 1)) {
            atomicOr(P.status, kDevTimeout);
            misc[0] = 1;
        }
        named_sync<C::CONS>();  // every consumer warp takes the same branch
        if (misc[0]) break;
        const uint32_t end = desc[is].end;
        // The previous item's partial, if it left one: handed to the merge
        // warp, or, when no item follows in this CTA (the kernel's tail, where
        // the consumers would idle), counted and merged here by all consumer
        // threads with one round of loads.  Both paths compute the same bits.
        if (pend[0]) {
            const uint32_t pb = pend[1], pkvh = pend[2], pns = pend[3];
            if (!end || pns > static_cast<uint32_t>(HD)) {
                if (warp == W - 1) {
                    if (lane == 0) {
                        const uint32_t hs = handed % NMS;
                        if (handed < NMS || mbar_wait(hfree0 + 8 * hs, ((handed / NMS) - 1) & 1)) {
                            hand[hs].b = pb;
                            hand[hs].kvh = pkvh;
                            hand[hs].nsplit = pns;
                            hand[hs].end = 0;
                            mbar_arrive(handed0 + 8 * hs);
                        } else {
                            atomicOr(P.status, kDevTimeout);
                            misc[0] = 1;
                        }
                    }
                    ++handed;
                }
            } else {
                uint32_t* counter = P.counters + static_cast<size_t>(pb) * P.n_kv_head + pkvh;
                if (tid == 0) {
                    const uint32_t old = atomic_add_acq_rel(counter, 1u);
                    const uint32_t last = old == pns - 1 ? 1u : 0u;
                    if (last) *counter = 0u;  // every split has arrived
                    pend[4] = last;
                }
                named_sync<C::CONS>();
                if (pend[4]) {
                    const size_t MS = P.max_splits;
                    const uint32_t hq0 = pkvh * G;
                    float* wts = chain;             // split weights [G][pns]
                    float* invl = chain + G * pns;  // 1 / L per head
                    for (int h = warp; h < G; h += W) {
                        const size_t hb = (static_cast<size_t>(pb) * P.n_head + hq0 + h) * MS;
                        float M1[1], L1[1];
                        merge_stats<1>(P.ws_ml + hb * 2, 0, 1, pns,
                                       P.sinks ? P.sinks + hq0 + h : nullptr, lane, M1, L1);
                        for (uint32_t s2 = lane; s2 < pns; s2 += 32)
                            wts[h * pns + s2] = exp2f(__ldcg(P.ws_ml + (hb + s2) * 2) - M1[0]);
                        if (lane == 0) invl[h] = __frcp_rn(L1[0]);
                    }
                    named_sync<C::CONS>();
                    // out = sum over the splits, in split order, of w * acc, times 1 / L
                    for (int c = tid; c < G * (HD / 4); c += C::CONS) {
                        const int h = c / (HD / 4), d4 = c % (HD / 4);
                        const size_t hb = (static_cast<size_t>(pb) * P.n_head + hq0 + h) * MS;
                        const float* wsa = P.ws_acc + hb * HD;
                        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (uint32_t s0 = 0; s0 < pns; s0 += 8) {
                            float4 v[8];
                            float wv[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const bool in = s0 + u < pns;
                                v[u] = in ? __ldcg(reinterpret_cast<const float4*>(wsa + (s0 + u) * HD) + d4)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                                wv[u] = in ? wts[h * pns + s0 + u] : 0.f;
                            }
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                a.x = __fmaf_rn(wv[u], v[u].x, a.x);
                                a.y = __fmaf_rn(wv[u], v[u].y, a.y);
                                a.z = __fmaf_rn(wv[u], v[u].z, a.z);
                                a.w = __fmaf_rn(wv[u], v[u].w, a.w);
                            }
                        }
                        const float inv = invl[h];
                        float* orow = P.out + (static_cast<size_t>(pb) * P.n_head + hq0 + h) * HD;
                        reinterpret_cast<float4*>(orow)[d4] =
                            make_float4(__fmul_rn(a.x, inv), __fmul_rn(a.y, inv),
                                        __fmul_rn(a.z, inv), __fmul_rn(a.w, inv));
                    }
                }
                named_sync<C::CONS>();  // the chain scratch is free again
            }
        }
        if (end) {
            // tell the merge warp there is nothing more
            if (warp == W - 1 && lane == 0) {
                const uint32_t hs = handed % NMS;
                if (handed < NMS || mbar_wait(hfree0 + 8 * hs, ((handed / NMS) - 1) & 1)) {
                    hand[hs].end = 1;
                    mbar_arrive(handed0 + 8 * hs);
                } else {
                    atomicOr(P.status, kDevTimeout);
                    misc[0] = 1;
                }
            }
            break;
        }
        const uint32_t b = desc[is].b, kvh = desc[is].kvh, split = desc[is].split;
        const uint32_t nsplit = desc[is].nsplit, p = desc[is].p, prow = desc[is].prow;
        const uint32_t k0 = desc[is].k0, hist_end = desc[is].hist_end;
        const uint32_t ntiles = desc[is].ntiles;
        const bool is_last = desc[is].is_last != 0;
        const float* qs = qbuf + is * G * HD;
        const float* ks = kbuf + is * HD;
        const float* vs = vbuf + is * HD;

        float q[G][E], m[G], l[G], acc[G][E];
        float m_t[C::CNT], l_t[C::CNT];
#pragma unroll
        for (int j = 0; j < C::CNT; ++j) {
            m_t[j] = -CUDART_INF_F;
            l_t[j] = 0.f;
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int c = 0; c < E / 4; ++c) {
                const float4 v =
                    *reinterpret_cast<const float4*>(qs + h * HD + c * 4 * L + li * 4);
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

        for (uint32_t t = 0; t < ntiles; ++t, ++tile_g) {
            const int st = tile_g % S;
            if (misc[0] || !mbar_wait(full0 + 8 * st, (tile_g / S) & 1)) {
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
                if constexpr (C::TR)
                    attend_rows_tr<HD, G, E, L, C::RC, C::GP, C::CNT>(
                        Kt, Vt, row, valid, li, lane, q, m_t, l_t, acc,
                        reinterpret_cast<float*>(smem + C::OFF_PBUF) + gid * C::NV);
                else
                    attend_rows<HD, G, E, L, C::RC>(Kt, Vt, row, valid, li, q, m, l, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
        }
        // an abort by any warp must send every consumer warp to the drain
        named_sync<C::CONS>();
        if (misc[0]) break;
        if constexpr (C::TR) tr_state_to_heads<G, L, C::RC, C::GP, C::CNT>(li, lane, m_t, l_t, m, l);

        if (is_last && warp == 0) {
            const int row1[1] = {0};
            const bool valid1[1] = {gid == 0};
            attend_rows<HD, G, E, L, 1>(ks, vs, row1, valid1, li, q, m, l, acc);
            // key p's K and V rows go to row prow: (slot*slot_ctx + p) in a slot,
            // (block*block_size + p % block_size) in paged mode
            const size_t at = static_cast<size_t>(prow) * P.n_kv_head + kvh;
            float4* kd = reinterpret_cast<float4*>(P.K + at * HD);
            float4* vd = reinterpret_cast<float4*>(P.V + at * HD);
            for (int i = lane; i < HD / 4; i += 32) {
                kd[i] = reinterpret_cast<const float4*>(ks)[i];
                vd[i] = reinterpret_cast<const float4*>(vs)[i];
            }
        }

        // ------------------------------------ merge the groups of each warp
        constexpr int EF = HD / 32;
        const int e0 = merge_warp_groups<G, E, L>(lane, m, l, acc);
        // element t < EF of this lane's slice sits at dimension dim(t) of a head
        // (pairs t, t + 1 are adjacent: EF and e0 are even)
        auto dim = [&](int t) { return ((e0 + t) >> 2) * 4 * L + 4 * li + ((e0 + t) & 3); };
        // ------------------------------------ chain the four warps: 0 -> 1 -> 2 -> 3
        for (int w2 = 0; w2 < W; ++w2) {
            if (warp == w2) {
                if (w2 > 0) {
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float Mc = chain_m[h], Lc = chain_l[h];
                        const float M = fmaxf(m[h], Mc);
                        const float c1 = partial_weight(m[h], M), c2 = partial_weight(Mc, M);
                        l[h] = __fmaf_rn(l[h], c1, __fmul_rn(Lc, c2));
#pragma unroll
                        for (int t = 0; t < EF; t += 2) {
                            const float2 v = *reinterpret_cast<const float2*>(chain + h * HD + dim(t));
                            acc[h][t] = __fmaf_rn(acc[h][t], c1, __fmul_rn(v.x, c2));
                            acc[h][t + 1] = __fmaf_rn(acc[h][t + 1], c1, __fmul_rn(v.y, c2));
                        }
                        m[h] = M;
                    }
                    __syncwarp();
                }
                if (w2 < W - 1) {
#pragma unroll
                    for (int h = 0; h < G; ++h) {
#pragma unroll
                        for (int t = 0; t < EF; t += 2)
                            *reinterpret_cast<float2*>(chain + h * HD + dim(t)) =
                                make_float2(acc[h][t], acc[h][t + 1]);
                        if (lane == 0) {
                            chain_m[h] = m[h];
                            chain_l[h] = l[h];
                        }
                    }
                }
            }
            if (w2 < W - 1) named_sync<C::CONS>();
        }

        // ------------------------------------ warp 3 holds the item's result
        if (warp == W - 1) {
            const uint32_t hq0 = kvh * G;  // first query head of this kv head
            if (nsplit == 1) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float c = 1.f, Ls = l[h];
                    if (P.sinks) {
                        const float sk = P.sinks[hq0 + h] * kLog2e;
                        const float M2 = fmaxf(m[h], sk);
                        c = exp2f(m[h] - M2);
                        Ls = Ls * c + exp2f(sk - M2);
                    }
                    float* o = P.out + (static_cast<size_t>(b) * P.n_head + hq0 + h) * HD;
                    const float f = __fmul_rn(c, __frcp_rn(Ls));  // one reciprocal per head
#pragma unroll
                    for (int t = 0; t < EF; t += 2)
                        *reinterpret_cast<float2*>(o + dim(t)) =
                            make_float2(acc[h][t] * f, acc[h][t + 1] * f);
                }
            } else {
                const size_t MS = P.max_splits;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const size_t base = (static_cast<size_t>(b) * P.n_head + hq0 + h) * MS + split;
                    float* a = P.ws_acc + base * HD;
#pragma unroll
                    for (int t = 0; t < EF; t += 2)
                        *reinterpret_cast<float2*>(a + dim(t)) = make_float2(acc[h][t], acc[h][t + 1]);
                    if (lane == 0) {
                        P.ws_ml[base * 2 + 0] = m[h];
                        P.ws_ml[base * 2 + 1] = l[h];
                    }
                }
                __syncwarp();
            }
            // the partial's merge is arranged at the next item's start
            if (lane == 0) {
                pend[1] = b;
                pend[2] = kvh;
                pend[3] = nsplit;
                pend[0] = nsplit > 1 ? 1u : 0u;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(free0 + 8 * is);  // this warp is done with the slot
    }

    if (misc[0]) {
        // drain this CTA's own copies that may still be in flight: the newest
        // tile of each stage and the newest staged items
        named_sync<C::CONS>();
        if (tid == 0) {
            const uint32_t tiles = static_cast<uint32_t>(misc[2]);
            for (uint32_t u = tiles > static_cast<uint32_t>(S) ? tiles - S : 0; u < tiles; ++u)
                mbar_wait(full0 + 8 * (u % S), (u / S) & 1, 1ll << 28);
            const uint32_t items = static_cast<uint32_t>(misc[3]);
            for (uint32_t u = items > 2u ? items - 2 : 0; u < items; ++u)
                mbar_wait(staged0 + 8 * (u & 1), (u >> 1) & 1, 1ll << 28);
        }
    }
}

// ------------------------------------------------------------ prefill KV write
// One warp per (token, kv head): k' = RoPE(RMSnorm(k_new)) and v (or its
// weightless norm) into the slot row (slot*slot_ctx + pos).  Out-of-range
// tokens are skipped (the plan kernel raises the flag).
template <int HD>
__global__ void __launch_bounds__(128) slotkv_write_kv_kernel(const DecodeParams P) {
    const int lane = threadIdx.x & 31;
    const uint32_t wg = blockIdx.x * 4 + (threadIdx.x >> 5);
    const uint32_t tok = wg / P.n_kv_head, kvh = wg % P.n_kv_head;
    if (tok >= P.B) return;
    const uint32_t p = P.positions[tok], slot = P.slots[tok];
    if (slot >= P.n_slots || p >= P.slot_ctx) return;
    float cs[HD / 64], sn[HD / 64];
    warp_rope_angles<HD>(p, P.inv_freq, cs, sn, lane);
    const float w1 = (P.flags & kOptNormPlusOne) ? 1.0f : 0.0f;
    const size_t src = (static_cast<size_t>(tok) * P.n_kv_head + kvh) * HD;
    const size_t dst = ((static_cast<size_t>(slot) * P.slot_ctx + p) * P.n_kv_head + kvh) * HD;
    warp_norm_rope<HD>(P.k_new + src, P.K + dst, P.k_norm_w, w1, 1.0f, P.eps, cs, sn, lane);
    if (P.flags & kOptVNorm) {
        warp_rms_norm_plain<HD>(P.v_new + src, P.V + dst, P.eps, lane);
    } else {
#pragma unroll
        for (int j = 0; j < HD / 32; ++j) P.V[dst + lane + 32 * j] = P.v_new[src + lane + 32 * j];
    }
}

template <int HD, int G>
int launch_one(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
               unsigned ctas, cudaStream_t stream) {
    using C = KCfg<HD, G>;
    // kernel attributes belong to each device's copy of the kernels: set them
    // once per device (bit d of the mask; devices past 63 set them every time)
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!(configured.load(std::memory_order_acquire) & bit) || bit == 0) {
        cudaError_t e = cudaFuncSetAttribute(slotkv_decode_attn_kernel<HD, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return static_cast<int>(e);
        // one shared-memory carve-out for every kernel of a call, so the SMs
        // need no reconfiguration between them
        const int carve = cudaSharedmemCarveoutMaxShared;
        if ((e = cudaFuncSetAttribute(slotkv_decode_attn_kernel<HD, G>,
                                      cudaFuncAttributePreferredSharedMemoryCarveout, carve)) !=
                cudaSuccess ||
            (e = cudaFuncSetAttribute(slotkv_plan_kernel<C::T>,
                                      cudaFuncAttributePreferredSharedMemoryCarveout, carve)) !=
                cudaSuccess ||
            (e = cudaFuncSetAttribute(slotkv_write_kv_kernel<HD>,
                                      cudaFuncAttributePreferredSharedMemoryCarveout, carve)) !=
                cudaSuccess)
            return static_cast<int>(e);
        // the register hand-over assumes the launch gives every thread 128
        // registers; with fewer, the consumers' request could never be met
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, slotkv_decode_attn_kernel<HD, G>);
        if (e != cudaSuccess) return static_cast<int>(e);
        if (fa.numRegs != 128) return static_cast<int>(cudaErrorInvalidConfiguration);
        // the grid (two CTAs per SM) and its static items assume that both
        // CTAs of an SM are resident at once
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, slotkv_decode_attn_kernel<HD, G>,
                                                          C::THREADS, C::SMEM);
        if (e != cudaSuccess) return static_cast<int>(e);
        if (per_sm < 2) return static_cast<int>(cudaErrorInvalidConfiguration);
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    if (p.prefill) {
        const uint32_t warps = p.B * p.n_kv_head;
        slotkv_write_kv_kernel<HD><<<(warps + 3) / 4, 128, 0, stream>>>(p);
    }
    cudaError_t e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (!p.no_plan) {
        // a programmatic dependent of the preceding work (see the plan kernel)
        cudaLaunchConfig_t pc = {};
        pc.gridDim = dim3(1);
        pc.blockDim = dim3(kPlanThreads);
        pc.stream = stream;
        pc.attrs = attr;
        pc.numAttrs = 1;
        e = cudaLaunchKernelEx(&pc, slotkv_plan_kernel<C::T>, p);
        if (e != cudaSuccess) return static_cast<int>(e);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = p.no_plan ? 0 : 1;  // programmatic dependent of the plan kernel
    e = cudaLaunchKernelEx(&cfg, slotkv_decode_attn_kernel<HD, G>, tmK, tmV, p);
    return static_cast<int>(e);
}

template <int HD>
int launch_hd(int G, const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
              unsigned ctas, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_one<HD, 1>(p, tmK, tmV, ctas, stream);
        case 2: return launch_one<HD, 2>(p, tmK, tmV, ctas, stream);
        case 3: return launch_one<HD, 3>(p, tmK, tmV, ctas, stream);
        case 4: return launch_one<HD, 4>(p, tmK, tmV, ctas, stream);
        case 5: return launch_one<HD, 5>(p, tmK, tmV, ctas, stream);
        case 6: return launch_one<HD, 6>(p, tmK, tmV, ctas, stream);
        case 7: return launch_one<HD, 7>(p, tmK, tmV, ctas, stream);
        case 8: return launch_one<HD, 8>(p, tmK, tmV, ctas, stream);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace slotkv

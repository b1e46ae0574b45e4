// prefill_tc.cuh -- batched causal prefill on the tensor cores, for head dims
// 64 and 128 ("Forward Cuda Gemma", prefillBatched: all prompt tokens of a
// call at once, equal to running them one decode step at a time; "Forward
// Cuda", batched prefill into the given slot).
//
// Three kernels per call, on one stream (the plan launched first, prep
// beside it as a programmatic dependent, the attention kernel after both):
//   * slotkv_prefill_prep_kernel: one warp per (token, 8 query heads or 4 kv
//     heads).  Query heads:
//     q' = RoPE(RMSnorm(q) * w) * scale * log2(e) into a workspace; kv heads:
//     k' = RoPE(RMSnorm(k_new) * w) and v into the token's slot row.  The
//     vector routines are the decode kernel's, so q' and k' are the same
//     bits as a decode step's.
//   * slotkv_prefill_plan_kernel (one CTA): cuts each run of consecutive
//     same-slot tokens into tiles of MT = 128 / G tokens -- a tile's G query
//     heads per token make the 128 rows of one MMA -- and lists the tiles,
//     handed out in reverse (each run from its last tile to its first).  A
//     work item is one (tile, kv head): keys 0 .. the tile's largest
//     position, read once for all its rows.
//   * slotkv_prefill_tc_kernel (persistent, one CTA per SM): flash attention
//     of each item with f32 accuracy from TF32 tensor-core products, split
//     in three: a = a_hi + a_lo with a_hi = a with its low 13 mantissa bits
//     cleared (exact in TF32) and a_lo = a - a_hi (exact in f32), and
//     a.b ~ a_hi.b_hi + a_hi.b_lo + a_lo.b_hi (the dropped a_lo.b_lo and the
//     TF32 rounding of the lo parts are ~2^-20 relative).
//       - warp 8 (producer): claims items and streams each key tile's K
//         and then V (BK = 64 keys x hd, 128-byte swizzled boxes of 32
//         floats) with TMA into a ring of half-stage slots (one operand's
//         hi and lo buffers each: 3 slots for hd 128, 6 for hd 64);
//       - warps 10-13 (converters): write each landed K tile's lo part
//         beside it (the tensor core reads a TF32 operand's f32 bits with the
//         low 13 mantissa bits ignored, so the landed tile is its own hi
//         part), and transpose each landed V tile into
//         a keys-contiguous layout while splitting it (TF32 MMA operands
//         in shared memory are K-major: for O += P V that is V^T, [hd][keys]);
//         keys past the item's last are zeroed;
//       - warp 9 (MMA issuer, one thread): S = Q K^T into a TMEM score
//         buffer (A = Q from TMEM), then O += P V (A = P from TMEM, B = the
//         transposed V tile).  With two score buffers (hd 64) the issue order
//         is QK(t+1), PV(t), QK(t+2), ...; with one (hd 128, where Q's hi and
//         lo parts take half of tensor memory) QK(t), PV(t), QK(t+1), ....
//         MMAs from one thread run in issue order, so a QK reuses a buffer
//         only after the PV before it has read it;
//       - warps 0-7 (softmax; two threads per query row = TMEM lane, each
//         with half of the columns, combining maxima and sums at pairwise
//         named barriers): put the item's q rows (hi, lo) into TMEM -- the
//         next item's as soon as the current item's last P is written, so
//         the next item's first QK overlaps the current item's epilogue --
//         then per key tile read S,
//         apply the causal mask (key <= the row's position), run a base-2
//         online softmax with a lazily raised max, write P (hi over S, lo
//         beside it) into the same buffer and, only when the max moves,
//         wait for the previous PV and rescale O in TMEM; at the end read O,
//         normalise (sink included) and store out.
// Every mbarrier wait is bounded; on expiry the CTA raises SLOTKV_DEV_TIMEOUT
// and every role leaves its loop; the MMA thread waits for its MMAs and the
// producer for its copies before tensor memory is freed.  The test option
// SLOTKV_OPT_TEST_STALL withholds each CTA's first score-ready signal to
// exercise that path.
#pragma once

#include "decode_attn.cuh"
#include "tc_ops.cuh"

namespace slotkv {

template <int HD, int G>
struct PCfg {
    static constexpr int M = 128;               // query rows per tile (MMA M)
    static constexpr int MT = M / G;            // tokens per tile
    static constexpr int ROWS = MT * G;         // rows in use (<= 128)
    static constexpr int BK = prefill_tile_keys(HD);  // keys per tile (QK's N)
    static constexpr int NB = HD / 32;          // 128-byte column blocks per key row
    static constexpr int BLK = BK * 128;        // one column block: BK rows x 128 B
    static constexpr int BUF = NB * BLK;        // one operand buffer, [BK][HD] f32
    static constexpr int SLOT = 2 * BUF;        // half-stage slot: hi | lo of K or V
    static constexpr int NSLOT = (192 * 1024) / SLOT;  // 3 (hd 128) or 6 (hd 64)
    // V transposed: KB column blocks of 32 keys, each [HD rows][128 B]; the
    // 32 x 32 sub-block (key block kb, dim block db) lands at kb * VT_BLK +
    // db * 4096 (TMA put it at db * BLK + kb * 4096)
    static constexpr int KB = BK / 32;
    static constexpr int VT_BLK = HD * 128;
    // softmax warps: two per tensor-memory lane quarter (warps q and q + 4),
    // each taking half of a score tile's columns
    static constexpr int NSW = 8;
    static constexpr int WARP_TMA = 8, WARP_MMA = 9, WARP_CONV = 10, NCONV = 4;
    static constexpr int SB_PER_WARP = KB * NB / NCONV;  // V sub-blocks per converter warp
    static constexpr int THREADS = 32 * (WARP_CONV + NCONV);
    // tensor memory columns: Q hi | Q lo | O | NBUF buffers of (S, then P hi
    // over it | P lo)
    static constexpr uint32_t C_QHI = 0, C_QLO = HD, C_O = 2 * HD, C_S = 3 * HD;
    static constexpr uint32_t C_BUF = 2 * BK;   // columns per score buffer
    static constexpr int NBUF = (512 - 3 * HD) / (2 * BK) >= 2 ? 2 : 1;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(3 * HD + NBUF * 2 * BK <= 512, "tensor memory columns");
    static_assert(BK % 32 == 0 && HD % 32 == 0, "32-column tensor memory accesses");
    // shared memory after the ring: item descriptors [2][8] | slot meta
    // [NSLOT][4] | barriers | tensor memory address | flags
    static constexpr int OFF_DESC = NSLOT * SLOT;
    static constexpr int OFF_META = OFF_DESC + 2 * 32;
    static constexpr int OFF_BAR = OFF_META + NSLOT * 16;
    // full[NSLOT], conv[NSLOT], empty[NSLOT], s_full[2], p_ready[2],
    // pv_done[2], q_ready, item_full[2], item_free[2], drain
    static constexpr int NBAR = 3 * NSLOT + 12;
    static constexpr int OFF_TSLOT = OFF_BAR + NBAR * 8;
    static constexpr int OFF_MISC = OFF_TSLOT + 16;
    // misc[0]: abort; misc[2 + w]: converter warp w's stop flag
    // the softmax halves' exchange: row maxima [2 parities][2 halves][M],
    // row sums [2 halves][M], and a stop flag beside each
    static constexpr int OFF_XCH = OFF_MISC + 64;
    static constexpr int SMEM_USED = OFF_XCH + 2 * 6 * M * 4;
    static constexpr int SMEM = SMEM_USED + 1024;   // slack to align the ring to 1 KiB
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(BLK % 1024 == 0 && SLOT % 1024 == 0, "128-byte swizzle atoms stay 1 KiB aligned");
    static constexpr uint32_t IDESC_QK = tc::idesc_tf32(M, BK, false);
    static constexpr uint32_t IDESC_PV = tc::idesc_tf32(M, HD, false);
    static_assert(KB * NB == SB_PER_WARP * NCONV, "V sub-blocks split evenly over the converters");
};

// Named barrier 2 over the converter warps (N threads).
template <int N>
__device__ __forceinline__ void named_sync_conv() {
    asm volatile("bar.sync 2, %0;" ::"n"(N) : "memory");
}

// 2^x by the hardware's approximate base-2 exponential (PTX ex2.approx.ftz:
// a few ulp of relative error, subnormal results flushed to zero), far
// inside the f32 tolerance of the step.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Split x into an exactly-TF32 high part and the f32 remainder.
__device__ __forceinline__ void tf32_split(float x, uint32_t& hi, uint32_t& lo) {
    const uint32_t h = __float_as_uint(x) & 0xFFFFE000u;
    hi = h;
    lo = __float_as_uint(x - __uint_as_float(h));
}

// ------------------------------------------------------------------ prep
// One warp per (token, group of heads): kPrepHeads query heads, or
// kPrepKvHeads kv heads (their k_new and v_new rows), so that every warp
// stages kPrepHeads rows.  The group's rows are staged into the warp's
// shared memory with cp.async, all in flight at once, while the warp forms
// the token's RoPE angles; then each row goes through the decode kernel's
// vector routine (the same arithmetic on the same values, so the same bits
// as a decode step).
constexpr int kPrepHeads = 8, kPrepKvHeads = kPrepHeads / 2;

__device__ __forceinline__ void prep_cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)),
                 "l"(gmem_src)
                 : "memory");
}

template <int HD>
__host__ __device__ constexpr int prep_smem_bytes() {
    return 4 * kPrepHeads * HD * 4;  // four warps x kPrepHeads rows
}

// query-head groups and kv-head groups per token
__host__ __device__ inline uint32_t prep_q_groups(uint32_t n_head) {
    return (n_head + kPrepHeads - 1) / kPrepHeads;
}
__host__ __device__ inline uint32_t prep_groups(uint32_t n_head, uint32_t n_kv_head) {
    return prep_q_groups(n_head) + (n_kv_head + kPrepKvHeads - 1) / kPrepKvHeads;
}

template <int HD>
__global__ void __launch_bounds__(128) slotkv_prefill_prep_kernel(const PrefillParams P) {
    extern __shared__ __align__(16) uint8_t prep_smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t qg = prep_q_groups(P.n_head), groups = prep_groups(P.n_head, P.n_kv_head);
    const uint32_t wg = blockIdx.x * 4 + warp;
    const uint32_t tok = wg / groups, grp = wg % groups;
    if (tok >= P.n_tok) return;
    const uint32_t p = P.positions[tok], slot = P.slots[tok];
    if (slot >= P.n_slots || p >= P.slot_ctx) return;  // the plan raises the flag
    const bool is_q = grp < qg;
    // the group's first head (a query head, or a kv head) and its size
    const uint32_t x0 = is_q ? grp * kPrepHeads : (grp - qg) * kPrepKvHeads;
    const uint32_t left = (is_q ? P.n_head : P.n_kv_head) - x0;
    const uint32_t cap = is_q ? kPrepHeads : kPrepKvHeads;
    const uint32_t nx = left < cap ? left : cap;
    float* rows = reinterpret_cast<float*>(prep_smem) + warp * kPrepHeads * HD;
    float* vrows = rows + kPrepKvHeads * HD;  // kv groups: v rows after the k rows
    for (uint32_t i = 0; i < nx; ++i) {
        const uint32_t x = x0 + i;
        if (is_q) {
            const float* src = P.q + (static_cast<size_t>(tok) * P.n_head + x) * HD;
            for (int c = lane; c < HD / 4; c += 32) prep_cp_async16(rows + i * HD + 4 * c, src + 4 * c);
        } else {
            const size_t at = (static_cast<size_t>(tok) * P.n_kv_head + x) * HD;
            for (int c = lane; c < HD / 4; c += 32) {
                prep_cp_async16(rows + i * HD + 4 * c, P.k_new + at + 4 * c);
                prep_cp_async16(vrows + i * HD + 4 * c, P.v_new + at + 4 * c);
            }
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    float cs[HD / 64], sn[HD / 64];
    warp_rope_angles<HD>(p, P.inv_freq, cs, sn, lane);
    const float w1 = (P.flags & kOptNormPlusOne) ? 1.0f : 0.0f;
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
    for (uint32_t i = 0; i < nx; ++i) {
        const uint32_t x = x0 + i;
        if (is_q) {
            const size_t at = (static_cast<size_t>(tok) * P.n_head + x) * HD;
            warp_norm_rope<HD>(rows + i * HD, P.q_rot + at, P.q_norm_w, w1, P.scale_log2, P.eps,
                               cs, sn, lane);
            continue;
        }
        const size_t dst = ((static_cast<size_t>(slot) * P.slot_ctx + p) * P.n_kv_head + x) * HD;
        warp_norm_rope<HD>(rows + i * HD, P.K + dst, P.k_norm_w, w1, 1.0f, P.eps, cs, sn, lane);
        if (P.flags & kOptVNorm) {
            warp_rms_norm_plain<HD>(vrows + i * HD, P.V + dst, P.eps, lane);
        } else {
#pragma unroll
            for (int j = 0; j < HD / 32; ++j) P.V[dst + lane + 32 * j] = vrows[i * HD + lane + 32 * j];
        }
    }
}

// ------------------------------------------------------------------ plan
// One CTA of 1024 threads, tokens in rounds of 1024.  A run is a maximal
// sequence of consecutive in-range tokens with the same slot; token i starts
// a tile when its index within its run is a multiple of MT.  Tile records:
// (first token, tokens, slot, largest position).  Out-of-range tokens raise
// SLOTKV_DEV_RANGE and belong to no tile.  Then the tiles' hand-out order.

template <int MT>
__global__ void __launch_bounds__(1024, 1) slotkv_prefill_plan_kernel(const PrefillParams P) {
    __shared__ int warp_max[32];
    __shared__ uint32_t warp_sum[32];
    __shared__ int carry_start;
    __shared__ uint32_t carry_tiles;
    // The prep kernel, launched next as a programmatic dependent, may start
    // at once: it reads none of what this kernel writes and writes none of
    // what it reads, and the attention kernel after both waits for both.
    grid_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry_start = -1;
        carry_tiles = 0;
    }
    __syncthreads();
    uint4* tiles = reinterpret_cast<uint4*>(P.tiles);
    for (uint32_t r0 = 0; r0 < P.n_tok; r0 += 1024) {
        const uint32_t i = r0 + tid;
        bool valid = false, start = false;
        uint32_t slot = 0;
        if (i < P.n_tok) {
            slot = P.slots[i];
            valid = slot < P.n_slots && P.positions[i] < P.slot_ctx;
            if (!valid) atomicOr(P.status, kDevRange);
            if (valid) {
                if (i == 0) {
                    start = true;
                } else {
                    const uint32_t ps = P.slots[i - 1];
                    start = ps != slot || P.positions[i - 1] >= P.slot_ctx;
                }
            }
        }
        // the latest run start at or before i: an inclusive prefix max
        int a = start ? static_cast<int>(i) : -1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, a, off);
            if (lane >= off) a = a > o ? a : o;
        }
        if (lane == 31) warp_max[warp] = a;
        __syncthreads();
        if (warp == 0) {
            int v = warp_max[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v = v > o ? v : o;
            }
            warp_max[lane] = v;
        }
        __syncthreads();
        int rs = warp > 0 ? warp_max[warp - 1] : -1;
        rs = rs > carry_start ? rs : carry_start;
        rs = rs > a ? rs : a;
        const bool tflag = valid && ((i - static_cast<uint32_t>(rs)) % MT) == 0;
        // tile index: an inclusive prefix sum of the tile starts
        uint32_t c = tflag ? 1u : 0u;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, c, off);
            if (lane >= off) c += o;
        }
        if (lane == 31) warp_sum[warp] = c;
        __syncthreads();
        if (warp == 0) {
            uint32_t v = warp_sum[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t o = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += o;
            }
            warp_sum[lane] = v;
        }
        __syncthreads();
        const uint32_t incl = c + (warp > 0 ? warp_sum[warp - 1] : 0u) + carry_tiles;
        if (tflag) tiles[incl - 1] = make_uint4(i, 0u, slot, 0u);
        if (i < P.n_tok) P.tile_of[i] = valid ? incl - 1 : 0xFFFFFFFFu;
        __syncthreads();  // every thread has read the carries
        if (tid == 1023) {
            carry_start = rs;
            carry_tiles = incl;
        }
        __syncthreads();
    }
    // each tile's token count and largest position
    for (uint32_t i = tid; i < P.n_tok; i += 1024) {
        const uint32_t t = P.tile_of[i];
        if (t == 0xFFFFFFFFu) continue;
        uint32_t* rec = P.tiles + 4 * static_cast<size_t>(t);
        atomicAdd(rec + 1, 1u);
        atomicMax(rec + 3, P.positions[i]);
    }
    __syncthreads();
    // The hand-out order, into tile_of (its per-token use is over): the
    // tiles in reverse, so each run is handed out from its last tile (the
    // most keys, when its positions increase) to its first, one run after
    // the other -- the attention kernel ends on small items while a run's
    // keys stay in L2 across its tiles.  (Any order gives the same bits:
    // items are independent.)
    const uint32_t n_tiles = carry_tiles;
    for (uint32_t t = tid; t < n_tiles; t += 1024) P.tile_of[t] = n_tiles - 1 - t;
    __syncthreads();
    if (tid == 0) {
        P.plan[0] = carry_tiles * P.n_kv_head;
        P.plan[1] = 0;
    }
}

// ------------------------------------------------------------------ attention
// Half-tile h of the CTA's stream of key tiles: h = 2g is tile g's K, h = 2g + 1
// its V; it lives in slot h % NSLOT.
template <int HD, int G>
__global__ void __launch_bounds__(PCfg<HD, G>::THREADS, 1)
    slotkv_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const PrefillParams P) {
    using C = PCfg<HD, G>;
    constexpr int BK = C::BK, NB = C::NB, NSLOT = C::NSLOT, NBUF = C::NBUF;
    constexpr float kLog2e = 1.4426950408889634f;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile uint32_t* desc = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_DESC);
    volatile uint32_t* meta = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_META);
    volatile int* misc = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + C::OFF_TSLOT);
    const uint32_t ring = smem_addr(smem);
    const uint32_t bar0 = smem_addr(smem + C::OFF_BAR);
    const uint32_t FULL = bar0, CONV = bar0 + 8 * NSLOT, EMPTY = bar0 + 16 * NSLOT;
    const uint32_t SFULL = bar0 + 24 * NSLOT, PREADY = SFULL + 16;
    const uint32_t PVDONE = PREADY + 16, QREADY = PVDONE + 16, IFULL = QREADY + 8;
    const uint32_t IFREE = IFULL + 16, DRAIN = IFREE + 16;
    // hi and lo operand buffers of a slot
    auto slot_hi = [&](uint32_t sl) { return ring + sl * C::SLOT; };
    auto slot_lo = [&](uint32_t sl) { return ring + sl * C::SLOT + C::BUF; };

    if (tid == 0) {
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(FULL + 8 * i, 1);
            mbar_init(CONV + 8 * i, C::NCONV);
            mbar_init(EMPTY + 8 * i, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(SFULL + 8 * b, 1);
            mbar_init(PREADY + 8 * b, C::NSW);
            mbar_init(PVDONE + 8 * b, 1);
            mbar_init(IFULL + 8 * b, 1);
            mbar_init(IFREE + 8 * b, C::NSW + 1);
        }
        mbar_init(QREADY, C::NSW);
        mbar_init(DRAIN, 1);
        misc[0] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        tc::tmem_alloc(smem_addr(tslot), C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;
    auto timeout = [&]() {
        atomicOr(P.status, kDevTimeout);
        misc[0] = 1;
    };

    if (warp == C::WARP_TMA) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t n_items = __ldcg(P.plan);
            const uint4* tiles = reinterpret_cast<const uint4*>(P.tiles);
            uint32_t h = 0;  // half-tiles issued
            // wait until slot h % NSLOT is free again
            auto slot_free = [&](uint32_t hh) {
                return hh < static_cast<uint32_t>(NSLOT) ||
                       mbar_wait(EMPTY + 8 * (hh % NSLOT), ((hh / NSLOT) - 1) & 1);
            };
            for (uint32_t k = 0;; ++k) {
                const uint32_t is = k & 1;
                if (k >= 2 && !mbar_wait(IFREE + 8 * is, ((k >> 1) - 1) & 1)) {
                    timeout();
                    break;
                }
                if (misc[0]) break;
                volatile uint32_t* d = desc + 8 * is;
                const uint32_t it = atomicAdd(P.plan + 1, 1u);
                if (it >= n_items) {
                    d[6] = 1;
                    mbar_arrive(IFULL + 8 * is);
                    // tell the converters: an end marker in the next slot
                    if (!slot_free(h)) {
                        timeout();
                        break;
                    }
                    meta[4 * (h % NSLOT) + 1] = 1;
                    mbar_arrive(FULL + 8 * (h % NSLOT));
                    break;
                }
                // in the plan's hand-out order
                const uint4 rec = __ldcg(tiles + __ldcg(P.tile_of + it / P.n_kv_head));
                const uint32_t kvh = it % P.n_kv_head;
                const uint32_t max_pos = rec.w;
                const uint32_t ntiles = (max_pos + BK) / BK;  // keys 0 .. max_pos
                d[0] = rec.x;
                d[1] = rec.y;
                d[2] = rec.z;
                d[3] = max_pos;
                d[4] = kvh;
                d[5] = ntiles;
                d[6] = 0;
                mbar_arrive(IFULL + 8 * is);
                const int y0 = static_cast<int>(rec.z * P.slot_ctx);
                for (uint32_t t = 0; t < ntiles && !misc[0]; ++t) {
                    const uint32_t left = max_pos + 1 - t * BK;
                    const int y = y0 + static_cast<int>(t * BK);
                    for (int which = 0; which < 2; ++which, ++h) {  // K, then V
                        if (!slot_free(h)) {
                            timeout();
                            break;
                        }
                        const uint32_t sl = h % NSLOT;
                        meta[4 * sl + 0] = left < static_cast<uint32_t>(BK) ? left : BK;
                        meta[4 * sl + 1] = 0;
                        mbar_expect_tx(FULL + 8 * sl, C::BUF);
#pragma unroll
                        for (int c = 0; c < NB; ++c)
                            tma_load_2d(slot_hi(sl) + c * C::BLK, which ? &tmV : &tmK,
                                        static_cast<int>(kvh * HD) + 32 * c, y, FULL + 8 * sl);
                    }
                }
                if (misc[0]) break;
            }
            if (misc[0]) {
                // drain this CTA's copies that may still be in flight
                for (uint32_t u = h > static_cast<uint32_t>(NSLOT) ? h - NSLOT : 0; u < h; ++u)
                    mbar_wait(FULL + 8 * (u % NSLOT), (u / NSLOT) & 1, 1ll << 28);
            }
        }
    } else if (warp >= C::WARP_CONV) {
        // ------------------------------------------------------------ converters
        const int ct = tid - C::WARP_CONV * 32;
        const int w = ct >> 5;
        constexpr int NT = C::NCONV * 32;
        for (uint32_t h = 0;; ++h) {
            const uint32_t sl = h % NSLOT;
            // The converter warps meet at named barriers below, so they must
            // all stop at the same half-tile: each publishes its own reason
            // to stop (a wait that expired, an abort, the end marker) and all
            // decide from the published flags.
            const bool ok = mbar_wait(FULL + 8 * sl, (h / NSLOT) & 1);
            if (!ok) timeout();
            if (lane == 0) misc[2 + w] = (!ok || misc[0] || meta[4 * sl + 1]) ? 1 : 0;
            named_sync_conv<NT>();
            int stop = 0;
#pragma unroll
            for (int w2 = 0; w2 < C::NCONV; ++w2) stop |= misc[2 + w2];
            if (stop) break;
            const uint32_t rows = meta[4 * sl + 0];
            uint8_t* hib = smem + sl * C::SLOT;
            uint8_t* lob = hib + C::BUF;
            if ((h & 1) == 0) {
                // K: the landed f32 tile is its own hi part (the tensor core
                // reads a TF32 operand's f32 bits with the low 13 mantissa
                // bits ignored, i.e. as x & 0xFFFFE000), so only the lo part
                // is written beside it (K-major, as TMA laid the tile out);
                // rows past the item's last key are zeroed in both
                float4* hi = reinterpret_cast<float4*>(hib);
                float4* lo = reinterpret_cast<float4*>(lob);
#pragma unroll
                for (int i = ct; i < C::BUF / 16; i += NT) {
                    // each 128-byte row of a column block is 8 float4s
                    const uint32_t row = static_cast<uint32_t>(i % (C::BLK / 16)) / 8;
                    if (row >= rows) {
                        hi[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                        lo[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                        continue;
                    }
                    const float4 x = hi[i];
                    uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
                    tf32_split(x.x, h0, l0);
                    tf32_split(x.y, h1, l1);
                    tf32_split(x.z, h2, l2);
                    tf32_split(x.w, h3, l3);
                    lo[i] = make_float4(__uint_as_float(l0), __uint_as_float(l1),
                                        __uint_as_float(l2), __uint_as_float(l3));
                }
            } else {
                // V: every 32 x 32 sub-block transposed (keys along the
                // 128-byte rows), hi in place, lo into the lo buffer.  All
                // converter threads read their sub-blocks (lane = dim, one
                // key per load) before any writes, so the in-place
                // permutation is safe whatever its cycles.
                float x[C::SB_PER_WARP][32];
#pragma unroll
                for (int j = 0; j < C::SB_PER_WARP; ++j) {
                    const int sb = w + C::NCONV * j;
                    const int kb = sb / NB, db = sb % NB;
                    const uint8_t* src = hib + db * C::BLK + kb * 4096;
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const uint32_t off = (k / 8) * 1024 + (k % 8) * 128 +
                                             (((lane / 4) ^ (k % 8)) * 16) + (lane % 4) * 4;
                        const float v = *reinterpret_cast<const float*>(src + off);
                        x[j][k] = static_cast<uint32_t>(kb * 32 + k) < rows ? v : 0.f;
                    }
                }
                named_sync_conv<NT>();
#pragma unroll
                for (int j = 0; j < C::SB_PER_WARP; ++j) {
                    const int sb = w + C::NCONV * j;
                    const int kb = sb / NB, db = sb % NB;
                    const uint32_t base = kb * C::VT_BLK + db * 4096 + (lane / 8) * 1024 +
                                          (lane % 8) * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t hh[4], ll[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) tf32_split(x[j][4 * c + e], hh[e], ll[e]);
                        const uint32_t off = base + ((c ^ (lane % 8)) * 16);
                        *reinterpret_cast<uint4*>(hib + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                        *reinterpret_cast<uint4*>(lob + off) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                    }
                }
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(CONV + 8 * sl);
        }
    } else if (warp == C::WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t g = 0;  // key tiles whose QK was issued
            bool ok = true;
            auto converted = [&](uint32_t hh) {
                return mbar_wait(CONV + 8 * (hh % NSLOT), (hh / NSLOT) & 1);
            };
            // O += P V for tile t of the item (global tile gp)
            auto issue_pv = [&](uint32_t t, uint32_t gp) {
                const uint32_t hv = 2 * gp + 1;
                if (!converted(hv) || !mbar_wait(PREADY + 8 * (gp & 1), (gp >> 1) & 1)) {
                    timeout();
                    return false;
                }
                tc::fence_after_sync();
                const uint32_t sl = hv % NSLOT;
                const uint32_t pcol0 = C::C_S + (gp % NBUF) * C::C_BUF;
                // O += P_lo V_hi + P_hi V_hi + P_hi V_lo, K-step by K-step
                // (consecutive products share their B, then their A, slice)
#pragma unroll
                for (int kk = 0; kk < BK / 8; ++kk) {
                    const uint32_t off = (kk / 4) * C::VT_BLK + (kk % 4) * 32;
                    const uint64_t bh = tc::smem_desc(slot_hi(sl) + off, 16, 1024, tc::kSwizzle128B);
                    const uint64_t bl = tc::smem_desc(slot_lo(sl) + off, 16, 1024, tc::kSwizzle128B);
                    tc::mma_tf32_ts(tbase + C::C_O, tbase + pcol0 + BK + kk * 8, bh, C::IDESC_PV,
                                    (t | kk) != 0 ? 1u : 0u);
                    tc::mma_tf32_ts(tbase + C::C_O, tbase + pcol0 + kk * 8, bh, C::IDESC_PV, 1u);
                    tc::mma_tf32_ts(tbase + C::C_O, tbase + pcol0 + kk * 8, bl, C::IDESC_PV, 1u);
                }
                tc::mma_commit(PVDONE + 8 * (gp & 1));
                tc::mma_commit(EMPTY + 8 * sl);
                return true;
            };
            for (uint32_t k = 0; ok; ++k) {
                const uint32_t is = k & 1;
                if (!mbar_wait(IFULL + 8 * is, (k >> 1) & 1)) {
                    timeout();
                    break;
                }
                const uint32_t ntiles = desc[8 * is + 5], end = desc[8 * is + 6];
                mbar_arrive(IFREE + 8 * is);
                if (end || misc[0]) break;
                if (!mbar_wait(QREADY, k & 1)) {
                    timeout();
                    break;
                }
                tc::fence_after_sync();
                for (uint32_t t = 0; t < ntiles; ++t, ++g) {
                    const uint32_t hk = 2 * g;
                    if (!converted(hk)) {
                        timeout();
                        ok = false;
                        break;
                    }
                    if (misc[0]) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    // S = Q_lo K_hi + Q_hi K_hi + Q_hi K_lo, K-step by K-step
                    // (consecutive products share their B, then their A, slice)
                    const uint32_t sl = hk % NSLOT;
                    const uint32_t scol = C::C_S + (g % NBUF) * C::C_BUF;
#pragma unroll
                    for (int kk = 0; kk < HD / 8; ++kk) {
                        const uint32_t off = (kk / 4) * C::BLK + (kk % 4) * 32;
                        const uint64_t bh = tc::smem_desc(slot_hi(sl) + off, 16, 1024, tc::kSwizzle128B);
                        const uint64_t bl = tc::smem_desc(slot_lo(sl) + off, 16, 1024, tc::kSwizzle128B);
                        tc::mma_tf32_ts(tbase + scol, tbase + C::C_QLO + kk * 8, bh, C::IDESC_QK,
                                        kk != 0 ? 1u : 0u);
                        tc::mma_tf32_ts(tbase + scol, tbase + C::C_QHI + kk * 8, bh, C::IDESC_QK, 1u);
                        tc::mma_tf32_ts(tbase + scol, tbase + C::C_QHI + kk * 8, bl, C::IDESC_QK, 1u);
                    }
                    // (the failure-path test option withholds the CTA's first
                    // score-ready signal, so the softmax's bounded wait runs out)
                    if (!(g == 0 && (P.flags & kOptTestStall))) tc::mma_commit(SFULL + 8 * (g & 1));
                    tc::mma_commit(EMPTY + 8 * sl);  // K slot free once QK has read it
                    // one buffer: this tile's PV next; two: the previous tile's
                    if (NBUF == 1) {
                        if (!issue_pv(t, g)) {
                            ok = false;
                            break;
                        }
                    } else if (t >= 1 && !issue_pv(t - 1, g - 1)) {
                        ok = false;
                        break;
                    }
                }
                if (NBUF == 2 && ok && ntiles && !misc[0] && !issue_pv(ntiles - 1, g - 1)) ok = false;
            }
            // every MMA issued above has completed before tensor memory is freed
            tc::mma_commit(DRAIN);
            mbar_wait(DRAIN, 0, 1ll << 28);
        }
    } else {
        // ------------------------------------------------------------ softmax
        // Warps q and q + 4 share tensor-memory lane quarter q (rows 32 q ..
        // 32 q + 31); half hf = warp / 4 takes columns [hf BK/2, (hf+1) BK/2)
        // of each score tile and columns [hf HD/2, (hf+1) HD/2) of Q and O.
        // The two halves of a row meet at a pairwise named barrier to combine
        // their maxima (every tile) and their sums (at an item's end); both
        // keep the same running max.  Every exit from the loops is decided
        // at one of these meetings from both halves' published state (a
        // failed bounded wait or the CTA's abort flag is published, never
        // acted on alone), so neither half can leave its partner waiting at
        // the barrier.
        constexpr int HB = BK / 2, HH = HD / 2;
        static_assert(HB == 32 && HH % 32 == 0, "one 32-column access per half of a score tile");
        const int quarter = warp & 3, hf = warp >> 2;
        const uint32_t r = static_cast<uint32_t>(quarter * 32 + lane);  // query row = TMEM lane
        const uint32_t lrow = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t t_local = r / G, h_local = r % G;
        float* xmax = reinterpret_cast<float*>(smem + C::OFF_XCH);   // [2 parities][2][M]
        float* xsum = xmax + 4 * C::M;                               // [2][M]
        int* xflag = reinterpret_cast<int*>(xmax + 6 * C::M);       // beside each value
        auto pair_sync = [&]() {
            asm volatile("bar.sync %0, 64;" ::"r"(3 + quarter) : "memory");
        };
        // Publish v and this warp's stop flag (any lane's) in slot [hf][r] of
        // buf, meet, and return the partner's value; stop becomes the pair's
        // decision (either warp's flag), the same in all 64 threads.
        auto exchange = [&](float* buf, float v, bool& stop) {
            const int at = static_cast<int>(buf - xmax);
            stop = __any_sync(0xffffffffu, stop);
            buf[hf * C::M + r] = v;
            xflag[at + hf * C::M + r] = stop ? 1 : 0;
            pair_sync();
            stop = stop || xflag[at + (1 - hf) * C::M + r] != 0;
            return buf[(1 - hf) * C::M + r];
        };
        uint32_t g = 0;  // key tiles processed
        // Meeting 1 opens item k: both halves hold its descriptor (xsum is
        // free: every meeting on it is followed by a pair barrier).  stop
        // carries a failure not yet published and becomes the pair's
        // decision; on success the descriptor's slot is released.
        auto open_item = [&](uint32_t k, bool stop, uint32_t (&d)[5]) {
            const uint32_t is = k & 1;
            stop = stop || misc[0];
            if (!stop && !mbar_wait(IFULL + 8 * is, (k >> 1) & 1)) {
                timeout();
                stop = true;
            }
            exchange(xsum, 0.f, stop);
            if (stop) return false;
            d[0] = desc[8 * is + 0];  // first token
            d[1] = desc[8 * is + 1];  // tokens
            d[2] = desc[8 * is + 4];  // kv head
            d[3] = desc[8 * is + 5];  // key tiles
            d[4] = desc[8 * is + 6];  // end marker
            pair_sync();  // both have read meeting 1 before xsum is written again
            __syncwarp();
            if (lane == 0) mbar_arrive(IFREE + 8 * is);
            return true;
        };
        struct ItemRow {
            bool valid;
            uint32_t tok, pos, head;
        };
        auto row_of = [&](const uint32_t (&d)[5]) {
            ItemRow w;
            w.valid = r < static_cast<uint32_t>(C::ROWS) && t_local < d[1];
            w.tok = d[0] + t_local;
            w.pos = w.valid ? __ldg(P.positions + w.tok) : 0u;
            w.head = d[2] * G + h_local;
            return w;
        };
        // this half of the item's q rows into tensor memory, split hi / lo
        auto load_q = [&](const ItemRow& w) {
            const float* qrow = P.q_rot + (static_cast<size_t>(w.valid ? w.tok : 0) * P.n_head + w.head) * HD;
#pragma unroll
            for (int c0 = hf * HH; c0 < (hf + 1) * HH; c0 += 32) {
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 x = w.valid ? __ldcg(reinterpret_cast<const float4*>(qrow + c0 + c))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    tf32_split(x.x, hi[c + 0], lo[c + 0]);
                    tf32_split(x.y, hi[c + 1], lo[c + 1]);
                    tf32_split(x.z, hi[c + 2], lo[c + 2]);
                    tf32_split(x.w, hi[c + 3], lo[c + 3]);
                }
                tc::tmem_st32(lrow + C::C_QHI + c0, hi);
                tc::tmem_st32(lrow + C::C_QLO + c0, lo);
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(QREADY);
        };
        uint32_t d[5];
        if (open_item(0, false, d) && !d[4]) {
            ItemRow cur = row_of(d);
            load_q(cur);
            for (uint32_t k = 0;; ++k) {
                const uint32_t ntiles = d[3];
                float m = -CUDART_INF_F, l = 0.f;  // l: this half's share of the row sum
                bool failed = false;
                for (uint32_t t = 0; t < ntiles; ++t, ++g) {
                    if (!mbar_wait(SFULL + 8 * (g & 1), (g >> 1) & 1)) {
                        timeout();
                        failed = true;
                    }
                    tc::fence_after_sync();
                    const uint32_t scol = C::C_S + (g % NBUF) * C::C_BUF + hf * HB;
                    float s[HB];
                    {
                        uint32_t v[32];
                        tc::tmem_ld32(lrow + scol, v);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < HB; ++c) s[c] = __uint_as_float(v[c]);
                    }
                    // causal mask: key kbase + c is attended iff it is <= cur.pos
                    const uint32_t kbase = t * BK + hf * HB;
                    float mx = -CUDART_INF_F;
                    if (kbase + HB - 1 <= cur.pos) {
#pragma unroll
                        for (int c = 0; c < HB; ++c) mx = fmaxf(mx, s[c]);
                    } else {
#pragma unroll
                        for (int c = 0; c < HB; ++c) {
                            s[c] = kbase + static_cast<uint32_t>(c) <= cur.pos ? s[c] : -CUDART_INF_F;
                            mx = fmaxf(mx, s[c]);
                        }
                    }
                    // meeting 2 (every tile): the row's max over both halves
                    // (double-buffered by tile parity: a half writes parity p
                    // again only after the next meeting, which its partner
                    // reaches after reading p)
                    bool stop2 = failed || misc[0];
                    const float other = exchange(xmax + (g & 1) * 2 * C::M, mx, stop2);
                    if (stop2) {
                        failed = true;
                        break;
                    }
                    mx = fmaxf(mx, other);
                    // lazy running max: raised only when a score passes it by 2^8
                    float corr = 1.f;
                    bool rescale = false;
                    if (mx > m + 8.f) {
                        corr = m == -CUDART_INF_F ? 0.f : fast_exp2(m - mx);
                        rescale = t > 0;
                        l *= corr;
                        m = mx;
                    }
#pragma unroll
                    for (int c = 0; c < HB; ++c) {
                        s[c] = s[c] == -CUDART_INF_F ? 0.f : fast_exp2(s[c] - m);
                        l += s[c];
                    }
                    // O may be rescaled only once the previous tile's O += P V
                    // (global tile g - 1) has completed.  PV(j) completes a phase
                    // of pv_done[j % 2]; at any wait for PV(j), PV(j - 2) has
                    // completed (the S this softmax already read was committed
                    // after it) and PV(j + 2) cannot start (it needs P from this
                    // softmax), so the parity of phase j / 2 is unambiguous.
                    // (One barrier for all PVs would not do: with two score
                    // buffers PV(j - 1) may still be running at the wait for
                    // PV(j), and its parity would read as already complete.)
                    // Both halves of a row take the same decision; a wait that
                    // runs out is published at the next meeting.
                    if (__any_sync(0xffffffffu, rescale)) {
                        if (!mbar_wait(PVDONE + 8 * ((g - 1) & 1), ((g - 1) >> 1) & 1)) {
                            timeout();
                            failed = true;
                        } else {
                            tc::fence_after_sync();
#pragma unroll
                            for (int c0 = hf * HH; c0 < (hf + 1) * HH; c0 += 32) {
                                uint32_t v[32];
                                tc::tmem_ld32(lrow + C::C_O + c0, v);
                                tc::tmem_ld_wait();
#pragma unroll
                                for (int c = 0; c < 32; ++c)
                                    v[c] = __float_as_uint(__uint_as_float(v[c]) * corr);
                                tc::tmem_st32(lrow + C::C_O + c0, v);
                            }
                        }
                    }
                    {
                        uint32_t hi[32], lo[32];
#pragma unroll
                        for (int c = 0; c < HB; ++c) tf32_split(s[c], hi[c], lo[c]);
                        tc::tmem_st32(lrow + scol, hi);
                        tc::tmem_st32(lrow + scol + BK, lo);
                    }
                    tc::tmem_st_wait();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(PREADY + 8 * (g & 1));
                }
                // The next item opens before this one ends: every QK of this
                // item has completed (its last S was read above), so the next
                // item's Q may replace this one's in tensor memory while the
                // last O += P V runs, and the next item's first QK overlaps
                // this item's epilogue.  Its first O += P V overwrites O only
                // after its P is published, which this softmax does after
                // reading O below.  A failure so far is published at this
                // meeting, and both halves leave together.
                if (!open_item(k + 1, failed, d)) break;
                const bool last = d[4] != 0;
                ItemRow nxt{};
                if (!last) {
                    nxt = row_of(d);
                    load_q(nxt);
                }
                // This item's last O += P V (global tile g - 1; its commit
                // covers every earlier MMA), then out = O / l (both halves'
                // sums, sink included).  Meeting 3, the sums, publishes a
                // wait that ran out.
                bool stop3 = !mbar_wait(PVDONE + 8 * ((g - 1) & 1), ((g - 1) >> 1) & 1);
                if (stop3) timeout();
                const float l_other = exchange(xsum, l, stop3);
                pair_sync();  // both have read the sums before xsum is written again
                if (stop3) break;
                tc::fence_after_sync();
                const float lt = l + l_other;
                float f = 1.f / lt;
                if (P.sinks) {
                    const float sk = __ldg(P.sinks + cur.head) * kLog2e;
                    const float M2 = fmaxf(m, sk);
                    const float c = exp2f(m - M2);
                    f = c / (lt * c + exp2f(sk - M2));
                }
                float* orow = P.out + (static_cast<size_t>(cur.tok) * P.n_head + cur.head) * HD;
#pragma unroll
                for (int c0 = hf * HH; c0 < (hf + 1) * HH; c0 += 32) {
                    uint32_t v[32];
                    tc::tmem_ld32(lrow + C::C_O + c0, v);
                    tc::tmem_ld_wait();
                    if (cur.valid) {
#pragma unroll
                        for (int c = 0; c < 32; c += 4)
                            *reinterpret_cast<float4*>(orow + c0 + c) =
                                make_float4(__uint_as_float(v[c]) * f, __uint_as_float(v[c + 1]) * f,
                                            __uint_as_float(v[c + 2]) * f, __uint_as_float(v[c + 3]) * f);
                    }
                }
                tc::fence_before_sync();
                if (last) break;
                cur = nxt;
            }
        }
    }
    // ---------------------------------------------------------------- teardown
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tbase, C::TMEM_COLS);
}

template <int HD, int G>
int launch_prefill_one(const PrefillParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       unsigned ctas, cudaStream_t stream) {
    using C = PCfg<HD, G>;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!(configured.load(std::memory_order_acquire) & bit) || bit == 0) {
        cudaError_t e = cudaFuncSetAttribute(slotkv_prefill_tc_kernel<HD, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return static_cast<int>(e);
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const uint32_t warps = p.n_tok * prep_groups(p.n_head, p.n_kv_head);
    // the plan (one CTA) first, then prep beside it as its programmatic
    // dependent; the attention kernel, launched in stream order, waits for
    // both.  Prep starts only once the plan runs, hence after the previous
    // call's attention kernel has finished reading the rows and q workspace
    // that prep overwrites.
    slotkv_prefill_plan_kernel<C::MT><<<1, 1024, 0, stream>>>(p);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((warps + 3) / 4);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = prep_smem_bytes<HD>();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, slotkv_prefill_prep_kernel<HD>, p);
    if (e != cudaSuccess) return static_cast<int>(e);
    slotkv_prefill_tc_kernel<HD, G><<<ctas, C::THREADS, C::SMEM, stream>>>(tmK, tmV, p);
    return static_cast<int>(cudaGetLastError());
}

template <int HD>
int launch_prefill_hd(int G, const PrefillParams& p, const CUtensorMap& tmK,
                      const CUtensorMap& tmV, unsigned ctas, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_prefill_one<HD, 1>(p, tmK, tmV, ctas, stream);
        case 2: return launch_prefill_one<HD, 2>(p, tmK, tmV, ctas, stream);
        case 3: return launch_prefill_one<HD, 3>(p, tmK, tmV, ctas, stream);
        case 4: return launch_prefill_one<HD, 4>(p, tmK, tmV, ctas, stream);
        case 5: return launch_prefill_one<HD, 5>(p, tmK, tmV, ctas, stream);
        case 6: return launch_prefill_one<HD, 6>(p, tmK, tmV, ctas, stream);
        case 7: return launch_prefill_one<HD, 7>(p, tmK, tmV, ctas, stream);
        case 8: return launch_prefill_one<HD, 8>(p, tmK, tmV, ctas, stream);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace slotkv

/*
 * slotkv.h -- C ABI of libslotkv: batched multi-sequence decode attention over
 * slot-based KV caches, for NVIDIA GB300 (sm_103a).
 *
 * Source of the semantics: the zinc engine's API pages,
 *   "Forward Cuda Gemma" -- allocSlotKv, slotKvOffsetBytes, slotKvSmoke and
 *     decodeBatch (per-row Q/K norm, RoPE, KV write, causal softmax over the
 *     row's own slot history, and the fused batched-seq attention kernel
 *     named there as the next step);
 *   "Forward Cuda" -- slot state allocation, the slot KV byte offset, the
 *     upload of inv_freq and attention sinks at init, and the note that
 *     attention slot KV needs no reset between occupants.
 *
 * Conventions for every call:
 *   - All tensors are f32, row-major and contiguous.  positions and slots are
 *     u32.  Notation: hd = head_dim, kv_dim = n_kv_head * hd,
 *     G = n_head / n_kv_head (query heads per kv head).
 *   - "device" pointers must be CUDA device memory on the handle's device;
 *     "host" pointers are ordinary (preferably pinned) host memory.
 *   - The caller owns every buffer it passes.  The library owns only what
 *     slot_kv_alloc allocates (the KV buffers when none were adopted, the
 *     split-K workspace and small staging buffers).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns without synchronising, unless stated otherwise.
 *   - Calls that use one handle must be ordered on the GPU (same stream, or
 *     synchronised): they share the handle's workspace.
 *   - A handle belongs to the device that was current at slot_kv_alloc; calls
 *     that enqueue work or synchronise on it need that device current
 *     (SLOTKV_ERR_STATE otherwise).  slot_kv_free switches to it by itself.
 *   - Every call returns SLOTKV_OK (0) or an SLOTKV_ERR_* code and never
 *     aborts the process; slot_kv_last_error() gives a message for the
 *     calling thread's last failure.
 */
#ifndef SLOTKV_H
#define SLOTKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct slotkv_s* slotkv_t;
typedef struct slotkv_host_call_s* slotkv_host_call_t;
typedef void* slotkv_stream_t; /* a cudaStream_t */

enum slotkv_status {
    SLOTKV_OK = 0,
    SLOTKV_ERR_ARG = 1,         /* bad pointer, size or geometry */
    SLOTKV_ERR_CUDA = 2,        /* a CUDA runtime or driver call failed */
    SLOTKV_ERR_UNSUPPORTED = 3, /* geometry outside the compiled kernels */
    SLOTKV_ERR_STATE = 4        /* handle not allocated / already freed */
};

/* The most parts prefill_batch_attn_host cuts a call into. */
#define SLOTKV_PREFILL_HOST_MAX_PARTS 8u

/* Sticky device-side flags, read and cleared by slot_kv_get_status. */
enum slotkv_device_flags {
    SLOTKV_DEV_RANGE = 1u,  /* some row had slots[b] >= n_slots or
                               positions[b] >= slot_ctx: that row was skipped,
                               its out rows and the KV were left untouched */
    SLOTKV_DEV_TIMEOUT = 2u /* a pipeline wait ran out its limit; that call's
                               results are not valid */
};

/*
 * slot_kv_alloc -- allocate (or adopt) one attention layer's slot KV and the
 * decode workspace.  "Forward Cuda Gemma", allocSlotKv; "Forward Cuda", slot
 * state allocation.
 *
 *   *handle    in/out.  Must be NULL or a live handle on entry; a live handle
 *              is freed first, so re-calling is allowed (the pages' allocSlotKv
 *              frees any prior slot KV first).  Receives the new handle.
 *   n_slots    number of concurrent sequences (slots), >= 1.
 *   slot_ctx   positions per slot, >= 1; n_slots * slot_ctx < 2^31 - 256.
 *   n_kv_head  kv heads per position, 1..256.
 *   head_dim   64, 128 or 256.
 *   k_buf, v_buf
 *              NULL, NULL: the library allocates both buffers (zero-filled)
 *              and frees them in slot_kv_free.  Otherwise both must be device
 *              buffers of n_slots*slot_ctx*kv_dim f32, 16-byte aligned; they are
 *              adopted (used in place, never freed by the library).
 *              Layout of each: [n_slots][slot_ctx][n_kv_head][head_dim].
 *   max_rows   the largest B a decode call will pass, 1..65535.
 *   max_n_head the largest n_head a decode call will pass; G = n_head /
 *              n_kv_head must be 1..8.
 *
 * Errors: SLOTKV_ERR_ARG for a bad size or a half-given buffer pair,
 * SLOTKV_ERR_CUDA if an allocation or the TMA descriptor set-up fails (nothing
 * is leaked and *handle is set to NULL).
 */
int slot_kv_alloc(slotkv_t* handle, uint32_t n_slots, uint32_t slot_ctx,
                  uint32_t n_kv_head, uint32_t head_dim, float* k_buf, float* v_buf,
                  uint32_t max_rows, uint32_t max_n_head);

/* slot_kv_free -- release what slot_kv_alloc allocated (not adopted
 * buffers).  NULL is a no-op.  Synchronises the device. */
int slot_kv_free(slotkv_t handle);

/*
 * slot_kv_offset_bytes -- byte offset of (slot, pos) in the K (and V) buffer:
 * (slot * slot_ctx + pos) * kv_dim * sizeof(float).  "Forward Cuda Gemma",
 * slotKvOffsetBytes; "Forward Cuda", slot KV offset.  The kernels index the
 * buffers exactly this way.  Returns SIZE_MAX for a NULL handle,
 * slot >= n_slots or pos >= slot_ctx.  Host only; no device work.
 */
size_t slot_kv_offset_bytes(slotkv_t handle, uint32_t slot, uint32_t pos);

/*
 * slot_kv_reset -- zero every position of one slot's K and V (asynchronous,
 * on `stream`).  The pages note that attention slot KV needs no reset when a
 * slot is reused ("Forward Cuda", slot state reset on admit): a step reads
 * only positions 0..pos of its own slot, which the sequence wrote itself.
 * This call exists for hygiene and tests; no result depends on it.
 * SLOTKV_ERR_ARG if slot >= n_slots.
 */
int slot_kv_reset(slotkv_t handle, uint32_t slot, slotkv_stream_t stream);

/* slot_kv_k_ptr / slot_kv_v_ptr -- device address of the K / V buffer. */
int slot_kv_k_ptr(slotkv_t handle, float** k);
int slot_kv_v_ptr(slotkv_t handle, float** v);

/* slot_kv_geometry -- the handle's sizes (any output pointer may be NULL). */
int slot_kv_geometry(slotkv_t handle, uint32_t* n_slots, uint32_t* slot_ctx,
                     uint32_t* n_kv_head, uint32_t* head_dim, uint32_t* max_rows,
                     uint32_t* max_n_head);

/*
 * decode_batch_attn -- one batched decode attention step for B independent
 * rows.  "Forward Cuda Gemma", decodeBatch (the attention inner part, fused
 * across rows as the batched-seq attention kernel).  For each row b, with
 * p = positions[b], s = slots[b], and each kv head g:
 *   1. q' = RoPE_p(RMSnorm(q[b][h]) * q_norm_w) for the query heads h of g,
 *      k' = RoPE_p(RMSnorm(k_new[b][g]) * k_norm_w); RMSnorm(x) =
 *      x / sqrt(mean(x^2) + eps); RoPE_p rotates the pairs (i, i + hd/2) by
 *      the f32 angle fl32((float)p * inv_freq[i]).
 *   2. K[s][p][g] = k', V[s][p][g] = v_new[b][g] (raw), at the byte offset
 *      slot_kv_offset_bytes(s, p).
 *   3. out[b][h] = sum_{t=0..p} w_t V[s][t][g] with w = softmax over
 *      scale * <q', K[s][t][g]> for t = 0..p, where a non-NULL sinks[h] adds
 *      one logit to the normaliser (it joins the max and the denominator,
 *      is not scaled, and carries no value).  Query head h uses kv head
 *      h / G.  Positions after p in the slot are never read.
 *
 *   handle      from slot_kv_alloc.
 *   B           rows, 0 <= B <= max_rows (B = 0 does nothing).
 *   n_head      query heads, a multiple of n_kv_head, <= max_n_head.
 *   q           device, [B][n_head][hd].
 *   k_new       device, [B][n_kv_head][hd].
 *   v_new       device, [B][n_kv_head][hd].
 *   positions   device, u32[B]; the slot must already hold 0..p-1.
 *   slots       device, u32[B]; pairwise distinct within one call
 *               (duplicates give an undefined result, never a fault).
 *   q_norm_w    device, [hd].        k_norm_w  device, [hd].
 *   inv_freq    device, [hd/2].      sinks     device [n_head], or NULL.
 *   out         device, [B][n_head][hd]; written for every in-range row.
 *   eps         RMS-norm epsilon.    scale     softmax scale (e.g. 1/sqrt(hd)).
 * q, k_new, v_new and out must be 16-byte aligned (the kernel stages them with
 * bulk copies and writes out in 16-byte stores), the other arrays 4-byte
 * aligned.
 *
 * Out-of-range rows (slots[b] >= n_slots or positions[b] >= slot_ctx, the
 * decodeBatch precondition) are skipped on the device and raise
 * SLOTKV_DEV_RANGE.  Host-side errors: SLOTKV_ERR_ARG (NULL or misaligned
 * pointer, B or n_head too large, n_head not a multiple of n_kv_head),
 * SLOTKV_ERR_UNSUPPORTED (G outside 1..8), SLOTKV_ERR_CUDA (launch failure,
 * including a GPU on which two of the persistent decode CTAs do not fit on
 * one SM).
 *
 * Which kernels run (slot_kv_call_shape reports it): under the default split
 * policy, a call of at most two CTAs' worth of (row, kv head) pairs per SM
 * over slots of at most 8 * 4096 / hd keys runs one CTA per pair; any other
 * call runs a plan kernel and the persistent decode kernel (the decode kernel
 * alone when every row fits in one chunk and the pairs fit in its CTAs).
 * Stream order holds as for any kernel, with one addition: the persistent
 * decode kernel lets a programmatic dependent launch (a kernel launched with
 * cudaLaunchAttributeProgrammaticStreamSerialization right after the call)
 * once every CTA has run out of work, before the kernel has finished; such a
 * dependent must wait for it (cudaGridDependencySynchronize) before reading
 * out, K or V.  The next call's plan kernel is such a dependent, and waits.
 */
int decode_batch_attn(slotkv_t handle, uint32_t B, uint32_t n_head, const float* q,
                      const float* k_new, const float* v_new, const uint32_t* positions,
                      const uint32_t* slots, const float* q_norm_w,
                      const float* k_norm_w, const float* inv_freq, const float* sinks,
                      float* out, float eps, float scale, slotkv_stream_t stream);

/*
 * prefill_batch_attn -- batched causal prefill into slots: n_tok new tokens,
 * each with its own slot and position, written and attended in one call.
 * "Forward Cuda Gemma", prefillBatched (batched causal attention and
 * batched norm/RoPE/KV write, equal to running the tokens one decode step
 * at a time) and "Forward Cuda", batched prefill into the given slot.
 * Tokens may share a slot; within a slot their positions must be distinct,
 * and the slot must already hold every position below its tokens' that is
 * not itself a token of this call.  The result for every token equals
 * decode_batch_attn run on the tokens one at a time in increasing position
 * (up to f32 rounding): first every token's k' and v go into its slot row,
 * then each token attends keys 0..pos of its slot, new rows included.
 * Arguments as decode_batch_attn with B = n_tok (<= max_rows); q, k_new,
 * v_new, positions, slots and out are indexed by token.  The options of
 * slot_kv_set_options apply.  Errors as decode_batch_attn.
 *
 * Head dims 64 and 128 run on the tensor cores: consecutive tokens of one
 * slot (a run; give each sequence's tokens one after another) are cut into
 * tiles of 128 / G tokens, and each tile reads its slot's keys once for all
 * its rows.  Products are formed from three TF32 tensor-core products (high
 * and low parts of both operands), which keeps them within f32 rounding of
 * the f32 result.  Tokens in any order stay correct; interleaved slots only
 * make the tiles smaller.  This path keeps a workspace in the handle (the
 * rotated queries and the tile list), grown to the largest n_tok * n_head
 * seen: a call larger than any before allocates (and synchronises the
 * device) first.  Head dim 256 runs the decode kernel once per token.
 */
int prefill_batch_attn(slotkv_t handle, uint32_t n_tok, uint32_t n_head, const float* q,
                       const float* k_new, const float* v_new, const uint32_t* positions,
                       const uint32_t* slots, const float* q_norm_w, const float* k_norm_w,
                       const float* inv_freq, const float* sinks, float* out, float eps,
                       float scale, slotkv_stream_t stream);

/*
 * prefill_batch_attn_host -- prefill_batch_attn for callers whose per-call
 * inputs and output live in host memory ("Forward Cuda Gemma",
 * prefillBatched, with the prompt's tensors on the host).  q, k_new, v_new,
 * positions, slots and out are HOST pointers; q_norm_w, k_norm_w, inv_freq
 * and sinks stay device pointers.  The inputs move to handle-owned device
 * staging with cudaMemcpyAsync (the copy engines: a prefill's tens of MB move
 * faster that way than through a gather kernel), the prefill runs (the same
 * kernels as prefill_batch_attn, the same bits) into device staging, out
 * moves back the same way, and `stream` is synchronised before the call
 * returns (page-locked buffers make the copies asynchronous DMA).  n_tok <=
 * max_rows.  Errors as prefill_batch_attn, plus SLOTKV_ERR_CUDA for a failed
 * copy.
 *
 * At head dims 64 and 128 a call of 1024 tokens or more is cut into parts
 * whose tokens share no slot (slot_kv_prefill_host_parts says where): each
 * part is a prefill of its own, with the same tiles and so the same bits,
 * its own rows of the handle's workspace and its own plan counters.  Inputs
 * go in on a copy stream owned by the handle, the parts' kernels run on
 * `stream` and a second stream of the handle by turns (a part's kernels
 * start on the SMs the previous part frees), and each part's output comes
 * back on a second copy stream while later parts run.  A call that cannot
 * be cut that way runs as one part.
 */
int prefill_batch_attn_host(slotkv_t handle, uint32_t n_tok, uint32_t n_head, const float* q,
                            const float* k_new, const float* v_new, const uint32_t* positions,
                            const uint32_t* slots, const float* q_norm_w,
                            const float* k_norm_w, const float* inv_freq, const float* sinks,
                            float* out, float eps, float scale, slotkv_stream_t stream);

/*
 * slot_kv_prefill_host_parts -- where prefill_batch_attn_host cuts a call of
 * n_tok tokens with these slots (HOST pointer, by token) at head dims 64 and
 * 128.  A cut before token m is allowed when no slot has tokens on both
 * sides; the call gets one part per 512 tokens, at most
 * SLOTKV_PREFILL_HOST_MAX_PARTS, none under 256 tokens, each cut the allowed
 * one nearest its target (fewer parts when too few cuts are allowed).  The
 * targets n_tok (2j - 1) / (2 (parts - 1)), j = 1 .. parts - 1, make the
 * first and the last part half the size of the others, since the first
 * part's input copies and the last part's output copies overlap nothing.
 * Writes the part boundaries cuts[0] = 0 < cuts[1] < ... < cuts[*n_parts] =
 * n_tok and the count to *n_parts (an empty call: one part, cuts {0, 0}).
 * cuts_len is the number of entries cuts holds, at least
 * SLOTKV_PREFILL_HOST_MAX_PARTS + 1.  Host only: no handle, no device work.
 * Returns SLOTKV_ERR_ARG for a null pointer or a cuts_len below that.
 */
int slot_kv_prefill_host_parts(uint32_t n_tok, const uint32_t* slots, uint32_t* cuts,
                               uint32_t cuts_len, uint32_t* n_parts);

/*
 * decode_batch_attn_paged -- the decode step over a paged KV pool: instead of
 * one contiguous slot per sequence, each row's keys live in fixed-size blocks
 * named by its block table (the paged cache with per-sequence block tables of
 * the Qwen3SsmLayer page, decode_multi_seq; the same step as "Forward Cuda
 * Gemma", decodeBatch, with only the addressing changed).
 *
 * The handle's buffers are the pool: allocate it with n_slots = the number of
 * blocks and slot_ctx = the block size, so K and V are
 * f32[n_blocks][block_size][n_kv_head][head_dim].  The block size must be a
 * multiple of 4096/head_dim (64 for head_dim 64, 32 for 128, 16 for 256), the
 * keys of one pipeline tile, else SLOTKV_ERR_UNSUPPORTED.
 *
 *   block_tables  device u32[B][bt_stride]: row b's key t (0 <= t <= pos) is at
 *                 block block_tables[b*bt_stride + t/block_size], offset
 *                 t % block_size.  Entries past a row's last used block are
 *                 never read.  Rows may share blocks they only read, but the
 *                 block holding a row's key pos must belong to that row alone
 *                 in this call, and appear once in its table.
 *   bt_stride     entries per row of block_tables (>= 1): the longest context
 *                 is bt_stride*block_size keys.
 * The other arguments are those of decode_batch_attn (slots is replaced by
 * the tables).  The step writes key pos's K' and V into its block, then
 * attends keys 0..pos through the table.  Per row the result equals
 * decode_batch_attn on a slot holding the same keys, bit for bit.  A row whose
 * pos >= bt_stride*block_size, or whose used entries (blocks 0..pos/block_size)
 * hold an id >= n_blocks, is skipped: nothing of it is written and
 * SLOTKV_DEV_RANGE is raised.  The options of slot_kv_set_options apply.
 * Errors as decode_batch_attn.
 */
int decode_batch_attn_paged(slotkv_t handle, uint32_t B, uint32_t n_head, const float* q,
                            const float* k_new, const float* v_new,
                            const uint32_t* positions, const uint32_t* block_tables,
                            uint32_t bt_stride, const float* q_norm_w,
                            const float* k_norm_w, const float* inv_freq,
                            const float* sinks, float* out, float eps, float scale,
                            slotkv_stream_t stream);

/*
 * decode_batch_attn_host -- decode_batch_attn for callers whose per-step
 * inputs and output live in host memory.  q, k_new, v_new, positions, slots
 * and out are HOST pointers with the layouts above; q_norm_w, k_norm_w,
 * inv_freq and sinks stay device pointers (resident parameters).  The call
 * moves the inputs into handle-owned device staging buffers on `stream`,
 * runs the step, moves out back and synchronises `stream` before returning,
 * so out is ready on return.  When all six host buffers are page-locked
 * (pinned, hence mapped into the device's address space) one copy kernel
 * gathers the inputs over the host link and the step writes out straight into
 * host memory (through a second copy kernel if out is not 16-byte aligned);
 * otherwise each buffer is copied with cudaMemcpyAsync.  Host buffers need only 4-byte
 * alignment.
 * Errors as decode_batch_attn, plus SLOTKV_ERR_CUDA for a failed copy.
 */
int decode_batch_attn_host(slotkv_t handle, uint32_t B, uint32_t n_head, const float* q,
                           const float* k_new, const float* v_new,
                           const uint32_t* positions, const uint32_t* slots,
                           const float* q_norm_w, const float* k_norm_w,
                           const float* inv_freq, const float* sinks, float* out,
                           float eps, float scale, slotkv_stream_t stream);

/*
 * decode_batch_attn_paged_host -- decode_batch_attn_paged for callers whose
 * per-step inputs and output live in host memory (the paged counterpart of
 * decode_batch_attn_host; the Qwen3SsmLayer page, decode_multi_seq over a
 * paged cache).  q, k_new, v_new, positions, block_tables (u32[B][bt_stride])
 * and out are HOST pointers; q_norm_w, k_norm_w, inv_freq and sinks stay
 * device pointers.  The inputs move to handle-owned device staging (one
 * gather kernel when all six host buffers are pinned, else cudaMemcpyAsync),
 * the step runs, out moves back and `stream` is synchronised before the call
 * returns.  The tables' staging grows to the largest B * bt_stride seen: a
 * call with a larger table than any before allocates (and synchronises the
 * device) first.  Errors as decode_batch_attn_paged, plus SLOTKV_ERR_CUDA
 * for a failed copy or staging allocation.
 */
int decode_batch_attn_paged_host(slotkv_t handle, uint32_t B, uint32_t n_head, const float* q,
                                 const float* k_new, const float* v_new,
                                 const uint32_t* positions, const uint32_t* block_tables,
                                 uint32_t bt_stride, const float* q_norm_w,
                                 const float* k_norm_w, const float* inv_freq,
                                 const float* sinks, float* out, float eps, float scale,
                                 slotkv_stream_t stream);

/*
 * slot_kv_host_call_create / _run / _enqueue / _free -- a prepared host step: the
 * arguments of decode_batch_attn_host (bt_stride = 0, idx = slots) or of
 * decode_batch_attn_paged_host (bt_stride >= 1, idx = block_tables), checked
 * once and with the device aliases of the page-locked host buffers resolved
 * once, for a serving loop that refills the same host buffers every step
 * ("Forward Cuda Gemma", decodeBatch, with the per-step inputs in host
 * memory; "Forward Cuda", the decode graph keyed by its buffers).
 *   create   checks the arguments as the host entry does (errors as there;
 *            B >= 1), grows the block-table staging once in paged mode, and
 *            returns *call (owned by the caller).  Only the pointers are
 *            kept: the buffers must stay allocated, at the same addresses,
 *            until the call is freed.
 *   run      one step on `stream` exactly as the host entry with these
 *            arguments would run it (the same kernels, the same bits): it
 *            reads the host buffers' current contents, writes out and K/V,
 *            and synchronises `stream` before returning.  SLOTKV_ERR_STATE
 *            once the handle has been freed (slot_kv_free detaches its
 *            calls), or when another device is current.
 *   enqueue  the same step (the same kernels, the same bits) without the
 *            final synchronisation.  While work is in flight on `stream`, the
 *            inputs are copied by the copy engines into device staging owned
 *            by the call (allocated by its first such enqueue) on a copy
 *            stream of the handle, so they overlap that work, and the step
 *            runs on `stream` after them; on an idle stream the step takes
 *            run's lower-latency path (one gather kernel).  The call returns
 *            without waiting.  out and K/V are complete, and the host
 *            input buffers may be refilled, only once `stream` has been
 *            synchronised (cudaStreamSynchronize, or an event recorded after
 *            the call); a caller running several steps synchronises once,
 *            when it needs the results.  Enqueuing the same call again
 *            orders its copies after its previous step.  With pageable (not
 *            page-locked) buffers the copies themselves may block.
 *   free     releases the call and its staging, after its last enqueued
 *            step has run (NULL is a no-op); a handle may be freed before or
 *            after its calls.
 */
int slot_kv_host_call_create(slotkv_t handle, slotkv_host_call_t* call, uint32_t B,
                             uint32_t n_head, const float* q, const float* k_new,
                             const float* v_new, const uint32_t* positions,
                             const uint32_t* idx, uint32_t bt_stride, const float* q_norm_w,
                             const float* k_norm_w, const float* inv_freq, const float* sinks,
                             float* out, float eps, float scale);
int slot_kv_host_call_run(slotkv_host_call_t call, slotkv_stream_t stream);
int slot_kv_host_call_enqueue(slotkv_host_call_t call, slotkv_stream_t stream);
int slot_kv_host_call_free(slotkv_host_call_t call);

/*
 * decode_batch_attn_noalloc -- the same decode step as decode_batch_attn for
 * callers that cannot allocate device memory.  The pages have no counterpart
 * to this entry point.
 *
 * Who needs it: code that runs under a host framework which owns every byte
 * of device memory (its own pool or a fixed budget), and code paths that
 * cannot afford the device-wide synchronisation cudaMalloc and cudaFree may
 * cause.  decode_batch_attn needs a handle, and slot_kv_alloc allocates.
 * This call needs no handle and allocates nothing, directly or through any
 * library.
 *
 * Scratch: the split-K partials, the merge counters and a status word live in
 * one fixed device array of SLOTKV_NOALLOC_SCRATCH_BYTES inside the library.
 * Every GPU that loads the library holds it until the process exits.  A batch
 * needs 256 + align256(4*B*n_kv_head) + align256(256*B*n_kv_head) +
 * align256(128*B*n_head) + 64*B*n_head*head_dim bytes of it (work list and
 * partials for up to 16 splits per row).  A batch that needs more is rejected
 * with SLOTKV_ERR_ARG and a message naming both sizes; use decode_batch_attn
 * with a handle then.
 * All calls in the process share the array, which keeps the last call's
 * contents.  Each call clears the status word and the counters first, on
 * `stream`.  Calls that overlap on the GPU (different streams, or different
 * host threads without ordering) race on it: order them.
 *
 * Set-up: the first call on each device looks up the array's device address
 * with that device current and caches it, keyed on the current CUDA context
 * (a new context -- after cudaDeviceReset, or a driver-API context made
 * current -- looks it up again on its first call).  Make that first call
 * before any stream capture begins.
 *
 *   K, V        device slot buffers, [n_slots][slot_ctx][n_kv_head][head_dim]
 *               f32, 16-byte aligned (the caller owns them).
 *   n_slots, slot_ctx, n_kv_head, head_dim
 *               their geometry (head_dim 64, 128 or 256; n_slots*slot_ctx
 *               < 2^31 - 256).
 *   B, n_head, q ... out, eps, scale, stream
 *               as decode_batch_attn (B <= 65535; G = n_head/n_kv_head 1..8).
 *   dev_flags   device u32 that receives the SLOTKV_DEV_* flags raised by
 *               this call (OR-ed in; the caller clears it), or NULL to
 *               discard them.  With NULL an out-of-range row (slots[b] >=
 *               n_slots or positions[b] >= slot_ctx) is skipped silently:
 *               its out rows keep their previous contents and nothing
 *               signals it, so pass dev_flags wherever the inputs are not
 *               validated already.
 *
 * Returns SLOTKV_OK, SLOTKV_ERR_ARG, SLOTKV_ERR_UNSUPPORTED or
 * SLOTKV_ERR_CUDA; slot_kv_last_error() says why.  Results match
 * decode_batch_attn's within f32 rounding: rows with more than 16 chunks of
 * the default size are split into 16 larger chunks instead.
 */
#define SLOTKV_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int decode_batch_attn_noalloc(float* K, float* V, uint32_t n_slots, uint32_t slot_ctx,
                              uint32_t n_kv_head, uint32_t head_dim, uint32_t B,
                              uint32_t n_head, const float* q, const float* k_new,
                              const float* v_new, const uint32_t* positions,
                              const uint32_t* slots, const float* q_norm_w,
                              const float* k_norm_w, const float* inv_freq,
                              const float* sinks, float* out, uint32_t* dev_flags,
                              float eps, float scale, slotkv_stream_t stream);

/*
 * slot_kv_advance_positions -- positions[b] += delta for b < B, on the device
 * (asynchronous, on `stream`).  "Forward Cuda Gemma", decodeBatch: after a
 * step the caller advances each sequence's position and feeds it back; doing
 * it on the device keeps a multi-step decode free of host work, so a run of
 * steps (decode_batch_attn, slot_kv_advance_positions, ...) can be captured
 * into one CUDA graph and replayed.  Make one decode_batch_attn call on the
 * handle before capturing (it sets kernel attributes on first use).
 * positions: device u32[B].  SLOTKV_ERR_ARG for a NULL pointer.
 */
int slot_kv_advance_positions(uint32_t* positions, uint32_t B, uint32_t delta,
                              slotkv_stream_t stream);

/*
 * Slot-ownership sharding over several GPUs.  The rows of a decode step are
 * independent sequences in disjoint slots ("Forward Cuda Gemma", decodeBatch:
 * B sequences each advance by one token over their own slot; allocSlotKv:
 * one slot per concurrent sequence), so the step shards by slot ownership:
 * each rank (one GPU) holds the KV of a contiguous range of the global slots
 * in its own handle and runs the rows whose slots it owns.  No rank reads
 * another's memory and the step needs no collective; only a consumer that
 * wants every row's output on one device gathers out afterwards.
 *
 * slot_kv_shard_range -- the global slots rank `rank` of n_ranks owns:
 * [*first, *first + *count) with first = floor(rank * n_slots / n_ranks)
 * (balanced contiguous ranges; count >= 1).  Global slot s is local slot
 * s - first of its owner, which allocates a handle of `count` slots.
 * SLOTKV_ERR_ARG unless 1 <= n_ranks <= n_slots and rank < n_ranks.  Host
 * only; first and count may be NULL.
 */
int slot_kv_shard_range(uint32_t n_ranks, uint32_t n_slots, uint32_t rank, uint32_t* first,
                        uint32_t* count);

/*
 * slot_kv_shard_route -- route one step's rows to the ranks that own their
 * slots.  slots: HOST u32[B], global slot ids.  Outputs (host, caller-owned):
 *   order[B]            the row indices grouped by owning rank, in
 *                       increasing order within a rank (a permutation of
 *                       0..B-1);
 *   offsets[n_ranks+1]  rank r's rows are order[offsets[r] .. offsets[r+1]);
 *   local_slots[B]      local_slots[i] = the owner's local slot of row
 *                       order[i].
 * A row whose slot is >= n_slots goes to the last rank with a local slot
 * past that rank's range, so its decode step skips it and raises
 * SLOTKV_DEV_RANGE, as for an out-of-range slot on one GPU.  Host only.
 * SLOTKV_ERR_ARG unless 1 <= n_ranks <= n_slots, or for a NULL pointer.
 */
int slot_kv_shard_route(uint32_t n_ranks, uint32_t n_slots, uint32_t B, const uint32_t* slots,
                        uint32_t* order, uint32_t* offsets, uint32_t* local_slots);

/*
 * slot_kv_get_status -- synchronise `stream`, return the sticky device flags
 * (SLOTKV_DEV_*) raised since the last call in *flags, and clear them.  After
 * SLOTKV_DEV_TIMEOUT the workspace is also cleared so later calls are valid.
 */
int slot_kv_get_status(slotkv_t handle, slotkv_stream_t stream, uint32_t* flags);

/*
 * slot_kv_set_split -- fix the split-K policy.  A row with n = p + 1 keys is
 * cut into nsplit = ceil(n / C) chunks of C = max(min_chunk_keys, ceil(n /
 * max_splits) rounded up to the tile) keys; chunks run on separate CTAs and
 * are merged by the last one to finish.  After this call C depends only on n
 * and the geometry, never on B or on the other rows, so a row's result is the
 * same bits in any batch.
 * min_chunk_keys must be a positive multiple of the tile (4096 / head_dim
 * keys); max_splits 1..256.  Reallocates the workspace (synchronises).
 * Until it is called, a handle uses the default policy: max_splits = 64 and
 * min_chunk_keys chosen per call from the batch's shape (B, n_kv_head, the
 * context capacity, the SM count), between 512 KiB and 2 MiB of K+V per kv
 * head, so that large batches run fewer, larger chunks.  Results are then
 * deterministic for a given batch size but may differ in the last bits
 * between batch sizes (within f32 rounding).
 */
int slot_kv_set_split(slotkv_t handle, uint32_t min_chunk_keys, uint32_t max_splits);

/*
 * slot_kv_call_shape -- how a call of B rows on this handle runs, without
 * running it (host only): *chunk_keys the split chunk C of the current policy,
 * *ctas the persistent CTAs of the decode kernel, *kernels the kernels the
 * call launches on its stream (KV write for prefill, work-list plan unless
 * every item is a CTA's first item, decode).  For a tensor-core prefill
 * (head dims 64 and 128): the keys per pipeline stage, one CTA per SM, and
 * three kernels (prep, plan, attention).  bt_stride: 0 for slot calls,
 * the table width for decode_batch_attn_paged; prefill: nonzero for
 * prefill_batch_attn.  Any output pointer may be NULL.  SLOTKV_ERR_ARG for
 * B = 0 or B > max_rows.
 */
int slot_kv_call_shape(slotkv_t handle, uint32_t B, uint32_t bt_stride, uint32_t prefill,
                       uint32_t* chunk_keys, uint32_t* ctas, uint32_t* kernels);

/*
 * slot_kv_set_options -- norm options of the per-head "V/Q/K norm" of the
 * Gemma path ("Forward Cuda Gemma", decodeBatch), for later decode calls on
 * this handle.  flags is a bitwise OR of:
 *   SLOTKV_OPT_VNORM          normalise v_new with a weightless RMS norm
 *                             (x / sqrt(mean(x^2) + eps)) before it is cached
 *                             and attended;
 *   SLOTKV_OPT_NORM_PLUS_ONE  apply the Q and K norm weights as (1 + w);
 *   SLOTKV_OPT_TEST_STALL     for testing the failure path only: the first
 *                             work item of every CTA is never marked ready,
 *                             so the consumers' bounded wait expires (after
 *                             about a second), every CTA abandons its work
 *                             and the call ends with SLOTKV_DEV_TIMEOUT set,
 *                             having written nothing.  The context stays
 *                             usable; clear the flags with
 *                             slot_kv_get_status and the option with
 *                             slot_kv_set_options(handle, 0).
 * 0 (the default) is the plain form of decode_batch_attn.  SLOTKV_ERR_ARG for
 * unknown bits.  Host only; takes effect at the next call.
 */
#define SLOTKV_OPT_VNORM 1u
#define SLOTKV_OPT_NORM_PLUS_ONE 2u
#define SLOTKV_OPT_TEST_STALL 0x80000000u
int slot_kv_set_options(slotkv_t handle, uint32_t flags);

/* slot_kv_last_error -- message for the calling thread's last failed call
 * ("" if none).  The pointer stays valid until that thread's next call. */
const char* slot_kv_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* SLOTKV_H */

"""Batched causal prefill ("Forward Cuda Gemma", prefillBatched; "Forward
Cuda", batched prefill into the given slot) against the oracle: the result
must equal running the prompt tokens one decode step at a time in position
order.  Several sequences share one call, with different history lengths
and prompt lengths, their tokens interleaved in the batch."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_harness import assert_close, to_dev
from sequence_slot_kv_gb300 import SlotKV

pytestmark = pytest.mark.gpu


def _setup(hd, G, idx, seqs, contiguous=False):
    """seqs: [(slot, history_len, prompt_len)].  Returns the geometry and the
    token arrays: interleaved round-robin, or one sequence after another."""
    n_kv = 2
    n_tok = sum(t for _, _, t in seqs)
    ctx = max(h + t for _, h, t in seqs) + 5
    n_slots = max(s for s, _, _ in seqs) + 2
    w = synth.Workload(f"prefill_hd{hd}", 700 + idx, B=n_tok, n_slots=n_slots, slot_ctx=ctx,
                       n_head=G * n_kv, n_kv_head=n_kv, head_dim=hd, theta=1e4, sinks=True,
                       pos_rule="fixed", fixed_positions=tuple([0] * n_tok), slot_rule="perm")
    order = []
    if contiguous:
        for i, (_, _, t) in enumerate(seqs):
            order.extend((i, j) for j in range(t))
    else:
        # interleave the sequences' tokens round-robin
        cursor = [0] * len(seqs)
        while len(order) < n_tok:
            for i, (_, _, t) in enumerate(seqs):
                if cursor[i] < t:
                    order.append((i, cursor[i]))
                    cursor[i] += 1
    slots = np.array([seqs[i][0] for i, _ in order], dtype=np.uint32)
    pos = np.array([seqs[i][1] + j for i, j in order], dtype=np.uint32)
    return w, slots, pos


def _oracle(w, slots, pos, flags=0):
    """The tokens as single decode steps in position order, on host copies of
    the used slots."""
    o = oracle.default()
    K = synth.normal(w.kv_elems(), w.seed, synth.S_HIST_K).reshape(
        w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    V = synth.normal(w.kv_elems(), w.seed, synth.S_HIST_V).reshape(K.shape)
    q, kn, vn = w.q(), w.k_new(), w.v_new()
    out = np.empty((w.B, w.n_head, w.head_dim), dtype=np.float32)
    for i in np.lexsort((pos, slots)):
        r, _, _ = o.decode_batch(K, V, q[i:i + 1], kn[i:i + 1], vn[i:i + 1], pos[i:i + 1],
                                 slots[i:i + 1], w.q_norm_w(), w.k_norm_w(), w.inv_freq(),
                                 w.sink_logits(), w.eps, w.scale, flags=flags)
        out[i] = r[0]
    return out, K, V


CASES = [(64, 8), (128, 4), (128, 5), (256, 2)]


@pytest.mark.parametrize("hd,G", CASES, ids=[f"hd{h}_g{g}" for h, g in CASES])
def test_prefill_equals_token_by_token_decode(hd, G):
    T = 4096 // hd
    seqs = [(2, 0, 3 * T + 5), (0, 37, 1), (3, 5 * T + 1, 2 * T - 3)]
    w, slots, pos = _setup(hd, G, CASES.index((hd, G)), seqs)
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    K = torch.empty(shape, device="cuda")
    V = torch.empty(shape, device="cuda")
    w.dev_fill_history(K.data_ptr(), V.data_ptr(), torch.cuda.current_stream().cuda_stream)
    kv = SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head, k_buf=K, v_buf=V)
    try:
        kv.set_split(T, 8)   # several splits per row: the cross-CTA merge runs too
        out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        kv.prefill_batch_attn(to_dev(w.q()), to_dev(w.k_new()), to_dev(w.v_new()),
                              to_dev(pos.astype(np.int32)), to_dev(slots.astype(np.int32)),
                              to_dev(w.q_norm_w()), to_dev(w.k_norm_w()), to_dev(w.inv_freq()),
                              to_dev(w.sink_logits()), out, w.eps, w.scale)
        torch.cuda.synchronize()
        assert kv.get_status() == 0
        ref, Kr, Vr = _oracle(w, slots, pos)
        assert_close(out.cpu().numpy(), ref, f"prefill out hd={hd} G={G}")
        # the slot buffers: written rows within tolerance (K) / exact (V),
        # every other byte untouched
        Kg, Vg = K.cpu().numpy(), V.cpu().numpy()
        mask = np.zeros(shape[:2], dtype=bool)
        mask[slots, pos] = True
        assert_close(Kg[mask], Kr[mask], "prefill written K")
        assert np.array_equal(Vg[mask].view(np.uint32), Vr[mask].view(np.uint32))
        assert np.array_equal(Kg[~mask].view(np.uint32), Kr[~mask].view(np.uint32))
        assert np.array_equal(Vg[~mask].view(np.uint32), Vr[~mask].view(np.uint32))
    finally:
        kv.free()


GROUPED = [(128, 4), (128, 3), (64, 2), (64, 1), (256, 1)]


@pytest.mark.parametrize("hd,G", GROUPED, ids=[f"hd{h}_g{g}" for h, g in GROUPED])
def test_prefill_contiguous_sequences(hd, G):
    """Sequences given one after another (the usual layout of a prompt
    chunk), with a one-token sequence and a position gap: every token must
    still equal one decode step at a time."""
    T = 4096 // hd
    seqs = [(1, 37, 7), (4, 5 * T + 3, 6), (0, 0, 2 * T + 1), (3, 200, 1), (5, 11, 9)]
    idx = 40 + GROUPED.index((hd, G))
    w, slots, pos = _setup(hd, G, idx, seqs, contiguous=True)
    pos = pos.copy()
    last = len(pos) - 1
    pos[last] += 3          # a gap: the last sequence's final token sits 3 positions on
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    K = torch.empty(shape, device="cuda")
    V = torch.empty(shape, device="cuda")
    w.dev_fill_history(K.data_ptr(), V.data_ptr(), torch.cuda.current_stream().cuda_stream)
    kv = SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head, k_buf=K, v_buf=V)
    try:
        out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        kv.prefill_batch_attn(to_dev(w.q()), to_dev(w.k_new()), to_dev(w.v_new()),
                              to_dev(pos.astype(np.int32)), to_dev(slots.astype(np.int32)),
                              to_dev(w.q_norm_w()), to_dev(w.k_norm_w()), to_dev(w.inv_freq()),
                              to_dev(w.sink_logits()), out, w.eps, w.scale)
        torch.cuda.synchronize()
        assert kv.get_status() == 0
        ref, Kr, Vr = _oracle(w, slots, pos)
        assert_close(out.cpu().numpy(), ref, f"contiguous prefill hd={hd} G={G}")
        Kg, Vg = K.cpu().numpy(), V.cpu().numpy()
        mask = np.zeros(shape[:2], dtype=bool)
        mask[slots, pos] = True
        assert_close(Kg[mask], Kr[mask], "prefill written K")
        assert np.array_equal(Vg[mask].view(np.uint32), Vr[mask].view(np.uint32))
        assert np.array_equal(Kg[~mask].view(np.uint32), Kr[~mask].view(np.uint32))
    finally:
        kv.free()


@pytest.mark.parametrize("flags", [1, 2, 3], ids=["vnorm", "plus_one", "both"])
def test_prefill_with_norm_options(flags):
    """Prefill with the Gemma norm forms: the KV-write kernel caches the
    weightless-normed V and the (1 + w) norms apply to q and k, as in one
    decode step at a time with the same options."""
    import sequence_slot_kv_gb300 as skv
    hd, G = 128, 4
    T = 4096 // hd
    w, slots, pos = _setup(hd, G, 60 + flags, [(2, 9, T + 3), (0, 40, 5)], contiguous=True)
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    K = torch.empty(shape, device="cuda")
    V = torch.empty(shape, device="cuda")
    w.dev_fill_history(K.data_ptr(), V.data_ptr(), torch.cuda.current_stream().cuda_stream)
    kv = SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head, k_buf=K, v_buf=V)
    try:
        kv.set_options(flags)
        assert skv.OPT_VNORM == 1 and skv.OPT_NORM_PLUS_ONE == 2
        out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        kv.prefill_batch_attn(to_dev(w.q()), to_dev(w.k_new()), to_dev(w.v_new()),
                              to_dev(pos.astype(np.int32)), to_dev(slots.astype(np.int32)),
                              to_dev(w.q_norm_w()), to_dev(w.k_norm_w()), to_dev(w.inv_freq()),
                              to_dev(w.sink_logits()), out, w.eps, w.scale)
        torch.cuda.synchronize()
        assert kv.get_status() == 0
        ref, Kr, Vr = _oracle(w, slots, pos, flags=flags)
        assert_close(out.cpu().numpy(), ref, f"prefill options {flags}")
        Kg, Vg = K.cpu().numpy(), V.cpu().numpy()
        mask = np.zeros(shape[:2], dtype=bool)
        mask[slots, pos] = True
        assert_close(Kg[mask], Kr[mask], "prefill written K")
        assert_close(Vg[mask], Vr[mask], "prefill written V")
        assert np.array_equal(Kg[~mask].view(np.uint32), Kr[~mask].view(np.uint32))
    finally:
        kv.free()


def test_prefill_of_one_token_matches_decode():
    """A one-token prefill is a decode step: same written rows bit for bit."""
    hd, G = 128, 4
    w, slots, pos = _setup(hd, G, 9, [(1, 100, 1), (0, 0, 1), (2, 700, 1)])
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    outs = []
    bufs = []
    for mode in ("decode", "prefill"):
        K = torch.empty(shape, device="cuda")
        V = torch.empty(shape, device="cuda")
        w.dev_fill_history(K.data_ptr(), V.data_ptr(), torch.cuda.current_stream().cuda_stream)
        kv = SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head,
                    k_buf=K, v_buf=V)
        out = torch.empty((w.B, w.n_head, w.head_dim), device="cuda")
        args = (to_dev(w.q()), to_dev(w.k_new()), to_dev(w.v_new()),
                to_dev(pos.astype(np.int32)), to_dev(slots.astype(np.int32)),
                to_dev(w.q_norm_w()), to_dev(w.k_norm_w()), to_dev(w.inv_freq()),
                to_dev(w.sink_logits()), out, w.eps, w.scale)
        if mode == "decode":
            kv.decode_batch_attn(*args)
        else:
            kv.prefill_batch_attn(*args)
        torch.cuda.synchronize()
        assert kv.get_status() == 0
        outs.append(out.cpu().numpy())
        bufs.append((K.cpu(), V.cpu()))
        kv.free()
    assert_close(outs[1], outs[0], "one-token prefill vs decode")
    assert torch.equal(bufs[0][0], bufs[1][0]) and torch.equal(bufs[0][1], bufs[1][1])


HOST_CASES = [(64, 4), (128, 2), (256, 2)]


@pytest.mark.parametrize("hd,G", HOST_CASES, ids=[f"hd{h}_g{g}" for h, g in HOST_CASES])
def test_prefill_host_entry_every_head_dim(hd, G):
    """prefill_batch_attn_host with pageable host tensors, at every head
    dim (hd 256 runs the decode kernel once per token behind it): the same
    output and slot bytes as the device entry, bit for bit, and the oracle's
    token-by-token result within tolerance."""
    T = 4096 // hd
    seqs = [(2, 3, 2 * T + 7), (0, 4 * T + 1, T - 2), (1, 0, 5)]
    w, slots, pos = _setup(hd, G, 80 + HOST_CASES.index((hd, G)), seqs)
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    outs, kvs = [], []
    for host in (False, True):
        K = torch.empty(shape, device="cuda")
        V = torch.empty(shape, device="cuda")
        w.dev_fill_history(K.data_ptr(), V.data_ptr(), torch.cuda.current_stream().cuda_stream)
        kv = SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head, k_buf=K,
                    v_buf=V)
        try:
            put = (lambda a: torch.from_numpy(np.ascontiguousarray(a))) if host else to_dev
            out = put(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32))
            fn = kv.prefill_batch_attn_host if host else kv.prefill_batch_attn
            fn(put(w.q()), put(w.k_new()), put(w.v_new()), put(pos.astype(np.int32)),
               put(slots.astype(np.int32)), to_dev(w.q_norm_w()), to_dev(w.k_norm_w()),
               to_dev(w.inv_freq()), to_dev(w.sink_logits()), out, w.eps, w.scale)
            torch.cuda.synchronize()
            assert kv.get_status() == 0
            outs.append(out.cpu().numpy())
            kvs.append((K, V))
        finally:
            kv.free()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert torch.equal(kvs[0][0], kvs[1][0]) and torch.equal(kvs[0][1], kvs[1][1])
    ref, _, _ = _oracle(w, slots, pos)
    assert_close(outs[1], ref, f"host-entry prefill hd={hd} G={G}")

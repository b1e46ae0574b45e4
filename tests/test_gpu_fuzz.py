"""Seeded random configurations against the oracle.

Decode: head dims, group sizes, kv heads, batch sizes, ragged positions (some
rows out of range), default and fixed split policies, slot and paged layouts
with random block sizes, and the norm options.  Prefill: random sequences in
one call, tokens in random order.  Each case checks every in-range row's
output, the range flag, the written rows and that no other byte changed."""
import os

import numpy as np
import pytest
import torch

import oracle
import sequence_slot_kv_gb300 as skv
import synth
from gpu_harness import assert_close, to_dev

pytestmark = pytest.mark.gpu

N_CASES = 200
# SLOTKV_FUZZ_OFFSET shifts every case's seed, for a stress run over fresh
# configurations; the suite's own cases are offset 0.
OFFSET = int(os.environ.get("SLOTKV_FUZZ_OFFSET", "0"))


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    hd = int(rng.choice([64, 128, 256]))
    T = 4096 // hd
    G = int(rng.integers(1, 9))
    nkv = int(rng.integers(1, 5))
    B = int(rng.integers(1, 41))
    paged = bool(rng.integers(0, 2))
    bs = T * int(rng.integers(1, 4)) if paged else 0
    per = int(rng.integers(1, 7))
    slot_ctx = (bs * per) if paged else int(rng.integers(1, 7 * T))
    n_slots = B + int(rng.integers(0, 4))
    pos = rng.integers(0, slot_ctx, size=B)
    # the edges: 0, the last position, tile boundaries
    for i, v in enumerate((0, slot_ctx - 1, min(T, slot_ctx - 1), max(0, min(T - 1, slot_ctx - 1)))):
        if i < B and rng.random() < 0.5:
            pos[int(rng.integers(0, B))] = v
    split = None
    if rng.random() < 0.5:
        split = (T * int(rng.integers(1, 5)), int(rng.integers(1, 17)))
    flags = int(rng.integers(0, 4)) if rng.random() < 0.3 else 0
    w = synth.Workload(f"fuzz{seed}", 2000 + seed, B=B, n_slots=n_slots, slot_ctx=slot_ctx,
                       n_head=G * nkv, n_kv_head=nkv, head_dim=hd, theta=1e4,
                       sinks=bool(rng.integers(0, 2)), pos_rule="fixed",
                       fixed_positions=tuple(int(x) for x in pos), slot_rule="perm")
    bad = []
    if B > 1 and rng.random() < 0.3:
        bad = [int(rng.integers(0, B))]
    return w, bs, split, flags, bad


@pytest.mark.parametrize("seed", range(OFFSET, OFFSET + N_CASES))
def test_random_configuration(seed):
    w, bs, split, flags, bad = _case(seed)
    o = oracle.default()
    T = 4096 // w.head_dim
    pos = w.positions(0).astype(np.uint32)
    q, kn, vn = w.q(), w.k_new(), w.v_new()
    K0 = synth.normal(w.kv_elems(), w.seed, synth.S_HIST_K).reshape(
        w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    V0 = synth.normal(w.kv_elems(), w.seed, synth.S_HIST_V).reshape(K0.shape)
    if bs:
        per = w.slot_ctx // bs
        nb = w.n_slots * per
        perm = w.block_perm(bs)
        Kh = np.empty((nb, bs, w.n_kv_head, w.head_dim), dtype=np.float32)
        Vh = np.empty_like(Kh)
        Kh[perm] = K0.reshape(Kh.shape)
        Vh[perm] = V0.reshape(Vh.shape)
        addr = w.block_tables(bs).astype(np.uint32)
        if bad:
            addr = addr.copy()
            addr[bad[0], int(pos[bad[0]]) // bs] = nb + 1     # a block outside the pool
    else:
        Kh, Vh = K0.copy(), V0.copy()
        addr = w.slots().astype(np.uint32)
        if bad:
            addr = addr.copy()
            addr[bad[0]] = w.n_slots + 3                       # a slot outside the buffer
    Kd, Vd = to_dev(Kh), to_dev(Vh)
    rows, per_row = Kh.shape[0], Kh.shape[1]
    kv = skv.SlotKV(rows, per_row, w.n_kv_head, w.head_dim, w.B, w.n_head, k_buf=Kd, v_buf=Vd)
    try:
        if split:
            kv.set_split(*split)
        if flags:
            kv.set_options(flags)
        out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        args = (to_dev(q), to_dev(kn), to_dev(vn), to_dev(pos.astype(np.int32)),
                to_dev(addr.astype(np.int32)), to_dev(w.q_norm_w()), to_dev(w.k_norm_w()),
                to_dev(w.inv_freq()), None if w.sink_logits() is None else to_dev(w.sink_logits()),
                out, w.eps, w.scale)
        if bs:
            kv.decode_batch_attn_paged(*args)
        else:
            kv.decode_batch_attn(*args)
        torch.cuda.synchronize()
        flags_dev = kv.get_status()
        assert flags_dev == (skv.DEV_RANGE if bad else 0), flags_dev
        Kr, Vr = Kh.copy(), Vh.copy()
        common = (q, kn, vn, pos)
        tail = (w.q_norm_w(), w.k_norm_w(), w.inv_freq(), w.sink_logits(), w.eps, w.scale)
        if bs:
            ref, _, skipped = o.decode_batch_paged(Kr, Vr, *common, addr, *tail,
                                                   n_threads=8, flags=flags)
        else:
            ref, _, skipped = o.decode_batch(Kr, Vr, *common, addr, *tail, n_threads=8,
                                             flags=flags)
        assert skipped == len(bad)
        good = [b for b in range(w.B) if b not in bad]
        got = out.cpu().numpy()
        assert np.all(np.isnan(got[bad]))
        assert_close(got[good], ref[good], f"fuzz case {seed}")
        Kg, Vg = Kd.cpu().numpy(), Vd.cpu().numpy()
        assert_close(Kg, Kr, f"fuzz case {seed} K")        # written rows within tolerance
        same = np.all(Kr == Kh, axis=(2, 3))                # rows the step did not write
        assert np.array_equal(Kg[same].view(np.uint32), Kh[same].view(np.uint32))
        assert np.array_equal(Vg[same].view(np.uint32), Vh[same].view(np.uint32))
        if flags & 1:
            assert_close(Vg, Vr, f"fuzz case {seed} V")
        else:
            assert np.array_equal(Vg.view(np.uint32), Vr.view(np.uint32))
    finally:
        kv.free()


N_PREFILL = 60


def _prefill_case(seed):
    rng = np.random.default_rng(5000 + seed)
    hd = int(rng.choice([64, 128, 256]))
    T = 4096 // hd
    G = int(rng.integers(1, 9))
    nkv = int(rng.integers(1, 4))
    n_seq = int(rng.integers(1, 6))
    hist = rng.integers(0, 3 * T, size=n_seq)
    plen = rng.integers(1, 2 * T + 1, size=n_seq)
    slot_ctx = int((hist + plen).max()) + int(rng.integers(1, 9))
    n_slots = n_seq + int(rng.integers(0, 3))
    slots_of = rng.permutation(n_slots)[:n_seq]
    toks = [(int(slots_of[i]), int(hist[i]) + j) for i in range(n_seq) for j in range(int(plen[i]))]
    order = rng.permutation(len(toks))
    slots = np.array([toks[k][0] for k in order], dtype=np.uint32)
    pos = np.array([toks[k][1] for k in order], dtype=np.uint32)
    split = (T * int(rng.integers(1, 4)), int(rng.integers(1, 9))) if rng.random() < 0.5 else None
    flags = int(rng.integers(0, 4)) if rng.random() < 0.3 else 0
    w = synth.Workload(f"pfuzz{seed}", 3000 + seed, B=len(toks), n_slots=n_slots,
                       slot_ctx=slot_ctx, n_head=G * nkv, n_kv_head=nkv, head_dim=hd,
                       theta=1e4, sinks=bool(rng.integers(0, 2)), pos_rule="fixed",
                       fixed_positions=tuple([0] * len(toks)), slot_rule="perm")
    return w, slots, pos, split, flags


@pytest.mark.parametrize("seed", range(OFFSET, OFFSET + N_PREFILL))
def test_random_prefill(seed):
    """Random sequences (history, prompt length, slot) as one prefill call
    with their tokens in random order: every token equals one decode step at
    a time in position order; written rows and untouched bytes as for decode."""
    w, slots, pos, split, flags = _prefill_case(seed)
    o = oracle.default()
    q, kn, vn = w.q(), w.k_new(), w.v_new()
    Kh = synth.normal(w.kv_elems(), w.seed, synth.S_HIST_K).reshape(
        w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    Vh = synth.normal(w.kv_elems(), w.seed, synth.S_HIST_V).reshape(Kh.shape)
    Kd, Vd = to_dev(Kh), to_dev(Vh)
    kv = skv.SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head,
                    k_buf=Kd, v_buf=Vd)
    try:
        if split:
            kv.set_split(*split)
        if flags:
            kv.set_options(flags)
        out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        kv.prefill_batch_attn(to_dev(q), to_dev(kn), to_dev(vn), to_dev(pos.astype(np.int32)),
                              to_dev(slots.astype(np.int32)), to_dev(w.q_norm_w()),
                              to_dev(w.k_norm_w()), to_dev(w.inv_freq()),
                              None if w.sink_logits() is None else to_dev(w.sink_logits()),
                              out, w.eps, w.scale)
        torch.cuda.synchronize()
        assert kv.get_status() == 0
        Kr, Vr = Kh.copy(), Vh.copy()
        ref = np.empty((w.B, w.n_head, w.head_dim), dtype=np.float32)
        for i in np.lexsort((pos, slots)):
            r, _, _ = o.decode_batch(Kr, Vr, q[i:i + 1], kn[i:i + 1], vn[i:i + 1], pos[i:i + 1],
                                     slots[i:i + 1], w.q_norm_w(), w.k_norm_w(), w.inv_freq(),
                                     w.sink_logits(), w.eps, w.scale, flags=flags)
            ref[i] = r[0]
        assert_close(out.cpu().numpy(), ref, f"prefill fuzz case {seed}")
        Kg, Vg = Kd.cpu().numpy(), Vd.cpu().numpy()
        mask = np.zeros(Kh.shape[:2], dtype=bool)
        mask[slots, pos] = True
        assert_close(Kg[mask], Kr[mask], f"prefill fuzz case {seed} K")
        assert_close(Vg[mask], Vr[mask], f"prefill fuzz case {seed} V")
        if not flags & 1:
            assert np.array_equal(Vg[mask].view(np.uint32), Vr[mask].view(np.uint32))
        assert np.array_equal(Kg[~mask].view(np.uint32), Kh[~mask].view(np.uint32))
        assert np.array_equal(Vg[~mask].view(np.uint32), Vh[~mask].view(np.uint32))
    finally:
        kv.free()

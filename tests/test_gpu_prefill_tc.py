"""The tensor-core prefill (head dims 64 and 128) on the shapes it tiles:
long runs of consecutive same-slot tokens cut into tiles of 128 / G tokens
(several tiles per run, a partial last tile, tiles whose 128 rows are not all
used when G does not divide 128), histories spanning many key tiles (every
stage of the ring reused), positions out of order within a run, and the
benchmark's prefill workload at full size.  Every token must equal one decode
step at a time in position order ("Forward Cuda Gemma", prefillBatched), as
the oracle computes it."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_harness import assert_close, to_dev
from sequence_slot_kv_gb300 import SlotKV, slot_kv_prefill_host_parts

pytestmark = pytest.mark.gpu


def _workload(hd, G, n_kv, idx, n_tok, n_slots, slot_ctx, sinks=True):
    return synth.Workload(f"pftc_hd{hd}_g{G}", 900 + idx, B=n_tok, n_slots=n_slots,
                          slot_ctx=slot_ctx, n_head=G * n_kv, n_kv_head=n_kv, head_dim=hd,
                          theta=1e4, sinks=sinks, pos_rule="fixed",
                          fixed_positions=tuple([0] * n_tok), slot_rule="perm")


def _run(w, slots, pos):
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    K = torch.empty(shape, device="cuda")
    V = torch.empty(shape, device="cuda")
    w.dev_fill_history(K.data_ptr(), V.data_ptr(), torch.cuda.current_stream().cuda_stream)
    kv = SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head, k_buf=K, v_buf=V)
    try:
        assert kv.call_shape(w.B, prefill=True)[2] == 3     # prep, plan, tensor-core kernel
        out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        s = w.sink_logits()
        kv.prefill_batch_attn(to_dev(w.q()), to_dev(w.k_new()), to_dev(w.v_new()),
                              to_dev(pos.astype(np.int32)), to_dev(slots.astype(np.int32)),
                              to_dev(w.q_norm_w()), to_dev(w.k_norm_w()), to_dev(w.inv_freq()),
                              None if s is None else to_dev(s), out, w.eps, w.scale)
        torch.cuda.synchronize()
        assert kv.get_status() == 0
        return out.cpu().numpy(), K, V
    finally:
        kv.free()


def _oracle_rows(w, slots, pos, rows):
    """The oracle for tokens ``rows``: every token's k' and v written into
    host copies of the slots first (what the earlier tokens of the sequential
    definition leave there; a token reads only positions <= its own), then
    one decode step per sampled token."""
    o = oracle.default()
    used = sorted(set(int(s) for s in slots))
    Kh = np.stack([w.hist_rows("k", s, 0, w.slot_ctx) for s in used])
    Vh = np.stack([w.hist_rows("v", s, 0, w.slot_ctx) for s in used])
    at = {s: i for i, s in enumerate(used)}
    kn, vn = w.k_new(), w.v_new()
    kw, inv = w.k_norm_w(), w.inv_freq()
    for i in range(w.B):
        c, p = at[int(slots[i])], int(pos[i])
        for g in range(w.n_kv_head):
            Kh[c, p, g] = o.norm_rope_head(kn[i, g], kw, w.eps, p, inv).astype(np.float32)
        Vh[c, p] = vn[i]
    rows = list(rows)
    compact = np.array([at[int(slots[i])] for i in rows], dtype=np.uint32)
    ref, _, skipped = o.decode_batch(Kh, Vh, w.q()[rows], kn[rows], vn[rows], pos[rows], compact,
                                     w.q_norm_w(), kw, inv, w.sink_logits(), w.eps, w.scale,
                                     n_threads=min(len(rows), 32))
    assert skipped == 0
    return ref


SHAPES = [(hd, G) for hd in (64, 128) for G in range(1, 9)]


@pytest.mark.parametrize("hd,G", SHAPES, ids=[f"hd{h}_g{g}" for h, g in SHAPES])
def test_long_runs_every_group_size(hd, G):
    """Three sequences given one after another: a run of 2.5 tiles after a
    history of several key tiles, a one-token run, and a run starting at
    position 0; the tokens of each run in increasing position."""
    MT = 128 // G
    BK = 64  # keys per key tile of the tensor-core prefill
    seqs = [(3, 7 * BK + 5, MT * 2 + MT // 2), (0, 41, 1), (1, 0, MT + 3)]
    slots = np.concatenate([np.full(n, s, np.uint32) for s, _, n in seqs])
    pos = np.concatenate([np.arange(h, h + n, dtype=np.uint32) for _, h, n in seqs])
    w = _workload(hd, G, 2, SHAPES.index((hd, G)), len(pos), 5, int(pos.max()) + 7,
                  sinks=(G % 2 == 1))
    got, K, V = _run(w, slots, pos)
    ref = _oracle_rows(w, slots, pos, range(w.B))
    assert_close(got, ref, f"tensor-core prefill hd={hd} G={G}")
    # the written rows: V exact, K as a decode step writes it
    Vg = V[torch.from_numpy(slots.astype(np.int64)).cuda(),
           torch.from_numpy(pos.astype(np.int64)).cuda()].cpu().numpy()
    assert np.array_equal(Vg.view(np.uint32), w.v_new().view(np.uint32))


@pytest.mark.parametrize("hd", [64, 128])
def test_unordered_positions_within_a_run(hd):
    """One slot's tokens in a shuffled order (a run is consecutive tokens of
    one slot, in any position order): each row's causal mask follows its own
    position."""
    G, n = 4, 150
    rng = np.random.default_rng(hd)
    pos = (300 + rng.permutation(n)).astype(np.uint32)
    slots = np.full(n, 2, np.uint32)
    w = _workload(hd, G, 2, 40 + hd, n, 3, 300 + n + 3)
    got, _, _ = _run(w, slots, pos)
    ref = _oracle_rows(w, slots, pos, range(n))
    assert_close(got, ref, f"unordered run hd={hd}")


def test_bench_prefill_workload_full_size():
    """The benchmark's prefill: 8 sequences, a 512-token chunk each after
    1536 positions of history, 32 query / 8 kv heads, head dim 128; sampled
    tokens of every sequence against the oracle."""
    import bench
    w, slots, pos = bench.prefill_workload()
    got, _, _ = _run(w, slots.astype(np.uint32), pos.astype(np.uint32))
    assert np.all(np.isfinite(got))
    chunk = bench.PREFILL_CHUNK
    rows = sorted({s * chunk + j for s in range(bench.PREFILL_SEQ) for j in (0, 31, 32, 257, 511)})
    ref = _oracle_rows(w, slots, pos, rows)
    assert_close(got[rows], ref, "prefill workload sampled tokens")


def _run_host(w, slots, pos, pinned):
    """prefill_batch_attn_host on fresh slots holding the same history."""
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    K = torch.empty(shape, device="cuda")
    V = torch.empty(shape, device="cuda")
    w.dev_fill_history(K.data_ptr(), V.data_ptr(), torch.cuda.current_stream().cuda_stream)
    kv = SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head, k_buf=K, v_buf=V)
    try:
        host = lambda a: (torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
                          if pinned else torch.from_numpy(np.ascontiguousarray(a)))
        out = host(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32))
        s = w.sink_logits()
        kv.prefill_batch_attn_host(host(w.q()), host(w.k_new()), host(w.v_new()),
                                   host(pos.astype(np.int32)), host(slots.astype(np.int32)),
                                   to_dev(w.q_norm_w()), to_dev(w.k_norm_w()),
                                   to_dev(w.inv_freq()), None if s is None else to_dev(s), out,
                                   w.eps, w.scale)
        assert kv.get_status() == 0
        return out.numpy(), K, V
    finally:
        kv.free()


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_prefill_host_entry_equals_device_entry(pinned):
    """prefill_batch_attn_host (tokens' tensors and out in host memory) runs
    the same kernels as the device entry on the same values: the same output
    and the same slot bytes, bit for bit."""
    hd, G = 128, 4
    slots = np.concatenate([np.full(70, 1, np.uint32), np.full(33, 3, np.uint32)])
    pos = np.concatenate([np.arange(200, 270, dtype=np.uint32), np.arange(0, 33, dtype=np.uint32)])
    w = _workload(hd, G, 2, 95, len(pos), 5, 300)
    got_dev, Kd, Vd = _run(w, slots, pos)
    got, K, V = _run_host(w, slots, pos, pinned)
    assert np.array_equal(got.view(np.uint32), got_dev.view(np.uint32))
    assert torch.equal(K, Kd) and torch.equal(V, Vd)


# (head dim, G, run lengths, the runs' slots, parts the host entry makes)
PART_LAYOUTS = {
    "equal_hd128": (128, 4, [512] * 8, None, 8),
    "uneven_hd64": (64, 8, [1500, 100, 900, 1700], None, 3),
    "returning_slot_hd128": (128, 2, [800] * 4, [0, 1, 0, 2], 2),
    "interleaved_hd64": (64, 4, [1] * 2048, [0, 1] * 1024, 1),
}


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("name", list(PART_LAYOUTS))
def test_prefill_host_entry_in_parts_equals_device_entry(name, pinned):
    """A host call of 1024 tokens or more is cut into parts whose tokens
    share no slot, each run as a prefill of its own while the others' copies
    move: the output and the slot bytes stay those of one device call, bit
    for bit (the parts hold the same runs, so the same tiles)."""
    hd, G, lengths, ids, n_parts = PART_LAYOUTS[name]
    ids = list(range(len(lengths))) if ids is None else ids
    slots = np.concatenate([np.full(n, s, np.uint32) for s, n in zip(ids, lengths)])
    # each slot's runs continue its positions after a history of its own
    nxt, pos = {}, []
    for s_, n in zip(ids, lengths):
        p0 = nxt.get(s_, 40 + 13 * s_)
        pos.append(np.arange(p0, p0 + n, dtype=np.uint32))
        nxt[s_] = p0 + n
    pos = np.concatenate(pos)
    assert len(slot_kv_prefill_host_parts(slots)) - 1 == n_parts
    w = _workload(hd, G, 2, 960 + list(PART_LAYOUTS).index(name), len(pos), int(slots.max()) + 1,
                  int(pos.max()) + 3)
    got_dev, Kd, Vd = _run(w, slots, pos)
    got, K, V = _run_host(w, slots, pos, pinned)
    assert np.array_equal(got.view(np.uint32), got_dev.view(np.uint32))
    assert torch.equal(K, Kd) and torch.equal(V, Vd)


@pytest.mark.parametrize("seed", range(8))
def test_prefill_host_in_parts_random_layouts(seed):
    """Seeded random calls of 2048 to 3500 tokens: runs of random lengths on
    slots that may come back later in the call, at either head dim and a
    random G; the host entry (cut where its parts allow) equals one device
    call bit for bit."""
    rng = np.random.default_rng(7100 + seed)
    hd = (64, 128)[seed % 2]
    G = int(rng.integers(1, 9))
    n_target = int(rng.integers(2048, 3500))
    lengths, ids = [], []
    n_slots = int(rng.integers(3, 10))
    while sum(lengths) < n_target:
        lengths.append(int(rng.integers(1, 900)))
        ids.append(int(rng.integers(0, n_slots)))
    lengths[-1] -= sum(lengths) - n_target
    if lengths[-1] == 0:
        lengths.pop()
        ids.pop()
    slots = np.concatenate([np.full(n, s, np.uint32) for s, n in zip(ids, lengths)])
    nxt, pos = {}, []
    for s_, n in zip(ids, lengths):
        p0 = nxt.get(s_, int(rng.integers(0, 200)))
        pos.append(np.arange(p0, p0 + n, dtype=np.uint32))
        nxt[s_] = p0 + n
    pos = np.concatenate(pos)
    cuts = slot_kv_prefill_host_parts(slots)
    for m in cuts[1:-1]:
        assert not set(slots[:m].tolist()) & set(slots[m:].tolist())
    w = _workload(hd, G, 2, 980 + seed, len(pos), n_slots, int(pos.max()) + 3,
                  sinks=(seed % 3 == 0))
    got_dev, Kd, Vd = _run(w, slots, pos)
    got, K, V = _run_host(w, slots, pos, pinned=True)
    assert np.array_equal(got.view(np.uint32), got_dev.view(np.uint32))
    assert torch.equal(K, Kd) and torch.equal(V, Vd)


@pytest.mark.parametrize("hd", [64, 128])
def test_out_of_range_tokens_are_skipped(hd):
    """Tokens whose slot or position is out of range raise SLOTKV_DEV_RANGE,
    join no tile and write nothing (their out rows keep their contents);
    every other token is the oracle's, as if the bad ones were not in the
    call, and only the good tokens' slot rows change."""
    import sequence_slot_kv_gb300 as skv
    G, n_slots, ctx = 4, 5, 240
    slots = np.concatenate([np.full(60, 1, np.uint32), np.full(40, 3, np.uint32)])
    pos = np.concatenate([np.arange(100, 160, dtype=np.uint32), np.arange(0, 40, dtype=np.uint32)])
    bad = [10, 70, 99]
    pos[10] = ctx              # position past the slot
    slots[70] = n_slots        # slot past the pool
    pos[99] = ctx + 5
    good = [i for i in range(len(pos)) if i not in bad]
    w = _workload(hd, G, 2, 60 + hd, len(pos), n_slots, ctx)
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    K = torch.empty(shape, device="cuda")
    V = torch.empty(shape, device="cuda")
    w.dev_fill_history(K.data_ptr(), V.data_ptr(), torch.cuda.current_stream().cuda_stream)
    K0, V0 = K.cpu().numpy(), V.cpu().numpy()
    kv = SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head, k_buf=K, v_buf=V)
    try:
        out = torch.full((w.B, w.n_head, w.head_dim), 7.0, device="cuda")
        s = w.sink_logits()
        kv.prefill_batch_attn(to_dev(w.q()), to_dev(w.k_new()), to_dev(w.v_new()),
                              to_dev(pos.astype(np.int32)), to_dev(slots.astype(np.int32)),
                              to_dev(w.q_norm_w()), to_dev(w.k_norm_w()), to_dev(w.inv_freq()),
                              None if s is None else to_dev(s), out, w.eps, w.scale)
        torch.cuda.synchronize()
        assert kv.get_status() == skv.DEV_RANGE
        got = out.cpu().numpy()
        Kg, Vg = K.cpu().numpy(), V.cpu().numpy()
    finally:
        kv.free()
    assert np.all(got[bad] == 7.0)
    # the oracle on host copies of the two slots, the good tokens' rows
    # written first, then one decode step per good token
    o = oracle.default()
    Kh, Vh = K0[[1, 3]].copy(), V0[[1, 3]].copy()
    at = {1: 0, 3: 1}
    kn, vn = w.k_new(), w.v_new()
    for i in good:
        c, p = at[int(slots[i])], int(pos[i])
        for g in range(w.n_kv_head):
            Kh[c, p, g] = o.norm_rope_head(kn[i, g], w.k_norm_w(), w.eps, p,
                                           w.inv_freq()).astype(np.float32)
        Vh[c, p] = vn[i]
    compact = np.array([at[int(slots[i])] for i in good], dtype=np.uint32)
    ref, _, skipped = o.decode_batch(Kh, Vh, w.q()[good], kn[good], vn[good], pos[good], compact,
                                     w.q_norm_w(), w.k_norm_w(), w.inv_freq(), s, w.eps,
                                     w.scale, n_threads=16)
    assert skipped == 0
    assert_close(got[good], ref, f"prefill with out-of-range tokens hd={hd}")
    # only the good tokens' rows changed; the bad tokens wrote nothing
    mask = np.zeros(shape[:2], dtype=bool)
    mask[slots[good], pos[good]] = True
    assert np.array_equal(Kg[~mask].view(np.uint32), K0[~mask].view(np.uint32))
    assert np.array_equal(Vg[~mask].view(np.uint32), V0[~mask].view(np.uint32))
    assert np.array_equal(Vg[mask].view(np.uint32), vn[good].view(np.uint32).reshape(Vg[mask].shape))

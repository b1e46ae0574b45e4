"""Paged KV: decode_batch_attn_paged against the paged oracle, through the C
ABI.  The paged cache with per-sequence block tables of the Qwen3SsmLayer
page (decode_multi_seq), running the step of "Forward Cuda Gemma",
decodeBatch.

The pool is the workload's slot history cut into blocks and shuffled (the
generator's block recipe), so each row reads blocks scattered over the pool.
Paging changes addresses only: the result must also equal the slot kernel's
on the same keys bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import sequence_slot_kv_gb300 as skv
import synth
from gpu_harness import DeviceRun, assert_close, to_dev

pytestmark = pytest.mark.gpu


class PagedRun:
    """A workload's history scattered into a device block pool, with a handle
    adopting the pool (n_slots = blocks, slot_ctx = block size)."""

    def __init__(self, w, bs, split=None):
        self.w, self.bs = w, bs
        self.per = w.slot_ctx // bs
        self.n_blocks = w.n_slots * self.per
        self.pshape = (self.n_blocks, bs, w.n_kv_head, w.head_dim)
        self.perm = torch.from_numpy(w.block_perm(bs).astype(np.int64)).cuda()
        self.K, self.V = self.fresh_pool()
        self.kv = skv.SlotKV(self.n_blocks, bs, w.n_kv_head, w.head_dim, w.B, w.n_head,
                             k_buf=self.K, v_buf=self.V)
        if split is not None:
            self.kv.set_split(*split)
        self.tables_np = w.block_tables(bs)
        self.tables = to_dev(self.tables_np.astype(np.int32))
        self.qw, self.kw, self.inv = to_dev(w.q_norm_w()), to_dev(w.k_norm_w()), to_dev(w.inv_freq())
        s = w.sink_logits()
        self.sinks = None if s is None else to_dev(s)

    def fresh_pool(self):
        w = self.w
        shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
        pools = []
        Ks = torch.empty(shape, device="cuda")
        Vs = torch.empty(shape, device="cuda")
        w.dev_fill_history(Ks.data_ptr(), Vs.data_ptr(), torch.cuda.current_stream().cuda_stream)
        for src in (Ks, Vs):
            dst = torch.empty(self.pshape, device="cuda")
            dst[self.perm] = src.view(self.pshape)
            pools.append(dst)
        del Ks, Vs
        return pools

    def step(self, step=0, positions=None, tables=None, out=None):
        w = self.w
        pos = w.positions(step) if positions is None else positions
        if out is None:
            out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        self.kv.decode_batch_attn_paged(
            to_dev(w.q(step)), to_dev(w.k_new(step)), to_dev(w.v_new(step)),
            to_dev(pos.astype(np.int32)), self.tables if tables is None else tables,
            self.qw, self.kw, self.inv, self.sinks, out, w.eps, w.scale)
        return out

    def close(self):
        self.kv.free()


def host_pool(w, bs):
    """Host copy of the whole shuffled pool (small workloads only)."""
    perm = w.block_perm(bs)
    shape = (w.n_slots * (w.slot_ctx // bs), bs, w.n_kv_head, w.head_dim)
    pools = []
    for stream in (synth.S_HIST_K, synth.S_HIST_V):
        src = synth.normal(w.kv_elems(), w.seed, stream).reshape(shape)
        dst = np.empty_like(src)
        dst[perm] = src
        pools.append(dst)
    return pools


def oracle_paged(w, bs, K, V, tables, positions=None, step=0, flags=0):
    o = oracle.default()
    pos = w.positions(step) if positions is None else positions
    out, _, skipped = o.decode_batch_paged(
        K, V, w.q(step), w.k_new(step), w.v_new(step), pos, tables, w.q_norm_w(),
        w.k_norm_w(), w.inv_freq(), w.sink_logits(), w.eps, w.scale,
        n_threads=min(w.B, 32), flags=flags)
    return out, skipped


def check_pool(run, Kr, Vr, written):
    """Pool after the step: the written rows' K within tolerance and V exact
    against the oracle's pool, every other byte bit-identical."""
    Kg, Vg = run.K.cpu().numpy(), run.V.cpu().numpy()
    assert_close(Kg[written], Kr[written], "paged written K")
    assert np.array_equal(Vg[written].view(np.uint32), Vr[written].view(np.uint32))
    assert np.array_equal(Kg[~written].view(np.uint32), Kr[~written].view(np.uint32))
    assert np.array_equal(Vg[~written].view(np.uint32), Vr[~written].view(np.uint32))


def written_mask(run, tables, pos, rows=None):
    m = np.zeros(run.pshape[:2], dtype=bool)
    for b in (range(len(pos)) if rows is None else rows):
        p = int(pos[b])
        m[tables[b, p // run.bs], p % run.bs] = True
    return m


def small_paged_workload(hd, G, bs_tiles, idx, sinks):
    T = 4096 // hd
    bs = bs_tiles * T
    slot_ctx = 6 * bs
    positions = (0, 1, T - 1, T, bs - 1, bs, bs + 1, 3 * bs + 7, slot_ctx - 2, slot_ctx - 1)
    w = synth.Workload(
        f"paged_hd{hd}_g{G}", 800 + idx, B=len(positions), n_slots=len(positions) + 2,
        slot_ctx=slot_ctx, n_head=2 * G, n_kv_head=2, head_dim=hd, theta=10000.0, sinks=sinks,
        pos_rule="fixed", fixed_positions=positions, slot_rule="perm")
    return w, bs


GEOMS = [(64, 8, 1), (64, 1, 2), (128, 4, 1), (128, 5, 2), (128, 2, 4), (256, 2, 1),
         (256, 8, 3)]


@pytest.mark.parametrize("policy", ["many_splits", "default"])
@pytest.mark.parametrize("hd,G,bt", GEOMS, ids=[f"hd{h}_g{g}_bs{b}T" for h, g, b in GEOMS])
def test_paged_small_geometry_matches_oracle(hd, G, bt, policy):
    idx = GEOMS.index((hd, G, bt))
    w, bs = small_paged_workload(hd, G, bt, idx, sinks=(idx % 2 == 0))
    split = (4096 // hd, 8) if policy == "many_splits" else None
    run = PagedRun(w, bs, split=split)
    try:
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.kv.get_status() == 0
        Kr, Vr = host_pool(w, bs)
        ref, skipped = oracle_paged(w, bs, Kr, Vr, run.tables_np)
        assert skipped == 0
        assert_close(out.cpu().numpy(), ref, f"paged out hd={hd} G={G} bs={bs} {policy}")
        check_pool(run, Kr, Vr, written_mask(run, run.tables_np, w.positions(0)))
    finally:
        run.close()


@pytest.mark.parametrize("split", [None, (32, 8)], ids=["default", "many_splits"])
def test_paged_equals_slot_kernel_bit_for_bit(split):
    """The same keys through a slot and through a shuffled block pool give the
    same output bits and the same written rows."""
    w = synth.Workload("paged_vs_slot", 820, B=16, n_slots=20, slot_ctx=2048, n_head=32,
                       n_kv_head=8, head_dim=128, theta=1e6, sinks=True, slot_rule="subset")
    bs = 64
    run_s = DeviceRun(w, split=split)
    run_p = PagedRun(w, bs, split=split)
    try:
        out_s = run_s.step(0)
        out_p = run_p.step(0)
        torch.cuda.synchronize()
        assert run_s.status() == 0 and run_p.kv.get_status() == 0
        assert torch.equal(out_s, out_p)
        # the pool, read back in slot order, equals the slot buffers
        shape = run_s.K.shape
        assert torch.equal(run_p.K[run_p.perm].view(shape), run_s.K)
        assert torch.equal(run_p.V[run_p.perm].view(shape), run_s.V)
    finally:
        run_s.close()
        run_p.close()


def _compact(w, bs, rows, pos):
    """Host pool holding only the blocks rows `rows` use, with tables into it."""
    slots = w.slots()
    used = [int(pos[r]) // bs + 1 for r in rows]
    width = max(used)
    Kc = np.empty((sum(used), bs, w.n_kv_head, w.head_dim), dtype=np.float32)
    Vc = np.empty_like(Kc)
    tab = np.zeros((len(rows), width), dtype=np.uint32)
    base = 0
    for i, r in enumerate(rows):
        s = int(slots[r])
        Kc[base:base + used[i]] = w.hist_rows("k", s, 0, used[i] * bs).reshape(
            used[i], bs, w.n_kv_head, w.head_dim)
        Vc[base:base + used[i]] = w.hist_rows("v", s, 0, used[i] * bs).reshape(
            used[i], bs, w.n_kv_head, w.head_dim)
        tab[i, :used[i]] = np.arange(base, base + used[i], dtype=np.uint32)
        base += used[i]
    return Kc, Vc, tab


def test_paged_full_size_mid():
    """The batch-32 workload at full size (4096-key slots, 32 query / 8 kv
    heads, head dim 128) in 64-key blocks under the default split policy:
    sampled rows against the paged oracle, every written row, every other byte."""
    w = synth.WORKLOADS["mid"]
    bs = 64
    run = PagedRun(w, bs)
    try:
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.kv.get_status() == 0
        got = out.cpu().numpy()
        pos = w.positions(0)
        rows = sorted({int(np.argmin(pos)), int(np.argmax(pos)), 3, 11, 20, 27})
        Kc, Vc, tab = _compact(w, bs, rows, pos)
        o = oracle.default()
        sub = lambda a: a[rows]  # noqa: E731
        ref, _, skipped = o.decode_batch_paged(
            Kc, Vc, sub(w.q()), sub(w.k_new()), sub(w.v_new()), pos[rows], tab, w.q_norm_w(),
            w.k_norm_w(), w.inv_freq(), w.sink_logits(), w.eps, w.scale, n_threads=len(rows))
        assert skipped == 0
        assert_close(got[rows], ref, f"paged mid rows {rows}")
        # every written row: V exact, K against the oracle's write
        for i, r in enumerate(rows):
            p = int(pos[r])
            blk = int(run.tables_np[r, p // bs])
            cb = int(tab[i, p // bs])
            assert_close(run.K[blk, p % bs].cpu().numpy(), Kc[cb, p % bs], f"K row {r}")
        Vw = run.V[torch.from_numpy(run.tables_np[np.arange(w.B), pos // bs].astype(np.int64)),
                   torch.from_numpy((pos % bs).astype(np.int64))].cpu().numpy()
        assert np.array_equal(Vw.view(np.uint32), w.v_new(0).view(np.uint32))
        # every other byte untouched
        K0, V0 = run.fresh_pool()
        mask = torch.from_numpy(written_mask(run, run.tables_np, pos)).cuda()
        K0[mask] = run.K[mask]
        V0[mask] = run.V[mask]
        assert torch.equal(K0.view(torch.int32), run.K.view(torch.int32))
        assert torch.equal(V0.view(torch.int32), run.V.view(torch.int32))
    finally:
        run.close()


def test_paged_out_of_range_rows_are_skipped_and_flagged():
    """A row whose used blocks include an id outside the pool, or whose pos is
    past its table, gets nothing written and raises the range flag; an
    out-of-pool id in an entry the row does not use is never read."""
    w, bs = small_paged_workload(128, 4, 1, 30, sinks=True)
    run = PagedRun(w, bs, split=(32, 8))
    try:
        pos = w.positions(0).copy()
        tabs = run.tables_np.copy()
        nb = np.uint32(run.n_blocks)
        rows_bad = [2, 7]
        tabs[2, int(pos[2]) // bs] = nb + 5            # the block holding key p
        tabs[7, 0] = nb                                # the first history block
        tabs[5, -1] = 0xFFFFFFFF                        # an entry row 5 never uses
        assert int(pos[5]) // bs < tabs.shape[1] - 1
        narrow = tabs[:, :4].copy()                    # 4 blocks: rows with pos >= 4*bs overflow
        over = [b for b in range(w.B) if int(pos[b]) >= 4 * bs]
        assert over
        for tables_np, bad in ((tabs, rows_bad), (narrow, sorted(set(rows_bad) | set(over)))):
            if tables_np is narrow:                    # start again from the fresh pool
                K0, V0 = run.fresh_pool()
                run.K.copy_(K0)
                run.V.copy_(V0)
                del K0, V0
            out = run.step(0, tables=to_dev(tables_np.astype(np.int32)))
            torch.cuda.synchronize()
            assert run.kv.get_status() == skv.DEV_RANGE
            got = out.cpu().numpy()
            good = [b for b in range(w.B) if b not in bad]
            assert np.all(np.isnan(got[bad]))
            Kr, Vr = host_pool(w, bs)
            ref, skipped = oracle_paged(w, bs, Kr, Vr, tables_np)
            assert skipped == len(bad)
            assert_close(got[good], ref[good], "paged rows beside skipped rows")
            check_pool(run, Kr, Vr, written_mask(run, tables_np, pos, rows=good))
    finally:
        run.close()


def test_paged_argument_errors():
    w, bs = small_paged_workload(128, 2, 1, 31, sinks=False)
    run = PagedRun(w, bs)
    try:
        out = torch.empty((w.B, w.n_head, w.head_dim), device="cuda")
        args = (to_dev(w.q()), to_dev(w.k_new()), to_dev(w.v_new()),
                to_dev(w.positions(0).astype(np.int32)))
        # a block size that is not a multiple of the 32-key tile
        K = torch.zeros((8, 48, w.n_kv_head, w.head_dim), device="cuda")
        kv48 = skv.SlotKV(8, 48, w.n_kv_head, w.head_dim, w.B, w.n_head, k_buf=K, v_buf=K.clone())
        try:
            with pytest.raises(skv.SlotKVError) as ei:
                kv48.decode_batch_attn_paged(*args, run.tables, run.qw, run.kw, run.inv, None, out,
                                             w.eps, w.scale)
            assert ei.value.code == 3
        finally:
            kv48.free()
        # a table stride of zero
        rc = skv._lib.decode_batch_attn_paged(
            run.kv._h, w.B, w.n_head, args[0].data_ptr(), args[1].data_ptr(),
            args[2].data_ptr(), args[3].data_ptr(), run.tables.data_ptr(), 0,
            run.qw.data_ptr(), run.kw.data_ptr(), run.inv.data_ptr(), None, out.data_ptr(),
            w.eps, w.scale, None)
        assert rc == 1
        # a null table
        rc = skv._lib.decode_batch_attn_paged(
            run.kv._h, w.B, w.n_head, args[0].data_ptr(), args[1].data_ptr(),
            args[2].data_ptr(), args[3].data_ptr(), None, 4,
            run.qw.data_ptr(), run.kw.data_ptr(), run.inv.data_ptr(), None, out.data_ptr(),
            w.eps, w.scale, None)
        assert rc == 1
        assert run.kv.get_status() == 0
    finally:
        run.close()


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_paged_host_entry_matches_device_entry_and_oracle(pinned):
    """decode_batch_attn_paged_host (inputs, tables and out in host memory)
    against the device entry with the same table on the same pool, bit for
    bit, and against the paged oracle; twice, so the second call reuses the
    table staging, and a wider table grows it.  (The table's width is the
    call's context capacity, which the default policy may size its work
    from -- here the narrow table takes the small-call kernel, the wide one
    the persistent kernel -- so each width is compared with its own device
    call.)"""
    w, bs = small_paged_workload(128, 4, 1, 40, sinks=True)
    run_d = PagedRun(w, bs)
    run_h = PagedRun(w, bs)
    try:
        Kr, Vr = host_pool(w, bs)
        ref, skipped = oracle_paged(w, bs, Kr, Vr, run_d.tables_np)
        assert skipped == 0
        host = lambda a: (torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
                          if pinned else torch.from_numpy(np.ascontiguousarray(a)))
        hq, hk, hv = host(w.q()), host(w.k_new()), host(w.v_new())
        hp = host(w.positions(0).astype(np.int32))
        for width in (run_d.tables_np.shape[1], run_d.tables_np.shape[1] + 5):
            # padded tables: entries past a row's last used block are never read
            tab = np.full((w.B, width), 2**31 - 1, dtype=np.int32)
            tab[:, :run_d.tables_np.shape[1]] = run_d.tables_np
            K0, V0 = run_h.fresh_pool()
            for r in (run_d, run_h):
                r.K.copy_(K0)
                r.V.copy_(V0)
            del K0, V0
            want = run_d.step(0, tables=to_dev(tab))
            torch.cuda.synchronize()
            assert run_d.kv.get_status() == 0
            out = host(np.full((w.B, w.n_head, w.head_dim), np.nan, dtype=np.float32))
            run_h.kv.decode_batch_attn_paged_host(hq, hk, hv, hp, host(tab), run_h.qw, run_h.kw,
                                                  run_h.inv, run_h.sinks, out, w.eps, w.scale)
            assert run_h.kv.get_status() == 0
            assert torch.equal(out, want.cpu()), f"table width {width}"
            assert_close(out.numpy(), ref, f"paged host entry, table width {width}")
            assert torch.equal(run_h.K, run_d.K) and torch.equal(run_h.V, run_d.V)
    finally:
        run_d.close()
        run_h.close()

"""The small-call decode kernel: a call whose (row, kv head) pairs fit in two
CTAs per SM and whose slots hold at most eight tiles of keys runs one CTA per
pair over all of the row's keys, instead of the persistent pipeline and its
plan ("Forward Cuda Gemma", decodeBatch: the same step).  It is taken under
the default split policy only.  Checked against the oracle (outputs and every
byte of K and V), against the persistent kernel on the same inputs, and for
the semantics the persistent kernel keeps: skipped out-of-range rows, stale
history never read, rows independent of each other, paged equal to slot.
"""
import numpy as np
import pytest
import torch

import oracle
import sequence_slot_kv_gb300 as skv
import synth
from gpu_harness import DeviceRun, assert_close, check_kv_after, oracle_rows, to_dev

pytestmark = pytest.mark.gpu


def _wl(hd, G, idx, sinks=True, nkv=2, ctx_tiles=8):
    """Rows at the chunk edges of a slot of ctx_tiles tiles: no history, one
    key, a ragged first chunk, exactly one chunk, one past it, and the last
    two positions of the slot."""
    T = 4096 // hd
    ctx = ctx_tiles * T
    pos = sorted({p for p in (0, 1, 3, T - 1, T, T + 1, 2 * T + 5, ctx - 2, ctx - 1) if p < ctx})
    return synth.Workload(f"small_hd{hd}_g{G}", 900 + idx, B=len(pos), n_slots=len(pos) + 2,
                          slot_ctx=ctx, n_head=G * nkv, n_kv_head=nkv, head_dim=hd, theta=1e4,
                          sinks=sinks, pos_rule="fixed", fixed_positions=tuple(pos),
                          slot_rule="perm")


def _is_small(kv, B, bt_stride=0):
    """The small kernel reports one kernel, a CTA per (row, kv head) and a
    chunk of one tile; the persistent kernel without a plan also launches
    alone, but its default chunk is at least 512 KiB of K+V per kv head."""
    chunk, ctas, kernels = kv.call_shape(B, bt_stride=bt_stride)
    return kernels == 1 and ctas == B * kv.n_kv_head and chunk == 4096 // kv.head_dim


@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8])
def test_small_matches_oracle(hd, G):
    w = _wl(hd, G, 8 * [64, 128, 256].index(hd) + G, sinks=G % 2 == 0)
    run = DeviceRun(w)
    try:
        assert _is_small(run.kv, w.B)
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.status() == 0
        ref, _, _ = oracle_rows(w, range(w.B))
        assert_close(out.cpu().numpy(), ref[0], f"small out hd={hd} G={G}")
        check_kv_after(run)
    finally:
        run.close()


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_small_equals_persistent_within_tolerance(hd):
    """The same inputs through the small kernel (default policy) and the
    persistent kernel (a fixed policy of one-tile chunks, several splits):
    outputs within tolerance, written K and V rows bit-identical (the same
    vector routines form them)."""
    w = _wl(hd, 4, 40 + hd // 64, sinks=True, nkv=3)
    a, b = DeviceRun(w), DeviceRun(w, split=(4096 // hd, 8))
    try:
        assert _is_small(a.kv, w.B) and not _is_small(b.kv, w.B)
        oa, ob = a.step(0), b.step(0)
        torch.cuda.synchronize()
        assert a.status() == 0 and b.status() == 0
        assert_close(oa.cpu().numpy(), ob.cpu().numpy(), f"small vs persistent hd={hd}")
        assert torch.equal(a.K, b.K) and torch.equal(a.V, b.V)
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("name", ["vnorm", "plus_one", "both"])
def test_small_options_match_oracle(name):
    gflags, oflags = {"vnorm": (skv.OPT_VNORM, oracle.VNORM),
                      "plus_one": (skv.OPT_NORM_PLUS_ONE, oracle.NORM_PLUS_ONE),
                      "both": (skv.OPT_VNORM | skv.OPT_NORM_PLUS_ONE,
                               oracle.VNORM | oracle.NORM_PLUS_ONE)}[name]
    w = _wl(128, 3, 50 + ["vnorm", "plus_one", "both"].index(name))
    run = DeviceRun(w)
    try:
        run.kv.set_options(gflags)
        assert _is_small(run.kv, w.B)
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.status() == 0
        ref, Kr, Vr = oracle_rows(w, range(w.B), flags=oflags)
        assert_close(out.cpu().numpy(), ref[0], f"small out {name}")
        pos = w.positions(0)
        for b in range(w.B):
            s, p = int(run.slots_np[b]), int(pos[b])
            assert_close(run.K[s, p].cpu().numpy(), Kr[b, p], f"written K {name}")
            assert_close(run.V[s, p].cpu().numpy(), Vr[b, p], f"written V {name}")
    finally:
        run.close()


def test_small_out_of_range_rows_are_skipped_and_flagged():
    w = _wl(64, 4, 60)
    run = DeviceRun(w)
    try:
        assert _is_small(run.kv, w.B)
        q, kn, vn, pos = run.inputs(0)
        pos = pos.copy()
        slots = run.slots_np.copy()
        pos[1] = w.slot_ctx                 # position out of range
        slots[4] = w.n_slots                # slot out of range
        bad = [1, 4]
        good = [b for b in range(w.B) if b not in bad]
        K0 = run.K.clone()
        out = torch.full((w.B, w.n_head, w.head_dim), 7.0, device="cuda")
        run.kv.decode_batch_attn(to_dev(q), to_dev(kn), to_dev(vn), to_dev(pos.astype(np.int32)),
                                 to_dev(slots.astype(np.int32)), run.qw, run.kw, run.inv,
                                 run.sinks, out, w.eps, w.scale)
        torch.cuda.synchronize()
        assert run.status() == skv.DEV_RANGE
        got = out.cpu().numpy()
        assert np.all(got[bad] == 7.0)
        ref, _, _ = oracle_rows(w, good)
        assert_close(got[good], ref[0], "in-range rows")
        changed = torch.nonzero((run.K != K0).any(-1).any(-1)).cpu().numpy().tolist()
        assert sorted(changed) == sorted([int(slots[b]), int(pos[b])] for b in good)
    finally:
        run.close()


def test_small_stale_history_is_never_read():
    """NaN in every slot position after each row's pos changes no bit."""
    w = _wl(128, 4, 61, sinks=False)
    run = DeviceRun(w)
    try:
        K0, V0 = run.K.clone(), run.V.clone()
        a = run.step(0).cpu()
        run.K.copy_(K0)
        run.V.copy_(V0)
        pos = w.positions(0)
        for b in range(w.B):
            s = int(run.slots_np[b])
            run.K[s, pos[b] + 1:] = float("nan")
            run.V[s, pos[b] + 1:] = float("nan")
        assert torch.equal(a, run.step(0).cpu())
        assert run.status() == 0
    finally:
        run.close()


def test_small_rows_are_independent_bit_exact():
    """Every call here takes the small kernel: a B-row call equals B one-row
    calls bit for bit, and permuting rows permutes outputs."""
    w = _wl(256, 2, 62)
    run = DeviceRun(w)
    try:
        q, kn, vn, pos = run.inputs(0)
        K0, V0 = run.K.clone(), run.V.clone()
        full = run.step(0).cpu()
        Kfull, Vfull = run.K.clone(), run.V.clone()
        run.K.copy_(K0)
        run.V.copy_(V0)
        for b in range(w.B):
            out1 = torch.full((1, w.n_head, w.head_dim), float("nan"), device="cuda")
            run.kv.decode_batch_attn(to_dev(q[b:b + 1]), to_dev(kn[b:b + 1]),
                                     to_dev(vn[b:b + 1]), to_dev(pos[b:b + 1].astype(np.int32)),
                                     run.slots[b:b + 1].contiguous(), run.qw, run.kw, run.inv,
                                     run.sinks, out1, w.eps, w.scale)
            assert torch.equal(out1.cpu()[0], full[b]), f"row {b} differs alone"
        assert torch.equal(run.K, Kfull) and torch.equal(run.V, Vfull)
        perm = np.random.default_rng(62).permutation(w.B)
        run.K.copy_(K0)
        run.V.copy_(V0)
        outp = torch.full_like(full.cuda(), float("nan"))
        run.kv.decode_batch_attn(to_dev(q[perm]), to_dev(kn[perm]), to_dev(vn[perm]),
                                 to_dev(pos[perm].astype(np.int32)),
                                 to_dev(run.slots_np[perm].astype(np.int32)), run.qw, run.kw,
                                 run.inv, run.sinks, outp, w.eps, w.scale)
        assert torch.equal(outp.cpu(), full[perm])
        assert run.status() == 0
    finally:
        run.close()


def test_small_host_entry_equals_device_entry():
    w = _wl(64, 8, 63)
    run = DeviceRun(w)
    try:
        K0, V0 = run.K.clone(), run.V.clone()
        dev = run.step(0).cpu()
        Kd, Vd = run.K.clone(), run.V.clone()
        run.K.copy_(K0)
        run.V.copy_(V0)
        q, kn, vn, pos = run.inputs(0)
        h = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        out_h = h(np.full((w.B, w.n_head, w.head_dim), np.nan, dtype=np.float32))
        run.kv.decode_batch_attn_host(h(q), h(kn), h(vn), h(pos.astype(np.int32)),
                                      h(run.slots_np.astype(np.int32)), run.qw, run.kw,
                                      run.inv, run.sinks, out_h, w.eps, w.scale)
        assert torch.equal(out_h, dev)
        assert torch.equal(run.K, Kd) and torch.equal(run.V, Vd)
        assert run.status() == 0
    finally:
        run.close()


def test_small_path_limits():
    """The small kernel up to its limits -- (row, kv head) pairs filling two
    CTAs per SM, a slot of exactly eight tiles -- and the persistent kernel
    one step past each limit; both against the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nkv, hd = 8, 128
    T = 4096 // hd
    rng = np.random.default_rng(64)
    for B, ctx, small in ((2 * sms // nkv, 8 * T, True), (2 * sms // nkv + 1, 8 * T, False),
                          (4, 8 * T + 1, False)):
        pos = tuple(int(x) for x in rng.integers(0, ctx, size=B))
        w = synth.Workload(f"small_lim{B}_{ctx}", 964, B=B, n_slots=B + 1, slot_ctx=ctx,
                           n_head=4 * nkv, n_kv_head=nkv, head_dim=hd, theta=1e6, sinks=True,
                           pos_rule="fixed", fixed_positions=pos, slot_rule="perm")
        run = DeviceRun(w)
        try:
            assert _is_small(run.kv, B) == small, (B, ctx)
            out = run.step(0)
            torch.cuda.synchronize()
            assert run.status() == 0
            ref, _, _ = oracle_rows(w, range(B))
            assert_close(out.cpu().numpy(), ref[0], f"B={B} ctx={ctx}")
        finally:
            run.close()


def test_small_paged_equals_slot_bit_for_bit():
    """One-tile blocks, eight per table: the paged call takes the small
    kernel as the slot call does and gives the same bits, and the pool read
    back in slot order equals the slot buffers."""
    from test_gpu_paged import PagedRun
    w = _wl(128, 4, 65, nkv=2)
    bs = 4096 // 128
    run_s, run_p = DeviceRun(w), PagedRun(w, bs)
    try:
        assert _is_small(run_s.kv, w.B)
        assert _is_small(run_p.kv, w.B, bt_stride=w.slot_ctx // bs)
        out_s, out_p = run_s.step(0), run_p.step(0)
        torch.cuda.synchronize()
        assert run_s.status() == 0 and run_p.kv.get_status() == 0
        assert torch.equal(out_s, out_p)
        shape = run_s.K.shape
        assert torch.equal(run_p.K[run_p.perm].view(shape), run_s.K)
        assert torch.equal(run_p.V[run_p.perm].view(shape), run_s.V)
    finally:
        run_s.close()
        run_p.close()


def test_small_paged_bad_tables_are_skipped_and_flagged():
    """A used table entry outside the pool, or a pos past the table: the row
    is skipped (out untouched, nothing written) and the range flag raised;
    an out-of-pool id in an entry the row does not use is never read."""
    from test_gpu_paged import PagedRun, check_pool, host_pool, oracle_paged, written_mask
    w = _wl(64, 2, 66, nkv=2)
    bs = 4096 // 64
    run = PagedRun(w, bs)
    try:
        pos = w.positions(0)
        tabs = run.tables_np.copy()
        nb = np.uint32(run.n_blocks)
        b_last = int(np.argmax(pos))
        b_mid = [b for b in range(w.B) if bs < int(pos[b]) < 3 * bs][0]
        b_short = [b for b in range(w.B) if int(pos[b]) < bs][1]
        tabs[b_last, int(pos[b_last]) // bs] = nb          # the block holding key p
        tabs[b_mid, 0] = nb + 3                             # a history block
        tabs[b_short, -1] = 0xFFFFFFFF                      # an entry never used
        bad = sorted([b_last, b_mid])
        good = [b for b in range(w.B) if b not in bad]
        assert _is_small(run.kv, w.B, bt_stride=tabs.shape[1])
        out = run.step(0, tables=to_dev(tabs.astype(np.int32)))
        torch.cuda.synchronize()
        assert run.kv.get_status() == skv.DEV_RANGE
        got = out.cpu().numpy()
        assert np.all(np.isnan(got[bad]))
        Kr, Vr = host_pool(w, bs)
        ref, skipped = oracle_paged(w, bs, Kr, Vr, tabs)
        assert skipped == len(bad)
        assert_close(got[good], ref[good], "paged rows beside skipped rows")
        check_pool(run, Kr, Vr, written_mask(run, tabs, pos, rows=good))
    finally:
        run.close()


def test_small_repeated_calls_are_identical():
    w = _wl(128, 8, 67)
    run = DeviceRun(w)
    try:
        outs = [run.step(0).cpu() for _ in range(3)]
        assert all(torch.equal(o, outs[0]) for o in outs[1:])
        assert run.status() == 0
    finally:
        run.close()

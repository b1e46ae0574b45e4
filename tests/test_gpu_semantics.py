"""Properties of the CUDA path that hold at any size: slot addressing and
non-overlap, batch and permutation invariance, stale history, precondition
violations, the host-pointer entry, reset, repeatability."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import sequence_slot_kv_gb300 as skv
import synth
from gpu_harness import DeviceRun, assert_close, check_kv_after, oracle_rows, to_dev

pytestmark = pytest.mark.gpu


def _wl(B=8, slot_ctx=700, hd=128, G=4, sinks=True, idx=300):
    rng = np.random.default_rng(idx)
    pos = tuple(int(x) for x in rng.integers(0, slot_ctx, size=B))
    return synth.Workload(f"sem{idx}", idx, B=B, n_slots=B + 4, slot_ctx=slot_ctx,
                          n_head=2 * G, n_kv_head=2, head_dim=hd, theta=10000.0,
                          sinks=sinks, pos_rule="fixed", fixed_positions=pos,
                          slot_rule="perm")


def test_slot_kv_smoke_offsets_and_no_overlap():
    """The pages' slotKvSmoke: a sentinel at (slot 0, pos 0) and a pattern at
    the last (slot, pos) of K, read back; neither clobbers the other.  The
    offsets agree with the oracle's everywhere we look."""
    n_slots, ctx, nkv, hd = 5, 37, 3, 64
    kv = skv.SlotKV(n_slots, ctx, nkv, hd, max_rows=4, max_n_head=nkv)
    try:
        K, V = kv.kv_tensors()
        assert torch.count_nonzero(K) == 0 and torch.count_nonzero(V) == 0
        o = oracle.default()
        for s, p in ((0, 0), (1, 3), (4, 36), (2, 17)):
            assert kv.offset_bytes(s, p) == o.offset_bytes(s, p, ctx, nkv * hd)
        assert kv.offset_bytes(n_slots, 0) is None and kv.offset_bytes(0, ctx) is None
        row = nkv * hd
        flatK = K.view(-1)
        first = kv.offset_bytes(0, 0) // 4
        last = kv.offset_bytes(n_slots - 1, ctx - 1) // 4
        flatK[first: first + row] = 1234.5
        flatK[last: last + row] = torch.arange(row, dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        assert torch.all(flatK[first: first + row] == 1234.5)
        assert torch.equal(flatK[last: last + row], torch.arange(row, dtype=torch.float32,
                                                                  device="cuda"))
        assert last + row == flatK.numel()
        assert torch.count_nonzero(flatK[first + row: last]) == 0
    finally:
        kv.free()


@pytest.mark.parametrize("split", [(512, 64), (32, 8)])
def test_rows_are_independent_bit_exact(split):
    """Under a fixed split policy one B-row call equals B one-row calls bit
    for bit (the split depends on the row's own position only), and
    permuting rows permutes outputs."""
    w = _wl()
    run = DeviceRun(w, split=split)
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
        perm = np.array([3, 0, 7, 1, 6, 2, 5, 4])
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


def test_default_policy_batch_and_alone():
    """The default policy sizes chunks from the batch's shape: a 64-row batch
    (8 kv heads, 4096-key slots) runs larger chunks than one row alone.  Each
    row alone then agrees with its row of the batch within tolerance, and a
    permutation of the batch (same size, same chunks) permutes the outputs
    bit for bit."""
    B = 64
    rng = np.random.default_rng(310)
    pos = tuple(int(x) for x in rng.integers(0, 4096, size=B))
    w = synth.Workload("sem_auto", 310, B=B, n_slots=B, slot_ctx=4096, n_head=32, n_kv_head=8,
                       head_dim=128, theta=1e6, sinks=True, pos_rule="fixed",
                       fixed_positions=pos, slot_rule="perm")
    run = DeviceRun(w)
    try:
        q, kn, vn, p = run.inputs(0)
        K0, V0 = run.K.clone(), run.V.clone()
        full = run.step(0).cpu()
        rows = [int(np.argmax(p)), int(np.argmin(p)), 5, 17, 40]
        for b in rows:
            run.K.copy_(K0)
            run.V.copy_(V0)
            out1 = torch.full((1, w.n_head, w.head_dim), float("nan"), device="cuda")
            run.kv.decode_batch_attn(to_dev(q[b:b + 1]), to_dev(kn[b:b + 1]),
                                     to_dev(vn[b:b + 1]), to_dev(p[b:b + 1].astype(np.int32)),
                                     run.slots[b:b + 1].contiguous(), run.qw, run.kw, run.inv,
                                     run.sinks, out1, w.eps, w.scale)
            assert_close(out1.cpu().numpy()[0], full[b].numpy(), f"row {b} alone")
        perm = rng.permutation(B)
        run.K.copy_(K0)
        run.V.copy_(V0)
        outp = torch.full_like(full.cuda(), float("nan"))
        run.kv.decode_batch_attn(to_dev(q[perm]), to_dev(kn[perm]), to_dev(vn[perm]),
                                 to_dev(p[perm].astype(np.int32)),
                                 to_dev(run.slots_np[perm].astype(np.int32)), run.qw, run.kw,
                                 run.inv, run.sinks, outp, w.eps, w.scale)
        assert torch.equal(outp.cpu(), full[perm])
        assert run.status() == 0
    finally:
        run.close()


@pytest.mark.parametrize("layout", ["slots", "paged"])
def test_many_rows(layout):
    """3000 rows with short, mixed contexts: the plan kernel takes rows in
    rounds of 1024 threads, so its later rounds (which re-read each row) and
    many more items than CTAs run; every row against the oracle, every
    written row, every other byte."""
    B = 3000
    w = synth.Workload("many_rows", 330, B=B, n_slots=B + 16, slot_ctx=192, n_head=4,
                       n_kv_head=2, head_dim=64, theta=1e4, sinks=True, slot_rule="perm")
    if layout == "slots":
        run = DeviceRun(w)
        try:
            out = run.step(0)
            torch.cuda.synchronize()
            assert run.status() == 0
            ref, _, _ = oracle_rows(w, range(B), n_threads=32)
            assert_close(out.cpu().numpy(), ref[0], "3000 rows")
            check_kv_after(run)
        finally:
            run.close()
        return
    from test_gpu_paged import PagedRun, check_pool, host_pool, oracle_paged, written_mask
    run = PagedRun(w, 64)
    try:
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.kv.get_status() == 0
        Kr, Vr = host_pool(w, 64)
        ref, skipped = oracle_paged(w, 64, Kr, Vr, run.tables_np)
        assert skipped == 0
        assert_close(out.cpu().numpy(), ref, "3000 paged rows")
        check_pool(run, Kr, Vr, written_mask(run, run.tables_np, w.positions(0)))
    finally:
        run.close()


def test_maximum_rows():
    """65535 rows, the most a call takes: the plan kernel's 64 rounds, row
    indices in all 16 bits of a work record; sampled rows against the oracle,
    every written row, every other byte."""
    B = 65535
    w = synth.Workload("max_rows", 331, B=B, n_slots=B, slot_ctx=64, n_head=1, n_kv_head=1,
                       head_dim=64, theta=1e4, sinks=False, slot_rule="perm")
    run = DeviceRun(w)
    try:
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.status() == 0
        rng = np.random.default_rng(331)
        rows = sorted({0, 1, 1023, 1024, 32767, 32768, B - 2, B - 1}
                      | set(int(r) for r in rng.choice(B, size=400, replace=False)))
        ref, _, _ = oracle_rows(w, rows, n_threads=32)
        assert_close(out.cpu().numpy()[rows], ref[0], "sampled rows of 65535")
        check_kv_after(run)
    finally:
        run.close()


def test_maximum_splits():
    """256 splits, the most a row can have (split indices in all 8 bits of a
    work record): a fixed policy of one tile per split and rows at 256, 255
    and fewer tiles."""
    hd = 64
    T = 4096 // hd
    ctx = 256 * T
    pos = (ctx - 1, ctx - T - 1, ctx - T, 255 * T - 1, 100 * T + 3, T - 1, 0)
    w = synth.Workload("max_splits", 332, B=len(pos), n_slots=len(pos) + 1, slot_ctx=ctx,
                       n_head=2, n_kv_head=1, head_dim=hd, theta=1e4, sinks=True,
                       pos_rule="fixed", fixed_positions=pos, slot_rule="perm")
    run = DeviceRun(w, split=(T, 256))
    try:
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.status() == 0
        ref, _, _ = oracle_rows(w, range(w.B))
        assert_close(out.cpu().numpy(), ref[0], "256 splits")
        check_kv_after(run)
    finally:
        run.close()


def test_maximum_kv_heads():
    """256 kv heads, the most a handle takes (kv head indices in all 8 bits
    of a work record), one query head each."""
    w = synth.Workload("max_kvh", 333, B=3, n_slots=4, slot_ctx=200, n_head=256, n_kv_head=256,
                       head_dim=64, theta=1e4, sinks=True, pos_rule="fixed",
                       fixed_positions=(199, 64, 0), slot_rule="perm")
    run = DeviceRun(w)
    try:
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.status() == 0
        ref, _, _ = oracle_rows(w, range(w.B))
        assert_close(out.cpu().numpy(), ref[0], "256 kv heads")
        check_kv_after(run)
    finally:
        run.close()


def test_call_shape():
    """slot_kv_call_shape reports what a call launches: the decode kernel
    alone when every item is a CTA's first item (a few short rows), with the
    plan kernel otherwise, plus the KV-write kernel for prefill; and the
    fixed policy's chunk once slot_kv_set_split is called."""
    tiny = synth.WORKLOADS["tiny"]
    run = DeviceRun(tiny)
    try:
        chunk, ctas, kernels = run.kv.call_shape(tiny.B)
        assert kernels == 1 and ctas == tiny.B * tiny.n_kv_head
        # head dim 64 prefills on the tensor cores: prep, plan, attention
        assert run.kv.call_shape(tiny.B, prefill=True)[2] == 3
        run.kv.set_split(64, 8)
        assert run.kv.call_shape(tiny.B)[0] == 64
    finally:
        run.close()
    mid = synth.WORKLOADS["mid"].replace(n_slots=40, B=32)
    kv = skv.SlotKV(mid.n_slots, mid.slot_ctx, mid.n_kv_head, mid.head_dim, mid.B, mid.n_head)
    try:
        chunk, ctas, kernels = kv.call_shape(mid.B)
        assert kernels == 2 and chunk % (4096 // mid.head_dim) == 0
        assert kv.call_shape(mid.B, prefill=True)[2] == 3
        with pytest.raises(skv.SlotKVError):
            kv.call_shape(0)
    finally:
        kv.free()


@pytest.mark.parametrize("split", [None, (64, 16)])
def test_spare_ctas_start_on_second_splits(split):
    """With fewer (row, kv head) pairs than persistent CTAs, the CTAs past
    the pairs start on split 1 of the first pairs: rows with one split, a
    row out of range and a row whose kv heads straddle the end of that range
    all come out as the oracle says, and the other rows too."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nkv, hd = 7, 64
    B = (2 * sms - 24) // nkv          # 24 CTAs to spare: 3 rows and 3 kv heads
    rng = np.random.default_rng(311)
    pos = rng.integers(0, 2500, size=B)
    pos[0], pos[2], pos[3], pos[4] = 5, 2499, 1024, 1023   # 1024 keys: one default chunk
    w = synth.Workload("sem311", 311, B=B, n_slots=B + 3, slot_ctx=2500, n_head=2 * nkv,
                       n_kv_head=nkv, head_dim=hd, theta=1e4, sinks=True, pos_rule="fixed",
                       fixed_positions=tuple(int(x) for x in pos), slot_rule="perm")
    run = DeviceRun(w, split=split)
    try:
        chunk, ctas, kernels = run.kv.call_shape(B)
        assert kernels == 2 and ctas == 2 * sms > B * nkv
        q, kn, vn, p = run.inputs(0)
        slots = run.slots_np.copy()
        slots[1] = w.n_slots + 1            # out of range, among the second splits
        out = torch.full((B, w.n_head, hd), 7.0, device="cuda")
        run.kv.decode_batch_attn(to_dev(q), to_dev(kn), to_dev(vn), to_dev(p.astype(np.int32)),
                                 to_dev(slots.astype(np.int32)), run.qw, run.kw, run.inv,
                                 run.sinks, out, w.eps, w.scale)
        torch.cuda.synchronize()
        assert run.status() == skv.DEV_RANGE
        got = out.cpu().numpy()
        assert np.all(got[1] == 7.0)
        rows = [b for b in range(B) if b != 1]
        ref, _, _ = oracle_rows(w, rows)
        assert_close(got[rows], ref[0], "rows")
    finally:
        run.close()


def test_stale_history_is_never_read():
    """NaN in every position after pos of each row's slot changes nothing."""
    w = _wl(sinks=False, idx=301)
    run = DeviceRun(w)
    try:
        K0, V0 = run.K.clone(), run.V.clone()
        a = run.step(0).cpu()
        run.K.copy_(K0)
        run.V.copy_(V0)
        pos = w.positions0()
        for b in range(w.B):
            s = int(run.slots_np[b])
            run.K[s, pos[b] + 1:] = float("nan")
            run.V[s, pos[b] + 1:] = float("nan")
        b_ = run.step(0).cpu()
        assert torch.equal(a, b_)
    finally:
        run.close()


def test_out_of_range_rows_are_skipped_and_flagged():
    w = _wl(B=4, idx=302)
    run = DeviceRun(w)
    try:
        q, kn, vn, pos = run.inputs(0)
        pos = pos.copy()
        slots = run.slots_np.copy()
        pos[1] = w.slot_ctx                 # position out of range
        slots[2] = w.n_slots + 7            # slot out of range
        K0, V0 = run.K.clone(), run.V.clone()
        out = torch.full((w.B, w.n_head, w.head_dim), 7.0, device="cuda")
        run.kv.decode_batch_attn(to_dev(q), to_dev(kn), to_dev(vn), to_dev(pos.astype(np.int32)),
                                 to_dev(slots.astype(np.int32)), run.qw, run.kw, run.inv,
                                 run.sinks, out, w.eps, w.scale)
        torch.cuda.synchronize()
        assert run.status() & skv.DEV_RANGE
        assert run.status() == 0            # read-and-clear
        got = out.cpu().numpy()
        assert np.all(got[1] == 7.0) and np.all(got[2] == 7.0)
        ref, _, _ = oracle_rows(w, [0, 3])
        assert_close(got[[0, 3]], ref[0], "in-range rows")
        # only rows 0 and 3 wrote
        changed = torch.nonzero((run.K != K0).any(-1).any(-1)).cpu().numpy().tolist()
        want = sorted([[int(slots[b]), int(pos[b])] for b in (0, 3)])
        assert sorted(changed) == want
    finally:
        run.close()


def test_zero_rows_is_a_no_op():
    w = _wl(B=2, idx=303)
    run = DeviceRun(w)
    try:
        e = torch.empty(0, device="cuda")
        rc = skv._lib.decode_batch_attn(run.kv._h, 0, w.n_head, e.data_ptr(), e.data_ptr(),
                                        e.data_ptr(), e.data_ptr(), e.data_ptr(),
                                        run.qw.data_ptr(), run.kw.data_ptr(), run.inv.data_ptr(),
                                        None, e.data_ptr(), w.eps, w.scale, None)
        assert rc == 0
    finally:
        run.close()


def _host_tensor(a, kind):
    """A host copy of array a: pinned, pageable, or pinned but starting one
    element into its allocation (4-byte aligned only)."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    if kind == "pageable":
        return t.clone()
    if kind == "pinned":
        return t.pin_memory()
    buf = torch.empty(t.numel() + 1, dtype=t.dtype).pin_memory()
    view = buf[1:].view(t.shape)
    view.copy_(t)
    return view


@pytest.mark.parametrize("kind", ["pinned", "pageable", "pinned_offset"])
def test_host_entry_equals_device_entry(kind):
    """decode_batch_attn_host equals the device entry bit for bit, whether
    its buffers are pinned (gathered and returned by copy kernels over the
    host link), pageable (copy-engine transfers), or pinned at an address
    that allows only 4-byte accesses."""
    w = _wl(idx=304)
    run = DeviceRun(w)
    try:
        K0, V0 = run.K.clone(), run.V.clone()
        dev = run.step(0).cpu()
        Kd, Vd = run.K.clone(), run.V.clone()
        for rep in range(2):
            run.K.copy_(K0)
            run.V.copy_(V0)
            q, kn, vn, pos = run.inputs(0)
            h = lambda a: _host_tensor(a, kind)  # noqa: E731
            out_h = h(np.full((w.B, w.n_head, w.head_dim), np.nan, dtype=np.float32))
            run.kv.decode_batch_attn_host(h(q), h(kn), h(vn), h(pos.astype(np.int32)),
                                          h(run.slots_np.astype(np.int32)), run.qw, run.kw,
                                          run.inv, run.sinks, out_h, w.eps, w.scale)
            assert torch.equal(out_h, dev), f"{kind} call {rep}"
            assert torch.equal(run.K, Kd) and torch.equal(run.V, Vd)
        assert run.status() == 0
    finally:
        run.close()


def test_reset_zeroes_exactly_one_slot():
    w = _wl(B=2, idx=305)
    run = DeviceRun(w)
    try:
        K0 = run.K.clone()
        run.kv.reset(3)
        torch.cuda.synchronize()
        assert torch.count_nonzero(run.K[3]) == 0 and torch.count_nonzero(run.V[3]) == 0
        keep = [s for s in range(w.n_slots) if s != 3]
        assert torch.equal(run.K[keep], K0[keep])
    finally:
        run.close()


@pytest.mark.parametrize("split", [None, (32, 16)])
def test_repeated_calls_are_identical(split):
    """Re-running a step at the same positions rewrites the same bytes and
    gives the same output (the merge counters reset themselves)."""
    w = _wl(idx=306, slot_ctx=3000)
    run = DeviceRun(w, split=split)
    try:
        outs = [run.step(0).cpu() for _ in range(4)]
        for o in outs[1:]:
            assert torch.equal(o, outs[0])
        assert run.status() == 0
    finally:
        run.close()


def test_argument_errors():
    w = _wl(B=2, idx=307)
    run = DeviceRun(w)
    try:
        q, kn, vn, pos = run.inputs(0)
        out = torch.empty((w.B, w.n_head, w.head_dim), device="cuda")
        with pytest.raises(skv.SlotKVError) as ei:      # B > max_rows
            big = [to_dev(np.concatenate([a] * 3)) for a in (q, kn, vn, pos.astype(np.int32))]
            run.kv.decode_batch_attn(*big, run.slots.repeat(3), run.qw, run.kw, run.inv, None,
                                     torch.empty((3 * w.B, w.n_head, w.head_dim), device="cuda"),
                                     w.eps, w.scale)
        assert ei.value.code == 1
        with pytest.raises(skv.SlotKVError):            # null output
            rc = skv._lib.decode_batch_attn(run.kv._h, w.B, w.n_head, 1, 1, 1, 1, 1, 1, 1, 1,
                                            None, None, w.eps, w.scale, None)
            skv._check(rc, "decode_batch_attn")
        # a q, k_new, v_new or out that is not 16-byte aligned is refused on
        # the host (the kernel's bulk copies and 16-byte stores need it)
        def misaligned(a):
            base = torch.empty(a.size + 4, dtype=torch.float32, device="cuda")
            view = base[1:1 + a.size].view(a.shape)
            view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
            return view
        args = [to_dev(q), to_dev(kn), to_dev(vn), to_dev(pos.astype(np.int32)), run.slots,
                run.qw, run.kw, run.inv, None, out, w.eps, w.scale]
        for i, a in ((0, q), (1, kn), (2, vn), (9, np.zeros(out.shape, np.float32))):
            bad = list(args)
            bad[i] = misaligned(a)
            with pytest.raises(skv.SlotKVError) as ei:
                run.kv.decode_batch_attn(*bad)
            assert ei.value.code == 1 and "aligned" in str(ei.value)
        with pytest.raises(skv.SlotKVError) as ei:
            skv.decode_batch_attn_noalloc(run.K, run.V, misaligned(q), to_dev(kn), to_dev(vn),
                                          to_dev(pos.astype(np.int32)), run.slots, run.qw,
                                          run.kw, run.inv, None, out, w.eps, w.scale)
        assert ei.value.code == 1 and "aligned" in str(ei.value)
        # tensors in the wrong place are refused by the binding
        with pytest.raises(ValueError, match="CUDA"):
            run.kv.decode_batch_attn(torch.from_numpy(q), to_dev(kn), to_dev(vn),
                                     to_dev(pos.astype(np.int32)), run.slots, run.qw, run.kw,
                                     run.inv, None, out, w.eps, w.scale)
        with pytest.raises(ValueError, match="CPU"):
            run.kv.decode_batch_attn_host(to_dev(q), torch.from_numpy(kn), torch.from_numpy(vn),
                                          torch.from_numpy(pos.astype(np.int32)),
                                          torch.from_numpy(run.slots_np.astype(np.int32)),
                                          run.qw, run.kw, run.inv, None,
                                          torch.empty(out.shape), w.eps, w.scale)
        with pytest.raises(skv.SlotKVError):
            run.kv.set_split(5, 8)                       # not a multiple of the tile
        h = ctypes.c_void_p()
        rc = skv._lib.slot_kv_alloc(ctypes.byref(h), 4, 16, 2, 96, None, None, 2, 2)
        assert rc == 3 and not h.value                   # head_dim 96 unsupported
    finally:
        run.close()


def test_realloc_frees_first():
    """slot_kv_alloc on a live handle frees it and allocates anew (the pages'
    allocSlotKv is re-callable)."""
    h = ctypes.c_void_p()
    assert skv._lib.slot_kv_alloc(ctypes.byref(h), 4, 64, 2, 64, None, None, 4, 8) == 0
    first = h.value
    assert skv._lib.slot_kv_alloc(ctypes.byref(h), 8, 32, 2, 128, None, None, 4, 8) == 0
    assert h.value
    ctx = ctypes.c_uint32()
    hd = ctypes.c_uint32()
    assert skv._lib.slot_kv_geometry(h, None, ctypes.byref(ctx), None, ctypes.byref(hd),
                                     None, None) == 0
    assert (ctx.value, hd.value) == (32, 128)
    assert skv._lib.slot_kv_free(h) == 0
    del first

"""Prepared host calls (slot_kv_host_call_create / _run / _free): a serving
loop's step with its inputs and output in host memory ("Forward Cuda
Gemma", decodeBatch), its arguments checked and its pinned buffers resolved
once.  Each run must equal the host entry with the same arguments bit for
bit (the same kernels run) -- slot and paged, pinned and pageable, the
persistent and the small-call kernel -- on whatever the buffers hold when it
runs; and a call whose handle was freed is refused."""
import numpy as np
import pytest
import torch

import sequence_slot_kv_gb300 as skv
import synth
from gpu_harness import DeviceRun, assert_close, oracle_rows, to_dev

pytestmark = pytest.mark.gpu


def _wl(idx, slot_ctx=700, B=8, hd=128, G=4):
    rng = np.random.default_rng(idx)
    pos = tuple(int(x) for x in rng.integers(0, slot_ctx - 4, size=B))
    return synth.Workload(f"hostcall{idx}", idx, B=B, n_slots=B + 3, slot_ctx=slot_ctx,
                          n_head=2 * G, n_kv_head=2, head_dim=hd, theta=1e4, sinks=True,
                          pos_rule="fixed", fixed_positions=pos, slot_rule="perm")


def _host(a, pinned):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pinned else t.clone()


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("shape", ["persistent", "small"])
def test_host_call_equals_host_entry(pinned, shape):
    """Three steps at advancing positions, the same host buffers refilled in
    place before each run: every output and the final K/V equal the host
    entry's bit for bit, and the outputs match the oracle."""
    w = _wl(1100 + (shape == "small"), slot_ctx=700 if shape == "persistent" else 256)
    ref, run = DeviceRun(w), DeviceRun(w)
    try:
        hq = _host(w.q(0), pinned)
        hk = _host(w.k_new(0), pinned)
        hv = _host(w.v_new(0), pinned)
        hp = _host(w.positions(0).astype(np.int32), pinned)
        hs = _host(run.slots_np.astype(np.int32), pinned)
        hout = _host(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32), pinned)
        call = run.kv.prepare_host_call(hq, hk, hv, hp, hs, run.qw, run.kw, run.inv, run.sinks,
                                        hout, w.eps, w.scale)
        for t in range(3):
            q, kn, vn, pos = w.q(t), w.k_new(t), w.v_new(t), w.positions(t).astype(np.int32)
            for dst, src in ((hq, q), (hk, kn), (hv, vn), (hp, pos)):
                dst.copy_(torch.from_numpy(src))
            got = call().clone()
            want = _host(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32), pinned)
            ref.kv.decode_batch_attn_host(_host(q, pinned), _host(kn, pinned), _host(vn, pinned),
                                          _host(pos, pinned), hs, ref.qw, ref.kw, ref.inv,
                                          ref.sinks, want, w.eps, w.scale)
            assert torch.equal(got, want), f"step {t}"
        assert torch.equal(run.K, ref.K) and torch.equal(run.V, ref.V)
        assert run.status() == 0 and ref.status() == 0
        oref, _, _ = oracle_rows(w, range(w.B), steps=3)
        assert_close(got.numpy(), oref[2], "last step vs the oracle")
        call.free()
    finally:
        ref.close()
        run.close()


def test_paged_host_call_equals_paged_host_entry():
    from test_gpu_paged import PagedRun, small_paged_workload
    w, bs = small_paged_workload(128, 4, 1, 60, sinks=True)
    ref, run = PagedRun(w, bs), PagedRun(w, bs)
    try:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        hq, hk, hv = pin(w.q(0)), pin(w.k_new(0)), pin(w.v_new(0))
        hp, ht = pin(w.positions(0).astype(np.int32)), pin(run.tables_np.astype(np.int32))
        hout = pin(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32))
        call = run.kv.prepare_host_call(hq, hk, hv, hp, None, run.qw, run.kw, run.inv,
                                        run.sinks, hout, w.eps, w.scale, block_tables=ht)
        got = call().clone()
        want = pin(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32))
        ref.kv.decode_batch_attn_paged_host(hq, hk, hv, hp, ht, ref.qw, ref.kw, ref.inv,
                                            ref.sinks, want, w.eps, w.scale)
        assert torch.equal(got, want)
        assert torch.equal(run.K, ref.K) and torch.equal(run.V, ref.V)
        assert run.kv.get_status() == 0 and ref.kv.get_status() == 0
        call.free()
    finally:
        ref.close()
        run.close()


def test_host_call_refused_after_its_handle_is_freed():
    w = _wl(1110, B=2)
    run = DeviceRun(w)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    hout = pin(np.zeros((w.B, w.n_head, w.head_dim), np.float32))
    call = run.kv.prepare_host_call(pin(w.q(0)), pin(w.k_new(0)), pin(w.v_new(0)),
                                    pin(w.positions(0).astype(np.int32)),
                                    pin(run.slots_np.astype(np.int32)), run.qw, run.kw, run.inv,
                                    run.sinks, hout, w.eps, w.scale)
    call()
    run.close()
    with pytest.raises(skv.SlotKVError) as e:
        call()
    assert e.value.code == 4
    call.free()


def test_host_call_argument_errors():
    w = _wl(1111, B=2)
    run = DeviceRun(w)
    try:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        hq, hk, hv = pin(w.q(0)), pin(w.k_new(0)), pin(w.v_new(0))
        hp, hs = pin(w.positions(0).astype(np.int32)), pin(run.slots_np.astype(np.int32))
        bad_out = pin(np.zeros((w.B, w.n_head + 1, w.head_dim), np.float32))
        with pytest.raises(ValueError):
            run.kv.prepare_host_call(hq, hk, hv, hp, hs, run.qw, run.kw, run.inv, run.sinks,
                                     bad_out, w.eps, w.scale)
        with pytest.raises(ValueError):   # device tensors where host ones are expected
            run.kv.prepare_host_call(to_dev(w.q(0)), hk, hv, hp, hs, run.qw, run.kw, run.inv,
                                     run.sinks, pin(np.zeros((w.B, w.n_head, w.head_dim),
                                                             np.float32)), w.eps, w.scale)
    finally:
        run.close()


def test_enqueued_host_calls_equal_synchronous_runs():
    """Three steps at advancing positions, each a prepared call with buffers
    of its own, enqueued back to back with one synchronisation at the end:
    every output and the final K/V equal three synchronous runs bit for
    bit."""
    w = _wl(1120)
    runs = [DeviceRun(w), DeviceRun(w)]
    try:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        outs = {}
        for mode, run in zip(("sync", "enqueue"), runs):
            calls, houts = [], []
            for t in range(3):
                hout = pin(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32))
                calls.append(run.kv.prepare_host_call(
                    pin(w.q(t)), pin(w.k_new(t)), pin(w.v_new(t)),
                    pin(w.positions(t).astype(np.int32)), pin(run.slots_np.astype(np.int32)),
                    run.qw, run.kw, run.inv, run.sinks, hout, w.eps, w.scale))
                houts.append(hout)
            stream = torch.cuda.Stream()
            for c in calls:
                c(stream=stream, sync=(mode == "sync"))
            stream.synchronize()
            outs[mode] = [h.clone() for h in houts]
            for c in calls:
                c.free()
        for t in range(3):
            assert torch.equal(outs["sync"][t], outs["enqueue"][t]), f"step {t}"
        assert torch.equal(runs[0].K, runs[1].K) and torch.equal(runs[0].V, runs[1].V)
        assert runs[0].status() == 0 and runs[1].status() == 0
    finally:
        for r in runs:
            r.close()


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_enqueued_call_twice_in_flight_and_paged(pinned):
    """The same prepared call enqueued twice before one synchronisation (the
    first on an idle stream takes the gather path, the second, with work in
    flight, the copy-engine path; the step is idempotent at the same
    positions) equals one synchronous run; and a paged call enqueued the same
    way equals the paged host entry."""
    from test_gpu_paged import PagedRun, small_paged_workload
    host = lambda a: (torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
                      if pinned else torch.from_numpy(np.ascontiguousarray(a)))
    w = _wl(1130 + pinned)
    a, b = DeviceRun(w), DeviceRun(w)
    try:
        args = lambda r: (host(w.q(0)), host(w.k_new(0)), host(w.v_new(0)),  # noqa: E731
                          host(w.positions(0).astype(np.int32)), host(r.slots_np.astype(np.int32)),
                          r.qw, r.kw, r.inv, r.sinks)
        oa = host(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32))
        ca = a.kv.prepare_host_call(*args(a), oa, w.eps, w.scale)
        ca()
        ob = host(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32))
        cb = b.kv.prepare_host_call(*args(b), ob, w.eps, w.scale)
        stream = torch.cuda.Stream()
        cb(stream=stream, sync=False)
        cb(stream=stream, sync=False)
        stream.synchronize()
        assert torch.equal(oa, ob)
        assert torch.equal(a.K, b.K) and torch.equal(a.V, b.V)
        assert a.status() == 0 and b.status() == 0
        ca.free()
        cb.free()
    finally:
        a.close()
        b.close()
    w, bs = small_paged_workload(128, 4, 1, 61, sinks=True)
    ref, run = PagedRun(w, bs), PagedRun(w, bs)
    try:
        hq, hk, hv = host(w.q(0)), host(w.k_new(0)), host(w.v_new(0))
        hp, ht = host(w.positions(0).astype(np.int32)), host(run.tables_np.astype(np.int32))
        out = host(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32))
        call = run.kv.prepare_host_call(hq, hk, hv, hp, None, run.qw, run.kw, run.inv, run.sinks,
                                        out, w.eps, w.scale, block_tables=ht)
        stream = torch.cuda.Stream()
        call(stream=stream, sync=False)   # an idle stream: the gather path
        call(stream=stream, sync=False)   # work in flight: the copy-engine path
        stream.synchronize()
        want = host(np.full((w.B, w.n_head, w.head_dim), np.nan, np.float32))
        ref.kv.decode_batch_attn_paged_host(hq, hk, hv, hp, ht, ref.qw, ref.kw, ref.inv,
                                            ref.sinks, want, w.eps, w.scale)
        assert torch.equal(out, want)
        assert torch.equal(run.K, ref.K) and torch.equal(run.V, ref.V)
        assert run.kv.get_status() == 0 and ref.kv.get_status() == 0
        call.free()
    finally:
        ref.close()
        run.close()

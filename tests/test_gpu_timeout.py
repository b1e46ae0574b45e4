"""The failure paths of the decode and tensor-core prefill kernels, exercised
without a GPU fault.

Every wait in the kernel is bounded (about a second).  With the test option
SLOTKV_OPT_TEST_STALL no CTA's first item is ever marked ready, so the
consumers' wait on that flag runs out: the kernel must end by itself, report
SLOTKV_DEV_TIMEOUT through slot_kv_get_status, write nothing, and leave the
context and the handle usable for the next call.
"""
import time

import numpy as np
import pytest
import torch

import sequence_slot_kv_gb300 as skv
import synth
from gpu_harness import DeviceRun, assert_close, check_kv_after, oracle_rows

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_recovers():
    w = synth.Workload("timeout", 900, B=6, n_slots=8, slot_ctx=900, n_head=8, n_kv_head=2,
                       head_dim=128, theta=1e4, sinks=True, pos_rule="fixed",
                       fixed_positions=(0, 31, 32, 200, 517, 899), slot_rule="perm")
    run = DeviceRun(w, split=(128, 8))   # several splits per row: merges are pending too
    try:
        K0, V0 = run.K.clone(), run.V.clone()
        run.kv.set_options(skv.OPT_TEST_STALL)
        out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        t0 = time.perf_counter()
        run.step(0, out=out)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        flags = run.status()
        assert flags & skv.DEV_TIMEOUT, flags
        assert elapsed < 30.0
        # nothing was written: the output keeps its fill, the slots their bytes
        assert torch.isnan(out).all()
        assert torch.equal(run.K, K0) and torch.equal(run.V, V0)
        assert run.status() == 0          # the flags were cleared by the read

        # the same handle then runs a normal step correctly
        run.kv.set_options(0)
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.status() == 0
        ref, _, _ = oracle_rows(w, range(w.B))
        assert_close(out.cpu().numpy(), ref[0], "step after a timeout")
        check_kv_after(run)
    finally:
        run.close()


@pytest.mark.parametrize("hd", [64, 128])
def test_prefill_expired_wait_reports_timeout_and_recovers(hd):
    """The tensor-core prefill's failure path: with SLOTKV_OPT_TEST_STALL the
    MMA thread withholds each CTA's first score-ready signal, so the softmax
    warps' bounded wait runs out; both halves of every row leave together,
    the MMA thread's wait for P runs out, the producer's and converters'
    waits run out in turn.  The call must end by itself with
    SLOTKV_DEV_TIMEOUT, write no output, and leave the handle usable: the
    same prefill then matches the oracle."""
    from test_gpu_prefill_tc import _oracle_rows, _workload
    from gpu_harness import to_dev
    G = 4
    slots = np.concatenate([np.full(70, 1, np.uint32), np.full(40, 3, np.uint32)])
    pos = np.concatenate([np.arange(300, 370, dtype=np.uint32),
                          np.arange(0, 40, dtype=np.uint32)])
    w = _workload(hd, G, 2, 70 + hd, len(pos), 5, 380)
    shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    K = torch.empty(shape, device="cuda")
    V = torch.empty(shape, device="cuda")
    w.dev_fill_history(K.data_ptr(), V.data_ptr(), torch.cuda.current_stream().cuda_stream)
    kv = skv.SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head,
                    k_buf=K, v_buf=V)
    try:
        assert kv.call_shape(w.B, prefill=True)[2] == 3
        s = w.sink_logits()
        args = (to_dev(w.q()), to_dev(w.k_new()), to_dev(w.v_new()),
                to_dev(pos.astype(np.int32)), to_dev(slots.astype(np.int32)),
                to_dev(w.q_norm_w()), to_dev(w.k_norm_w()), to_dev(w.inv_freq()),
                None if s is None else to_dev(s))
        kv.set_options(skv.OPT_TEST_STALL)
        out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        t0 = time.perf_counter()
        kv.prefill_batch_attn(*args, out, w.eps, w.scale)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        flags = kv.get_status()
        assert flags & skv.DEV_TIMEOUT, flags
        assert elapsed < 60.0
        assert torch.isnan(out).all()
        assert kv.get_status() == 0
        kv.set_options(0)
        out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        kv.prefill_batch_attn(*args, out, w.eps, w.scale)
        torch.cuda.synchronize()
        assert kv.get_status() == 0
        ref = _oracle_rows(w, slots, pos, range(w.B))
        assert_close(out.cpu().numpy(), ref, f"prefill after a timeout hd={hd}")
    finally:
        kv.free()

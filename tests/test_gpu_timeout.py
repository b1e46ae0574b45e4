"""The failure path of the decode kernel, exercised without a GPU fault.

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

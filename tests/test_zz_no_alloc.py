"""decode_batch_attn_noalloc, the entry point for callers that cannot allocate
device memory (a framework that owns all device memory, or a path that
cannot take cudaMalloc's synchronisation), against decode_batch_attn.

It is called through the C ABI twice in a row on the same inputs; both
outputs must match the regular entry point's within the parity tolerance.
The second call also shows that the shared scratch left behind by the first
does not leak into the next result.  This file is collected last, so a run
that stops at its first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

import sequence_slot_kv_gb300 as skv
import synth
from gpu_harness import DeviceRun, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(run, dev_flags, out):
    w = run.w
    q, kn, vn, pos = run.inputs(0)
    # hold every device tensor until the call has finished
    dq, dk, dv = to_dev(q), to_dev(kn), to_dev(vn)
    dpos = to_dev(pos.astype(np.int32))
    rc = skv._lib.decode_batch_attn_noalloc(
        run.K.data_ptr(), run.V.data_ptr(), w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim,
        w.B, w.n_head, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dpos.data_ptr(),
        run.slots.data_ptr(), run.qw.data_ptr(), run.kw.data_ptr(), run.inv.data_ptr(),
        None if run.sinks is None else run.sinks.data_ptr(), out.data_ptr(),
        dev_flags.data_ptr(), w.eps, w.scale, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0, skv.last_error()
    del dq, dk, dv, dpos
    return out


LONG = synth.Workload("long_rows", 400, B=4, n_slots=6, slot_ctx=8192, n_head=16, n_kv_head=4,
                      head_dim=128, theta=1e6, sinks=True, pos_rule="fixed",
                      fixed_positions=(8191, 5000, 4200, 77), slot_rule="perm")


@pytest.mark.parametrize("name", ["mid", "long_rows"])
def test_noalloc_matches_regular_entry_twice(name):
    w = synth.WORKLOADS["mid"] if name == "mid" else LONG
    run = DeviceRun(w)
    try:
        K0, V0 = run.K.clone(), run.V.clone()
        ref = run.step(0).cpu().numpy()
        assert run.status() == 0
        K_ref, V_ref = run.K.clone(), run.V.clone()
        run.K.copy_(K0)
        run.V.copy_(V0)
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        for call in range(2):
            out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
            got = _noalloc(run, flags, out).cpu().numpy()
            assert_close(got, ref, f"{name} no-alloc call {call + 1}")
            assert int(flags.item()) == 0
            assert torch.equal(run.V, V_ref)
            assert_close(run.K[run.slots.long(), torch.from_numpy(
                w.positions(0).astype(np.int64)).cuda()].cpu().numpy(),
                K_ref[run.slots.long(), torch.from_numpy(
                    w.positions(0).astype(np.int64)).cuda()].cpu().numpy(),
                f"{name} written K, call {call + 1}")
    finally:
        run.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    w = synth.WORKLOADS["large"]           # 256 rows x 40 heads x hd 128 needs ~85 MB
    e = torch.empty(16, device="cuda")
    p = e.data_ptr()
    rc = skv._lib.decode_batch_attn_noalloc(p, p, w.n_slots, w.slot_ctx, w.n_kv_head,
                                            w.head_dim, w.B, w.n_head, p, p, p, p, p, p, p, p,
                                            None, p, None, w.eps, w.scale, None)
    assert rc == 1
    msg = skv.last_error()
    assert "scratch" in msg and str(64 * 1024 * 1024) in msg

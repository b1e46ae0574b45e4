"""decode_batch_attn_noalloc, the entry point for callers that cannot allocate
device memory (a framework that owns all device memory, or a path that
cannot take cudaMalloc's synchronisation), against decode_batch_attn and
against the oracle.

Each case calls the entry point twice in a row on the same inputs: once
through the raw C ABI, once through the Python binding.  Both outputs must
match the regular entry point's and the oracle's within the parity
tolerance, and the written K/V rows must match too.  The second call also
shows that the shared scratch left behind by the first does not leak into
the next result.  The cases cover every head dim, G from 1 to 8, one split
per row, and rows that need more than the entry point's 16 splits at the
default chunk (so it takes larger chunks).  This file is collected last, so
a run that stops at its first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

import sequence_slot_kv_gb300 as skv
import synth
from gpu_harness import DeviceRun, assert_close, expected_written_k, oracle_rows, to_dev

pytestmark = pytest.mark.gpu


def _raw_call(run, dq, dk, dv, dpos, out, flags):
    w = run.w
    return skv._lib.decode_batch_attn_noalloc(
        run.K.data_ptr(), run.V.data_ptr(), w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim,
        w.B, w.n_head, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dpos.data_ptr(),
        run.slots.data_ptr(), run.qw.data_ptr(), run.kw.data_ptr(), run.inv.data_ptr(),
        None if run.sinks is None else run.sinks.data_ptr(), out.data_ptr(),
        flags.data_ptr(), w.eps, w.scale, torch.cuda.current_stream().cuda_stream)


def _wl(name, idx, B, n_slots, slot_ctx, n_head, n_kv_head, hd, sinks=False, positions=None):
    kw = dict(pos_rule="fixed", fixed_positions=tuple(positions)) if positions else {}
    return synth.Workload(name, idx, B=B, n_slots=n_slots, slot_ctx=slot_ctx, n_head=n_head,
                          n_kv_head=n_kv_head, head_dim=hd, theta=1e4, sinks=sinks,
                          slot_rule="perm", **kw)


CASES = {
    "tiny": synth.WORKLOADS["tiny"],
    "mid": synth.WORKLOADS["mid"],
    # one row past 16 default chunks (8191 keys, 512-key chunks at hd 128)
    "long_rows": _wl("long_rows", 400, 4, 6, 8192, 16, 4, 128, sinks=True,
                     positions=(8191, 5000, 4200, 77)),
    "sinks": synth.WORKLOADS["sinks"],
    # the skewed workload's head geometry on 8 slots: 4 rows at 16, 4 at 32767
    "skewed_8": synth.WORKLOADS["skewed"].replace(name="skewed_8", index=401, B=8, n_slots=8),
    "hd64_g1": _wl("hd64_g1", 402, 6, 8, 1024, 4, 4, 64),
    "hd128_g3": _wl("hd128_g3", 403, 6, 8, 1024, 6, 2, 128, sinks=True),
    "hd256_g5": _wl("hd256_g5", 404, 5, 8, 512, 10, 2, 256),
    "hd128_g8": _wl("hd128_g8", 405, 6, 8, 2048, 16, 2, 128),
    "hd256_g8": _wl("hd256_g8", 406, 3, 4, 1024, 8, 1, 256, sinks=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_regular_entry_and_oracle(name):
    w = CASES[name]
    run = DeviceRun(w)
    try:
        K0, V0 = run.K.clone(), run.V.clone()
        ref = run.step(0).cpu().numpy()
        assert run.status() == 0
        K_ref, V_ref = run.K.clone(), run.V.clone()
        q, kn, vn, pos = run.inputs(0)
        dq, dk, dv = to_dev(q), to_dev(kn), to_dev(vn)
        dpos = to_dev(pos.astype(np.int32))
        # the oracle on up to 16 rows spread over the batch
        rows = sorted(set(np.linspace(0, w.B - 1, min(w.B, 16)).round().astype(int).tolist()))
        want, _, _ = oracle_rows(w, rows)
        slots = torch.from_numpy(run.slots_np.astype(np.int64)).cuda()
        prow = torch.from_numpy(pos.astype(np.int64)).cuda()
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        run.K.copy_(K0)
        run.V.copy_(V0)
        for call in range(2):
            out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
            if call == 0:
                rc = _raw_call(run, dq, dk, dv, dpos, out, flags)
                assert rc == 0, skv.last_error()
            else:
                skv.decode_batch_attn_noalloc(run.K, run.V, dq, dk, dv, dpos, run.slots, run.qw,
                                              run.kw, run.inv, run.sinks, out, w.eps, w.scale,
                                              dev_flags=flags)
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            what = f"{name} no-alloc call {call + 1}"
            assert int(flags.item()) == 0, what
            assert_close(got, ref, what + " vs decode_batch_attn")
            assert_close(got[rows], want[0], what + " vs the oracle")
            # written rows: V bit-exact, K as the regular entry and the oracle
            assert torch.equal(run.V, V_ref), what
            gotK = run.K[slots, prow].cpu().numpy()
            assert_close(gotK, K_ref[slots, prow].cpu().numpy(), what + " written K")
            assert_close(gotK, expected_written_k(w, 0), what + " written K vs the oracle")
        del dq, dk, dv, dpos
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

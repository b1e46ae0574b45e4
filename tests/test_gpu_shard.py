"""Slot-ownership sharding on one GPU: the ranks of a sharded step run one
after another in this process, each through its own handle over its own
slot buffers (only the slots it owns), and their outputs are assembled at
the rows' original indices.  The result must match the oracle over the
whole batch, and every rank's buffers must hold exactly the rows its step
wrote.  (On several GPUs each rank is a process with its own device; the
step has no collective, so running the ranks in sequence exercises the same
kernels and routing.)"""
import numpy as np
import pytest
import torch

import synth
from gpu_harness import assert_close, expected_written_k, oracle_rows, to_dev
from sequence_slot_kv_gb300 import shard

pytestmark = pytest.mark.gpu


def _fill_local(w, first, count):
    """Device K/V of global slots [first, first + count), history recipe."""
    shape = (count, w.slot_ctx, w.n_kv_head, w.head_dim)
    K = torch.empty(shape, device="cuda")
    V = torch.empty(shape, device="cuda")
    n = count * w.slot_ctx * w.kv_dim
    s = torch.cuda.current_stream().cuda_stream
    synth.dev_fill_normal(K.data_ptr(), n, w.seed, synth.S_HIST_K, w.hist_index0(first), s)
    synth.dev_fill_normal(V.data_ptr(), n, w.seed, synth.S_HIST_V, w.hist_index0(first), s)
    return K, V


CASES = [(2, synth.Workload("shard_2", 70, B=16, n_slots=24, slot_ctx=1024, n_head=16,
                            n_kv_head=4, head_dim=128, theta=1e6, sinks=True,
                            slot_rule="subset")),
         (3, synth.Workload("shard_3", 71, B=20, n_slots=20, slot_ctx=512, n_head=16,
                            n_kv_head=2, head_dim=64, theta=1e4, sinks=False,
                            slot_rule="perm")),
         (2, synth.WORKLOADS["mid"])]


@pytest.mark.parametrize("n_ranks,w", CASES, ids=[c[1].name for c in CASES])
def test_sharded_step_matches_oracle(n_ranks, w):
    rt = shard.shard_route(n_ranks, w.n_slots, w.slots())
    q, kn, vn = to_dev(w.q()), to_dev(w.k_new()), to_dev(w.v_new())
    pos_np = w.positions(0)
    pos = to_dev(pos_np.astype(np.int32))
    qw, kw, inv = to_dev(w.q_norm_w()), to_dev(w.k_norm_w()), to_dev(w.inv_freq())
    sinks = None if not w.sinks else to_dev(w.sink_logits())
    ranks, outs = [], []
    try:
        for r in range(n_ranks):
            first, count = shard.shard_range(n_ranks, w.n_slots, r)
            K, V = _fill_local(w, first, count)
            sk = shard.ShardedSlotKV(n_ranks, r, w.n_slots, w.slot_ctx, w.n_kv_head,
                                     w.head_dim, w.B, w.n_head, k_buf=K, v_buf=V)
            ranks.append((sk, K, V))
            outs.append(sk.decode_batch_attn(rt, q, kn, vn, pos, qw, kw, inv, sinks, w.eps,
                                             w.scale))
        torch.cuda.synchronize()
        for sk, _, _ in ranks:
            assert sk.kv.get_status() == 0
        got = shard.assemble(rt, outs).cpu().numpy()
        rows = list(range(w.B)) if w.B <= 16 else \
            sorted(set(np.linspace(0, w.B - 1, 16).round().astype(int).tolist()))
        want, _, _ = oracle_rows(w, rows)
        assert_close(got[rows], want[0], f"sharded {w.name} over {n_ranks} ranks")
        # each rank's buffers: the rows it wrote (K as the oracle, V exact),
        # every other byte as the history recipe left it
        wk = expected_written_k(w, 0)
        for r, (sk, K, V) in enumerate(ranks):
            K0, V0 = _fill_local(w, sk.first, sk.count)
            mine = rt.rows(r).astype(np.int64)
            loc = torch.from_numpy(rt.local(r).astype(np.int64)).cuda()
            p = torch.from_numpy(pos_np[mine].astype(np.int64)).cuda()
            assert_close(K[loc, p].cpu().numpy(), wk[mine], f"rank {r} written K")
            assert np.array_equal(V[loc, p].cpu().numpy().view(np.uint32),
                                  w.v_new()[mine].view(np.uint32))
            K0[loc, p] = K[loc, p]
            V0[loc, p] = V[loc, p]
            assert torch.equal(K0.view(torch.int32), K.view(torch.int32))
            assert torch.equal(V0.view(torch.int32), V.view(torch.int32))
    finally:
        for sk, _, _ in ranks:
            sk.free()

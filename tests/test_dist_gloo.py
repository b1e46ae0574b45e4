"""The N>1 bench path on CPU: world size 2 over gloo.  Each rank runs its own
copy of the workload (rows are independent, so there is no data-path
collective); the only cross-rank step is the max over ranks of the timed
region, from which the whole-job rate is formed."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_setup() == (world, rank, rank)
        local_s = [0.5, 0.8][rank]
        mx = bench.max_over_ranks(local_s)
        value = bench.whole_job_rows_per_s(32, 10, world, mx)
        q.put((rank, mx, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_world_size_two_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, mx, value in got:
        assert mx == 0.8
        assert abs(value - 2 * 32 * 10 / 0.8) < 1e-9


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.whole_job_rows_per_s(32, 10, 1, 2.0) == 160.0


SHARD_W = dict(name="shard_gloo", index=60, B=12, n_slots=20, slot_ctx=64, n_head=8,
               n_kv_head=2, head_dim=64, theta=1e4, sinks=True, slot_rule="subset")


def _shard_worker(rank, world, port, q):
    """One rank of slot-ownership sharding over gloo: its own slots' buffers
    only, the rows routed to it, a local step, and the all-gather of out.
    The local step is the oracle (test infrastructure standing in for the
    rank's GPU step, which needs a device)."""
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    import synth
    from sequence_slot_kv_gb300 import shard
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.Workload(**SHARD_W)
        first, count = shard.shard_range(world, w.n_slots, rank)
        K = np.stack([w.hist_rows("k", s, 0, w.slot_ctx) for s in range(first, first + count)])
        V = np.stack([w.hist_rows("v", s, 0, w.slot_ctx) for s in range(first, first + count)])
        rt = shard.shard_route(world, w.n_slots, w.slots())
        rows = rt.rows(rank).astype(np.int64)
        out, _, skipped = oracle.default().decode_batch(
            K, V, w.q()[rows], w.k_new()[rows], w.v_new()[rows], w.positions(0)[rows],
            rt.local(rank), w.q_norm_w(), w.k_norm_w(), w.inv_freq(), w.sink_logits(), w.eps,
            w.scale)
        assert skipped == 0
        full = shard.all_gather_out(rt, torch.from_numpy(out))
        q.put((rank, first, count, len(rows), full.numpy(), K, V))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_slot_sharding_world_size_two_equals_one_process():
    import numpy as np

    import oracle
    import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=150) for _ in range(2)), key=lambda t: t[0])
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    # the whole step on one process, over all slots
    w = synth.Workload(**SHARD_W)
    K = np.stack([w.hist_rows("k", s, 0, w.slot_ctx) for s in range(w.n_slots)])
    V = np.stack([w.hist_rows("v", s, 0, w.slot_ctx) for s in range(w.n_slots)])
    ref, _, _ = oracle.default().decode_batch(
        K, V, w.q(), w.k_new(), w.v_new(), w.positions(0), w.slots(), w.q_norm_w(),
        w.k_norm_w(), w.inv_freq(), w.sink_logits(), w.eps, w.scale)
    assert sum(t[3] for t in got) == w.B and all(t[3] > 0 for t in got)
    for rank, first, count, _, full, Kr, Vr in got:
        # every rank holds every row's output, at the row's original index
        assert np.array_equal(full, ref)
        # its own slots hold what the one-process step wrote there
        assert np.array_equal(Kr, K[first:first + count])
        assert np.array_equal(Vr, V[first:first + count])
    # the ranks' slot ranges tile the global slots
    assert got[0][1] == 0 and got[0][1] + got[0][2] == got[1][1]
    assert got[1][1] + got[1][2] == w.n_slots

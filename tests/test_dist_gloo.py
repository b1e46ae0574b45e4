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

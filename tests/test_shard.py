"""Slot-ownership sharding on the CPU: the partition of the global slots over
ranks and the routing of a step's rows to the ranks that own their slots
(slot_kv_shard_range, slot_kv_shard_route through the C ABI), and the
reassembly of the ranks' outputs at the rows' original indices.

The rows of a step are independent sequences in disjoint slots ("Forward
Cuda Gemma", decodeBatch / allocSlotKv), so a correct routing is: every row
goes to exactly one rank, the one whose range holds its slot, with that
slot's local index; the ranks' rows together are a permutation of the step."""
import numpy as np
import pytest
import torch

import sequence_slot_kv_gb300 as skv
from sequence_slot_kv_gb300 import shard


@pytest.mark.parametrize("n_ranks,n_slots", [(1, 1), (1, 7), (2, 2), (2, 64), (3, 10),
                                             (4, 5), (8, 512), (7, 100), (8, 8)])
def test_ranges_partition_the_slots(n_ranks, n_slots):
    ranges = [shard.shard_range(n_ranks, n_slots, r) for r in range(n_ranks)]
    owned = np.concatenate([np.arange(f, f + c) for f, c in ranges])
    # contiguous, in rank order, every slot exactly once, none empty, balanced
    assert np.array_equal(owned, np.arange(n_slots))
    counts = [c for _, c in ranges]
    assert min(counts) >= 1 and max(counts) - min(counts) <= 1


def test_route_against_brute_force():
    rng = np.random.default_rng(7)
    for trial in range(300):
        n_ranks = int(rng.integers(1, 9))
        n_slots = int(rng.integers(n_ranks, 600))
        B = int(rng.integers(0, min(n_slots, 300) + 1))
        slots = rng.permutation(n_slots)[:B].astype(np.uint32)
        if trial % 5 == 0 and B:
            slots[rng.integers(0, B)] = n_slots + int(rng.integers(0, 1000))   # out of range
        rt = shard.shard_route(n_ranks, n_slots, slots)
        ranges = [shard.shard_range(n_ranks, n_slots, r) for r in range(n_ranks)]
        # a permutation of the rows, grouped by rank, increasing within a rank
        assert np.array_equal(np.sort(rt.order), np.arange(B))
        assert rt.offsets[0] == 0 and rt.offsets[-1] == B
        for r, (first, count) in enumerate(ranges):
            rows = rt.rows(r)
            assert np.all(np.diff(rows.astype(np.int64)) > 0)
            for b, loc in zip(rows, rt.local(r)):
                s = int(slots[b])
                if s < n_slots:
                    assert first <= s < first + count and loc == s - first
                else:       # out of range: the last rank, past its range
                    assert r == n_ranks - 1 and loc >= count
        # no slot owned twice: the (rank, local slot) pairs of in-range rows differ
        pairs = {(r, int(loc)) for r in range(n_ranks) for loc in rt.local(r)}
        assert len(pairs) == B


def test_route_argument_errors():
    with pytest.raises(skv.SlotKVError):
        shard.shard_range(0, 4, 0)
    with pytest.raises(skv.SlotKVError):
        shard.shard_range(5, 4, 0)
    with pytest.raises(skv.SlotKVError):
        shard.shard_range(2, 4, 2)
    with pytest.raises(skv.SlotKVError):
        shard.shard_route(3, 2, [0, 1])
    rt = shard.shard_route(3, 9, [])
    assert list(rt.offsets) == [0, 0, 0, 0]


def test_assemble_puts_rows_back_at_their_indices():
    rng = np.random.default_rng(3)
    n_ranks, n_slots, B = 3, 40, 17
    slots = rng.permutation(n_slots)[:B]
    rt = shard.shard_route(n_ranks, n_slots, slots)
    glob = torch.from_numpy(rng.standard_normal((B, 4, 8)).astype(np.float32))
    # each rank's output rows in route order, padded like an all-gather's
    outs = []
    for r in range(n_ranks):
        part = torch.full((rt.max_count(), 4, 8), float("nan"))
        part[:rt.count(r)] = glob[torch.from_numpy(rt.rows(r).astype(np.int64))]
        outs.append(part)
    assert torch.equal(shard.assemble(rt, outs), glob)

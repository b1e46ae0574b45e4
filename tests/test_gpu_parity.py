"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Small geometries cover every head dim and a spread of GQA group sizes with
positions at the tile and split edges and a ragged tail, under a split policy
that forces several splits per row (exercising the cross-CTA merge) and under
the default policy.  The five workloads run at full size with sampled rows
(the oracle computes those rows one by one) and every written K/V row.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_harness import DeviceRun, assert_close, check_kv_after, oracle_rows

pytestmark = pytest.mark.gpu


def small_workload(hd, G, sinks, idx, n_kv_head=2):
    T = 4096 // hd
    slot_ctx = 8 * T + 5
    positions = (0, 1, T - 1, T, T + 1, 3 * T + 7, slot_ctx - 2, slot_ctx - 1)
    return synth.Workload(
        f"small_hd{hd}_g{G}", 100 + idx, B=len(positions), n_slots=len(positions) + 3,
        slot_ctx=slot_ctx, n_head=G * n_kv_head, n_kv_head=n_kv_head, head_dim=hd,
        theta=10000.0, sinks=sinks, pos_rule="fixed", fixed_positions=positions,
        slot_rule="perm")


GEOMS = [(hd, G) for hd in (64, 128, 256) for G in (1, 2, 3, 4, 5, 8)]


@pytest.mark.parametrize("policy", ["many_splits", "default"])
@pytest.mark.parametrize("hd,G", GEOMS, ids=[f"hd{h}_g{g}" for h, g in GEOMS])
def test_small_geometry_matches_oracle(hd, G, policy):
    idx = GEOMS.index((hd, G))
    w = small_workload(hd, G, sinks=(idx % 2 == 1), idx=idx)
    split = (4096 // hd, 8) if policy == "many_splits" else None
    run = DeviceRun(w, split=split)
    try:
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.status() == 0
        ref, _, _ = oracle_rows(w, range(w.B))
        assert_close(out.cpu().numpy(), ref[0], f"out hd={hd} G={G} {policy}")
        check_kv_after(run)
    finally:
        run.close()


def test_tiny_workload_full():
    w = synth.WORKLOADS["tiny"]
    run = DeviceRun(w)
    try:
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.status() == 0
        ref, _, _ = oracle_rows(w, range(w.B))
        assert_close(out.cpu().numpy(), ref[0], "tiny out")
        check_kv_after(run)
    finally:
        run.close()


def _sample_rows(w, k, seed):
    """Rows to check one by one: the extremes of position plus a seeded spread."""
    pos = w.positions0()
    rows = {int(np.argmin(pos)), int(np.argmax(pos))}
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.choice(w.B, size=min(k, w.B), replace=False))
    return sorted(rows)[: max(k, 2)]


@pytest.mark.parametrize("name,k", [("mid", 32), ("skewed", 4), ("sinks", 24),
                                    ("gqa8_hd128", 12), ("gqa8_hd256", 12)])
def test_full_size_workload(name, k):
    w = {**synth.WORKLOADS, **synth.EXTRA_WORKLOADS}[name]
    run = DeviceRun(w)
    try:
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.status() == 0
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        rows = list(range(w.B)) if k >= w.B else _sample_rows(w, k, seed=5)
        if name == "skewed":
            rows = [0, 1, w.B - 2, w.B - 1]       # two short rows, two long rows
        ref, _, _ = oracle_rows(w, rows)
        assert_close(got[rows], ref[0], f"{name} out rows {rows}")
        check_kv_after(run)
    finally:
        run.close()


def test_large_batch_multi_step():
    """64 consecutive steps, positions advancing by one, fresh q/k/v each
    step; sampled rows against the oracle's sequential loop at every step,
    and the final slot contents (all written rows, all other bytes)."""
    w = synth.WORKLOADS["large"]
    run = DeviceRun(w)
    rows = _sample_rows(w, 6, seed=9)
    try:
        outs = []
        for t in range(w.steps):
            outs.append(run.step(t)[rows].cpu())
        torch.cuda.synchronize()
        assert run.status() == 0
        ref, _, _ = oracle_rows(w, rows, steps=w.steps)
        for t in range(w.steps):
            assert_close(outs[t].numpy(), ref[t], f"large step {t}")
        check_kv_after(run, steps=w.steps)
    finally:
        run.close()

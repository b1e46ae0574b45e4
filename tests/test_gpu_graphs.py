"""Multi-step decode captured in a CUDA graph: decode_batch_attn and
slot_kv_advance_positions on device-resident positions, with no host work
between steps ("Forward Cuda Gemma", decodeBatch: the caller advances each
position and feeds it back).  Graph replay must equal eager execution bit
for bit, and both must match the oracle's sequential steps."""
import numpy as np
import pytest
import torch

import sequence_slot_kv_gb300 as skv
import synth
from gpu_harness import DeviceRun, assert_close, oracle_rows, to_dev

pytestmark = pytest.mark.gpu

STEPS = 6
W = synth.Workload("graph_steps", 500, B=8, n_slots=12, slot_ctx=700, n_head=16, n_kv_head=4,
                   head_dim=128, theta=1e6, sinks=True, steps=STEPS, pos_rule="uniform_start",
                   start_hi=600, slot_rule="subset")


def _step_inputs(w):
    return [(to_dev(w.q(t)), to_dev(w.k_new(t)), to_dev(w.v_new(t))) for t in range(w.steps)]


def test_graph_replay_equals_eager_and_oracle():
    w = W
    run = DeviceRun(w)
    try:
        K0, V0 = run.K.clone(), run.V.clone()
        ins = _step_inputs(w)
        pos0 = to_dev(w.positions(0).astype(np.int32))
        outs_e = [torch.empty((w.B, w.n_head, w.head_dim), device="cuda") for _ in range(STEPS)]
        outs_g = [torch.empty_like(o) for o in outs_e]

        def steps(pos, outs):
            for t in range(STEPS):
                q, kn, vn = ins[t]
                run.kv.decode_batch_attn(q, kn, vn, pos, run.slots, run.qw, run.kw, run.inv,
                                         run.sinks, outs[t], w.eps, w.scale)
                skv.slot_kv_advance_positions(pos, 1)

        # eager
        pos = pos0.clone()
        steps(pos, outs_e)
        torch.cuda.synchronize()
        assert run.status() == 0
        K_e, V_e = run.K.clone(), run.V.clone()
        assert torch.equal(pos.cpu(), (pos0 + STEPS).cpu())

        # captured once, replayed from the initial state
        run.K.copy_(K0)
        run.V.copy_(V0)
        posg = pos0.clone()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                steps(posg, outs_g)
        torch.cuda.current_stream().wait_stream(s)
        run.K.copy_(K0)
        run.V.copy_(V0)
        posg.copy_(pos0)
        g.replay()
        torch.cuda.synchronize()
        assert run.status() == 0
        for t in range(STEPS):
            assert torch.equal(outs_g[t], outs_e[t]), f"step {t}"
        assert torch.equal(run.K, K_e) and torch.equal(run.V, V_e)
        assert torch.equal(posg.cpu(), (pos0 + STEPS).cpu())

        # a second replay continues from the advanced positions: rewind first
        run.K.copy_(K0)
        run.V.copy_(V0)
        posg.copy_(pos0)
        g.replay()
        torch.cuda.synchronize()
        for t in range(STEPS):
            assert torch.equal(outs_g[t], outs_e[t]), f"second replay, step {t}"

        ref, _, _ = oracle_rows(w, range(w.B), steps=STEPS)
        for t in range(STEPS):
            assert_close(outs_g[t].cpu().numpy(), ref[t], f"graph step {t} vs oracle")
    finally:
        run.close()


def test_graph_replay_paged():
    """Multi-step paged decode in a graph: each step writes its key into the
    row's block and the next step reads it through the table."""
    from test_gpu_paged import PagedRun, host_pool, oracle_paged
    steps, bs = 4, 32
    w = synth.Workload("graph_paged", 510, B=6, n_slots=8, slot_ctx=8 * bs, n_head=16,
                       n_kv_head=4, head_dim=128, theta=1e6, sinks=True, steps=steps,
                       pos_rule="uniform_start", start_hi=8 * bs - steps - 1, slot_rule="subset")
    run = PagedRun(w, bs, split=(32, 8))
    try:
        K0, V0 = run.K.clone(), run.V.clone()
        ins = [(to_dev(w.q(t)), to_dev(w.k_new(t)), to_dev(w.v_new(t))) for t in range(steps)]
        pos0 = to_dev(w.positions(0).astype(np.int32))
        outs_e = [torch.empty((w.B, w.n_head, w.head_dim), device="cuda") for _ in range(steps)]
        outs_g = [torch.empty_like(o) for o in outs_e]

        def run_steps(pos, outs):
            for t in range(steps):
                q, kn, vn = ins[t]
                run.kv.decode_batch_attn_paged(q, kn, vn, pos, run.tables, run.qw, run.kw,
                                               run.inv, run.sinks, outs[t], w.eps, w.scale)
                skv.slot_kv_advance_positions(pos, 1)

        pos = pos0.clone()
        run_steps(pos, outs_e)
        torch.cuda.synchronize()
        assert run.kv.get_status() == 0
        K_e, V_e = run.K.clone(), run.V.clone()
        run.K.copy_(K0)
        run.V.copy_(V0)
        posg = pos0.clone()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                run_steps(posg, outs_g)
        torch.cuda.current_stream().wait_stream(s)
        run.K.copy_(K0)
        run.V.copy_(V0)
        posg.copy_(pos0)
        g.replay()
        torch.cuda.synchronize()
        assert run.kv.get_status() == 0
        for t in range(steps):
            assert torch.equal(outs_g[t], outs_e[t]), f"paged step {t}"
        assert torch.equal(run.K, K_e) and torch.equal(run.V, V_e)
        Kr, Vr = host_pool(w, bs)
        for t in range(steps):
            ref, skipped = oracle_paged(w, bs, Kr, Vr, run.tables_np, step=t)
            assert skipped == 0
            assert_close(outs_g[t].cpu().numpy(), ref, f"paged graph step {t} vs oracle")
    finally:
        run.close()


def test_advance_positions():
    p = torch.arange(1000, dtype=torch.int32, device="cuda")
    skv.slot_kv_advance_positions(p, 3)
    skv.slot_kv_advance_positions(p[:0], 5)
    torch.cuda.synchronize()
    assert torch.equal(p.cpu(), torch.arange(3, 1003, dtype=torch.int32))

"""The norm options of the Gemma path ("Forward Cuda Gemma", decodeBatch:
per-head V/Q/K norm) against the oracle: a weightless RMS norm of v_new
before it is cached and attended, and norm weights applied as (1 + w)."""
import numpy as np
import pytest
import torch

import oracle
import sequence_slot_kv_gb300 as skv
import synth
from gpu_harness import DeviceRun, assert_close, oracle_rows

pytestmark = pytest.mark.gpu

FLAGS = {"vnorm": (skv.OPT_VNORM, oracle.VNORM),
         "plus_one": (skv.OPT_NORM_PLUS_ONE, oracle.NORM_PLUS_ONE),
         "both": (skv.OPT_VNORM | skv.OPT_NORM_PLUS_ONE, oracle.VNORM | oracle.NORM_PLUS_ONE)}


def _wl(hd, idx):
    T = 4096 // hd
    ctx = 6 * T + 3
    pos = (0, 1, T - 1, T + 2, 4 * T + 1, ctx - 1)
    return synth.Workload(f"opt_hd{hd}", 600 + idx, B=len(pos), n_slots=len(pos) + 2,
                          slot_ctx=ctx, n_head=16, n_kv_head=4, head_dim=hd, theta=1e4,
                          sinks=True, pos_rule="fixed", fixed_positions=pos, slot_rule="perm")


@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("name", list(FLAGS))
def test_options_match_oracle(hd, name):
    gflags, oflags = FLAGS[name]
    w = _wl(hd, [64, 128, 256].index(hd))
    run = DeviceRun(w, split=(4096 // hd, 8))
    try:
        run.kv.set_options(gflags)
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.status() == 0
        ref, Kr, Vr = oracle_rows(w, range(w.B), flags=oflags)
        assert_close(out.cpu().numpy(), ref[0], f"out {name} hd={hd}")
        pos = w.positions(0)
        for b in range(w.B):
            s, p = int(run.slots_np[b]), int(pos[b])
            assert_close(run.K[s, p].cpu().numpy(), Kr[b, p], f"written K {name}")
            assert_close(run.V[s, p].cpu().numpy(), Vr[b, p], f"written V {name}")
    finally:
        run.close()


@pytest.mark.parametrize("name", list(FLAGS))
def test_options_paged(name):
    """The options over the paged path (64-key blocks of a shuffled pool),
    against the paged oracle with the same flags."""
    from test_gpu_paged import PagedRun, host_pool, oracle_paged, written_mask
    gflags, oflags = FLAGS[name]
    hd, bs = 128, 64
    T = 4096 // hd
    pos = (0, 5, T + 1, bs, 3 * bs + 7, 6 * bs - 1)
    w = synth.Workload(f"opt_paged_{name}", 620 + list(FLAGS).index(name), B=len(pos),
                       n_slots=len(pos) + 2, slot_ctx=6 * bs, n_head=16, n_kv_head=4,
                       head_dim=hd, theta=1e4, sinks=True, pos_rule="fixed",
                       fixed_positions=pos, slot_rule="perm")
    run = PagedRun(w, bs, split=(T, 8))
    try:
        run.kv.set_options(gflags)
        out = run.step(0)
        torch.cuda.synchronize()
        assert run.kv.get_status() == 0
        Kr, Vr = host_pool(w, bs)
        ref, skipped = oracle_paged(w, bs, Kr, Vr, run.tables_np, flags=oflags)
        assert skipped == 0
        assert_close(out.cpu().numpy(), ref, f"paged out {name}")
        written = written_mask(run, run.tables_np, w.positions(0))
        Kg, Vg = run.K.cpu().numpy(), run.V.cpu().numpy()
        assert_close(Kg[written], Kr[written], f"paged written K {name}")
        assert_close(Vg[written], Vr[written], f"paged written V {name}")
        assert np.array_equal(Kg[~written].view(np.uint32), Kr[~written].view(np.uint32))
        assert np.array_equal(Vg[~written].view(np.uint32), Vr[~written].view(np.uint32))
    finally:
        run.close()


def test_unknown_option_bits_rejected():
    w = _wl(128, 9)
    run = DeviceRun(w)
    try:
        with pytest.raises(skv.SlotKVError):
            run.kv.set_options(4)
    finally:
        run.close()

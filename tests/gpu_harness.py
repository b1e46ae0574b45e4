"""Shared set-up for the GPU parity tests: device workloads, oracle runs on
host copies regenerated from the input generator, and the comparisons.

Nothing here computes a step of the method: expected values come from the
oracle only, inputs from ``synth`` only.
"""
import numpy as np
import torch

import oracle
import synth
from sequence_slot_kv_gb300 import SlotKV

ATOL = 1e-4
RTOL = 1e-4


def assert_close(got, want, what, atol=ATOL, rtol=RTOL):
    """Element-wise: |got - want| <= atol, or <= rtol * |want|."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    bad = (err > atol) & (err > rtol * np.abs(want))
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err, 0)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: got {got[i]!r} want {want[i]!r}")
    return float(err.max()) if err.size else 0.0


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


class DeviceRun:
    """A workload resident on the GPU: slot K/V filled with the history
    recipe, the parameters uploaded, and a SlotKV handle adopting the
    buffers."""

    def __init__(self, w, split=None):
        self.w = w
        shape = (w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
        self.K = torch.empty(shape, dtype=torch.float32, device="cuda")
        self.V = torch.empty(shape, dtype=torch.float32, device="cuda")
        w.dev_fill_history(self.K.data_ptr(), self.V.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
        self.kv = SlotKV(w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim, w.B, w.n_head,
                         k_buf=self.K, v_buf=self.V)
        if split is not None:
            self.kv.set_split(*split)
        self.qw = to_dev(w.q_norm_w())
        self.kw = to_dev(w.k_norm_w())
        self.inv = to_dev(w.inv_freq())
        s = w.sink_logits()
        self.sinks = None if s is None else to_dev(s)
        self.slots_np = w.slots()
        self.slots = to_dev(self.slots_np.astype(np.int32))

    def inputs(self, step):
        w = self.w
        return (w.q(step), w.k_new(step), w.v_new(step), w.positions(step))

    def step(self, step=0, out=None, inputs=None):
        w = self.w
        q, kn, vn, pos = self.inputs(step) if inputs is None else inputs
        if out is None:
            out = torch.full((w.B, w.n_head, w.head_dim), float("nan"), device="cuda")
        self.kv.decode_batch_attn(to_dev(q), to_dev(kn), to_dev(vn),
                                  to_dev(pos.astype(np.int32)), self.slots, self.qw, self.kw,
                                  self.inv, self.sinks, out, w.eps, w.scale)
        return out

    def status(self):
        return self.kv.get_status()

    def close(self):
        self.kv.free()


def oracle_rows(w, rows, steps=1, n_threads=None, first_step=0, flags=0):
    """Run the oracle for rows ``rows`` over ``steps`` consecutive steps on
    compact host slot buffers regenerated from the history recipe.
    Returns (outs [steps][len(rows)][n_head][hd], K, V, ctx_end) where K/V are
    the compact buffers after the last step (compact slot i = rows[i])."""
    o = oracle.default()
    rows = list(rows)
    slots = w.slots()
    p0 = w.positions(first_step)
    ctx = int(max(p0[r] for r in rows)) + steps
    K = np.empty((len(rows), ctx, w.n_kv_head, w.head_dim), dtype=np.float32)
    V = np.empty_like(K)
    for i, r in enumerate(rows):
        K[i] = w.hist_rows("k", slots[r], 0, ctx)
        V[i] = w.hist_rows("v", slots[r], 0, ctx)
    outs = []
    nt = n_threads or min(len(rows), 32)
    for t in range(first_step, first_step + steps):
        q, kn, vn, pos = w.q(t), w.k_new(t), w.v_new(t), w.positions(t)
        out, _, skipped = o.decode_batch(
            K, V, q[rows], kn[rows], vn[rows], pos[rows],
            np.arange(len(rows), dtype=np.uint32), w.q_norm_w(), w.k_norm_w(), w.inv_freq(),
            w.sink_logits(), w.eps, w.scale, n_threads=nt, flags=flags)
        assert skipped == 0
        outs.append(out)
    return np.stack(outs), K, V


def expected_written_k(w, step):
    """Oracle value of the K row each row writes at its position in ``step``:
    f32[B][n_kv_head][hd]."""
    o = oracle.default()
    kn, pos = w.k_new(step), w.positions(step)
    kw, inv = w.k_norm_w(), w.inv_freq()
    out = np.empty((w.B, w.n_kv_head, w.head_dim), dtype=np.float32)
    for b in range(w.B):
        for g in range(w.n_kv_head):
            out[b, g] = o.norm_rope_head(kn[b, g], kw, w.eps, int(pos[b]), inv).astype(np.float32)
    return out


def check_kv_after(run, steps=1, first_step=0):
    """The slot buffers after ``steps`` steps: the written rows against the
    oracle (K within tolerance, V bit-exact), every other byte bit-identical to
    the history recipe."""
    w = run.w
    shape = run.K.shape
    expK = torch.empty(shape, dtype=torch.float32, device="cuda")
    expV = torch.empty(shape, dtype=torch.float32, device="cuda")
    w.dev_fill_history(expK.data_ptr(), expV.data_ptr(), torch.cuda.current_stream().cuda_stream)
    slots = torch.from_numpy(run.slots_np.astype(np.int64)).cuda()
    for t in range(first_step, first_step + steps):
        pos = torch.from_numpy(w.positions(t).astype(np.int64)).cuda()
        # written rows: V bit-exact to v_new, K within tolerance of the oracle
        gotV = run.V[slots, pos].cpu().numpy()
        assert np.array_equal(gotV.view(np.uint32), w.v_new(t).view(np.uint32)), \
            f"V rows written at step {t} differ from v_new"
        gotK = run.K[slots, pos].cpu().numpy()
        assert_close(gotK, expected_written_k(w, t), f"K rows written at step {t}")
        expK[slots, pos] = run.K[slots, pos]
        expV[slots, pos] = run.V[slots, pos]
    torch.cuda.synchronize()
    assert torch.equal(expK.view(torch.int32), run.K.view(torch.int32)), \
        "K bytes outside the written rows changed"
    assert torch.equal(expV.view(torch.int32), run.V.view(torch.int32)), \
        "V bytes outside the written rows changed"
    del expK, expV

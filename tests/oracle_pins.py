"""Pins for the CPU oracle: facts fixed by the pages and by the mathematics.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a closed form, an invariant, a library routine on a
special case, or brute force on a tiny case.  ``test_oracle_pins.py`` runs
them on the real oracle; ``test_oracle_mutants.py`` runs them on copies of the
oracle with one planted mistake each and requires that some pin fails.

Page references name the zinc engine's API pages ("Forward Cuda",
"Forward Cuda Gemma") and the entry they document.
"""
import math
import os

import numpy as np
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# helpers (inputs only; no step of the method is computed here)
# --------------------------------------------------------------------------
class Case:
    """A small decode step: geometry, inputs and host slot buffers."""

    def __init__(self, n_slots=3, slot_ctx=16, n_head=4, n_kv_head=2, hd=8, B=1,
                 seed=7, eps=1e-6, scale=None):
        self.n_slots, self.slot_ctx = n_slots, slot_ctx
        self.n_head, self.n_kv_head, self.hd, self.B = n_head, n_kv_head, hd, B
        self.eps = eps
        self.scale = np.float32(1.0 / math.sqrt(hd)) if scale is None else np.float32(scale)
        rng = np.random.default_rng(seed)
        shape = (n_slots, slot_ctx, n_kv_head, hd)
        self.K = rng.standard_normal(shape).astype(np.float32)
        self.V = rng.standard_normal(shape).astype(np.float32)
        self.q = rng.standard_normal((B, n_head, hd)).astype(np.float32)
        self.k_new = rng.standard_normal((B, n_kv_head, hd)).astype(np.float32)
        self.v_new = rng.standard_normal((B, n_kv_head, hd)).astype(np.float32)
        self.q_norm_w = (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32)
        self.k_norm_w = (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32)
        i = np.arange(hd // 2, dtype=np.float64)
        self.inv_freq = (10000.0 ** (-2 * i / hd)).astype(np.float32)
        self.sinks = None
        self.positions = np.zeros(B, dtype=np.uint32)
        self.slots = np.arange(B, dtype=np.uint32) % n_slots

    def run(self, o, want64=True, flags=0, **over):
        K = over.pop("K", self.K)
        V = over.pop("V", self.V)
        args = dict(q=self.q, k_new=self.k_new, v_new=self.v_new,
                    positions=self.positions, slots=self.slots, q_norm_w=self.q_norm_w,
                    k_norm_w=self.k_norm_w, inv_freq=self.inv_freq, sinks=self.sinks,
                    eps=self.eps, scale=self.scale)
        args.update(over)
        return o.decode_batch(K, V, want64=want64, flags=flags, **args)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# --------------------------------------------------------------------------
# slot offsets ("Forward Cuda Gemma", slotKvOffsetBytes; "Forward Cuda")
# --------------------------------------------------------------------------
def pin_offsets_tile_the_buffer(o):
    """Offsets round-trip to (slot, pos), never overlap, and tile the buffer."""
    n_slots, slot_ctx, kv_dim = 4, 64, 128
    row = kv_dim * 4
    offs = []
    for s in range(n_slots):
        for p in range(slot_ctx):
            off = o.offset_bytes(s, p, slot_ctx, kv_dim)
            assert off % row == 0
            assert divmod(off // row, slot_ctx) == (s, p)
            offs.append(off)
    offs = np.sort(np.array(offs, dtype=np.int64))
    # disjoint [off, off+row) intervals covering [0, n_slots*slot_ctx*row) exactly
    assert np.array_equal(offs, np.arange(n_slots * slot_ctx, dtype=np.int64) * row)


def pin_offsets_golden(o):
    """Hand-worked offsets, including ones past 2^32 bytes."""
    path = os.path.join(GOLDEN, "slot_offsets.txt")
    n = 0
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            slot, pos, slot_ctx, kv_dim, want = (int(x) for x in line.split())
            assert o.offset_bytes(slot, pos, slot_ctx, kv_dim) == want, line
            n += 1
    assert n >= 4


# --------------------------------------------------------------------------
# per-head RMS norm and RoPE ("Forward Cuda Gemma", decodeBatch: per-head
# Q/K norm + RoPE)
# --------------------------------------------------------------------------
def pin_norm_is_library_rms_norm(o):
    """At pos 0 RoPE is the identity, so the result is torch's RMS norm."""
    rng = np.random.default_rng(1)
    for hd, eps in ((64, 1e-6), (128, 0.1), (256, 2.0)):
        x = rng.standard_normal(hd).astype(np.float32)
        w = (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32)
        inv = rng.random(hd // 2).astype(np.float32)
        y = o.norm_rope_head(x, w, eps, 0, inv)
        ref = torch.nn.functional.rms_norm(
            torch.from_numpy(x.astype(np.float64)), (hd,),
            torch.from_numpy(w.astype(np.float64)), eps=float(np.float32(eps))).numpy()
        _close(y, ref, 1e-12, f"rms norm hd={hd} eps={eps}")


def pin_rope_unit_vectors(o):
    """A scaled basis vector e_i (or e_{i+hd/2}) normalises to sqrt(hd) e_i and
    RoPE turns it by the f32 angle fl32(pos * inv_freq[i]) within pair
    (i, i + hd/2): the columns of the rotation matrix."""
    hd = 128
    half = hd // 2
    i_arr = np.arange(half, dtype=np.float64)
    inv = (1e6 ** (-2 * i_arr / hd)).astype(np.float32)
    w = np.ones(hd, dtype=np.float32)
    r = math.sqrt(hd)
    for pos in (0, 1, 7, 1000, 4095, 32767):
        for i in (0, 1, 5, half - 1):
            ang = float(np.float32(pos) * inv[i])        # one f32 rounding
            c, s = math.cos(ang), math.sin(ang)
            x = np.zeros(hd, dtype=np.float32)
            x[i] = 3.0
            y = o.norm_rope_head(x, w, 0.0, pos, inv)
            want = np.zeros(hd)
            want[i], want[i + half] = r * c, r * s
            _close(y, want, 1e-12, f"e_{i} pos={pos}")
            x = np.zeros(hd, dtype=np.float32)
            x[i + half] = -2.0
            y = o.norm_rope_head(x, w, 0.0, pos, inv)
            want = np.zeros(hd)
            want[i], want[i + half] = r * s, -r * c
            _close(y, want, 1e-12, f"e_{i + half} pos={pos}")


def pin_rope_preserves_norm(o):
    rng = np.random.default_rng(2)
    hd = 64
    x = rng.standard_normal(hd).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32)
    inv = rng.random(hd // 2).astype(np.float32)
    y0 = o.norm_rope_head(x, w, 1e-6, 0, inv)
    for pos in (1, 17, 999):
        y = o.norm_rope_head(x, w, 1e-6, pos, inv)
        assert abs(np.linalg.norm(y) - np.linalg.norm(y0)) < 1e-12
        # each pair keeps its own length
        half = hd // 2
        _close(np.hypot(y[:half], y[half:]), np.hypot(y0[:half], y0[half:]), 1e-12,
               "pair lengths")


def pin_rope_relative_position(o):
    """<R(p)q, R(j)k> depends on p - j only.  With power-of-two frequencies
    the f32 angles are exact, so the identity holds to f64 rounding."""
    rng = np.random.default_rng(3)
    hd = 32
    inv = (2.0 ** -np.arange(hd // 2)).astype(np.float32)
    w = np.ones(hd, dtype=np.float32)
    q = rng.standard_normal(hd).astype(np.float32)
    k = rng.standard_normal(hd).astype(np.float32)
    for p, j in ((5, 2), (9, 9), (3, 11)):
        base = np.dot(o.norm_rope_head(q, w, 0.0, p, inv), o.norm_rope_head(k, w, 0.0, j, inv))
        for d in (1, 4, 13):
            sh = np.dot(o.norm_rope_head(q, w, 0.0, p + d, inv),
                        o.norm_rope_head(k, w, 0.0, j + d, inv))
            assert abs(sh - base) < 1e-11, (p, j, d, sh, base)


# --------------------------------------------------------------------------
# the decode step ("Forward Cuda Gemma", decodeBatch)
# --------------------------------------------------------------------------
def pin_written_k_is_normed_rotated_k(o):
    """The row written at (slot, pos) is fl32(RoPE(norm(k_new))) for K and the
    raw v_new for V, at the offset slotKvOffsetBytes gives."""
    c = Case(B=3, n_slots=4)
    c.positions = np.array([0, 5, 15], dtype=np.uint32)
    c.slots = np.array([2, 0, 3], dtype=np.uint32)
    K, V = c.K.copy(), c.V.copy()
    c.run(o, K=K, V=V)
    kv_dim = c.n_kv_head * c.hd
    Kb, Vb = K.reshape(-1).view(np.uint8), V.reshape(-1).view(np.uint8)
    for b in range(c.B):
        off = o.offset_bytes(int(c.slots[b]), int(c.positions[b]), c.slot_ctx, kv_dim)
        krow = Kb[off: off + kv_dim * 4].view(np.float32).reshape(c.n_kv_head, c.hd)
        vrow = Vb[off: off + kv_dim * 4].view(np.float32).reshape(c.n_kv_head, c.hd)
        for g in range(c.n_kv_head):
            want = o.norm_rope_head(c.k_new[b, g], c.k_norm_w, c.eps,
                                    int(c.positions[b]), c.inv_freq).astype(np.float32)
            assert np.array_equal(krow[g], want)
            assert np.array_equal(vrow[g].view(np.uint32), c.v_new[b, g].view(np.uint32))
        # at pos 0, the written K is torch's RMS norm of k_new (RoPE is the identity)
        if c.positions[b] == 0:
            ref = torch.nn.functional.rms_norm(
                torch.from_numpy(c.k_new[b].astype(np.float64)), (c.hd,),
                torch.from_numpy(c.k_norm_w.astype(np.float64)), eps=float(np.float32(c.eps)))
            _close(krow, ref.numpy(), 1e-6, "pos-0 K vs rms_norm")


def pin_kv_write_set(o):
    """Exactly the rows (slots[b], positions[b]) change; all other bytes of K
    and V stay bit-identical."""
    c = Case(B=3, n_slots=5, slot_ctx=9)
    c.positions = np.array([8, 0, 3], dtype=np.uint32)
    c.slots = np.array([4, 1, 2], dtype=np.uint32)
    K, V = c.K.copy(), c.V.copy()
    c.run(o, K=K, V=V)
    mask = np.ones(K.shape[:2], dtype=bool)
    for b in range(c.B):
        mask[c.slots[b], c.positions[b]] = False
    assert np.array_equal(K[mask].view(np.uint32), c.K[mask].view(np.uint32))
    assert np.array_equal(V[mask].view(np.uint32), c.V[mask].view(np.uint32))
    for b in range(c.B):
        assert np.array_equal(V[c.slots[b], c.positions[b]].view(np.uint32),
                              c.v_new[b].view(np.uint32))


def pin_pos0_returns_own_v(o):
    """At pos 0 the only key is the new one: out[h] = v_new[kv head of h]."""
    c = Case(B=2, n_head=6, n_kv_head=3)
    c.slots = np.array([1, 0], dtype=np.uint32)
    out, out64, _ = c.run(o, K=c.K.copy(), V=c.V.copy())
    g = c.n_head // c.n_kv_head
    for b in range(c.B):
        for h in range(c.n_head):
            assert np.array_equal(out64[b, h], c.v_new[b, h // g].astype(np.float64))


def pin_pos0_sink_closed_form(o):
    """With q orthogonal to the new key the lone score is 0, so a sink logit
    s_h gives out[h] = v / (1 + e^{s_h}); the sink is not scaled."""
    c = Case(B=1, n_head=4, n_kv_head=2, hd=8, scale=0.37)
    c.q[:] = 0
    c.q[0, :, 0] = 1.0
    c.k_new[:] = 0
    c.k_new[0, :, 1] = 1.0
    c.sinks = np.array([-1.5, 0.0, 0.75, 3.0], dtype=np.float32)
    out, out64, _ = c.run(o, K=c.K.copy(), V=c.V.copy())
    for h in range(c.n_head):
        want = c.v_new[0, h // 2].astype(np.float64) / (1.0 + math.exp(float(c.sinks[h])))
        _close(out64[0, h], want, 1e-14, f"sink head {h}")


def pin_constant_v_history(o):
    """If every value row of a kv head is the same vector u, out = u."""
    c = Case(B=2, n_slots=2, slot_ctx=20, n_head=4, n_kv_head=2)
    c.positions = np.array([19, 7], dtype=np.uint32)
    c.slots = np.array([0, 1], dtype=np.uint32)
    u = np.random.default_rng(4).standard_normal((c.n_kv_head, c.hd)).astype(np.float32)
    V = np.broadcast_to(u, c.V.shape).copy()
    c.v_new = np.broadcast_to(u, c.v_new.shape).copy()
    out, out64, _ = c.run(o, K=c.K.copy(), V=V)
    for b in range(c.B):
        for h in range(c.n_head):
            _close(out64[b, h], u[h // 2], 1e-13, "constant V")


def pin_equal_scores_give_mean(o):
    """q = 0 gives every key the score 0: out is the mean of V over keys
    0..pos inclusive (history rows and the new row)."""
    c = Case(B=2, n_slots=2, slot_ctx=12, n_head=4, n_kv_head=2)
    c.q[:] = 0
    c.positions = np.array([11, 4], dtype=np.uint32)
    c.slots = np.array([1, 0], dtype=np.uint32)
    V0 = c.V.copy()
    out, out64, _ = c.run(o, K=c.K.copy(), V=c.V.copy())
    for b in range(c.B):
        p, s = int(c.positions[b]), int(c.slots[b])
        rows = np.concatenate([V0[s, :p].astype(np.float64),
                               c.v_new[b][None].astype(np.float64)], axis=0)
        want = rows.mean(axis=0)                      # [n_kv_head][hd]
        for h in range(c.n_head):
            _close(out64[b, h], want[h // 2], 1e-13, "uniform mean")


def pin_equal_scores_with_sink(o):
    """q = 0 with a sink s_h and constant values u: out = u (p+1)/(p+1+e^{s_h})."""
    c = Case(B=1, n_slots=1, slot_ctx=10, n_head=2, n_kv_head=1, scale=0.5)
    c.q[:] = 0
    c.positions = np.array([6], dtype=np.uint32)
    u = np.linspace(-1, 1, c.hd).astype(np.float32)
    V = np.broadcast_to(u, c.V.shape).copy()
    c.v_new = np.broadcast_to(u, c.v_new.shape).copy()
    c.sinks = np.array([0.3, -2.0], dtype=np.float32)
    out, out64, _ = c.run(o, K=c.K.copy(), V=V)
    for h in range(2):
        want = u.astype(np.float64) * 7 / (7 + math.exp(float(c.sinks[h])))
        _close(out64[0, h], want, 1e-14, "sink with equal scores")


def pin_two_keys_closed_form(o):
    """pos 1 with RoPE off (inv_freq = 0), unit weights, eps = 0:
    q = c e_0 normalises to sqrt(hd) e_0; history key a_g e_0 and new key e_0
    give scores s0 = scale sqrt(hd) a_g and s1 = scale hd.  Each kv head g has
    its own a_g, which pins which kv head a query head reads."""
    hd = 16
    c = Case(B=1, n_slots=1, slot_ctx=4, n_head=4, n_kv_head=2, hd=hd, eps=0.0,
             scale=0.11)
    c.q_norm_w[:] = 1
    c.k_norm_w[:] = 1
    c.inv_freq[:] = 0
    c.positions = np.array([1], dtype=np.uint32)
    c.q[:] = 0
    c.q[0, :, 0] = 2.5
    c.k_new[:] = 0
    c.k_new[0, :, 0] = 0.5
    a = [1.7, -0.9]
    K = c.K.copy()
    K[0, 0] = 0
    for g in range(2):
        K[0, 0, g, 0] = a[g]
    out, out64, _ = c.run(o, K=K, V=c.V.copy())
    for h in range(c.n_head):
        g = h // 2
        s0 = float(c.scale) * math.sqrt(hd) * float(np.float32(a[g]))
        s1 = float(c.scale) * hd
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        want = w0 * c.V[0, 0, g].astype(np.float64) + (1 - w0) * c.v_new[0, g].astype(np.float64)
        _close(out64[0, h], want, 1e-13, f"two keys head {h}")


def pin_query_scale_invariance(o):
    """With eps = 0, scaling q by c > 0 does not change out (per-head norm)."""
    c = Case(B=2, n_slots=2, slot_ctx=10, eps=0.0)
    c.positions = np.array([9, 3], dtype=np.uint32)
    c.slots = np.array([0, 1], dtype=np.uint32)
    _, a, _ = c.run(o, K=c.K.copy(), V=c.V.copy())
    _, b, _ = c.run(o, K=c.K.copy(), V=c.V.copy(), q=c.q * np.float32(8.0))
    _close(a, b, 1e-12, "q scale invariance")


def pin_stale_history_ignored(o):
    """Bytes past pos in a slot (an earlier occupant's) never reach the output."""
    c = Case(B=2, n_slots=2, slot_ctx=16)
    c.positions = np.array([5, 12], dtype=np.uint32)
    c.slots = np.array([1, 0], dtype=np.uint32)
    out_a, a64, _ = c.run(o, K=c.K.copy(), V=c.V.copy())
    K, V = c.K.copy(), c.V.copy()
    for b in range(c.B):
        K[c.slots[b], c.positions[b] + 1:] = np.nan
        V[c.slots[b], c.positions[b] + 1:] = np.nan
    out_b, b64, _ = c.run(o, K=K, V=V)
    assert np.array_equal(a64, b64)


def pin_out_of_range_rows_skipped(o):
    """A slot >= n_slots or a pos >= slot_ctx breaks the precondition: the
    row is skipped, nothing is written, the other rows are unaffected."""
    c = Case(B=3, n_slots=3, slot_ctx=8)
    c.positions = np.array([2, 8, 3], dtype=np.uint32)
    c.slots = np.array([0, 1, 3], dtype=np.uint32)
    K, V = c.K.copy(), c.V.copy()
    out, _, skipped = c.run(o, K=K, V=V)
    assert skipped == 2
    mask = np.ones(K.shape[:2], dtype=bool)
    mask[0, 2] = False
    assert np.array_equal(K[mask], c.K[mask]) and np.array_equal(V[mask], c.V[mask])
    assert not np.any(out[1]) and not np.any(out[2])
    c1 = Case(B=3, n_slots=3, slot_ctx=8)
    c1.positions, c1.slots = c.positions[:1].copy(), c.slots[:1].copy()
    c1.q, c1.k_new, c1.v_new = c.q[:1], c.k_new[:1], c.v_new[:1]
    c1.B = 1
    out1, _, _ = c1.run(o, K=c.K.copy(), V=c.V.copy())
    assert np.array_equal(out1[0], out[0])


def pin_rows_independent(o):
    """B rows in one call equal B one-row calls, and permuting the rows
    permutes the outputs (the serial per-sequence reference of "Forward
    Cuda")."""
    c = Case(B=4, n_slots=4, slot_ctx=24, n_head=8, n_kv_head=2, hd=16)
    c.positions = np.array([23, 0, 9, 16], dtype=np.uint32)
    c.slots = np.array([2, 3, 0, 1], dtype=np.uint32)
    K_all, V_all = c.K.copy(), c.V.copy()
    out_all, _, _ = c.run(o, K=K_all, V=V_all)
    K1, V1 = c.K.copy(), c.V.copy()
    for b in range(c.B):
        out1, _, _ = c.run(o, K=K1, V=V1, q=c.q[b:b + 1], k_new=c.k_new[b:b + 1],
                           v_new=c.v_new[b:b + 1], positions=c.positions[b:b + 1],
                           slots=c.slots[b:b + 1])
        assert np.array_equal(out1[0], out_all[b])
    assert np.array_equal(K1, K_all) and np.array_equal(V1, V_all)
    perm = np.array([2, 0, 3, 1])
    out_p, _, _ = c.run(o, K=c.K.copy(), V=c.V.copy(), q=c.q[perm], k_new=c.k_new[perm],
                        v_new=c.v_new[perm], positions=c.positions[perm],
                        slots=c.slots[perm])
    assert np.array_equal(out_p, out_all[perm])


def pin_shifted_two_step_sequence(o):
    """Two consecutive steps, at pos d and then d+1 (the second reads the
    first one's K/V write).  Attention over RoPE'd keys sees relative
    positions only, so the two live keys get the same scores for every d.
    The d rows before them hold K = 0 and V = 0: score 0, no value.  Hence
    out_d = N / (Z + d) with N and Z independent of d, i.e. per query head
    out_d / out_0 is one constant Z / (Z + d) over the head's elements.
    Power-of-two frequencies keep the f32 angles exact; the step-one key is
    stored in f32, which bounds the agreement at about 1e-7."""
    hd = 16
    rng = np.random.default_rng(12)
    q2 = rng.standard_normal((1, 2, hd)).astype(np.float32)
    k2 = rng.standard_normal((1, 1, hd)).astype(np.float32)
    v2 = rng.standard_normal((1, 1, hd)).astype(np.float32)
    outs = {}
    for d in (0, 3, 10):
        c = Case(B=1, n_slots=1, slot_ctx=16, n_head=2, n_kv_head=1, hd=hd, seed=11)
        c.inv_freq = (2.0 ** -np.arange(hd // 2)).astype(np.float32)
        K, V = c.K.copy(), c.V.copy()
        K[0, :d] = 0
        V[0, :d] = 0
        c.run(o, K=K, V=V, positions=np.array([d], dtype=np.uint32))
        _, outs[d], _ = c.run(o, K=K, V=V, q=q2, k_new=k2, v_new=v2,
                              positions=np.array([d + 1], dtype=np.uint32))
    for h in range(2):
        base = outs[0][0, h]
        big = np.abs(base) > 1e-3
        assert big.sum() > 4
        for d in (3, 10):
            r = outs[d][0, h][big] / base[big]
            assert np.ptp(r) < 1e-7, (h, d, np.ptp(r))
            assert 0.0 < r[0] < 1.0


def pin_one_dominant_key(o):
    """A history key far along q (score ~1e3 above the rest) takes all the
    weight: out equals that key's value row.  The scores are far beyond
    exp's range, so this also pins the max subtraction."""
    c = Case(B=1, n_slots=1, slot_ctx=12, n_head=2, n_kv_head=1, hd=8, eps=0.0)
    c.q_norm_w[:] = 1
    c.inv_freq[:] = 0
    c.positions = np.array([9], dtype=np.uint32)
    c.q[:] = 0
    c.q[0, :, 3] = 1.0
    K = c.K.copy()
    K[0, :10] = np.clip(K[0, :10], -1, 1)
    K[0, 6, 0, 3] = 4000.0
    out, out64, _ = c.run(o, K=K, V=c.V.copy())
    for h in range(2):
        _close(out64[0, h], c.V[0, 6, 0].astype(np.float64), 1e-300, "dominant key")


def pin_option_norm_plus_one(o):
    """Gemma's norm form: with NORM_PLUS_ONE the written K at pos 0 is torch's
    RMS norm with weight (1 + w), and the whole step equals the plain step
    run with weights fl32(1 + w) (up to that one rounding)."""
    import oracle as oracle_pkg
    c = Case(B=2, n_slots=2, slot_ctx=12, n_head=4, n_kv_head=2, hd=16)
    c.positions = np.array([0, 9], dtype=np.uint32)
    c.slots = np.array([1, 0], dtype=np.uint32)
    c.q_norm_w = (0.1 * np.random.default_rng(21).standard_normal(16)).astype(np.float32)
    c.k_norm_w = (0.1 * np.random.default_rng(22).standard_normal(16)).astype(np.float32)
    K, V = c.K.copy(), c.V.copy()
    _, a64, _ = c.run(o, K=K, V=V, flags=oracle_pkg.NORM_PLUS_ONE)
    ref = torch.nn.functional.rms_norm(
        torch.from_numpy(c.k_new[0].astype(np.float64)), (16,),
        torch.from_numpy(1.0 + c.k_norm_w.astype(np.float64)),
        eps=float(np.float32(c.eps))).numpy()
    _close(K[1, 0], ref, 1e-6, "(1+w) written K")
    c2 = Case(B=2, n_slots=2, slot_ctx=12, n_head=4, n_kv_head=2, hd=16)
    c2.positions, c2.slots = c.positions, c.slots
    c2.q_norm_w = (np.float32(1) + c.q_norm_w).astype(np.float32)
    c2.k_norm_w = (np.float32(1) + c.k_norm_w).astype(np.float32)
    _, b64, _ = c2.run(o, K=c.K.copy(), V=c.V.copy())
    _close(a64, b64, 1e-6, "(1+w) vs shifted weights")


def pin_option_vnorm(o):
    """With VNORM the cached V row is the weightless RMS norm of v_new, and at
    pos 0 (only that key) the output is that normed vector."""
    import oracle as oracle_pkg
    c = Case(B=2, n_slots=2, slot_ctx=10, n_head=4, n_kv_head=2, hd=16)
    c.positions = np.array([0, 7], dtype=np.uint32)
    c.slots = np.array([0, 1], dtype=np.uint32)
    K, V = c.K.copy(), c.V.copy()
    _, out64, _ = c.run(o, K=K, V=V, flags=oracle_pkg.VNORM)
    for b in range(2):
        ref = torch.nn.functional.rms_norm(torch.from_numpy(c.v_new[b].astype(np.float64)),
                                           (16,), eps=float(np.float32(c.eps))).numpy()
        _close(V[c.slots[b], c.positions[b]], ref, 1e-6, "normed V row")
        if c.positions[b] == 0:
            for h in range(4):
                assert np.array_equal(out64[b, h], V[0, 0, h // 2].astype(np.float64))
    # the history rows are used as stored
    mask = np.ones(K.shape[:2], dtype=bool)
    mask[0, 0] = mask[1, 7] = False
    assert np.array_equal(V[mask], c.V[mask])


def pin_brute_force_tiny(o):
    """The tiny workload against an all-at-once f64 formulation: scores
    materialised as one matrix, softmax from scipy, norm from torch."""
    import scipy.special

    w = synth.WORKLOADS["tiny"]
    K0 = synth.normal(w.kv_elems(), w.seed, synth.S_HIST_K).reshape(
        w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    V0 = synth.normal(w.kv_elems(), w.seed, synth.S_HIST_V).reshape(K0.shape)
    pos, slots = w.positions0(), w.slots()
    q, kn, vn = w.q(), w.k_new(), w.v_new()
    qw, kw, inv = w.q_norm_w(), w.k_norm_w(), w.inv_freq()
    K, V = K0.copy(), V0.copy()
    out, out64, _ = o.decode_batch(K, V, q, kn, vn, pos, slots, qw, kw, inv, None,
                                   w.eps, w.scale, want64=True)
    hd, half = w.head_dim, w.head_dim // 2
    g = w.n_head // w.n_kv_head

    def norm_t(x, wt):
        return torch.nn.functional.rms_norm(torch.from_numpy(x.astype(np.float64)), (hd,),
                                            torch.from_numpy(wt.astype(np.float64)),
                                            eps=float(np.float32(w.eps))).numpy()

    for b in range(w.B):
        p, s = int(pos[b]), int(slots[b])
        ang = (np.float32(p) * inv).astype(np.float64)          # f32 products
        rot = np.zeros((hd, hd))
        for i in range(half):
            c_, s_ = math.cos(ang[i]), math.sin(ang[i])
            rot[i, i], rot[i, i + half] = c_, -s_
            rot[i + half, i], rot[i + half, i + half] = s_, c_
        kr = norm_t(kn[b], kw) @ rot.T                          # [n_kv][hd]
        assert np.array_equal(K[s, p], kr.astype(np.float32))
        keys = K0[s, : p + 1].astype(np.float64).copy()
        keys[p] = kr.astype(np.float32)
        vals = V0[s, : p + 1].astype(np.float64).copy()
        vals[p] = vn[b]
        qr = norm_t(q[b], qw) @ rot.T                           # [n_head][hd]
        for h in range(w.n_head):
            scores = float(w.scale) * keys[:, h // g, :] @ qr[h]
            prob = scipy.special.softmax(scores)
            _close(out64[b, h], prob @ vals[:, h // g, :], 1e-12, f"brute b={b} h={h}")


def _paged_from_slots(c, bs, rng, spare=3):
    """Scatter the slot buffers of case ``c`` into a pool of blocks of ``bs``
    positions under a random block permutation (plus ``spare`` unused blocks
    filled with other data).  Returns (Kp, Vp, tables[n_slots][slot_ctx/bs])."""
    per = c.slot_ctx // bs
    n_blocks = c.n_slots * per + spare
    perm = rng.permutation(n_blocks)[: c.n_slots * per]
    tables = perm.reshape(c.n_slots, per).astype(np.uint32)
    Kp = rng.standard_normal((n_blocks, bs, c.n_kv_head, c.hd)).astype(np.float32)
    Vp = rng.standard_normal(Kp.shape).astype(np.float32)
    for s in range(c.n_slots):
        for i in range(per):
            Kp[tables[s, i]] = c.K[s, i * bs:(i + 1) * bs]
            Vp[tables[s, i]] = c.V[s, i * bs:(i + 1) * bs]
    return Kp, Vp, tables


def pin_paged_is_an_addressing_change(o):
    """Paged KV (the Qwen3SsmLayer page, decode_multi_seq over per-sequence
    block tables) changes where a key lives, not what is computed: scattering
    each slot's rows into shuffled blocks and passing the matching tables gives
    the slot step's output bit for bit, and the key/value write lands in block
    table[pos // bs] at offset pos % bs."""
    rng = np.random.default_rng(31)
    bs = 4
    c = Case(B=3, n_slots=3, slot_ctx=16, n_head=4, n_kv_head=2, hd=8)
    c.positions = np.array([13, 2, 8], dtype=np.uint32)
    c.slots = np.array([1, 2, 0], dtype=np.uint32)
    Kp, Vp, tables = _paged_from_slots(c, bs, rng)
    K, V = c.K.copy(), c.V.copy()
    _, ref64, _ = c.run(o, K=K, V=V)
    bt = tables[c.slots]
    Kp0, Vp0 = Kp.copy(), Vp.copy()
    _, got64, skipped = o.decode_batch_paged(
        Kp, Vp, c.q, c.k_new, c.v_new, c.positions, bt, c.q_norm_w, c.k_norm_w,
        c.inv_freq, None, c.eps, c.scale, want64=True)
    assert skipped == 0
    assert np.array_equal(got64, ref64)
    written = np.zeros(Kp.shape[:2], dtype=bool)
    for b in range(c.B):
        p = int(c.positions[b])
        blk, off = bt[b, p // bs], p % bs
        written[blk, off] = True
        assert np.array_equal(Kp[blk, off], K[c.slots[b], p])
        assert np.array_equal(Vp[blk, off], c.v_new[b])
    assert np.array_equal(Kp[~written], Kp0[~written])
    assert np.array_equal(Vp[~written], Vp0[~written])


def pin_paged_brute_force(o):
    """Paged step on a tiny case against keys gathered one by one through the
    table, softmax from scipy: every row reads only its own blocks."""
    import scipy.special

    rng = np.random.default_rng(32)
    bs, nb, hd = 2, 9, 8
    c = Case(B=2, n_slots=1, slot_ctx=2, n_head=2, n_kv_head=1, hd=hd)
    Kp = rng.standard_normal((nb, bs, 1, hd)).astype(np.float32)
    Vp = rng.standard_normal(Kp.shape).astype(np.float32)
    bt = np.array([[7, 2, 5, 0], [3, 8, 1, 6]], dtype=np.uint32)
    pos = np.array([6, 3], dtype=np.uint32)
    K, V = Kp.copy(), Vp.copy()
    _, out64, skipped = o.decode_batch_paged(
        K, V, c.q, c.k_new, c.v_new, pos, bt, c.q_norm_w, c.k_norm_w, c.inv_freq, None,
        c.eps, c.scale, want64=True)
    assert skipped == 0
    for b in range(2):
        p = int(pos[b])
        keys = np.stack([K[bt[b, t // bs], t % bs, 0] for t in range(p + 1)]).astype(np.float64)
        vals = np.stack([V[bt[b, t // bs], t % bs, 0] for t in range(p + 1)]).astype(np.float64)
        # the history rows come from the untouched pool, the last from the write
        for t in range(p):
            assert np.array_equal(keys[t], Kp[bt[b, t // bs], t % bs, 0])
        assert np.array_equal(vals[p], c.v_new[b, 0])
        for h in range(2):
            qr = o.norm_rope_head(c.q[b, h], c.q_norm_w, c.eps, p, c.inv_freq)
            prob = scipy.special.softmax(float(c.scale) * keys @ qr)
            _close(out64[b, h], prob @ vals, 1e-12, f"paged brute b={b} h={h}")


def pin_paged_out_of_range(o):
    """A row is skipped (nothing written, output zero) when a block it uses
    (blocks 0..pos // bs of its table) is not in the pool, or when pos is past
    its table; ids in table entries beyond its last used block are never read."""
    rng = np.random.default_rng(33)
    bs, nb, hd = 4, 6, 8
    c = Case(B=4, n_slots=1, slot_ctx=4, n_head=2, n_kv_head=1, hd=hd)
    Kp = rng.standard_normal((nb, bs, 1, hd)).astype(np.float32)
    Vp = rng.standard_normal(Kp.shape).astype(np.float32)
    bad = np.uint32(nb)
    bt = np.array([[0, 1, bad],       # pos 5 uses blocks 0, 1: fine, entry 2 unused
                   [2, bad, 3],       # pos 6 uses block entry 1: skipped
                   [4, 5, 3],         # pos 12 = 3 * bs, past the table: skipped
                   [bad, 3, 3]],      # pos 0 uses entry 0: skipped
                  dtype=np.uint32)
    pos = np.array([5, 6, 12, 0], dtype=np.uint32)
    c.q = rng.standard_normal((4, 2, hd)).astype(np.float32)
    c.k_new = rng.standard_normal((4, 1, hd)).astype(np.float32)
    c.v_new = rng.standard_normal((4, 1, hd)).astype(np.float32)
    K, V = Kp.copy(), Vp.copy()
    out, _, skipped = o.decode_batch_paged(
        K, V, c.q, c.k_new, c.v_new, pos, bt, c.q_norm_w, c.k_norm_w, c.inv_freq, None,
        c.eps, c.scale)
    assert skipped == 3
    assert np.any(out[0]) and not np.any(out[1:])
    mask = np.ones(K.shape[:2], dtype=bool)
    mask[1, 1] = False                # row 0's write: block 1, offset 1
    assert np.array_equal(K[mask], Kp[mask]) and np.array_equal(V[mask], Vp[mask])
    assert np.array_equal(V[1, 1], c.v_new[0])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

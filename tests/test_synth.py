"""The synthetic input generator: published hash values, moments, regeneration."""
import ctypes

import numpy as np
import pytest

import synth


def test_splitmix64_published_first_output():
    # SplitMix64 seeded with 0 first returns mix64(0 + golden) = 0xE220A8397B1DCDAF
    lib = synth.host_lib()
    # synth_key_of(seed, stream) = mix64(seed ^ mix64(stream + golden)); with
    # stream = 0 the inner value is that first output
    key = lib.synth_key_of(0, 0)
    assert key != 0
    inner = 0xE220A8397B1DCDAF
    z = inner
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & (2**64 - 1)
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & (2**64 - 1)
    z ^= z >> 31
    assert key == z


def test_normal_moments_and_support():
    x = synth.normal(1 << 20, 123, 1).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1.0) < 1e-2
    assert np.abs(x).max() <= 3.4642
    # symmetric, light-tailed, bell shaped: about 68% within one sd
    assert 0.66 < np.mean(np.abs(x) < 1) < 0.70


def test_values_regenerate_piecewise():
    full = synth.normal(10000, 99, 2)
    part = synth.normal(777, 99, 2, index0=1234)
    assert np.array_equal(full[1234:1234 + 777], part)
    assert not np.array_equal(synth.normal(100, 99, 3), full[:100])


def test_affine_is_two_rounded_ops():
    x = synth.normal(1000, 5, 6)
    y = synth.normal_affine(1000, 5, 6, 1.0, 0.1)
    want = (x * np.float32(0.1)).astype(np.float32) + np.float32(1.0)
    assert np.array_equal(y, want.astype(np.float32))


def test_subsets_and_permutations():
    p = synth.subset(100, 100, 1, 2)
    assert sorted(p.tolist()) == list(range(100))
    s = synth.subset(512, 256, 3, 4)
    assert len(set(s.tolist())) == 256 and s.max() < 512


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_shapes(name):
    w = synth.WORKLOADS[name]
    pos, slots = w.positions0(), w.slots()
    assert pos.shape == (w.B,) and slots.shape == (w.B,)
    assert len(set(slots.tolist())) == w.B and slots.max() < w.n_slots
    assert (pos + w.steps - 1).max() < w.slot_ctx
    assert w.q().shape == (w.B, w.n_head, w.head_dim)
    assert w.k_new(1).shape == (w.B, w.n_kv_head, w.head_dim)
    assert w.n_head % w.n_kv_head == 0
    if name == "tiny":
        assert pos.tolist() == [0, 5, 17, 63]
    if name == "skewed":
        assert pos[0::2].tolist() == [16] * 32 and pos[1::2].tolist() == [32767] * 32
    if name == "large":
        assert pos.max() <= 1983


def test_history_rows_match_flat_index():
    w = synth.WORKLOADS["tiny"]
    flat = synth.normal(w.kv_elems(), w.seed, synth.S_HIST_K).reshape(
        w.n_slots, w.slot_ctx, w.n_kv_head, w.head_dim)
    rows = w.hist_rows("k", 2, 5, 17)
    assert np.array_equal(rows, flat[2, 5:17])

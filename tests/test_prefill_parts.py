"""Where prefill_batch_attn_host cuts a call (slot_kv_prefill_host_parts,
host logic only): parts whose tokens share no slot, one per 512 tokens and
at most eight, none under 256 tokens, each cut the allowed one nearest its
target, the targets giving the first and the last part half the size of the
others; a call that cannot be cut that way stays whole.  Each part is a
prefill of its own, so a cut with a slot on both sides would let one part's
tokens miss keys the other part writes ("Forward Cuda Gemma", prefillBatched:
every token attends its own slot's keys 0..pos)."""
import numpy as np
import pytest

import sequence_slot_kv_gb300 as skv
from sequence_slot_kv_gb300 import slot_kv_prefill_host_parts as parts


def _seqs(lengths, slot_ids=None):
    ids = range(len(lengths)) if slot_ids is None else slot_ids
    return np.concatenate([np.full(n, s, np.uint32) for s, n in zip(ids, lengths)])


def _check_valid(slots, cuts):
    n = len(slots)
    assert cuts[0] == 0 and cuts[-1] == n
    assert all(a < b for a, b in zip(cuts, cuts[1:]))
    assert len(cuts) - 1 <= min(skv.PREFILL_HOST_MAX_PARTS, max(1, n // 512))
    if len(cuts) > 2:
        assert all(b - a >= 256 for a, b in zip(cuts, cuts[1:]))
    for m in cuts[1:-1]:
        assert not set(slots[:m].tolist()) & set(slots[m:].tolist())


def test_small_calls_stay_whole():
    assert parts([]) == [0, 0]  # one empty part
    assert parts(_seqs([400, 500])) == [0, 900]
    assert parts(_seqs([511, 512])) == [0, 1023]
    # from 1024 tokens on: two parts
    assert parts(_seqs([700, 700])) == [0, 700, 1400]


def test_equal_sequences_cut_at_their_boundaries():
    # eight parts, targets 4096 * (1, 3, .., 13) / 14 = 293, 878, .., 3803:
    # every sequence boundary is the nearest allowed cut of one target
    assert parts(_seqs([512] * 8)) == [0, 512, 1024, 1536, 2048, 2560, 3072, 3584, 4096]
    # four parts wanted (targets 341, 1024, 1707); one cut allowed
    assert parts(_seqs([1024] * 2)) == [0, 1024, 2048]
    # eight parts wanted, seven sequences: targets 500, 1500, ..; of two
    # cuts equally near, the first not too close to the previous cut
    assert parts(_seqs([1000] * 7)) == [0, 1000, 2000, 3000, 4000, 5000, 6000, 7000]


def test_half_size_ends():
    # sixteen 256-token sequences, eight parts: the targets 4096 * (1, 3, ..,
    # 13) / 14 = 292, 877, 1462, 2048, 2633, 3218, 3803 snap to the nearest
    # sequence boundaries, so the first and the last part hold one sequence
    # and the others two or three
    assert parts(_seqs([256] * 16)) == [0, 256, 768, 1536, 2048, 2560, 3328, 3840, 4096]


def test_no_allowed_cut_keeps_one_part():
    assert parts(np.full(3000, 5, np.uint32)) == [0, 3000]
    # two slots interleaved token by token: every prefix holds both
    assert parts(np.tile(np.array([1, 2], np.uint32), 2048)) == [0, 4096]
    # a slot at both ends
    assert parts(_seqs([10, 4000, 10], [7, 8, 7])) == [0, 4020]


def test_uneven_sequences_take_the_nearest_allowed_cuts():
    # targets 4200 * (1, 3, .., 13) / 14 = 300, 900, ..; allowed cuts 1500,
    # 1600, 2500: the first two targets take 1500 and 2500, and no allowed
    # cut is left for the others
    assert parts(_seqs([1500, 100, 900, 1700])) == [0, 1500, 2500, 4200]


def test_a_slot_returning_later_joins_its_part():
    # slot 0 again after slot 1: nothing may cut between its runs
    s = _seqs([800, 800, 800, 800], [0, 1, 0, 2])
    cuts = parts(s)
    _check_valid(s, cuts)
    assert cuts == [0, 2400, 3200]


@pytest.mark.parametrize("seed", range(40))
def test_random_layouts(seed):
    rng = np.random.default_rng(seed)
    k = int(rng.integers(1, 12))
    lengths = rng.integers(1, 1500, size=k)
    ids = rng.integers(0, max(1, k - int(rng.integers(0, 3))), size=k)
    s = _seqs(lengths, ids)
    if seed % 4 == 0:  # a few tokens moved to other places
        idx = rng.choice(len(s), size=min(len(s), 5), replace=False)
        s[idx] = s[rng.permutation(idx)]
    _check_valid(s, parts(s))


def test_bad_arguments_are_refused():
    import ctypes
    n = ctypes.c_uint32()
    k = skv.PREFILL_HOST_MAX_PARTS + 1
    cuts = (ctypes.c_uint32 * k)()
    assert skv._lib.slot_kv_prefill_host_parts(4, None, cuts, k, ctypes.byref(n)) == 1
    assert skv._lib.slot_kv_prefill_host_parts(0, None, None, k, ctypes.byref(n)) == 1
    # a cuts array too short for the most parts a call can have
    s = _seqs([512] * 8)
    assert skv._lib.slot_kv_prefill_host_parts(len(s), s.ctypes.data, cuts, k - 1,
                                               ctypes.byref(n)) == 1
    assert skv._lib.slot_kv_prefill_host_parts(0, None, cuts, k, ctypes.byref(n)) == 0
    assert n.value == 1 and cuts[0] == 0 and cuts[1] == 0


def test_python_constant_matches_the_header():
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "include", "slotkv.h")) as f:
        m = re.search(r"#define SLOTKV_PREFILL_HOST_MAX_PARTS (\d+)u", f.read())
    assert m and int(m.group(1)) == skv.PREFILL_HOST_MAX_PARTS

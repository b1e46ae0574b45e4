"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is a copy of ``oracle/oracle.c`` with one plausible mistake
(a dropped term, a wrong sign or index, a swapped operand), compiled into a
temporary directory.  The real oracle is never modified.  A mutant that
passes every pin would mean the pins leave that part of the oracle unchecked.
"""
import os
import shutil
import subprocess
import sys

import pytest

import oracle
import oracle_pins
from oracle import build as obuild

# (name, original snippet, mutated snippet, replace every occurrence?)
MUTANTS = [
    ("sink_dropped_from_denominator",
     "if (j->sinks) denom += exp(sink - m);", ";", False),
    ("sink_scaled_like_a_score",
     "sink = (double)j->sinks[h];", "sink = (double)j->scale * j->sinks[h];", False),
    ("rope_first_row_sign",
     "y[i] = x0 * c - x1 * s;", "y[i] = x0 * c + x1 * s;", False),
    ("rope_second_row_sign",
     "y[i + half] = x1 * c + x0 * s;", "y[i + half] = x1 * c - x0 * s;", False),
    ("rope_adjacent_pairs",
     "uint32_t half = hd / 2;", "uint32_t half = 1;", False),
    ("rope_angle_in_f64",
     "float angle_f32 = (float)pos * inv_freq[i];",
     "double angle_f32 = (double)pos * (double)inv_freq[i];", False),
    ("range_excludes_pos",
     "t <= p;", "t < p;", True),
    ("values_read_from_k",
     "const float* v_row = j->V + key_offset", "const float* v_row = j->K + key_offset", False),
    ("gqa_interleaved_heads",
     "const uint32_t g = h / group;", "const uint32_t g = h % j->n_kv_head;", False),
    ("score_unscaled",
     "score[t] = (double)j->scale * dot;", "score[t] = dot;", False),
    ("norm_weight_plus_one",
     "y[i] = (double)x[i] * inv_rms * (double)w[i];",
     "y[i] = (double)x[i] * inv_rms * (1.0 + (double)w[i]);", False),
    ("eps_outside_sqrt",
     "1.0 / sqrt(sum_sq / (double)n + eps);", "1.0 / (sqrt(sum_sq / (double)n) + eps);",
     True),
    ("norm_over_sum_not_mean",
     "sqrt(sum_sq / (double)n + eps)", "sqrt(sum_sq + eps)", True),
    ("cached_k_not_rotated",
     "oracle_norm_rope_head(k_in, j->k_norm_w, hd, j->eps, p, j->inv_freq, kv);",
     "oracle_norm_rope_head(k_in, j->k_norm_w, hd, j->eps, 0, j->inv_freq, kv);", False),
    ("query_not_rotated",
     "oracle_norm_rope_head(q_in, j->q_norm_w, hd, j->eps, p, j->inv_freq, qv);",
     "oracle_norm_rope_head(q_in, j->q_norm_w, hd, j->eps, 0, j->inv_freq, qv);", False),
    ("query_uses_k_norm_weight",
     "oracle_norm_rope_head(q_in, j->q_norm_w,", "oracle_norm_rope_head(q_in, j->k_norm_w,",
     False),
    ("cached_v_not_raw",
     "j->V[at_p + (uint64_t)g * hd + i] = v_in[i];",
     "j->V[at_p + (uint64_t)g * hd + i] = (float)kv[i];", False),
    ("offset_missing_slot_ctx",
     "return ((uint64_t)slot * slot_ctx + pos)", "return ((uint64_t)slot + pos)", False),
    ("row_base_ignores_slot",
     "return ((uint64_t)j->slots[b] * j->slot_ctx + t) * kv_dim;",
     "return ((uint64_t)t) * kv_dim;", False),
    ("paged_table_ignored",
     "if (j->block_tables) {", "if (0) {", False),
    ("paged_block_index_dropped",
     "j->block_tables[(uint64_t)b * j->bt_stride + t / j->slot_ctx];",
     "j->block_tables[(uint64_t)b * j->bt_stride];", False),
    ("paged_block_and_offset_swapped",
     "j->block_tables[(uint64_t)b * j->bt_stride + t / j->slot_ctx];",
     "j->block_tables[(uint64_t)b * j->bt_stride + t % j->slot_ctx];", False),
    ("paged_table_row_stride_dropped",
     "j->block_tables[(uint64_t)b * j->bt_stride + t / j->slot_ctx];",
     "j->block_tables[t / j->slot_ctx];", False),
    ("paged_range_checks_first_block_only",
     "for (uint32_t i = 0; i <= p / j->slot_ctx; ++i)",
     "for (uint32_t i = 0; i < 1; ++i)", False),
    ("vnorm_with_weight",
     "rms_norm_gemma(v_in, NULL, hd,", "rms_norm_gemma(v_in, j->k_norm_w, hd,", False),
    ("vnorm_ignored",
     "if (j->flags & ORACLE_VNORM) {", "if (0) {", False),
    ("plus_one_dropped",
     "(w ? 1.0 + (double)w[i] : 1.0)", "(w ? (double)w[i] : 1.0)", False),
    ("exp_without_max_subtraction",
     "score[t] = exp(score[t] - m);", "score[t] = exp(score[t]);", False),
    ("max_taken_over_first_key_only",
     "if (score[t] > m) m = score[t];", "if (t == 0) m = score[t];", False),
]


# Mutants of the paged addressing can index outside the pool (or, with the
# table ignored, the absent slot array): their pins run in a child process, and
# a crash there counts as caught.
ISOLATED = {"paged_table_ignored", "paged_block_and_offset_swapped",
            "paged_table_row_stride_dropped", "paged_range_checks_first_block_only",
            "paged_block_index_dropped"}

_CHILD = """
import sys
import oracle, oracle_pins
lib = oracle.Oracle(sys.argv[1])
caught = 0
for pin in oracle_pins.ALL_PINS:
    try:
        pin(lib)
    except Exception:
        caught += 1
sys.exit(3 if caught else 0)
"""


def _mutant_lib(tmp_path, name, old, new, every):
    src = open(obuild.SRC).read()
    n = src.count(old)
    assert n >= 1, f"mutant {name}: snippet not found in oracle.c"
    if not every:
        assert n == 1, f"mutant {name}: snippet is not unique in oracle.c"
    mutated = src.replace(old, new) if every else src.replace(old, new, 1)
    d = tmp_path / name
    d.mkdir()
    shutil.copy(os.path.join(obuild.HERE, "oracle.h"), d / "oracle.h")
    (d / "oracle.c").write_text(mutated)
    return obuild.build_oracle(str(d / "oracle.c"), str(d / "liboracle.so"), str(d))


@pytest.mark.parametrize("name,old,new,every", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, every):
    path = _mutant_lib(tmp_path, name, old, new, every)
    if name in ISOLATED:
        here = os.path.dirname(os.path.abspath(__file__))
        env = dict(os.environ)
        env["PYTHONPATH"] = os.pathsep.join([here, os.path.dirname(here),
                                             env.get("PYTHONPATH", "")])
        r = subprocess.run([sys.executable, "-c", _CHILD, path], cwd=here, env=env,
                           capture_output=True, timeout=600)
        assert r.returncode != 0, f"mutant {name} passed every pin"
        return
    lib = oracle.Oracle(path)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except Exception:  # noqa: BLE001 -- any failure counts as caught
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"

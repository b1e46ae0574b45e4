"""bench.py's reference arm (the CPU oracle) keeps the line the benchmark
contract asks for, for the decode, paged, norm-option and prefill
workloads; and the line's rate is the rows the sample holds over the time
it took.  CPU only: the arm never touches a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e"}


def _run(*flags):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3", *flags],
                         cwd=ROOT, capture_output=True, text=True, timeout=600,
                         env=dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0"))
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("flags", [(), ("--paged", "64", "--options", "both"), ("--prefill",)],
                         ids=["decode", "paged_options", "prefill"])
def test_reference_line(flags):
    d = _run(*flags)
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["warmup"] >= 3 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and cb["sample"]
    # value = units in one step's sample / the step's time
    per_step = d["value"] * d["ms_per_step"] / 1e3
    if "--prefill" in flags:
        assert d["unit"] == "tokens/s" and d["config"]["workload"] == "prefill"
        assert per_step == pytest.approx(8)
        # one sequence per thread: the threads the oracle actually ran
        assert cb["cores"] == min(os.cpu_count() or 1, 8)
    else:
        assert d["unit"] == "rows/s" and d["config"]["workload"] == "large"
        assert per_step == pytest.approx(min(256, cb["cores"]))
    if "--paged" in flags:
        assert d["config"]["kv_layout"] == "paged" and d["config"]["block_size"] == 64
        assert "norm_options" in d["config"]

"""bench.py's CUDA arm keeps the line the benchmark contract asks for: one
JSON line with the metric, the whole-job value, the roofline block (bound,
achieved, peak, unit, fraction), the end-to-end rate through the host entry
with the bytes it copies, the launches it claims, the clocks it saw and the
CPU baseline; for decode (a small workload) and for the batched prefill."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
        "e2e", "gpu_launches", "clocks", "cpu_baseline"}


def _run(*flags):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3",
                          "--warmup", "3", "--cpu-budget", "0.3", *flags],
                         cwd=ROOT, capture_output=True, text=True, timeout=900,
                         env=dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0"))
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def _check_common(d):
    assert KEYS <= set(d), KEYS - set(d)
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["data"] == "synthetic" and d["value"] > 0 and d["ms_per_step"] > 0
    r = d["roofline"]
    assert r["bound"] in ("hbm", "tensor") and r["unit"] in ("GB/s", "TFLOP/s")
    assert r["achieved"] > 0 and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-6)
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= d["steps"]
    c = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(c)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    assert cb["single_thread"]["value"] > 0


def test_decode_line():
    d = _run("--workload", "tiny", "--no-per-config")
    _check_common(d)
    assert d["unit"] == "rows/s" and d["config"]["workload"] == "tiny"
    assert d["roofline"]["bound"] == "hbm" and d["roofline"]["unit"] == "GB/s"


def test_prefill_line():
    d = _run("--prefill")
    _check_common(d)
    assert d["unit"] == "tokens/s" and d["config"]["workload"] == "prefill"
    assert d["roofline"]["bound"] == "tensor" and d["roofline"]["unit"] == "TFLOP/s"

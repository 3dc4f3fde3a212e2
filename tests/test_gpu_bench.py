"""The benchmark's JSON contract on the GPU: the default (stage-3) line and
the other workload kinds' lines carry every key the contract asks for, on a
scaled-down case so that the test stays short."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
        "clocks", "e2e", "gpu_launches")


def _line(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [x for x in out.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,extra", [("llama-7b-stage3", ()), ("gpt2-small", ()),
                                            ("llama-1.4b", ()),
                                            ("llama-7b-stage3", ("--grad-dtype", "f32"))])
def test_bench_line_keys(cuda, workload, extra):
    d = _line("--workload", workload, "--scale", "16", "--steps", "3", "--warmup", "3",
              "--no-cpu-baseline", *extra)
    for k in KEYS:
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["unit"] == "Gparams/s"
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic", "peak_nominal_gbs"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["achieved"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in e, k
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0 and e["value"] > 0
    assert d["gpu_launches"] > 0 and "workload" in d["config"]
    if extra:
        assert d["config"]["grad_dtype"] == "f32" and "f32" in r["kernel"]
        assert d["config"]["bytes_per_step"] == d["config"]["psi"] * (16 * 4 + 26)
    if workload == "llama-7b-stage3":
        assert d["gpu_launches"] == 34 * 3 and d["config"]["groups"] == 34
        g = d["gather"]
        assert g["launches"] == 68 and g["gathers_only_ms"] > 0 and g["broadcast_ms"] > 0

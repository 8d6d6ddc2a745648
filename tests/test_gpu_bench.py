"""bench.py end to end on the GPU, on a small shape: one JSON line carrying
every key of the benchmark contract, with figures that agree with each other
(tokens/s with the step time, the roofline fraction with its achieved rate and
peak, the launch count, the end-to-end copy bytes)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         check=True, capture_output=True, text=True, timeout=900).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out[-2000:]
    return json.loads(lines[0])


def test_bench_line_small_shape():
    N, H, V, steps = 1024, 512, 4096, 3
    d = _bench("--shape", f"{N},{H},{V}", "--steps", str(steps), "--warmup", "3",
               "--cpu-baseline-rows", "16")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
              "cpu_baseline", "e2e", "gpu_launches", "clocks", "kernels", "step_roofline"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == 3
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] == pytest.approx(N * steps / (d["ms_per_step"] * steps / 1e3), rel=1e-6)
    cfg = d["config"]
    assert cfg["N"] == N and cfg["H"] == H and cfg["V"] == V
    assert cfg["workload"].startswith("llama3_n8192")
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-9)
    # a loop this short is stated against the burst peak
    assert r["peak"] == r["peak_burst"] and "burst" in r["peak_source"]
    assert r["kernel"] in d["kernels"] and r["achieved"] == d["kernels"][r["kernel"]]["tflops"]
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0
    e = d["e2e"]
    assert e["unit"] == "tokens/s" and e["value"] > 0
    assert e["h2d_bytes_per_step"] == N * H * 2 + V * H * 2 + N * 8
    assert e["d2h_bytes_per_step"] == 4
    # every step launches our kernels: at least the forward, merge, finalize and three per chunk
    assert d["gpu_launches"] >= steps * 6
    assert d["engine"]["vocab_chunk"] > 0

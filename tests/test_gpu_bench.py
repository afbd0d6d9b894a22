"""The benchmark's JSON line, end to end on the tiny workload: one line with
the contract's keys (metric, value, unit, steps, warmup, roofline with its
algorithmic bytes and measured peak, e2e with the bytes copied per step,
clocks, gpu_launches) and a per_config entry, and a reference arm that
reports the same config and step count."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_contract_on_the_tiny_workload():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = run_bench("--workload", "tiny", "--steps", "4", "--warmup", "3", "--configs", "llama7b_p1024",
                  "--no-cpu-baseline", "--no-context")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["steps"] == 4 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["higher_is_better"] is False
    assert d["value"] > 0 and abs(d["ms_per_step"] * 1e3 - d["value"]) < 1e-2
    assert d["gpu_launches"] == 2 * 4                       # attention + merge per timed step
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0 and rf["kernel_us"] > 0
    assert rf["algorithmic_bytes"] == d["config"]["unique_kv_bytes"] + 2 * 4 * 2 * 64 * 2
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert d["e2e"]["h2d_bytes_per_step"] == d["e2e"]["d2h_bytes_per_step"] == 4 * 2 * 64 * 2
    assert set(d["per_config"]) == {"tiny", "llama7b_p1024"}
    e = d["per_config"]["llama7b_p1024"]
    assert e["config"] == "2" and e["us_per_call"] > 0 and e["isolated_call_us"] > 0 and e["kernel_us"] > 0
    assert e["pool_copies"] >= 2                           # 272 MB of KV is under 4 x L2


def test_reference_arm_matches_the_config():
    ref = run_bench("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1")
    ours = run_bench("--workload", "tiny", "--steps", "2", "--warmup", "3", "--quick")
    assert ref["impl"] == "reference" and ref["steps"] == 2 and ref["config"] == ours["config"]

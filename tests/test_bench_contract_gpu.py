"""bench.py's JSON line on a GPU: one short run of the default workload must
print every key the measurement contract names, with consistent values."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_default_bench_line_has_the_contract_keys():
    res = subprocess.run([sys.executable, "bench.py", "--steps", "5", "--warmup", "3", "--cpu-seconds", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks",
                "gpu_launches"):
        assert key in line, f"missing {key}"
    assert line["steps"] == 5 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["config"]["workload"] == "bf16_gqa_causal_b2_hq32_hkv8_l4096_d128"
    r = line["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert 0.0 < r["frac"] < 1.5
    e = line["e2e"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0 and 0 < e["value"] <= line["value"] * 1.01
    c = line["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0
    assert line["gpu_launches"] >= line["steps"]
    assert set(line["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    # the clock record covers the timed steps themselves (and, beside them, a sustained soak)
    clk = line["clocks"]
    assert clk["window"] == "timed steps only" and clk["samples"] >= 1, clk
    assert clk["sm_mhz"] is not None and clk["soak"]["samples"] >= 1, clk


@pytest.mark.parametrize("workload,dtype,launches", [
    ("bf16_h8_l2000_d256", "bf16", 3),            # head dim 256
    ("fp32_b1_h2_l128_d64", "f32", 11),           # fp32 on the TF32 tensor cores
    ("bf16_bool_mask_h8_l2000_d128", "bf16", 4),  # the forward's mask (one more pre-pass)
])
def test_bwd_bench_lines(workload, dtype, launches):
    res = subprocess.run([sys.executable, "bench.py", "--pass", "bwd", "--workload", workload, "--steps", "3",
                          "--warmup", "3", "--cpu-seconds", "1"], cwd=ROOT, capture_output=True, text=True,
                         timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["metric"] == "attention bwd TFLOP/s" and line["dtype"] == dtype
    assert line["config"]["workload"] == workload and line["config"]["pass"] == "bwd"
    assert line["value"] > 0 and line["gpu_launches"] == launches * line["steps"]
    r = line["roofline"]
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9 and 0.0 < r["frac"] < 1.5
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] > 0

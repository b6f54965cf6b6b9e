"""bench.py on CPU: one short run of the reference arm (the fp64 oracle on the
host cores) for each pass prints the contract's JSON line on the metric of
the pass it was asked for; the secondary exponential roofline's arithmetic."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("pass_,workload,metric", [
    ("fwd", "fp32_b1_h2_l128_d64", "attention fwd TFLOP/s"),
    ("bwd", "bf16_causal_b4_h8_l1024_d64", "attention bwd TFLOP/s"),
    ("bwd", "bf16_bool_mask_h8_l2000_d128", "attention bwd TFLOP/s"),
])
def test_reference_line(pass_, workload, metric):
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--pass", pass_, "--workload", workload,
                          "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == metric
    assert line["config"]["workload"] == workload
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["higher_is_better"] is True and line["steps"] == 1 and line["warmup"] == 3


def test_exp_roofline_arithmetic():
    """One exponential per allowed score: the causal B2 H32 L4096 workload has 2*32*4096*4096/2 of them."""
    import bench
    import workloads
    w = workloads.WORKLOADS["bf16_gqa_causal_b2_hq32_hkv8_l4096_d128"]
    r = bench.exp_roofline(w, 0.2, 152, 2070.0)
    n_exp = 2 * 32 * 4096 * 4096 / 2
    assert abs(r["achieved"] - n_exp / 0.2e-3 / 1e9) < 1e-6 * r["achieved"]
    assert abs(r["peak"] - 152 * 32 * 2070e6 / 1e9) < 1e-9 * r["peak"]
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12 and r["unit"] == "Gexp/s"
    assert bench.exp_roofline(w, 0.2, 152, None)["frac"] is None

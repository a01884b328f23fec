"""CPU-only checks of bench.py's host logic: the algorithmic byte counts behind
the roofline figure, the choice of the dominant kernel, and the reference
arm's JSON line (the CPU oracle on a bounded sample), run end to end."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_of_the_dominant_gemm():
    m, n, k = 4096, 7168, 16384
    a, b, d = m * k, n * k, 2 * m * n
    scales = (m + n) * (k // 512) * 4  # packed UE8M0 words, one per 4 K blocks per row
    assert bench.algorithmic_bytes_gemm(m, n, k, False) == a + b + d + scales
    assert bench.algorithmic_bytes_gemm(m, n, k, True) == a + b + d + scales + 2 * m * n
    assert abs(bench.algorithmic_bytes_gemm(m, n, k, False) / 1e6 - 244.7) < 0.1


def test_roofline_takes_the_largest_launch_without_c():
    per_shape = [
        dict(m=4096, n=2112, k=7168, c=False, us=56.0, tflops=2213.0),
        dict(m=4096, n=7168, k=16384, c=False, us=320.0, tflops=3004.0),
        dict(m=4096, n=7168, k=16384, c=True, us=326.0, tflops=2953.0),
    ]
    r = bench.prefill_roofline({"per_shape": per_shape, "achieved": 2600.0}, 3901.4, "measured")
    assert r["achieved"] == 3004.0 and abs(r["frac"] - 3004.0 / 3901.4) < 1e-12
    assert r["traffic"] == bench.DOMINANT_TRAFFIC          # the captured shape
    assert abs(r["all_gemms"]["frac"] - 2600.0 / 3901.4) < 1e-12
    other = [dict(m=4096, n=2112, k=7168, c=False, us=56.0, tflops=2213.0)]
    assert bench.prefill_roofline({"per_shape": other, "achieved": 1.0}, 3901.4, "measured")["traffic"] is None


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOPS"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 1, 1)
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]

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
    assert bench.dominant_launch(per_shape) is per_shape[1]
    r = bench.prefill_roofline({"per_shape": per_shape, "achieved": 2600.0}, 3901.4, "measured", 1.5e8)
    assert r["achieved"] == 3004.0 and abs(r["frac"] - 3004.0 / 3901.4) < 1e-12
    assert r["traffic"] == 1.5e8
    assert abs(r["all_gemms"]["frac"] - 2600.0 / 3901.4) < 1e-12


class _FakePlanner:
    """Stands in for the binding's tile-choice query (pure host arithmetic)."""

    def __init__(self, plan):
        self.plan = plan

    def plan_fp8_gemm_nt_ws(self, m, n, k, has_c=False, num_sms=152):
        return dict(self.plan)


def test_traffic_only_for_the_captured_tile_configuration(monkeypatch):
    key = (4096, 7168, 16384, False, 256, 192, 1, 0, 1)
    monkeypatch.setitem(bench.CAPTURED_TRAFFIC, key, 4.0e8)
    m, n, k, c, bm, bn, sk, pair, mc = key
    same = _FakePlanner(dict(block_m=bm, block_n=bn, split_k=sk, cta_pair=bool(pair), multicast=bool(mc)))
    t, plan = bench.captured_traffic(same, m, n, k, c, 152)
    assert t == bench.CAPTURED_TRAFFIC[key] and plan["block_n"] == bn
    other = _FakePlanner(dict(block_m=bm, block_n=bn + 32, split_k=sk, cta_pair=bool(pair), multicast=bool(mc)))
    assert bench.captured_traffic(other, m, n, k, c, 152)[0] is None  # a changed tile: stale counters
    single = _FakePlanner(dict(block_m=bm, block_n=bn, split_k=sk, cta_pair=bool(pair), multicast=False))
    assert bench.captured_traffic(single, m, n, k, c, 152)[0] != 4.0e8  # the other kernel's counters
    assert bench.captured_traffic(same, m, n + 128, k, c, 152)[0] is None  # another shape


def test_grouped_byte_counts():
    # contiguous: valid rows of A and D, all experts' B, packed scale words
    assert bench.algorithmic_bytes_contiguous(1000, 8, 4096, 7168) == (
        1000 * 7168 + 8 * 4096 * 7168 + 2 * 1000 * 4096 + 4 * 14 * (1000 + 8 * 4096))
    # masked: only experts with rows read their B
    assert bench.algorithmic_bytes_masked(300, 3, 7168, 2048) == (
        300 * 2048 + 3 * 7168 * 2048 + 2 * 300 * 7168 + 4 * 4 * (300 + 3 * 7168))


def test_clock_summary_uses_samples_under_load():
    idle = ["0", "1000", "2070", "100.0", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]
    busy = ["0", "1900", "2070", "1300.0", "0x4", "Not Active", "Not Active", "Not Active", "Active"]
    c = bench.summarise_clocks([idle] * 5 + [busy] * 7 + [["garbage"]])
    assert c["samples"] == 12 and c["samples_under_load"] == 7
    assert c["sm_mhz"] == 1900.0 and c["sm_max_mhz"] == 2070.0 and c["reasons"] == ["sw_power_cap"]
    assert bench.summarise_clocks([]) is None


def test_cpu_baseline_of_the_small_config():
    cb = bench.cpu_baseline_config("small", __import__("moe_grouped_gemm_fp8_gb300.workloads",
                                                       fromlist=["x"]), seconds=0.2)
    assert cb["kind"] == "oracle" and cb["unit"] == "TFLOPS" and cb["value"] > 0 and cb["cores"] >= 1
    assert "repetitions" in cb["sample"]


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

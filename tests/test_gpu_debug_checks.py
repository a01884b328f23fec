"""The debug build of the library (libdg_debug.so: the same sources compiled
with DG_DEBUG_CHECKS=1, loaded by the binding when DG_DEBUG_LIBRARY=1).  Its
kernels check every TMA load's coordinates (16-byte aligned innermost
coordinate, rows, tiles and groups inside their tensors), the TMEM columns
the MMA issuer addresses, every row and column tile the epilogue stores, and
each stream-K slot and K range; a failed check records DG_ERR_DEVICE_CHECK
with its site in the error word and never traps.

Both tests run in child processes, since a process loads one of the two
libraries: one plants a failed check and reads it back; the other runs the
small-shape GPU suites (dense tiles of every width, 256-row tiles, split-K,
short A, CTA pairs, contiguous, masked, K-grouped, NN/TN/TT layouts, FP32
scales, stream-K, the bounded-wait timeouts) under the debug library, where
the conftest fixture fails any test that leaves a failed check behind."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_gemm.py", "tests/test_gpu_decode.py", "tests/test_gpu_stream_k.py", "tests/test_gpu_kgrouped.py",
          "tests/test_gpu_layouts.py", "tests/test_gpu_fp32_scales.py", "tests/test_gpu_fault.py"]

PLANTED = r"""
import torch
import moe_grouped_gemm_fp8_gb300 as dg
from moe_grouped_gemm_fp8_gb300 import _lib, workloads
assert _lib.LIB_PATH.endswith("libdg_debug.so"), _lib.LIB_PATH
w = workloads.dense(256, 512, 512, seed=3)  # 4 K blocks: single-CTA tiles, no split-K
qa, sfa = dg.quantize_fp8(w.a.cuda(), 1)
qb, sfb = dg.quantize_fp8(w.b.cuda(), 128)
ref = dg.fp8_gemm_nt(qa, sfa, qb, sfb)
assert dg.get_device_error()[0] == 0
dg.debug_plant_check(True)
try:
    d = dg.fp8_gemm_nt(qa, sfa, qb, sfb)
finally:
    dg.debug_plant_check(False)
st, word = dg.get_device_error()
assert st == 9 and (word >> 8) & 0xFFFF == 43, (st, hex(word))  # DG_ERR_DEVICE_CHECK, TMEM site
assert torch.equal(d.view(torch.int16), ref.view(torch.int16))  # nothing else changed
d = dg.fp8_gemm_nt(qa, sfa, qb, sfb)
assert dg.get_device_error()[0] == 0
print("planted check reported")
"""


@pytest.fixture(scope="module")
def debug_env():
    from moe_grouped_gemm_fp8_gb300 import build
    build.build(debug=True)
    env = dict(os.environ)
    env["DG_DEBUG_LIBRARY"] = "1"
    return env


def test_planted_check_reaches_the_caller(debug_env):
    r = subprocess.run([sys.executable, "-c", PLANTED], env=debug_env, cwd=ROOT, timeout=300,
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]


def test_release_library_refuses_the_planted_check():
    import moe_grouped_gemm_fp8_gb300 as dg
    from moe_grouped_gemm_fp8_gb300 import _lib
    if _lib.DEBUG:
        pytest.skip("this process loaded the debug library")
    with pytest.raises(dg.DGError):
        dg.debug_plant_check(True)
    dg.debug_plant_check(False)


def test_small_gpu_suites_pass_every_device_check(debug_env):
    if os.environ.get("DG_DEBUG_LIBRARY", "0") not in ("", "0"):
        pytest.skip("already running under the debug library")
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITES, "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider"], env=debug_env, cwd=ROOT, timeout=1800,
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-6000:] + r.stderr[-3000:]

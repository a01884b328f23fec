import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built CUDA library")


DG_ERR_DEVICE_CHECK = 9


@pytest.fixture(autouse=True)
def _device_checks_clean(request):
    """Under the debug library (DG_DEBUG_LIBRARY=1, kernels built with
    DG_DEBUG_CHECKS=1) every GPU test also ends with no failed device check:
    in-range load coordinates, TMEM columns, output rows and stream-K slots."""
    yield
    if os.environ.get("DG_DEBUG_LIBRARY", "0") in ("", "0") or request.node.get_closest_marker("gpu") is None:
        return
    import moe_grouped_gemm_fp8_gb300 as dg
    st, word = dg.get_device_error()
    assert st != DG_ERR_DEVICE_CHECK, "device check failed at site %d in block %d" % (
        (word >> 8) & 0xFFFF, word >> 32)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Per-tensor error figures of the full-size parity checks (GPU runs)."""
    try:
        import _parity
    except Exception:
        return
    if not _parity.REPORT:
        return
    tr = terminalreporter
    tr.section("parity: per-tensor error of every written element vs the oracle")
    tr.write_line("%-62s %12s %12s %12s" % ("tensor", "elements", "rel_sq_err", "max_err/max|o|"))
    for what, n, rel, mx in _parity.REPORT:
        tr.write_line("%-62s %12d %12.3e %12.3e" % (what[:62], n, rel, mx))
    path = os.environ.get("DG_PARITY_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump([dict(tensor=w, elements=n, rel_sq_err=r, max_err_ratio=m)
                       for w, n, r, m in _parity.REPORT], f, indent=1)

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built CUDA library")


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

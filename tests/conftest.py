import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Worst element-wise relative error per compared tensor (see gpu_util)."""
    try:
        from tests.gpu_util import REPORT
    except ImportError:
        return
    if not REPORT:
        return
    import json
    worst = {}
    for r in REPORT:
        k = (r["what"].split("[")[0].split(" ")[0], r["dtype"], r["elem_asserted"])
        if k not in worst or r["elem"] > worst[k]["elem"]:
            worst[k] = r
    terminalreporter.section("parity: worst element-wise relative error per tensor")
    for (what, dt, asserted), r in sorted(worst.items()):
        terminalreporter.write_line(
            f"{what:>22} {dt:>4}  elem {r['elem']:.2e}  inf {r['inf']:.2e}  "
            f"{'asserted' if asserted else 'reported'}  ({r['test']})")
    path = os.environ.get("TP_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(REPORT, f, indent=0)

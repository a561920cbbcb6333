import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libpnq.so")


@pytest.fixture(scope="session")
def oracle():
    import oracle as _o
    _o.lib()
    return _o


def pytest_terminal_summary(terminalreporter):
    """Worst error / bound ratio of the GEMV parity checks that ran (1.0 = at the bound)."""
    try:
        import gpu_util
    except Exception:
        return
    worst = getattr(gpu_util, "WORST_RATIO", {})
    if not worst:
        return
    tr = terminalreporter
    tr.write_sep("-", "GEMV error / bound (worst per check; 1.0 is the bound)")
    top = sorted(worst.items(), key=lambda kv: -kv[1])
    tr.write_line(f"checks: {len(worst)}  worst overall: {top[0][1]:.3g} ({top[0][0]})")
    full = {k: v for k, v in worst.items() if any(s in k for s in ("M=", "workload", "x"))}
    for k, v in sorted(full.items(), key=lambda kv: -kv[1])[:12]:
        tr.write_line(f"  {v:.3g}  {k}")

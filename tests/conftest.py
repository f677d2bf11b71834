import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built qmm library")
    config.addinivalue_line("markers", "slow: full-size workload checks")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Largest parity errors of the session as fractions of their tolerances
    (1.0 = at the bound), so the arithmetic's headroom is on record."""
    try:
        from tests._helpers import HEADROOM
    except ImportError:
        return
    if not HEADROOM:
        return
    rows = sorted(HEADROOM.items(), key=lambda kv: -kv[1])
    terminalreporter.write_sep("-", f"parity headroom: worst error / tolerance over {len(rows)} tests")
    for name, frac in rows[:25]:
        terminalreporter.write_line(f"{frac:8.4f}  {name}")
    fracs = np.array([f for _, f in rows])
    terminalreporter.write_line(f"median {float(np.median(fracs)):.4f}, max {float(fracs.max()):.4f}")

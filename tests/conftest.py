import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Print how often the GPU parity gates used the oracle's ambiguity term."""
    helpers = sys.modules.get("gpu_helpers")
    log = getattr(helpers, "AMB_LOG", None)
    if not log:
        return
    rows = sum(r[1] for r in log)
    used = sum(r[2] for r in log)
    tr = terminalreporter
    tr.write_sep("-", "ambiguity term of the per-row emulation gate")
    tr.write_line(f"{len(log)} comparisons, {rows} rows, {used} rows needed the term; largest amb "
                  f"among those {max(r[3] for r in log):.3e}, over all rows "
                  f"{max(r[4] for r in log):.3e}")
    for label, n, k, au, am in log:
        if k:
            tr.write_line(f"  {label}: {k} of {n} rows, largest amb used {au:.3e}")

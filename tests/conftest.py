import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")
    config.addinivalue_line("markers", "slow: full-size workload checks")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


def pytest_sessionfinish(session, exitstatus):
    """Write every parity comparison (max-norm and elementwise error) to $SSM_PARITY_REPORT, if set."""
    path = os.environ.get("SSM_PARITY_REPORT")
    if not path:
        return
    import json
    from tolerance import REPORT
    with open(path, "w") as f:
        json.dump([{"test": t, "maxnorm": m, "elementwise": e, "n": n} for t, m, e, n in REPORT], f, indent=0)

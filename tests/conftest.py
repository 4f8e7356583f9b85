import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the secondary parity metric (exact match wherever the gap exceeds 1e-5) collected
    by the GPU parity helpers, and write it as JSON to $DG_PARITY_REPORT if that is set."""
    mod = sys.modules.get("parity")
    if mod is None or not mod.STRICT_REPORT:
        return
    rep = {t: dict(c) for t, c in mod.STRICT_REPORT.items()}
    tot = {}
    for c in rep.values():
        for k, v in c.items():
            tot[k] = tot.get(k, 0) + v
    terminalreporter.write_sep("-", "parity: secondary metric (gap > 1e-5 exact), totals")
    terminalreporter.write_line(json.dumps(tot, sort_keys=True))
    path = os.environ.get("DG_PARITY_REPORT")
    if path:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "w") as f:
            json.dump({"totals": tot, "per_test": rep}, f, indent=1, sort_keys=True)

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built libls_reduce.so")
    config.addinivalue_line(
        "markers", "slow: full-size workload (still run by default)")


@pytest.fixture(scope="session")
def ref():
    """The CPU oracle (built on first use)."""
    import oracle
    oracle.build()
    return oracle


def pytest_sessionfinish(session, exitstatus):
    """With LS_PARITY_REPORT set, write the error statistics of every GPU-vs-
    oracle comparison of the session as JSON lines to that file."""
    path = os.environ.get("LS_PARITY_REPORT")
    if not path:
        return
    mod = sys.modules.get("_parity")
    if mod is None or not mod.REPORT:
        return
    import json
    with open(path, "w", encoding="utf-8") as f:
        for rec in mod.REPORT:
            f.write(json.dumps(rec) + "\n")

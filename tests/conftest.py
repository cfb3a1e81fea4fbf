import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT


def pytest_sessionfinish(session, exitstatus):
    """With ATTN_PARITY_REPORT set, write every parity comparison's error figures there."""
    path = os.environ.get("ATTN_PARITY_REPORT")
    if not path:
        return
    mod = sys.modules.get("gpu_util")
    if mod is None or not mod.REPORT:
        return
    import json
    with open(path, "w") as f:
        json.dump(mod.REPORT, f, indent=1, sort_keys=True)

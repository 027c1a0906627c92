import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.join(ROOT, "tests")):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libpkv.so")


def pytest_sessionfinish(session, exitstatus):
    """Write the parity records (raw max-abs error and excess over the output rounding, per test)
    to the file PKV_PARITY_LOG names, if any."""
    path = os.environ.get("PKV_PARITY_LOG")
    if path:
        import _parity
        _parity.dump(path)


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def read_golden_kv(path):
    """Parse 'key value...' lines of a golden fixture (comments start with '#')."""
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            out[k] = v
    return out

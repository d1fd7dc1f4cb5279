import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: minutes of CPU work")


def read_fixture(name):
    """Parse a golden text file: '#' lines are comments, other lines are 'key values...'."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        rows = []
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            out[key] = rest
            rows.append(line.split())
    out["_rows"] = rows
    return out

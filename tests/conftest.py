import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes of oracle time)")


def load_golden(name):
    """Parse a golden fixture: '# ...' comment lines, then 'key = rows' where
    rows are separated by ';' and numbers by whitespace."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            rows = [[float(t) for t in r.split()] for r in val.split(";")]
            arr = np.array(rows, dtype=np.float64)
            if arr.shape[0] == 1:
                arr = arr[0]
                if arr.shape[0] == 1:
                    arr = float(arr[0])
            out[key] = arr
    return out


@pytest.fixture
def golden():
    return load_golden

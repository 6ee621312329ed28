import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


def read_golden(name):
    """Parse a tests/golden fixture: '#' comments, 'key = values' lines and
    bare rows of numbers."""
    path = os.path.join(ROOT, "tests", "golden", name)
    kv, rows = {}, []
    with open(path, encoding="utf-8") as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if "=" in line:
                k, v = line.split("=", 1)
                kv[k.strip()] = [float(s) for s in v.split()]
            else:
                rows.append([float(s) for s in line.split()])
    return kv, rows


@pytest.fixture
def golden():
    return read_golden

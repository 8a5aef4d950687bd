import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def read_golden(name):
    """Parse a tests/golden fixture: '<key> v v | v v' lines, '#' comments."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, rest = line.partition(" ")
            out[key] = rest.strip()
    return out


def parse_matrix(text, consts=None):
    consts = consts or {}
    rows = []
    for r in text.split("|"):
        rows.append([float(consts.get(v, v)) for v in r.split()])
    return rows


@pytest.fixture(scope="session")
def golden():
    return read_golden

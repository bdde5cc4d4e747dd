import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden_rows(name):
    """Non-comment, non-empty lines of a golden fixture, split on whitespace."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def read_worked_examples():
    out = {}
    for row in read_golden_rows("worked_examples.txt"):
        out[row[0]] = {k: float(v) for k, v in (kv.split("=") for kv in row[1:])}
    return out


@pytest.fixture(scope="session")
def worked():
    return read_worked_examples()


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle

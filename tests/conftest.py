import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


def read_golden(name):
    """Non-comment, non-empty lines of a golden fixture (text after ';' is a
    worked note and is dropped)."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split(";", 1)[0].strip()
            if line and not line.startswith("#"):
                out.append(line)
    return out


def build_lib():
    """Build libbw.so (fast when up to date) and return its path."""
    import __graft_entry__
    return __graft_entry__.load_builder().build()

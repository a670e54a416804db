import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def read_golden(name: str) -> dict:
    """Parse a tests/golden fixture: '#' lines are the citation, other lines 'key v1 v2 ...'."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            nums = [float(v) for v in vals]
            out[key] = nums[0] if len(nums) == 1 else nums
    return out


@pytest.fixture(scope="session")
def golden():
    return read_golden

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name: str) -> dict:
    """Parse a ``key value [value ...]`` fixture; '#' lines are comments."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            nums = [float(x) for x in vals]
            out[key] = nums[0] if len(nums) == 1 else nums
    return out


@pytest.fixture(scope="session")
def golden():
    return read_golden


@pytest.fixture(scope="session")
def dev():
    """cuda:0 with the library built; GPU tests fail loudly without a device."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from exact_io_aware_order_gb300 import build

    build.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and runs libkivi kernels")
    config.addinivalue_line("markers", "slow: full-size workload parity (minutes)")


@pytest.fixture(scope="session")
def ref():
    """The CPU oracle (built with gcc on first use)."""
    from oracle import ref as R
    R.lib()
    return R


@pytest.fixture(scope="session")
def kivi_lib():
    """libkivi.so, built in-tree with nvcc if it is missing or stale."""
    from kivi_bit_kv_gb300 import build, abi
    build.build()
    return abi.load()


@pytest.fixture(scope="session")
def cuda(kivi_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def golden(name):
    """Rows of a '|'-separated fixture under tests/golden (comments skipped)."""
    path = os.path.join(ROOT, "tests", "golden", name)
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows

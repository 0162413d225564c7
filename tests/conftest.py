import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running check (minutes)")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly when no GPU is present instead of skipping: a GPU run that silently
    # skipped would read as a pass.
    pass


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    assert torch.cuda.is_available(), "this test needs a CUDA GPU"
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def qkvp(cuda_device):
    """The CUDA library's Python binding (built in-tree); fails if the extension is missing."""
    import quantized_kv_paged_gb300 as q
    q.load()
    return q


def read_golden(name):
    path = os.path.join(ROOT, "tests", "golden", name)
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def moelib():
    """The built library (built here if missing or stale; nvcc cross-compiles
    without a GPU)."""
    from bit_grouped_expert_moe_gb300 import _build
    _build.build()
    import bit_grouped_expert_moe_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="session")
def cuda_dev(moelib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def moe():
    """The CUDA library binding, built in-tree if needed (GPU tests only)."""
    if not gpu_available():
        pytest.skip("no GPU")
    from moe_expert_layer_counts_gb300 import build as b
    b.build()
    import moe_expert_layer_counts_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.build()
    return o

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large case (full-size workloads)")


@pytest.fixture(scope="session")
def oracle():
    import oracle as o

    o.build()
    return o


@pytest.fixture(scope="session")
def dsa_lib():
    """The built CUDA library (compiled on first use; nvcc cross-compiles without a GPU)."""
    from dsa_sparse_attention_mla_gb300 import _build
    import dsa_sparse_attention_mla_gb300 as dsa

    _build.build()
    return dsa.load_library()


@pytest.fixture(scope="session")
def gpu(dsa_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU")
    major, minor = torch.cuda.get_device_capability()
    assert (major, minor) == (10, 3), f"expected an sm_103 GPU, got sm_{major}{minor}"
    return torch.device("cuda:0")

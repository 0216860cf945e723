import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library on a visible GPU (skips when there is no GPU)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_gqa_online_gb300 import build as _b
    _b.build()
    import attention_gqa_online_gb300 as A
    A.load_library()
    return A

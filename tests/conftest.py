import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (CUDA) device")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library (building it if needed; nvcc cross-compiles here)."""
    from gqa_decode_attention_02_gb300 import build, _lib

    build.build()
    return _lib.lib()


@pytest.fixture(scope="session")
def gpu():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_decode_attention_02_gb300 import build

    build.build()
    return torch.device("cuda:0")

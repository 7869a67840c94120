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
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle

    return oracle.default()


@pytest.fixture(scope="session")
def jl():
    """The ctypes binding of libjetlong.so, built first if it is stale."""
    from zero_shot_rope_02_b300 import build

    build.build()
    from zero_shot_rope_02_b300 import binding

    return binding


@pytest.fixture(scope="session")
def dev(jl):
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test without a CUDA device")
    return torch.device("cuda:0")

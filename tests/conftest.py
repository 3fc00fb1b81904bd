import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def cpt():
    """The C-ABI binding, built in-tree if missing or stale. Under
    CPT_LIBRARY_VARIANT=checked it is the bounds-checked build, and the
    session ends with a check that no device bounds check failed."""
    from context_attention_token_gb300 import build as cpt_build

    cpt_build.build()
    from context_attention_token_gb300 import cpt as binding

    yield binding
    import torch

    if binding.cpt_bounds_checked() and torch.cuda.is_available() and torch.cuda.is_initialized():
        torch.cuda.synchronize()
        assert binding.cpt_bounds_violations() == 0, "a device bounds check failed during the session"


@pytest.fixture(scope="session")
def cuda_device():
    import torch

    if not torch.cuda.is_available():
        pytest.fail("the gpu-marked tests need a CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda", 0)

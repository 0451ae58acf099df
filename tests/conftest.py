import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libbgq.so")
    config.addinivalue_line("markers", "slow: long-running test")


@pytest.fixture(scope="session")
def cuda_device():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def guard_canaries(request):
    """GPU tests: every buffer the binding creates (outputs, workspaces) sits
    between guard regions of a known byte, checked when the test ends."""
    if request.node.get_closest_marker("gpu") is None:
        yield None
        return
    import torch

    if not torch.cuda.is_available():
        yield None
        return
    from bit_group_quantized_gb300 import lib
    from tests.helpers import GuardedAllocator

    g = GuardedAllocator()
    lib.set_allocator(g)
    try:
        yield g
        torch.cuda.synchronize()
        g.check()
    finally:
        lib.set_allocator(None)

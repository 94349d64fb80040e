import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: long-running")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def cuda():
    """cuda:0 with the CUDA library built and loaded (gpu tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test run without a CUDA device")
    from invariant_moe_gb300 import _build
    _build.build()
    import invariant_moe_gb300 as bm
    bm.load_library()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _no_device_error(request):
    """Every gpu test must leave the device error word clear."""
    yield
    if request.node.get_closest_marker("gpu") is not None and "cuda" in request.fixturenames:
        import invariant_moe_gb300 as bm
        code = bm.device_error()
        expected = getattr(request.node, "expected_device_error", 0)
        assert code == expected, f"device error word = {code}"

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """After every GPU test the library's device error word must be clear: a
    bounded wait that gave up would otherwise hide behind partial outputs."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    if request.node.name.startswith("test_bounded_wait"):
        return
    import torch
    if not torch.cuda.is_available():
        return
    from tensor_column_linear_gelu_b300 import tpla
    st = tpla.tp_device_status()
    assert st == tpla.TP_OK, f"device status after test: {tpla.status_string(st)}"

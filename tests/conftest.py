import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkda")
    config.addinivalue_line(
        "markers", "slow: long-running (full-size workloads)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """After every GPU test, libkda's device status word must be clear: a
    bounded wait inside a kernel that gave up (or a pool index out of range)
    is a failure even when the host call returned KDA_SUCCESS.  Tests that
    provoke such a status read and clear it themselves."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    from kimi_delta_attention_chunkwise_gb300 import binding
    if binding._lib is None:
        return
    st = binding.kda_device_status()
    assert st == binding.KDA_SUCCESS, \
        f"device status word after the test: {binding.kda_status_string(st)}"

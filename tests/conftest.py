import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running test")


def golden(name):
    import json
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        return json.load(f)


@pytest.fixture(autouse=True)
def _device_status(request):
    """After every GPU test: no bounded device wait may have expired."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import blockwise_attention_gb300 as ba
    rc = ba.sync_status()
    assert rc == 0, f"device status {rc} (a bounded wait expired) after {request.node.name}"

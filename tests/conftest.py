import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running full-size case")


@pytest.fixture(autouse=True)
def _short_device_waits(request):
    """GPU tests run with a 1 s limit on every device-side wait, so a broken
    pipeline reports MM_ERR_TIMEOUT quickly instead of after the default 2 s."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import moe_expert_layer_idx_gb300 as mm

    prev = mm.mm_get_wait_timeout_ns()
    mm.mm_set_wait_timeout_ns(1_000_000_000)
    yield
    mm.mm_set_wait_timeout_ns(prev)

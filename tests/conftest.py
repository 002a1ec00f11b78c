import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on a GB300)")


@pytest.fixture(scope="session")
def oracle():
    import oracle as orc
    orc.build()
    return orc


@pytest.fixture(autouse=True)
def device_error_word_stays_clear(request):
    """After every GPU test: no kernel's bounded pipeline wait gave up (the
    library's device error word reads 0; reading it also clears it)."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import residual_add_rmsnorm_fwd_gb300 as rn
    flags = rn.rmsnorm_read_device_errors()
    assert flags == 0, f"device error word {flags:#x}: a pipeline wait gave up during the test"

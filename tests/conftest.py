import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


@pytest.fixture(autouse=True)
def _bounds_flags_clear(request):
    """With the bounds-checked library loaded (BD_LIBRARY naming
    libbitdelta_bounds.so), every GPU test also requires that no kernel met
    an out-of-range index; with the normal library this does nothing."""
    yield
    if request.node.get_closest_marker("gpu") is None or not os.environ.get("BD_LIBRARY"):
        return
    from bit_weight_delta_bd_gb300 import bitdelta as bd

    if bd._lib is None or not bd.bd_debug_bounds_enabled():
        return
    st, bits = bd.bd_debug_bounds_check()
    assert st == bd.BD_OK, f"bounds check fired in kernels 0x{bits:x}"

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(autouse=True)
def _no_skipped_out_of_range_stores(request):
    """With MOEQ_CHECK_BOUNDS set (runs against a MOEQ_DEBUG_BOUNDS build of
    the library), every GPU test must end with no store skipped for lying
    outside its buffer."""
    yield
    if os.environ.get("MOEQ_CHECK_BOUNDS") and request.node.get_closest_marker("gpu"):
        from fp4_fp8_quantization_gb300 import moeq
        assert not moeq.get_device_error() & moeq.DEVERR_BOUNDS

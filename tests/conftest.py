import json
import os
import sys
import time

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


@pytest.fixture(autouse=True)
def _metrics_notes():
    from tests import _util
    _util.NOTES.clear()
    yield


def pytest_runtest_logreport(report):
    """With MOEQ_METRICS_LOG set, appends one JSON line per test to that file:
    test id (its parameters are the shapes), outcome, seconds, the device and
    host core count, and what the test noted (compared elements, largest
    error and its ratio to the tolerance for the GEMM comparisons)."""
    path = os.environ.get("MOEQ_METRICS_LOG")
    if not path or not (report.when == "call" or (report.when == "setup" and report.skipped)):
        return
    from tests import _util
    line = {"time": round(time.time(), 3), "test": report.nodeid, "outcome": report.outcome,
            "seconds": round(report.duration, 4), "gpu": "gpu" in report.keywords,
            "host_cores": len(os.sched_getaffinity(0))}
    if line["gpu"]:
        import torch
        if torch.cuda.is_available():
            line["device"] = torch.cuda.get_device_name(0)
    line.update(_util.NOTES)
    with open(path, "a") as f:
        f.write(json.dumps(line) + "\n")

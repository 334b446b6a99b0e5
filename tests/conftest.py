import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


# Sampled indices of the CUDA path that differ from the oracle's search of its
# own fp64 CDF (allowed only inside the boundary band), per workload: recorded
# by the GPU tests, printed at the end of the run.
_BAND_COUNTS = []


@pytest.fixture
def band_report():
    def record(workload, mismatches, samples, band):
        _BAND_COUNTS.append((workload, int(mismatches), int(samples), band))
    return record


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if not _BAND_COUNTS:
        return
    terminalreporter.section("indices differing from the oracle's own fp64 CDF (all inside the boundary band)")
    for workload, mism, samples, band in _BAND_COUNTS:
        terminalreporter.write_line(f"{workload}: {mism} of {samples} samples (band {band})")


def _cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libcosa.so")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The parity record of the GPU tests: per workload, skip-decision agreement with every
    disagreement and its oracle margin, output errors, mask rows compared and float64 ties."""
    gh = sys.modules.get("tests.gpu_helpers")
    lines = gh.parity_summary_lines() if gh is not None else []
    if not lines:
        return
    terminalreporter.write_sep("=", "parity record: GPU path against the float64 oracle")
    for line in lines:
        terminalreporter.write_line(line)

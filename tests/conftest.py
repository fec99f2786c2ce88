import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Print the largest errors of the full-size whole-output comparisons."""
    from tests.tolerances import LSE_TOL, O_TOL, PARITY_LOG
    if not PARITY_LOG:
        return
    terminalreporter.write_sep("-", f"full-size parity against the fp64 oracle "
                                    f"(limits: |dO| {O_TOL:g} (+ half a bf16 ulp for bf16 O), |dLSE| {LSE_TOL:g})")
    for what, eo, el in PARITY_LOG:
        terminalreporter.write_line(f"{what:<58s} max|dO| {eo:.3e}   max|dLSE| {el:.3e}")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built libdspark.so")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) on machines without a CUDA device
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    # near-tie divergences of the full-size chain parity tests: device tokens
    # that differ from the oracle's only where the oracle's top-2 margin is
    # below 1e-3 * |max|
    h = sys.modules.get("gpu_harness")
    log = getattr(h, "NEAR_TIE_LOG", None) if h else None
    if not log:
        return
    terminalreporter.write_line("near-tie divergences (case: count / rows x positions checked):")
    for case, near, checked in log:
        terminalreporter.write_line(f"  {case}: {near} / {checked}")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


def _has_gpu():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA GPU visible")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """How many compared attention elements needed the |O| >= 2 allowance
    (half a bf16 ulp + 4e-3 against the unrounded oracle)."""
    mod = sys.modules.get("_cases")
    if mod is None or not mod.WIDE["compared"]:
        return
    w = mod.WIDE
    terminalreporter.write_line(
        f"attention tolerance: {w['elements']} of {w['compared']} compared elements had |O| >= 2 and were held to "
        f"half a bf16 ulp + 4e-3 (largest |O| {w['max_abs_o']:.3f}, largest error {w['max_err']:.3e}); "
        f"all others to 4e-3 against the unrounded fp64 oracle")

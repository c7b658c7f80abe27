import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Totals of the GPU parity checks: max abs error, max rel error (over
    |oracle| >= 0.2) and the elements that passed only through the relative
    term while |oracle| < 0.2 (flagged)."""
    gu = sys.modules.get("gpu_util")
    if gu is None or not gu.STATS["checks"]:
        return
    st = gu.STATS
    terminalreporter.write_line(
        f"tolerance: {st['checks']} checks over {st['elements']} elements; max abs error {st['max_abs']:.3e} "
        f"(bound {gu.ATOL}), max rel error {st['max_rel']:.3e} over |ref| >= {gu.REL_FLOOR} (bound {gu.RTOL}); "
        f"flagged (abs > {gu.ATOL} with |ref| < {gu.REL_FLOOR}): {st['flagged']}"
        + (f", worst {st['worst_flagged'][0]:.3e} in {st['worst_flagged'][1]}" if st["worst_flagged"] else ""))

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")
    config.addinivalue_line("markers", "slow: large oracle runs")


def pytest_collection_modifyitems(config, items):
    # A GPU test on a machine without a GPU is skipped, never run on a fallback.
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


def pytest_terminal_summary(terminalreporter):
    # How the appended K/V rows of the tensor-core projections compared with
    # the oracle's fp32-sequential chain over the whole session.
    try:
        from tests.helpers import PROJECTION_TALLY as t
    except Exception:  # pragma: no cover
        return
    if t["elements"]:
        n = t["elements"]
        terminalreporter.write_line(
            f"projection appends vs oracle: {n} elements, bit-exact {t['bit_exact'] / n:.5f}, "
            f"within 1 ulp {t['within_1ulp'] / n:.6f}, accepted only through the fp32 "
            f"summation bound {t['fp32_bound_only']} (all near-cancellations; largest "
            f"|sum| / sum|x w| among them {t['max_cancellation_ratio']:.3g})")

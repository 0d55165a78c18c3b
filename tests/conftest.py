import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # Worst output error of every oracle comparison: the fixed rule's ratio
    # and the error in bf16 ulps of the reference.
    try:
        from _common import RESULTS
    except ImportError:  # pragma: no cover
        return
    if not RESULTS:
        return
    tr = terminalreporter
    tr.section("output errors against the oracle")
    tr.write_line(f"{'comparison':56s} {'elements':>9s} {'err/tol':>8s} {'worst ulp':>10s} {'median ulp':>10s}")
    for label, n, ratio, worst, med in RESULTS:
        tr.write_line(f"{label[:56]:56s} {n:9d} {ratio:8.3f} {worst:10.2f} {med:10.2f}")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped, not failed, on a machine without a GPU, unless
    # they were selected explicitly with -m gpu (then they must run).
    markexpr = config.getoption("-m") or ""
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu or "gpu" in markexpr and "not gpu" not in markexpr:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)

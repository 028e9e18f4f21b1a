import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libtq.so")
    config.addinivalue_line("markers", "slow: long-running CPU check")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def tqlib():
    """The ctypes handle of libtq.so, building it first if it is missing."""
    from turboquant_kv_cache_gb300 import binding, build
    if not os.path.exists(build.LIB):
        build.build()
    return binding.library()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Reports the boundary-tie mismatches of every GPU-vs-oracle code
    comparison: codes may differ from the oracle only for coordinates within
    1e-5 of a decision boundary (QJL bits: |S r| < 1e-5), and those are
    counted here per case."""
    try:
        from _parity import TIE_LOG
    except Exception:  # pragma: no cover
        return
    if not TIE_LOG:
        return
    tr = terminalreporter
    tr.section("boundary-tie mismatches (GPU vs oracle)")
    tot_bad = tot = 0
    for test, kind, bad, n in TIE_LOG:
        tr.write_line(f"{bad:6d} / {n:9d} {kind:5s} {test}")
        tot_bad += bad
        tot += n
    tr.write_line(f"total: {tot_bad} of {tot} compared codes/bits differ, every one a boundary tie")

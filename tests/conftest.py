import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload checks (tens of seconds of oracle work)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        # The GPU tests load the in-tree library: build it first (a no-op when current).
        import __graft_entry__
        __graft_entry__.build()
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The plain max-abs and mean-abs of every parity comparison of the session."""
    try:
        from tests._gpu import RECORDS
    except Exception:  # pragma: no cover
        return
    if not RECORDS:
        return
    tr = terminalreporter
    tr.section("parity against the oracle: max-abs, mean-abs, worst |x-ref|/bound, elements under a derived bound")
    for test, name, n, mx, mean, worst, derived in RECORDS:
        tr.write_line(f"{test} | {name} | {n} elements | max-abs {mx:.3g} | mean-abs {mean:.3g} | {worst:.3g} | "
                      f"{derived}")

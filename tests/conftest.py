import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _ensure_library():
    """Build libspec_tree.so when it is missing or older than its sources (nvcc is needed)."""
    from dynamic_tree_speculative_gb300 import build
    srcs = [os.path.join(build.CSRC, f) for f in os.listdir(build.CSRC)]
    srcs.append(os.path.join(build.INCLUDE, "spec_tree.h"))
    if not os.path.exists(build.LIB) or max(os.path.getmtime(f) for f in srcs) > os.path.getmtime(build.LIB):
        build.build()


def pytest_sessionstart(session):
    _ensure_library()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """One line with the session's GPU-vs-oracle parity counts (trees compared, near-ties adopted)."""
    mod = sys.modules.get("parity_compare")
    if mod is not None and (mod.TALLY["build_trees"] or mod.TALLY["verify_trees"]):
        terminalreporter.write_line(mod.tally_line())

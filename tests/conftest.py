"""Shared pytest setup.

Markers: ``gpu`` marks tests that launch CUDA kernels through the C ABI; the
CPU suite runs with ``-m "not gpu"``.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and libdflash2.so")


@pytest.fixture(scope="session")
def ora():
    import oracle
    oracle.build()
    return oracle


def pytest_collection_modifyitems(config, items):
    # GPU tests need a CUDA device; on a machine without one they are skipped.
    # On a GPU machine a missing or broken extension fails loudly instead.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def cuda():
    import torch
    import __graft_entry__ as g
    g.build_library()
    from block_draft_proposal_gb300 import dflash2
    dflash2.library()
    return torch.device("cuda:0")

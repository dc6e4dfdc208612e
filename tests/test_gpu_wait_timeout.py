"""Failure detection on the GPU without a fault: a pipeline wait that nothing
completes must give up after the library's limit (one second), set
DFLASH2_DEVERR_TIMEOUT, raise the CTA's abort flag and return, and the context
must stay usable for the next library call."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import __graft_entry__ as g
from block_draft_proposal_gb300 import dflash2

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe(cuda, tmp_path_factory):
    so = str(tmp_path_factory.mktemp("probe") / "wait_probe.so")
    cmd = [g._nvcc(), *g.NVCC_FLAGS, "-shared", os.path.join(HERE, "wait_probe.cu"), "-o", so]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    lib = ctypes.CDLL(so)
    lib.wait_probe.argtypes = [ctypes.c_void_p] * 3
    lib.wait_probe.restype = ctypes.c_int
    return lib


def test_bounded_wait_gives_up_and_reports(cuda, probe):
    err = torch.zeros(1, dtype=torch.int32, device=cuda)
    elapsed = torch.zeros(1, dtype=torch.int64, device=cuda)
    result = torch.zeros(1, dtype=torch.int32, device=cuda)
    rc = probe.wait_probe(err.data_ptr(), elapsed.data_ptr(), result.data_ptr())
    assert rc == 0                                   # the kernel returned normally
    assert int(result.item()) == 2                   # gave up, abort flag raised
    assert int(err.item()) & dflash2.DEVERR_TIMEOUT
    secs = int(elapsed.item()) / 1e9
    assert 1.0 <= secs < 3.0, secs                   # the one-second limit
    # the context is intact: an ordinary library call runs and is exact
    ids = torch.arange(10, dtype=torch.int64, device=cuda)
    out, e2 = dflash2.d2t_remap(ids, None, 100, 100)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), np.arange(10))
    assert int(e2.item()) == 0

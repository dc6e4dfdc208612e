"""The allocation-free selector walk (dflash2_selector_walk_noalloc).

Some callers cannot hand the library a device buffer when they call it: a
serving loop whose device memory belongs to another allocator, or a
latency-critical path that must never reach cudaMalloc / cudaFree (they can
synchronise the device).  This entry point serves them from a fixed 4 MiB
array inside the library.  The test checks, through the C ABI, that two
calls in a row give the same tokens, q and edges as the workspace entry
point, and that shapes needing more scratch are refused.  The file is named
to run last, so that a failure here leaves the rest of the suite already run.
"""
import numpy as np
import pytest
import torch

from block_draft_proposal_gb300 import dflash2, synth

pytestmark = pytest.mark.gpu


def _inputs(w, dev, seed):
    rng = np.random.default_rng(seed)
    inp = synth.make(w, parts=("h", "A", "B", "proj", "uniforms", "anchors"))
    cand = np.stack([rng.choice(w.draft_vocab, size=w.top_k, replace=False)
                     for _ in range(w.rows)]).reshape(w.batch, w.slots, w.top_k).astype(np.int64)
    cand_u = np.sort(rng.standard_normal((w.batch, w.slots, w.top_k)).astype(np.float32),
                     axis=-1)[..., ::-1].copy()
    t = {k: dflash2.to_device(v, dev) for k, v in inp.items() if v is not None}
    return (t["h"], t["proj"], t["A"], t["B"], t["anchors"], torch.from_numpy(cand).to(dev),
            torch.from_numpy(cand_u).to(dev), t["temperatures"], t["greedy"], t["uniforms"])


@pytest.mark.parametrize("name,scale", [("qwen3-8b-bf16", dict(batch=8, draft_vocab=20000,
                                                               target_vocab=20000)),
                                        ("stress-bf16", dict(batch=6, draft_vocab=20000,
                                                             target_vocab=20000)),
                                        ("tiny-fp32", {})])
def test_noalloc_walk_matches_the_workspace_walk_twice(name, scale):
    dev = torch.device("cuda:0")
    w = synth.BY_NAME[name].scaled(**scale)
    args = _inputs(w, dev, seed=123)
    ref_tok, ref_q, ref_ps, ref_err = dflash2.selector_walk(*args, with_path_scores=True)
    tol = 1e-5 if w.dtype == "f32" else 2e-2
    for _ in range(2):   # the second call reuses the scratch the first one left behind
        tok, q, ps, err = dflash2.selector_walk_noalloc(*args, with_path_scores=True)
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok)
        assert (q - ref_q).abs().max().item() <= tol
        assert (ps - ref_ps).abs().max().item() <= tol
        assert int(err.item()) == int(ref_err.item()) == 0


def test_noalloc_walk_refuses_shapes_beyond_its_scratch():
    dev = torch.device("cuda:0")
    # 1024 requests x 15 slots x rank 256 in bf16 need more than 4 MiB of scratch
    need = dflash2.selector_walk_workspace_size(1024, 15, 4096, 256, 16, dflash2.BF16)
    assert need > dflash2.NOALLOC_SCRATCH_BYTES
    lib = dflash2.library()
    status = lib.dflash2_selector_walk_noalloc(
        None, None, None, None, 1000, None, None, None, None, None, None, 1024, 15, 4096, 256,
        16, dflash2.BF16, None, None, None, None, None)
    assert status == 4   # DFLASH2_ERR_WORKSPACE, before any work is queued

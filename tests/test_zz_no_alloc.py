"""The allocation-free selector walk (dflash2_selector_walk_noalloc).

Some callers cannot hand the library a device buffer when they call it: a
serving loop whose device memory belongs to another allocator, or a
latency-critical path that must never reach cudaMalloc / cudaFree (they can
synchronise the device).  This entry point serves them from a fixed 4 MiB
array inside the library.  The tests check, through the C ABI, that two calls
in a row give bit for bit the tokens, q and edges of the workspace entry point
(the two run the same kernels on the same inputs), on the default stream and
on a stream of the caller's, including a shape whose scratch ends just short
of the array's end; and that shapes needing more scratch are refused.  The
file is named to run last, so that a failure here leaves the rest of the suite
already run.
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


def _largest_batch_that_fits(w):
    """The largest batch of w's other shapes whose walk scratch fits the array."""
    code = dflash2.BF16 if w.dtype == "bf16" else dflash2.F32
    batch = 1
    while dflash2.selector_walk_workspace_size(batch + 1, w.slots, w.hidden, w.rank, w.top_k,
                                               code) <= dflash2.NOALLOC_SCRATCH_BYTES:
        batch += 1
    return batch


CASES = [
    ("qwen3-8b-bf16", dict(batch=8, draft_vocab=20000, target_vocab=20000), False),
    ("stress-bf16", dict(batch=6, draft_vocab=20000, target_vocab=20000), True),
    ("tiny-fp32", {}, False),
    # the scratch (projection partials, then the lattice) ends within 32 KB (one request)
    # of the array's end
    ("reduced-vocab-bs12-bf16", dict(draft_vocab=20000, target_vocab=20000), True),
]


@pytest.mark.parametrize("name,scale,own_stream", CASES, ids=[c[0] for c in CASES])
def test_noalloc_walk_matches_the_workspace_walk_twice(name, scale, own_stream):
    dev = torch.device("cuda:0")
    w = synth.BY_NAME[name].scaled(**scale)
    if name == "reduced-vocab-bs12-bf16":
        w = w.scaled(batch=_largest_batch_that_fits(w))
        code = dflash2.BF16
        need = dflash2.selector_walk_workspace_size(w.batch, w.slots, w.hidden, w.rank, w.top_k,
                                                    code)
        assert dflash2.NOALLOC_SCRATCH_BYTES - 32768 < need <= dflash2.NOALLOC_SCRATCH_BYTES
    args = _inputs(w, dev, seed=123)
    ref_tok, ref_q, ref_ps, ref_err = dflash2.selector_walk(*args, with_path_scores=True)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream() if own_stream else None
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())
    for _ in range(2):   # the second call reuses the scratch the first one left behind
        tok, q, ps, err = dflash2.selector_walk_noalloc(*args, with_path_scores=True,
                                                        stream=stream)
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok)
        assert torch.equal(q, ref_q)
        assert torch.equal(ps, ref_ps)
        assert int(err.item()) == int(ref_err.item()) == 0


def test_noalloc_walk_refuses_shapes_beyond_its_scratch():
    # 1024 requests x 15 slots x rank 256 in bf16 need more than 4 MiB of scratch
    need = dflash2.selector_walk_workspace_size(1024, 15, 4096, 256, 16, dflash2.BF16)
    assert need > dflash2.NOALLOC_SCRATCH_BYTES
    lib = dflash2.library()
    status = lib.dflash2_selector_walk_noalloc(
        None, None, None, None, 1000, None, None, None, None, None, None, 1024, 15, 4096, 256,
        16, dflash2.BF16, None, None, None, None, None)
    assert status == 4   # DFLASH2_ERR_WORKSPACE, before any work is queued

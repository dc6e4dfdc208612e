"""GPU parity of the vocab-sharded unary top-K (dflash2_topk_merge).

Simulated shards on one GPU: each shard runs dflash2_unary_topk over its
slice of lm_head rows (dflash2.shard_topk), the lists are stacked as the
all-gather would stack them, and the merge must reproduce the unsharded
dflash2_unary_topk exactly (ids and u bit for bit): a vocab row's logits do
not depend on the slice that computes them.  The unsharded result itself is
pinned to the oracle by test_gpu_unary.py.  The merge's own edge cases
(absent entries, unsorted lists, short rows) are checked against a lexsort
of the union."""
import numpy as np
import pytest
import torch

from block_draft_proposal_gb300 import dflash2, synth

pytestmark = pytest.mark.gpu


def _sharded(w, t, shards):
    lists = [dflash2.shard_topk(t["h"], t["lm_head"][first:first + n], first, w.target_vocab,
                                w.mult, w.cap, w.top_k)
             for first, n, _ in (dflash2.vocab_shard(w.draft_vocab, w.target_vocab, shards, s)
                                 for s in range(shards))]
    ids = torch.stack([a for a, _ in lists])
    u = torch.stack([b for _, b in lists])
    offsets = [dflash2.vocab_shard(w.draft_vocab, w.target_vocab, shards, s)[0]
               for s in range(shards)]
    return dflash2.topk_merge(ids, u, offsets, w.top_k)


@pytest.mark.parametrize("name,scale,shards", [
    ("qwen3-8b-bf16", dict(batch=6, draft_vocab=30000, target_vocab=30000), 2),
    ("qwen3-8b-bf16", dict(batch=6, draft_vocab=30000, target_vocab=30000), 8),
    ("padded-vocab-bf16", dict(batch=3, draft_vocab=20000, target_vocab=12000), 3),
    ("stress-bf16", dict(batch=2, draft_vocab=9000, target_vocab=9000), 5),
    ("tiny-fp32", dict(draft_vocab=3000, target_vocab=2500), 2),
])
def test_simulated_shards_merge_to_the_unsharded_top_k(cuda, name, scale, shards):
    w = synth.BY_NAME[name].scaled(**scale)
    inp = synth.make(w, parts=("h", "lm_head"))
    t = {k: dflash2.to_device(v, cuda) for k, v in inp.items() if v is not None}
    ref_ids, ref_u, ref_err = dflash2.unary_topk(t["h"], t["lm_head"], w.target_vocab, w.mult,
                                                 w.cap, w.top_k)
    ids, u, err = _sharded(w, t, shards)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    if w.dtype == "bf16" and int(ref_err.item()) & dflash2.DEVINFO_TOPK_FALLBACK:
        # a row whose candidate list overflowed was recomputed on CUDA cores,
        # whose logits round differently from the tensor-core ones
        pytest.skip(f"{name}: a row took the CUDA-core recomputation")
    assert torch.equal(ids, ref_ids)
    assert torch.equal(u, ref_u)


def _lexsort_merge(ids, u, offsets, k_out):
    gid = ids + np.asarray(offsets)[:, None, None]
    gid = gid.transpose(1, 0, 2).reshape(ids.shape[1], -1)
    gu = u.transpose(1, 0, 2).reshape(ids.shape[1], -1).astype(np.float64)
    gu = np.where(np.isnan(gu), -np.inf, gu)
    order = np.lexsort((gid, -gu), axis=1)[:, :k_out]
    out_ids = np.take_along_axis(gid, order, axis=1)
    out_u = np.take_along_axis(gu, order, axis=1).astype(np.float32)
    out_ids[out_u == -np.inf] = 0
    return out_ids, out_u


@pytest.mark.parametrize("shards,rows,k_in,k_out", [(2, 5, 16, 16), (7, 3, 33, 20),
                                                    (4, 9, 128, 128), (32, 2, 128, 100),
                                                    (1, 4, 8, 8)])
def test_merge_of_unsorted_lists_with_absent_entries(cuda, shards, rows, k_in, k_out):
    rng = np.random.default_rng(1000 + shards * k_in)
    offsets = np.cumsum(rng.integers(2 * k_in, 3 * k_in, shards)) - 2 * k_in  # disjoint ranges
    ids = np.stack([np.stack([rng.choice(2 * k_in, size=k_in, replace=False) for _ in range(rows)])
                    for _ in range(shards)]).astype(np.int64)
    # few distinct values, so equal u across shards is common (ties by id)
    u = rng.integers(-6, 6, size=(shards, rows, k_in)).astype(np.float32) * 0.25
    u[rng.random(u.shape) < 0.2] = -np.inf
    u[rng.random(u.shape) < 0.05] = np.nan
    out_ids, out_u, err = dflash2.topk_merge(torch.from_numpy(ids).to(cuda),
                                             torch.from_numpy(u).to(cuda), offsets.tolist(), k_out)
    torch.cuda.synchronize()
    ref_ids, ref_u = _lexsort_merge(ids, u, offsets, k_out)
    np.testing.assert_array_equal(out_ids.cpu().numpy(), ref_ids)
    np.testing.assert_array_equal(out_u.cpu().numpy(), ref_u)
    present = (~np.isnan(u) & (u != -np.inf)).transpose(1, 0, 2).reshape(rows, -1).sum(1)
    assert bool(int(err.item()) & dflash2.DEVERR_SHORT) == bool((present < k_out).any())


def test_merge_drops_an_id_past_the_largest_vocab(cuda):
    ids = torch.tensor([[[5, 2]], [[0, 3]]], dtype=torch.int64, device=cuda)
    u = torch.tensor([[[1.0, 0.5]], [[2.0, 0.25]]], dtype=torch.float32, device=cuda)
    out_ids, out_u, err = dflash2.topk_merge(ids, u, [0, 2**31 - 1], 3)
    torch.cuda.synchronize()
    # global ids up to 2^32 - 2 fit a key: shard 1's land at 2^31 - 1 and 2^31 + 2
    assert out_ids.tolist() == [[2**31 - 1, 5, 2]] and int(err.item()) == 0
    # a global id below zero cannot: it is dropped and flagged
    ids[1, 0, 0] = -2**31 - 5
    out_ids, out_u, err = dflash2.topk_merge(ids, u, [0, 2**31 - 1], 3)
    torch.cuda.synchronize()
    assert out_ids.tolist() == [[5, 2, 2**31 + 2]]
    assert int(err.item()) & dflash2.DEVERR_ID_RANGE


def test_sharded_helper_through_a_process_group(cuda):
    """unary_topk_vocab_sharded end to end on a one-rank NCCL group: the shard
    is the whole head, the all-gather and the merge still run."""
    import os
    import socket
    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=cuda)
    try:
        w = synth.BY_NAME["qwen3-8b-bf16"].scaled(batch=4, draft_vocab=12000, target_vocab=11000)
        inp = synth.make(w, parts=("h", "lm_head"))
        t = {k: dflash2.to_device(v, cuda) for k, v in inp.items() if v is not None}
        ref_ids, ref_u, _ = dflash2.unary_topk(t["h"], t["lm_head"], w.target_vocab, w.mult,
                                               w.cap, w.top_k)
        ids, u, err = dflash2.unary_topk_vocab_sharded(t["h"], t["lm_head"], w.draft_vocab,
                                                       w.target_vocab, w.mult, w.cap, w.top_k)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(ids, ref_ids) and torch.equal(u, ref_u)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("shards,rows,k_in,k_out", [(64, 1, 1, 64), (64, 3, 64, 128),
                                                    (3, 1, 1, 1)])
def test_merge_edge_shapes(cuda, shards, rows, k_in, k_out):
    rng = np.random.default_rng(2000 + shards + k_in)
    offsets = np.arange(shards) * 1000
    ids = rng.integers(0, 1000, (shards, rows, k_in)).astype(np.int64)
    u = rng.normal(0, 1, (shards, rows, k_in)).astype(np.float32)
    out_ids, out_u, err = dflash2.topk_merge(torch.from_numpy(ids).to(cuda),
                                             torch.from_numpy(u).to(cuda), offsets.tolist(), k_out)
    torch.cuda.synchronize()
    ref_ids, ref_u = _lexsort_merge(ids, u, offsets, k_out)
    np.testing.assert_array_equal(out_ids.cpu().numpy(), ref_ids)
    np.testing.assert_array_equal(out_u.cpu().numpy(), ref_u)
    assert bool(int(err.item()) & dflash2.DEVERR_SHORT) == (shards * k_in < k_out)

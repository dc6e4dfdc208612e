"""The multi-rank host path of bench.py on CPU: two gloo ranks agree on the
slowest rank's step time, the job value counts every rank's proposals, and the
reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [1.0 + rank, 10.0 - rank]           # rank 1 is slower on the first value
    got = bench.reduce_max_over_ranks(mine)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, got, bench.job_value(world, 480, got[0])))


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [2.0, 10.0]
        assert value == pytest.approx(2 * 480 / 2.0e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from block_draft_proposal_gb300 import synth
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, gpus = 1, 3, 2

    assert bench.run_reference(Args, synth.BY_NAME["tiny-fp32"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_json_line(monkeypatch, capsys):
    import json
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from block_draft_proposal_gb300 import synth
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)

    class Args:
        steps, warmup, gpus = 2, 3, 1

    assert bench.run_reference(Args, synth.BY_NAME["tiny-fp32"]) == 0
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    line = json.loads(out[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == bench.UNIT
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_vocab_shards_partition_the_vocab():
    import sys
    sys.path.insert(0, ROOT)
    from block_draft_proposal_gb300 import dflash2
    for vd, vt in ((151936, 151936), (201024, 200058), (32768, 151936), (20000, 12000), (5, 5)):
        for world in (1, 2, 3, 7, 8):
            parts = [dflash2.vocab_shard(vd, vt, world, s) for s in range(world)]
            nxt = 0
            for first, n, valid in parts:
                assert first == nxt and n >= 0 and 0 <= valid <= n
                nxt = first + n
            assert nxt == vd
            assert sum(v for _, _, v in parts) == min(vd, vt)


def _shard_rank_main(rank, world, port, out):
    """One rank of a vocab-sharded top-K on CPU: the oracle's u over this
    rank's lm_head rows, its local top-K list, the product's all-gather."""
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import numpy as np
    import torch
    import torch.distributed as dist
    import oracle
    from block_draft_proposal_gb300 import dflash2, synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = synth.BY_NAME["tiny-fp32"].scaled(draft_vocab=3000, target_vocab=2500, batch=2)
    inp = synth.make(w, parts=("h", "lm_head"))
    k = w.top_k
    first, n, valid = dflash2.vocab_shard(w.draft_vocab, w.target_vocab, world, rank)
    ids = np.zeros((w.rows, k), dtype=np.int64)
    u = np.full((w.rows, k), -np.inf)
    if valid > 0:
        us = oracle.unary_rows(inp["h"], inp["lm_head"][first:first + n], valid, w.mult, w.cap)
        kk = min(k, valid)
        # this shard's k best in double, ties by the smaller id
        order = np.lexsort((np.arange(n)[None, :].repeat(w.rows, 0), -us), axis=1)[:, :kk]
        ids[:, :kk] = order
        u[:, :kk] = np.take_along_axis(us, order, axis=1)
    all_ids, all_u = dflash2.gather_shard_lists(torch.from_numpy(ids), torch.from_numpy(u))
    offsets = [dflash2.vocab_shard(w.draft_vocab, w.target_vocab, world, s)[0]
               for s in range(world)]
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, all_ids.numpy(), all_u.numpy(), offsets))


def test_vocab_sharded_lists_gather_into_the_unsharded_top_k():
    import sys
    sys.path.insert(0, ROOT)
    import numpy as np
    import oracle
    from block_draft_proposal_gb300 import synth
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = synth.BY_NAME["tiny-fp32"].scaled(draft_vocab=3000, target_vocab=2500, batch=2)
    inp = synth.make(w, parts=("h", "lm_head"))
    ref_ids, _ = oracle.topk(oracle.unary_rows(inp["h"], inp["lm_head"], w.target_vocab, w.mult,
                                               w.cap), w.top_k)
    for rank, all_ids, all_u, offsets in res:
        assert all_ids.shape == (world, w.rows, w.top_k)
        np.testing.assert_array_equal(all_u, res[0][2])        # every rank holds every list
        gid = all_ids + np.asarray(offsets)[:, None, None]
        gid = gid.transpose(1, 0, 2).reshape(w.rows, -1)
        gu = all_u.transpose(1, 0, 2).reshape(w.rows, -1)
        order = np.lexsort((gid, -gu), axis=1)[:, :w.top_k]    # u descending, then id
        np.testing.assert_array_equal(np.take_along_axis(gid, order, axis=1), ref_ids)

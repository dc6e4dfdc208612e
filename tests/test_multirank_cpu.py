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

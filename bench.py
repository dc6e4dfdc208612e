"""Benchmark of the DFlash2 draft-proposal hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
grouped conv, unary candidates (lm_head GEMM + transform + padded mask +
top-K), selector walk (projection + edges + walk) and d2t remap, through the
C ABI (dflash2.proposal_step, the input-only work on a second stream beside
the top-K), replayed from one captured CUDA graph.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME] [--stage conv|unary_topk|unary_topk_fp8|
                                               unary_topk_nvfp4|projection|walk]

The default workload is the largest one-GPU configuration, the large-batch,
large-K stress draft (batch 512, block 16, hidden 7168 = 896 groups x 8, taps
4, vocab 163840, rank 128, top-K 64, cap 30, mult 0.5, every row sampled at
T = 0.6); the other named workloads run with --workload.  The metric is
proposals per second (batch x slots proposed / step time).  L2 is flushed
before every timed step (a 256 MiB write, then a read of the same buffer, so
no dirty line is left) and the flush is outside the timed events.  Prints ONE JSON line (rank 0).

`--impl reference` times the CPU oracle (the method restated in plain C,
double accumulation) on a bounded sample of the same workload on the host
cores; it never touches the GPU.  Under torchrun every rank runs its own
replica of the workload (weak scaling; requests are independent, so there is
no data-path collective) and the step time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft blocks/sec (batch×slots proposed/s) + % HBM / tensor roofline per kernel"
UNIT = "proposals/s"
DEFAULT_WORKLOAD = "stress-bf16"
L2_FLUSH_BYTES = 256 << 20
# DRAM bytes of the unary top-K stage per workload, from one ncu capture of
# the stage's launches, keyed by the hash of the sources that make the stage
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def flush_l2(buf):
    """Evicts the L2 before a timed call: writes `buf` (larger than the L2),
    then reads it back, so that the L2 holds only clean lines of `buf` when the
    timer starts (after the write alone the timed kernel would pay for writing
    the flush's dirty lines back to HBM)."""
    import torch
    buf.zero_()
    buf.view(torch.int64).sum()


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max_over_ranks(values, device="cpu"):
    """Element-wise maximum of a list of floats over all ranks of the default
    process group (the step time of a job is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_value(world: int, rows_per_rank: int, ms: float) -> float:
    """Proposals per second of the whole job: every rank proposes rows_per_rank
    rows per step (weak scaling) and the step takes the slowest rank's time."""
    return world * rows_per_rank / (ms * 1e-3)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def algorithmic_work(w):
    """Per-call algorithmic work of each stage (bytes moved at minimum, or flops)."""
    e = 2 if w.dtype == "bf16" else 4
    n, hdim, g = w.n_tokens, w.hidden, w.groups
    conv_bytes = 2 * n * hdim * e + n * w.taps * g * e + w.taps * hdim * e
    gemm_flops = 2 * w.rows * w.draft_vocab * hdim
    # walk incl. projection: h and proj once, per slot K candidate B rows + one A
    # row, the unary values, ids, uniforms; outputs q and tokens
    walk_bytes = (w.rows * hdim * e + w.rank * hdim * e
                  + w.rows * (w.top_k + 1) * w.rank * e
                  + w.rows * w.top_k * (4 + 8) + w.rows * 4
                  + w.rows * w.top_k * 4 + w.rows * 8)
    d2t_bytes = w.rows * (8 + 8 + (8 if w.uses_d2t else 0))
    # conv prepare (beside the step): kernel projection n x hidden x 2*taps*groups
    kproj_flops = 2 * n * hdim * (2 * w.taps * g)
    # verify (beside the step): the target logits once, plus the per-chunk partials
    # (32 x 16 B per position, written and read) and the small per-slot inputs
    pos = w.batch * (w.slots + 1)
    verify_bytes = (pos * w.target_vocab * e + 2 * pos * ((w.target_vocab + 4095) // 4096) * 16
                    + w.rows * w.top_k * (8 + 4) + pos * (4 + 8))
    return dict(conv_bytes=conv_bytes, gemm_flops=gemm_flops, walk_bytes=walk_bytes,
                d2t_bytes=d2t_bytes, kproj_flops=kproj_flops, verify_bytes=verify_bytes)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _profile_traffic(workload: str, src_hash: str):
    """DRAM bytes (read + write) of one unary_topk stage (all its launches) of
    `workload` from the committed ncu record, or None when there is none or
    the stage's sources changed since the capture."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_sha16") != src_hash:
        return None
    return float(rec["unary_topk_dram_bytes"])


_NCU_BYTES = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}


def write_traffic(csv_path: str, workload: str, command: str):
    """Records in TRAFFIC_FILE the DRAM bytes (dram__bytes_read.sum +
    dram__bytes_write.sum) of every launch in an ncu --csv metrics log of one
    unary_topk stage call, keyed by workload and by the current hash of the
    stage's sources."""
    import csv
    with open(csv_path) as f:
        rows = [r for r in csv.reader(f) if len(r) > 10]
    head = rows[0]
    ik, im, iu, iv = (head.index("Kernel Name"), head.index("Metric Name"),
                      head.index("Metric Unit"), head.index("Metric Value"))
    iid = head.index("ID")
    total, kernels = 0.0, {}
    for r in rows[1:]:
        if r[im] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            b = float(r[iv].replace(",", "")) * _NCU_BYTES[r[iu]]
            total += b
            kernels.setdefault(r[iid], [r[ik].split("(")[0].split("::")[-1], 0.0])[1] += b
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        rec = {}
    src_hash, srcs = kernel_source_hash()
    rec[workload] = {"unary_topk_dram_bytes": total,
                     "launches": [{"kernel": k, "dram_bytes": v} for k, v in kernels.values()],
                     "source_sha16": src_hash,
                     "sources": [os.path.relpath(p, ROOT) for p in srcs],
                     "command": command}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(rec, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps({"workload": workload, "unary_topk_dram_bytes": total,
                      "launches": len(kernels)}))
    return 0


def kernel_source_hash():
    import hashlib
    srcs = [os.path.join(ROOT, "block_draft_proposal_gb300", "csrc", f)
            for f in ("gemm_tc.cu", "topk.cu", "common.cuh", "kernels.h")]
    h = hashlib.sha256()
    for path in srcs:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16], srcs


# ---------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------------------

def oracle_sample_time(w, inp, n_requests: int):
    """Time the oracle chain over the first n_requests requests of the workload."""
    import oracle
    rows = n_requests * w.slots
    t0 = time.perf_counter()
    nt = n_requests * w.block_size
    oracle.conv(inp["x"][:nt], inp["base"], inp["delta"][:nt], w.block_size, w.group_size, w.taps)
    u = oracle.unary_rows(inp["h"], inp["lm_head"], w.target_vocab, w.mult, w.cap,
                          rows=list(range(rows)))
    ids, vals = oracle.topk(u, w.top_k)
    sel = oracle.selector(inp["h"][:rows], inp["proj"], inp["A"], inp["B"], inp["anchors"][:n_requests],
                          ids.reshape(n_requests, w.slots, w.top_k),
                          vals.reshape(n_requests, w.slots, w.top_k), inp["uniforms"][:n_requests],
                          inp["temperatures"][:n_requests], inp["greedy"][:n_requests])
    oracle.d2t(sel["tokens"].reshape(-1), inp["d2t"], w.draft_vocab, w.target_vocab)
    return time.perf_counter() - t0


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, w):
    rank, world, _ = _dist()
    if rank != 0:
        return 0
    from block_draft_proposal_gb300 import synth
    inp = synth.make(w)
    n_req = 1
    for _ in range(args.warmup):
        oracle_sample_time(w, inp, n_req)
    times = [oracle_sample_time(w, inp, n_req) for _ in range(args.steps)]
    t = statistics.mean(times)
    value = n_req * w.slots / t
    sample = (f"{n_req} request ({n_req * w.slots} proposal rows) of {w.name} per step: conv of its "
              f"block, unary logits over the full vocab, full-sort top-K, lattice + walk, d2t")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(w):
    return {"workload": w.name, "batch": w.batch, "block_size": w.block_size, "slots": w.slots,
            "hidden": w.hidden, "group_size": w.group_size, "taps": w.taps,
            "draft_vocab": w.draft_vocab, "target_vocab": w.target_vocab, "rank": w.rank,
            "top_k": w.top_k, "mult": w.mult, "cap": w.cap, "sampling": w.sampling,
            "temperature": w.temperature,
            "l2": "value: flushed before every timed step (256 MiB write then read back, outside the "
                  "timed events); "
                  "e2e: a pipelined loop without flush, inputs larger than L2 (the lm_head streams "
                  "from HBM at every step)",
            "e2e": "double-buffered device inputs and outputs: the next step's H2D copy and the "
                   "previous step's D2H read-back overlap this step's compute; timed from the "
                   "first copy to the last D2H read-back",
            "graph": "one CUDA graph per step (replayed)"}


# ---------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------

def run_gpu(args, w):
    import numpy as np
    import torch

    rank, world, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)

    import __graft_entry__ as g
    g.build_library()
    from block_draft_proposal_gb300 import dflash2, synth

    inp = synth.make(w)
    t = {k: dflash2.to_device(v, dev) for k, v in inp.items() if v is not None}
    bufs = dflash2.ProposalBuffers(w, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    # the walk's uniforms are drawn on the device at every step; the counter
    # lives on the device so each graph replay draws a fresh sequence
    rng_counter = torch.zeros(1, dtype=torch.int64, device=dev)
    uniforms = t["uniforms"].view(-1)

    def step(record: bool, t=t, b=bufs):
        if not record:
            # the timed step: the public API, the input-only work (uniforms,
            # conv, selector projection) on a second stream beside the top-K
            dflash2.proposal_step(w, t, b, stream=stream, rng=(w.seed, rng_counter))
            return
        # the staged step: the same launches on one stream, with events
        # between the stages
        ev[0].record(stream)
        dflash2.grouped_conv(t["x"], t["base"], t["delta"], w.block_size, w.group_size, w.taps,
                             out=bufs.conv_out, stream=stream)
        ev[1].record(stream)
        dflash2.unary_topk(t["h"], t["lm_head"], w.target_vocab, w.mult, w.cap, w.top_k,
                           cand_ids=bufs.cand_ids, cand_u=bufs.cand_u, workspace=bufs.ws_topk,
                           err=bufs.err, stream=stream)
        ev[2].record(stream)
        dflash2.philox_uniforms(w.seed, w.rows, out=uniforms, counter=rng_counter, stream=stream)
        dflash2.selector_walk(t["h"], t["proj"], t["A"], t["B"], t["anchors"],
                              bufs.cand_ids.view(w.batch, w.slots, w.top_k),
                              bufs.cand_u.view(w.batch, w.slots, w.top_k), t["temperatures"],
                              t["greedy"], t["uniforms"], tokens=bufs.tokens, q=bufs.q,
                              workspace=bufs.ws_walk, err=bufs.err, stream=stream)
        ev[3].record(stream)
        dflash2.d2t_remap(bufs.tokens, t.get("d2t"), w.draft_vocab, w.target_vocab,
                          out=bufs.target_ids, err=bufs.err, stream=stream)
        ev[4].record(stream)

    # capture one step into a graph (stage events cannot be timed inside a graph)
    with torch.cuda.stream(stream):
        step(False)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    use_graph = True
    try:
        with torch.cuda.graph(graph, stream=stream):
            step(False)
    except Exception:
        use_graph = False
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2(flush)
            graph.replay() if use_graph else step(False)
            flush_l2(flush)
            step(True)
    stream.synchronize()

    # timed region: K graph replays (the value), then K eager steps with stage
    # events (the per-stage breakdown and the roofline); L2 flushed before each
    # step, outside the events.  Events are read after one final synchronize.
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush_l2(flush)
                gev[i][0].record(stream)
                graph.replay() if use_graph else step(False)
                gev[i][1].record(stream)
            for i in range(args.steps):
                flush_l2(flush)
                ev[:] = sev[i]
                step(True)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    graph_ms = [a.elapsed_time(b) for a, b in gev]
    stage_ms = {
        "conv": [e[0].elapsed_time(e[1]) for e in sev],
        "unary_topk": [e[1].elapsed_time(e[2]) for e in sev],
        "walk": [e[2].elapsed_time(e[3]) for e in sev],
        "d2t": [e[3].elapsed_time(e[4]) for e in sev],
        "step": [e[0].elapsed_time(e[4]) for e in sev],
    }
    ms = statistics.mean(graph_ms)
    eager_ms = statistics.mean(stage_ms["step"])
    err = int(bufs.err.item())

    # end to end through the public API, as a serving loop runs it: every step
    # copies its inputs from pinned host memory into one of two device input
    # sets on a copy stream (overlapping the previous step's compute), replays
    # the captured step on that set (each set has its own outputs), and reads
    # its tokens and q back into pinned host memory on a third stream, so the
    # next step's compute does not wait for the read-back.  Timed from the
    # first copy to the last read-back over K steps; the lm_head (1.2 GB and
    # more) streams from HBM at every step (inputs larger than L2), so this
    # loop runs without the flush.
    in_keys = ("x", "delta", "h", "temperatures", "greedy", "anchors")
    host_in = {k: torch.from_numpy(inp[k].view(np.int16) if inp[k].dtype == np.uint16 else inp[k])
               .pin_memory() for k in in_keys}
    t_b = dict(t)
    t_b.update({k: t[k].clone() for k in in_keys})  # valid inputs for the warm-up before capture
    sets = [t, t_b]
    outs = [bufs, dflash2.ProposalBuffers(w, dev)]
    graphs = [graph, None]
    if use_graph:
        with torch.cuda.stream(stream):
            step(False, t=t_b, b=outs[1])
        stream.synchronize()
        graphs[1] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[1], stream=stream):
            step(False, t=t_b, b=outs[1])
    host_tok = [torch.empty(bufs.target_ids.shape, dtype=torch.int64).pin_memory() for _ in range(2)]
    host_q = [torch.empty(bufs.q.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = host_tok[0].numel() * 8 + host_q[0].numel() * 4
    copy_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    ev_copied = [torch.cuda.Event() for _ in range(2)]   # set j's inputs are on the device
    ev_free = [torch.cuda.Event() for _ in range(2)]     # set j's step is done with its inputs
    ev_read = [torch.cuda.Event() for _ in range(2)]     # set j's outputs are on the host

    def e2e_steps(n):
        for i in range(n):
            j = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(ev_free[j])  # the step two back is done with set j
                for k, hv in host_in.items():
                    dv = sets[j][k]
                    if dv.dtype == torch.bfloat16:
                        dv = dv.view(torch.int16)
                    dv.copy_(hv, non_blocking=True)
                ev_copied[j].record(copy_stream)
            stream.wait_event(ev_copied[j])
            stream.wait_event(ev_read[j])  # the step two back has been read back
            with torch.cuda.stream(stream):
                if use_graph:
                    graphs[j].replay()
                else:
                    step(False, t=sets[j], b=outs[j])
                ev_free[j].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev_free[j])
                host_tok[j].copy_(outs[j].target_ids, non_blocking=True)
                host_q[j].copy_(outs[j].q, non_blocking=True)
                ev_read[j].record(d2h_stream)

    e2e_steps(args.warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(copy_stream)
    e2e_steps(args.steps)
    e1.record(d2h_stream)
    torch.cuda.synchronize()
    e2e = e0.elapsed_time(e1) / args.steps

    # NEXT-row kernels timed beside the step (not part of its value): the grouped
    # conv's prepare (kernel projection GEMM + input-side conv), L2 flushed
    next_rows = {}
    if w.dtype == "bf16":
        dk = synth.make(w, parts=("w_kp", "base2"))
        t_wkp, t_base2 = dflash2.to_device(dk["w_kp"], dev), dflash2.to_device(dk["base2"], dev)
        coef = torch.empty((w.n_tokens, 2, w.taps, w.groups), dtype=torch.bfloat16, device=dev)
        p_out = torch.empty_like(t["x"])
        p_err = torch.zeros(1, dtype=torch.int32, device=dev)
        reps = max(1, min(args.steps, 200))
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]

        def prep():
            dflash2.conv_prepare(t["x"], t_wkp, t_base2, w.block_size, w.group_size, w.taps,
                                 out=p_out, coef=coef, err=p_err, stream=stream)

        with torch.cuda.stream(stream):
            prep()
        stream.synchronize()
        pgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pgraph, stream=stream):
            prep()
        with torch.cuda.stream(stream):
            for i in range(args.warmup + reps):
                flush_l2(flush)
                if i >= args.warmup:
                    pev[i - args.warmup][0].record(stream)
                pgraph.replay()
                if i >= args.warmup:
                    pev[i - args.warmup][1].record(stream)
        torch.cuda.synchronize()
        next_rows["conv_prepare"] = {"ms": statistics.mean(a.elapsed_time(b) for a, b in pev),
                                     "calls": reps, "err": int(p_err.item())}

        # verification of the step's proposals against synthetic target logits
        # [B, S+1, V_t] (seeded, on the device), uniforms from the device generator
        gen = torch.Generator(device=dev)
        gen.manual_seed(w.seed)
        tlog = torch.randn((w.batch, w.slots + 1, w.target_vocab), generator=gen, device=dev,
                           dtype=torch.float32).to(torch.bfloat16)
        v_unif = torch.empty((w.batch, w.slots + 1), dtype=torch.float32, device=dev)
        v_counter = torch.full((1,), 1 << 40, dtype=torch.int64, device=dev)
        tgt_cand = torch.empty_like(bufs.cand_ids)
        v_acc = torch.empty(w.batch, dtype=torch.int64, device=dev)
        v_out = torch.empty((w.batch, w.slots + 1), dtype=torch.int64, device=dev)
        v_ws = torch.empty(dflash2.verify_workspace_size(w.batch, w.slots, w.target_vocab),
                           dtype=torch.uint8, device=dev)
        v_err = torch.zeros(1, dtype=torch.int32, device=dev)

        def ver():
            dflash2.d2t_remap(bufs.cand_ids, t.get("d2t"), w.draft_vocab, w.target_vocab,
                              out=tgt_cand, err=v_err, stream=stream)
            dflash2.philox_uniforms(w.seed + 1, v_unif.numel(), out=v_unif.view(-1),
                                    counter=v_counter, stream=stream)
            dflash2.verify(tlog, t["temperatures"], t["greedy"], bufs.target_ids,
                           tgt_cand.view(w.batch, w.slots, w.top_k), bufs.q, v_unif,
                           accept_len=v_acc, out_tokens=v_out, workspace=v_ws, err=v_err,
                           stream=stream)

        with torch.cuda.stream(stream):
            ver()
        stream.synchronize()
        vgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(vgraph, stream=stream):
            ver()
        vev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        with torch.cuda.stream(stream):
            for i in range(args.warmup + reps):
                flush_l2(flush)
                if i >= args.warmup:
                    vev[i - args.warmup][0].record(stream)
                vgraph.replay()
                if i >= args.warmup:
                    vev[i - args.warmup][1].record(stream)
        torch.cuda.synchronize()
        next_rows["verify"] = {"ms": statistics.mean(a.elapsed_time(b) for a, b in vev),
                               "calls": reps, "err": int(v_err.item()),
                               "mean_accept_len": float(v_acc.double().mean().item())}
        del tlog

        # the FP8 (E4M3) head: the same candidates from a W8A8 head (activation
        # quantization + kind::f8f6f4 top-K), one captured call replayed
        fq = synth.make(w, parts=("lm_head_fp8", "w_scale"))
        t_q8, t_sw = dflash2.to_device(fq["lm_head_fp8"], dev), dflash2.to_device(fq["w_scale"], dev)
        del fq
        f_ids = torch.empty_like(bufs.cand_ids)
        f_u = torch.empty_like(bufs.cand_u)
        f_ws = torch.empty(dflash2.unary_topk_fp8_workspace_size(w.rows, w.hidden, w.draft_vocab,
                                                                 w.top_k),
                           dtype=torch.uint8, device=dev)
        f_err = torch.zeros(1, dtype=torch.int32, device=dev)

        def fp8():
            dflash2.unary_topk_fp8(t["h"], t_q8, t_sw, w.target_vocab, w.mult, w.cap, w.top_k,
                                   cand_ids=f_ids, cand_u=f_u, workspace=f_ws, err=f_err,
                                   stream=stream)

        with torch.cuda.stream(stream):
            fp8()
        stream.synchronize()
        fgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(fgraph, stream=stream):
            fp8()
        fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        with torch.cuda.stream(stream):
            for i in range(args.warmup + reps):
                flush_l2(flush)
                if i >= args.warmup:
                    fev[i - args.warmup][0].record(stream)
                fgraph.replay()
                if i >= args.warmup:
                    fev[i - args.warmup][1].record(stream)
        torch.cuda.synchronize()
        next_rows["unary_topk_fp8"] = {"ms": statistics.mean(a.elapsed_time(b) for a, b in fev),
                                       "calls": reps, "err": int(f_err.item())}
        del t_q8

        # the NVFP4 head: W4A4 with E4M3 scales per 16 elements (activation
        # quantization + kind::mxf4nvf4 block-scaled top-K), one captured call
        if w.hidden % 64 == 0:
            nq = synth.make(w, parts=("lm_head_nvfp4", "w_scales_nvfp4"))
            t_q4 = dflash2.to_device(nq["lm_head_nvfp4"], dev)
            t_s4 = dflash2.nvfp4_tile_scales(dflash2.to_device(nq["w_scales_nvfp4"], dev),
                                             w.hidden)
            g4 = synth.nvfp4_w_global(w)
            del nq
            n_ws = torch.empty(dflash2.unary_topk_nvfp4_workspace_size(w.rows, w.hidden,
                                                                       w.draft_vocab, w.top_k),
                               dtype=torch.uint8, device=dev)

            def nvfp4():
                dflash2.unary_topk_nvfp4(t["h"], t_q4, t_s4, g4, w.target_vocab, w.mult, w.cap,
                                         w.top_k, cand_ids=f_ids, cand_u=f_u, workspace=n_ws,
                                         err=f_err, stream=stream)

            f_err.zero_()
            with torch.cuda.stream(stream):
                nvfp4()
            stream.synchronize()
            ngraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ngraph, stream=stream):
                nvfp4()
            nev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            with torch.cuda.stream(stream):
                for i in range(args.warmup + reps):
                    flush_l2(flush)
                    if i >= args.warmup:
                        nev[i - args.warmup][0].record(stream)
                    ngraph.replay()
                    if i >= args.warmup:
                        nev[i - args.warmup][1].record(stream)
            torch.cuda.synchronize()
            next_rows["unary_topk_nvfp4"] = {
                "ms": statistics.mean(a.elapsed_time(b) for a, b in nev), "calls": reps,
                "err": int(f_err.item())}
            del t_q4, t_s4, n_ws

    # max over ranks
    if world > 1:
        ms, e2e = reduce_max_over_ranks([ms, e2e], device=dev)

    # conv, unary (as the library reports for this device and shape), uniforms,
    # walk (projection, then rows + chase in lattice mode, top_k <= 32, or the
    # path-mode walk), d2t
    walk_launches = 3 if w.top_k <= 32 else 2
    unary_launches = dflash2.library().dflash2_unary_topk_launches(
        w.rows, w.draft_vocab, w.top_k, w.mult, dflash2.BF16 if w.dtype == "bf16" else dflash2.F32)
    launches_per_step = 1 + unary_launches + 1 + walk_launches + 1

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    hbm, tf_burst, tf_sust, peak_kind = _peaks()
    # The stage is timed across the whole eager phase: when that phase lasts
    # seconds, the GPU runs at its power-capped sustained rate, so the
    # sustained peak (a seconds-long cuBLAS loop) is the denominator; a short
    # phase is compared with the burst peak.
    eager_phase_s = statistics.mean(stage_ms["unary_topk"]) * 1e-3 * args.steps
    roof_kind = "sustained" if eager_phase_s >= 1.0 else "burst"
    roof_peak = tf_sust if roof_kind == "sustained" else tf_burst
    work = algorithmic_work(w)
    unary_ms = statistics.mean(stage_ms["unary_topk"])
    achieved_tf = work["gemm_flops"] / (unary_ms * 1e-3) / 1e12
    src_hash, _ = kernel_source_hash()
    traffic = _profile_traffic(w.name, src_hash)
    conv_ms = statistics.mean(stage_ms["conv"])
    walk_ms = statistics.mean(stage_ms["walk"])
    stages = {
        "conv": {"ms": conv_ms, "GB/s": work["conv_bytes"] / (conv_ms * 1e-3) / 1e9,
                 "frac_hbm": work["conv_bytes"] / (conv_ms * 1e-3) / 1e9 / hbm},
        "unary_topk": {"ms": unary_ms, "TFLOP/s": achieved_tf, "frac_bf16_burst": achieved_tf / tf_burst,
                       "frac_bf16_sustained": achieved_tf / tf_sust},
        "walk": {"ms": walk_ms, "GB/s": work["walk_bytes"] / (walk_ms * 1e-3) / 1e9,
                 "frac_hbm": work["walk_bytes"] / (walk_ms * 1e-3) / 1e9 / hbm},
        "d2t": {"ms": statistics.mean(stage_ms["d2t"])},
    }
    if "conv_prepare" in next_rows:
        cp = next_rows["conv_prepare"]
        cp["TFLOP/s"] = work["kproj_flops"] / (cp["ms"] * 1e-3) / 1e12
        cp["frac_bf16_burst"] = cp["TFLOP/s"] / tf_burst
        cp["what"] = ("kernel projection x.W_kp^T (2*N*H*2*taps*G flops) + input-side conv, "
                      "one captured call replayed, beside the step")
    if "verify" in next_rows:
        vr = next_rows["verify"]
        vr["GB/s"] = work["verify_bytes"] / (vr["ms"] * 1e-3) / 1e9
        vr["frac_hbm"] = vr["GB/s"] / hbm
        vr["what"] = ("speculative-sampling verify of the step's proposals against synthetic "
                      "bf16 target logits [B, S+1, V_t] (candidate remap + uniforms + 2 kernels), "
                      "one captured call replayed; bytes = logits once + partials")

    if "unary_topk_fp8" in next_rows:
        f8 = next_rows["unary_topk_fp8"]
        f8["TFLOP/s"] = work["gemm_flops"] / (f8["ms"] * 1e-3) / 1e12
        # fp8 peak: the measured bf16 peak times the nominal fp8 / bf16 ratio (2)
        f8["frac_fp8_burst"] = f8["TFLOP/s"] / (2 * tf_burst)
        f8["frac_fp8_sustained"] = f8["TFLOP/s"] / (2 * tf_sust)
        f8["speedup_vs_bf16_stage"] = unary_ms / f8["ms"]
        f8["what"] = ("unary top-K from an E4M3 head with per-row scales: activation "
                      "quantization + tcgen05 kind::f8f6f4 GEMM + top-K, one captured call "
                      "replayed; 2*M*V*H flops; peak = measured bf16 x 2 (nominal ratio)")

    if "unary_topk_nvfp4" in next_rows:
        f4 = next_rows["unary_topk_nvfp4"]
        f4["TFLOP/s"] = work["gemm_flops"] / (f4["ms"] * 1e-3) / 1e12
        # fp4 peak: the measured bf16 peak times the nominal dense fp4 / bf16
        # ratio of GB300 (13.5 / 2.25 = 6)
        f4["frac_fp4_burst"] = f4["TFLOP/s"] / (6 * tf_burst)
        f4["frac_fp4_sustained"] = f4["TFLOP/s"] / (6 * tf_sust)
        f4["speedup_vs_bf16_stage"] = unary_ms / f4["ms"]
        f4["what"] = ("unary top-K from an NVFP4 head (E2M1 codes, E4M3 scale per 16 elements, "
                      "fp32 tensor scale) with per-row NVFP4 activations: activation "
                      "quantization + tcgen05 kind::mxf4nvf4 block-scaled GEMM + top-K, one "
                      "captured call replayed; 2*M*V*H flops; peak = measured bf16 x 6 "
                      "(nominal dense ratio)")

    # CPU baseline: the oracle as it stands on a bounded sample (rank 0, N = 1)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        # about 1.9e11 multiply-adds of the lm_head (10-20 s on 16 cores): 20
        # requests of the Qwen3-8B-shaped draft, 10 of the stress draft
        per_req = w.slots * w.draft_vocab * w.hidden
        n_req = max(1, min(w.batch, 20, int(round(1.9e11 / per_req))))
        tc = oracle_sample_time(w, inp, n_req)
        import oracle
        threads = oracle.set_threads(0)
        # the same chain on one core, over one request
        oracle.set_threads(1)
        try:
            t1 = oracle_sample_time(w, inp, 1)
        finally:
            oracle.set_threads(threads)
        cpu = {"value": n_req * w.slots / tc, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n_req} requests ({n_req * w.slots} proposal rows) of {w.name}: the "
                         f"whole oracle chain, {tc:.1f} s on {threads} OpenMP threads "
                         f"({_cores()} cores available)",
               "value_single_thread": w.slots / t1,
               "sample_single_thread": f"1 request ({w.slots} rows), one thread, {t1:.1f} s"}

    value = job_value(world, w.rows, ms)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded; weights N(0,0.02), "
        "activations N(0,1); walk uniforms drawn on the device by Philox4x64-10)", "config": _config(w),
        "roofline": {"bound": "tensor", "achieved": achieved_tf, "peak": roof_peak,
                     "unit": "TFLOP/s", "frac": achieved_tf / roof_peak, "traffic": traffic,
                     "traffic_source": "profiles/traffic.json" if traffic is not None else None,
                     "kernel": "unary_topk stage (fused pilot + select + filter GEMM, then "
                               "finalize), 2*M*V*H flops over the stage time",
                     "peak_kind": f"{peak_kind} bf16 {roof_kind}"},
        "stages": stages,
        "next_rows": next_rows,
        "cpu_baseline": cpu,
        "e2e": {"value": job_value(world, w.rows, e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps * 2,  # graph phase + eager phase
        "clocks": clocks.summary(),
        "device_err_word": err,
        "graph": use_graph,
        "eager_ms_per_step": eager_ms,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_stage(args, w):
    """One stage of the path alone, `--steps` timed calls with L2 flushed
    before each (outside the events), on one stream; prints one JSON line with
    the median and minimum call time and the stage's algorithmic rate.  The
    walk runs on seeded synthetic candidates (distinct ids, descending u), so
    no lm_head is allocated: the command the committed ncu summaries of the
    conv, projection and walk kernels name."""
    import numpy as np
    import torch

    import __graft_entry__ as g
    g.build_library()
    from block_draft_proposal_gb300 import dflash2, synth

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    parts = {"conv": ("x", "base", "delta"),
             "unary_topk": ("h", "lm_head"),
             "unary_topk_fp8": ("h", "lm_head_fp8", "w_scale"),
             "unary_topk_nvfp4": ("h", "lm_head_nvfp4", "w_scales_nvfp4"),
             "projection": ("h", "proj"),
             "walk": ("h", "A", "B", "proj", "uniforms", "anchors")}[args.stage]
    inp = synth.make(w, parts=parts)
    t = {k: dflash2.to_device(v, dev) for k, v in inp.items() if v is not None}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)
    code = dflash2.BF16 if w.dtype == "bf16" else dflash2.F32
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    work = algorithmic_work(w)
    if args.stage == "conv":
        out = torch.empty_like(t["x"])
        fn = lambda: dflash2.grouped_conv(t["x"], t["base"], t["delta"], w.block_size,
                                          w.group_size, w.taps, out=out, stream=st)
        amount, unit = work["conv_bytes"], "GB/s"
    elif args.stage == "unary_topk":
        ids = torch.empty((w.rows, w.top_k), dtype=torch.int64, device=dev)
        u = torch.empty((w.rows, w.top_k), dtype=torch.float32, device=dev)
        ws = torch.empty(dflash2.unary_topk_workspace_size(w.rows, w.draft_vocab, w.top_k, code),
                         dtype=torch.uint8, device=dev)
        fn = lambda: dflash2.unary_topk(t["h"], t["lm_head"], w.target_vocab, w.mult, w.cap,
                                        w.top_k, cand_ids=ids, cand_u=u, workspace=ws, err=err,
                                        stream=st)
        amount, unit = work["gemm_flops"], "TFLOP/s"
    elif args.stage in ("unary_topk_fp8", "unary_topk_nvfp4"):
        ids = torch.empty((w.rows, w.top_k), dtype=torch.int64, device=dev)
        u = torch.empty((w.rows, w.top_k), dtype=torch.float32, device=dev)
        if args.stage == "unary_topk_fp8":
            ws = torch.empty(dflash2.unary_topk_fp8_workspace_size(w.rows, w.hidden, w.draft_vocab,
                                                                   w.top_k),
                             dtype=torch.uint8, device=dev)
            fn = lambda: dflash2.unary_topk_fp8(t["h"], t["lm_head_fp8"], t["w_scale"],
                                                w.target_vocab, w.mult, w.cap, w.top_k,
                                                cand_ids=ids, cand_u=u, workspace=ws, err=err,
                                                stream=st)
        else:
            ws = torch.empty(dflash2.unary_topk_nvfp4_workspace_size(w.rows, w.hidden,
                                                                     w.draft_vocab, w.top_k),
                             dtype=torch.uint8, device=dev)
            g4 = synth.nvfp4_w_global(w)
            tiles4 = dflash2.nvfp4_tile_scales(t["w_scales_nvfp4"], w.hidden)
            fn = lambda: dflash2.unary_topk_nvfp4(t["h"], t["lm_head_nvfp4"], tiles4,
                                                  g4, w.target_vocab, w.mult, w.cap, w.top_k,
                                                  cand_ids=ids, cand_u=u, workspace=ws, err=err,
                                                  stream=st)
        amount, unit = work["gemm_flops"], "TFLOP/s"
    else:
        ws = torch.empty(dflash2.selector_walk_workspace_size(w.batch, w.slots, w.hidden, w.rank,
                                                              w.top_k, code),
                         dtype=torch.uint8, device=dev)
        e = 2 if w.dtype == "bf16" else 4
        if args.stage == "projection":
            fn = lambda: dflash2.selector_project(t["h"], t["proj"], w.batch, w.slots, w.top_k,
                                                  ws, err=err, stream=st)
            amount, unit = w.rows * w.hidden * e + w.rank * w.hidden * e, "GB/s"
        else:
            rng = np.random.default_rng(w.seed + 1)
            cand = np.stack([rng.choice(w.draft_vocab, size=w.top_k, replace=False)
                             for _ in range(w.rows)]).astype(np.int64)
            cu = np.sort(rng.standard_normal((w.rows, w.top_k)).astype(np.float32),
                         axis=1)[:, ::-1].copy()
            tc = torch.from_numpy(cand).to(dev).view(w.batch, w.slots, w.top_k)
            tu = torch.from_numpy(cu).to(dev).view(w.batch, w.slots, w.top_k)
            tok = torch.empty((w.batch, w.slots), dtype=torch.int64, device=dev)
            q = torch.empty((w.batch, w.slots, w.top_k), dtype=torch.float32, device=dev)
            fn = lambda: dflash2.selector_walk(t["h"], t["proj"], t["A"], t["B"], t["anchors"], tc,
                                               tu, t["temperatures"], t["greedy"], t["uniforms"],
                                               tokens=tok, q=q, workspace=ws, err=err, stream=st)
            amount, unit = work["walk_bytes"], "GB/s"
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        for i in range(args.warmup + args.steps):
            flush_l2(flush)
            if i >= args.warmup:
                evs[i - args.warmup][0].record(st)
            fn()
            if i >= args.warmup:
                evs[i - args.warmup][1].record(st)
    torch.cuda.synchronize()
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    med = statistics.median(us)
    scale = 1e3 if unit == "GB/s" else 1e6
    print(json.dumps({"stage": args.stage, "workload": w.name, "calls": args.steps,
                      "us_median": med, "us_min": us[0], unit: amount / (med * scale),
                      "algorithmic": amount, "err": int(err.item())}), flush=True)
    return 0 if int(err.item()) & ~dflash2.DEVINFO_TOPK_FALLBACK == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--write-traffic", metavar="NCU_CSV",
                    help="record the DRAM bytes of an ncu --csv log of one unary_topk stage call "
                         "of --workload in profiles/traffic.json, then exit")
    ap.add_argument("--traffic-command", default="",
                    help="the ncu command that made the log (stored beside the bytes)")
    ap.add_argument("--stage", choices=["conv", "unary_topk", "unary_topk_fp8", "unary_topk_nvfp4",
                                        "projection", "walk"],
                    help="time one stage alone (one GPU) instead of the whole step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.write_traffic:
        return write_traffic(args.write_traffic, args.workload, args.traffic_command)
    from block_draft_proposal_gb300 import synth
    w = synth.BY_NAME[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.stage:
        return run_stage(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())

"""GPU parity of dflash2_selector_walk (projection, lattice edges, walk).

Staged parity: the oracle's projection, lattice and walk run on the GPU's own
candidates and unary values, so a near-tie in the top-K cannot cascade.
Tokens must equal the oracle's along each request until an accepted near-tie
(documented in parity.py); the edges the walk read (path_scores) must match
the oracle lattice row of the predecessor the GPU chose; q must match within
tolerance; greedy q is exactly one-hot and sampled q sums to one."""
import numpy as np
import pytest
import torch

import oracle
from block_draft_proposal_gb300 import dflash2, synth
from parity import compare_walk

pytestmark = pytest.mark.gpu


def _run_walk(dev, inp, cand, cand_u, with_ws=None):
    t = {k: dflash2.to_device(v, dev) for k, v in inp.items() if v is not None}
    tc = torch.from_numpy(np.ascontiguousarray(cand)).to(dev)
    tu = torch.from_numpy(np.ascontiguousarray(cand_u)).to(dev)
    tokens, q, ps, err = dflash2.selector_walk(t["h"], t["proj"], t["A"], t["B"], t["anchors"], tc,
                                               tu, t["temperatures"], t["greedy"], t["uniforms"],
                                               with_path_scores=True)
    torch.cuda.synchronize()
    return tokens.cpu().numpy(), q.cpu().numpy(), ps.cpu().numpy(), int(err.item())


def _compare(inp, cand, cand_u, tokens, q, ps, dtype, hidden):
    ora = oracle.selector(inp["h"], inp["proj"], inp["A"], inp["B"], inp["anchors"], cand, cand_u,
                          inp["uniforms"], inp["temperatures"], inp["greedy"])
    return compare_walk(inp, ora, cand, cand_u, tokens, q, ps, dtype, hidden)


def _named(name):
    w = synth.BY_NAME[name]
    inp = synth.make(w)
    return w, inp


@pytest.mark.parametrize("name", [c.name for c in synth.CONFIGS])
def test_walk_staged_parity_on_named_workloads(cuda, name):
    w, inp = _named(name)
    th, tw = dflash2.to_device(inp["h"], cuda), dflash2.to_device(inp["lm_head"], cuda)
    ids, vals, err = dflash2.unary_topk(th, tw, w.target_vocab, w.mult, w.cap, w.top_k)
    cand = ids.cpu().numpy().reshape(w.batch, w.slots, w.top_k)
    cand_u = vals.cpu().numpy().reshape(w.batch, w.slots, w.top_k)
    del th, tw
    tokens, q, ps, err2 = _run_walk(cuda, inp, cand, cand_u)
    assert int(err.item()) == 0 and err2 == 0
    ties = _compare(inp, cand, cand_u, tokens, q, ps, w.dtype, w.hidden)
    print(f"{name}: walk near-ties accepted {ties}")


def _random_candidates(w, seed, scale_ab=1.0):
    rng = np.random.default_rng(seed)
    inp = synth.make(w, parts=("h", "A", "B", "proj", "uniforms", "anchors"))
    if scale_ab != 1.0:
        for p in ("A", "B"):
            a = (synth.bf16_bits_to_f32(inp[p]) if w.dtype == "bf16" else inp[p]) * scale_ab
            inp[p] = synth.to_bf16_bits(a) if w.dtype == "bf16" else a.astype(np.float32)
    cand = np.stack([rng.choice(w.draft_vocab, size=w.top_k, replace=False)
                     for _ in range(w.rows)]).reshape(w.batch, w.slots, w.top_k).astype(np.int64)
    cand_u = np.sort(rng.standard_normal((w.batch, w.slots, w.top_k)).astype(np.float32),
                     axis=-1)[..., ::-1].copy()
    return inp, cand, cand_u


WALK_CASES = [
    dict(batch=6, block_size=9, hidden=192, rank=8, top_k=20, dtype="bf16", sampling="mixed", temperature=0.9),
    dict(batch=4, block_size=5, hidden=96, rank=16, top_k=1, dtype="bf16", sampling="sampled", temperature=1.0),
    dict(batch=5, block_size=17, hidden=128, rank=256, top_k=128, dtype="bf16", sampling="mixed", temperature=0.5),
    dict(batch=3, block_size=2, hidden=64, rank=32, top_k=33, dtype="f32", sampling="sampled", temperature=2.0),
    dict(batch=7, block_size=8, hidden=256, rank=16, top_k=8, dtype="f32", sampling="mixed", temperature=1e-7),
    # chain mode (bf16, 32 < top_k <= 128): ragged K under 64 with rank 40 (five
    # rank chunks, most lanes idle); one slot with K = 100 and rank 136 (a lane
    # with two chunks); 300 requests of K = 128 at rank 256 (whose buffers
    # exceed shared memory: the one-warp path walk), greedy rows with T below
    # its clamp
    dict(batch=9, block_size=6, hidden=160, rank=40, top_k=47, dtype="bf16", sampling="mixed", temperature=0.8),
    dict(batch=4, block_size=2, hidden=64, rank=136, top_k=100, dtype="bf16", sampling="sampled", temperature=0.3),
    dict(batch=300, block_size=4, hidden=96, rank=256, top_k=128, dtype="bf16", sampling="mixed", temperature=1e-7),
    dict(batch=5, block_size=16, hidden=128, rank=128, top_k=64, dtype="bf16", sampling="sampled", temperature=0.6),
    # chain mode with two shared B buffers: K <= 64 at rank 200, and K = 96 at rank 64
    dict(batch=7, block_size=7, hidden=96, rank=200, top_k=40, dtype="bf16", sampling="mixed", temperature=0.9),
    dict(batch=6, block_size=11, hidden=64, rank=64, top_k=96, dtype="bf16", sampling="sampled", temperature=0.4),
    # at least 4096 rows: the projection runs on CTA pairs with the tokens as the
    # weight side, split over hidden; hidden off the 128-element stage (1000)
    # and a rank off the 16-row tile (72), then chain mode at rank 128
    dict(batch=300, block_size=16, hidden=1000, rank=72, top_k=24, dtype="bf16", sampling="mixed", temperature=0.8),
    dict(batch=280, block_size=16, hidden=520, rank=128, top_k=48, dtype="bf16", sampling="sampled", temperature=0.7),
]


@pytest.mark.parametrize("case", WALK_CASES, ids=lambda c: f"r{c['rank']}-k{c['top_k']}-{c['dtype']}")
def test_walk_small_shapes(cuda, case):
    w = synth.BY_NAME["tiny-fp32"].scaled(draft_vocab=3000, target_vocab=3000, seed=97, **case)
    inp, cand, cand_u = _random_candidates(w, 98, scale_ab=20.0)
    tokens, q, ps, err = _run_walk(cuda, inp, cand, cand_u)
    assert err == 0
    _compare(inp, cand, cand_u, tokens, q, ps, w.dtype, w.hidden)


def test_out_of_range_ids_set_the_error_bit_and_use_zero_rows(cuda):
    w = synth.BY_NAME["tiny-fp32"].scaled(batch=3, block_size=4, hidden=64, rank=16, top_k=8, dtype="bf16",
                                draft_vocab=500, target_vocab=500, sampling="greedy", seed=99)
    inp, cand, cand_u = _random_candidates(w, 100, scale_ab=30.0)
    inp["anchors"] = inp["anchors"].copy()
    inp["anchors"][1] = 10_000
    cand[2, 1, 3] = -5
    tokens, q, ps, err = _run_walk(cuda, inp, cand, cand_u)
    assert err & dflash2.DEVERR_ID_RANGE
    ora = oracle.selector(inp["h"], inp["proj"], inp["A"], inp["B"], inp["anchors"], cand, cand_u,
                          inp["uniforms"], inp["temperatures"], inp["greedy"])
    assert ora["errors"] > 0
    # request 1's first slot falls back to the unary values alone
    np.testing.assert_allclose(ps[1, 0], cand_u[1, 0], rtol=0, atol=0)
    _compare(inp, cand, cand_u, tokens, q, ps, w.dtype, w.hidden)


def test_chain_mode_out_of_range_ids_set_the_error_bit_and_use_zero_rows(cuda):
    w = synth.BY_NAME["tiny-fp32"].scaled(batch=3, block_size=4, hidden=64, rank=16, top_k=40, dtype="bf16",
                                draft_vocab=500, target_vocab=500, sampling="mixed", seed=104)
    inp, cand, cand_u = _random_candidates(w, 105, scale_ab=30.0)
    inp["anchors"] = inp["anchors"].copy()
    inp["anchors"][1] = 10_000
    cand[2, 1, 3] = -5
    cand[0, 2, 39] = 500
    tokens, q, ps, err = _run_walk(cuda, inp, cand, cand_u)
    assert err & dflash2.DEVERR_ID_RANGE
    np.testing.assert_allclose(ps[1, 0], cand_u[1, 0], rtol=0, atol=0)
    _compare(inp, cand, cand_u, tokens, q, ps, w.dtype, w.hidden)


@pytest.mark.parametrize("top_k", [16, 48])
def test_greedy_rows_do_not_depend_on_other_rows(cuda, top_k):
    w = synth.BY_NAME["tiny-fp32"].scaled(batch=8, block_size=10, hidden=128, rank=32, top_k=top_k,
                                dtype="bf16", draft_vocab=2000, target_vocab=2000,
                                sampling="mixed", temperature=0.7, seed=101)
    inp, cand, cand_u = _random_candidates(w, 102, scale_ab=10.0)
    t1, q1, _, _ = _run_walk(cuda, inp, cand, cand_u)
    rng = np.random.default_rng(103)
    inp2 = dict(inp)
    inp2["uniforms"] = rng.random(inp["uniforms"].shape, dtype=np.float32)
    inp2["temperatures"] = np.where(inp["greedy"] == 1, np.float32(1.0),
                                    rng.uniform(0.1, 3.0, w.batch).astype(np.float32)).astype(np.float32)
    t2, q2, _, _ = _run_walk(cuda, inp2, cand, cand_u)
    g = inp["greedy"] == 1
    np.testing.assert_array_equal(t1[g], t2[g])
    np.testing.assert_array_equal(q1[g], q2[g])


@pytest.mark.parametrize("case", [WALK_CASES[0], WALK_CASES[2], WALK_CASES[3]],
                         ids=lambda c: f"r{c['rank']}-k{c['top_k']}-{c['dtype']}")
def test_projection_then_walk_equals_the_one_call_walk(cuda, case):
    """dflash2_selector_project on one stream, then dflash2_selector_walk_projected
    on another (ordered by an event), give exactly what dflash2_selector_walk gives."""
    w = synth.BY_NAME["tiny-fp32"].scaled(draft_vocab=3000, target_vocab=3000, seed=97, **case)
    inp, cand, cand_u = _random_candidates(w, 98, scale_ab=20.0)
    tokens, q, ps, err = _run_walk(cuda, inp, cand, cand_u)
    t = {k: dflash2.to_device(v, cuda) for k, v in inp.items() if v is not None}
    tc = torch.from_numpy(np.ascontiguousarray(cand)).to(cuda)
    tu = torch.from_numpy(np.ascontiguousarray(cand_u)).to(cuda)
    code = dflash2.BF16 if w.dtype == "bf16" else dflash2.F32
    ws = torch.full((dflash2.selector_walk_workspace_size(w.batch, w.slots, w.hidden, w.rank,
                                                          w.top_k, code),), 0xA5,
                    dtype=torch.uint8, device=cuda)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    dflash2.selector_project(t["h"], t["proj"], w.batch, w.slots, w.top_k, ws, stream=s1)
    done = torch.cuda.Event()
    done.record(s1)
    s2.wait_event(done)
    tok2, q2, ps2, err2 = dflash2.selector_walk_projected(
        t["A"], t["B"], t["anchors"], tc, tu, t["temperatures"], t["greedy"], t["uniforms"],
        w.hidden, ws, with_path_scores=True, stream=s2)
    torch.cuda.synchronize()
    assert int(err2.item()) == err == 0
    np.testing.assert_array_equal(tok2.cpu().numpy(), tokens)
    np.testing.assert_array_equal(q2.cpu().numpy(), q)
    np.testing.assert_array_equal(ps2.cpu().numpy(), ps)

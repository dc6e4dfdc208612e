"""GPU parity of dflash2_unary_topk (lm_head GEMM, transform, padded mask, top-K).

Ids must equal the oracle's except documented near-ties (see parity.py);
cand_u must lie within the fp32 forward-error bound of the exact u.  Small
cases cover several tiles with ragged tails in every dimension, compare every
row, and pin which path (the fused cooperative launch or the split passes) each
one takes; the named workloads run at full size with the oracle on every row
(three workloads) or on at least 64 rows that include each token tile's first
and last row (the padded-vocab and stress sizes); the candidate-list overflow
path, adversarial vocab orders, high padded logits and K equal to the logical
vocab are covered explicitly."""
import numpy as np
import pytest
import torch

import oracle
from block_draft_proposal_gb300 import dflash2, synth
from parity import compare_topk_rows

pytestmark = pytest.mark.gpu


def _check(h, W, target_vocab, mult, cap, k, ids, vals, rows):
    u = oracle.unary_rows(h, W, target_vocab, mult, cap, rows=rows)
    ora_ids, _ = oracle.topk(u, k)
    ties, _ = compare_topk_rows(h, W, u, ora_ids, mult, k, ids, vals, rows, target_vocab)
    return ties


def _launches(rows, vd, k, mult, dtype):
    return dflash2.library().dflash2_unary_topk_launches(
        rows, vd, k, mult, dflash2.BF16 if dtype == "bf16" else dflash2.F32)


def _gb300():
    return torch.cuda.get_device_properties(0).multi_processor_count == 152


def _run(dev, h, W, target_vocab, mult, cap, k, ws_bytes=None):
    th, tw = dflash2.to_device(h, dev), dflash2.to_device(W, dev)
    ws = None
    if ws_bytes is not None:
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ids, vals, err = dflash2.unary_topk(th, tw, target_vocab, mult, cap, k, workspace=ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), vals.cpu().numpy(), int(err.item())


# The last column is the number of kernels dflash2_unary_topk_launches reports on
# a 152-SM GB300: 2 = the fused cooperative launch (pilot, select and filter in
# one GEMM launch, then finalize), 3 / 4 = the split passes (pilot, select,
# filter when the pilot does not cover the vocab, finalize), None = fp32.  Every
# case compares all of its rows with the oracle, so both bf16 paths are pinned
# row by row.
SMALL = [
    # rows, hidden, draft_vocab, target_vocab, k, mult, cap, dtype, launches
    (37, 200, 5000, 4900, 16, 0.5, 30.0, "bf16", 2),      # ragged in every dimension
    (300, 264, 40000, 39990, 32, 1.0, 0.0, "bf16", 4),    # filter pass active, two token tiles
    (7, 512, 70000, 70000, 64, 1.0, 30.0, "bf16", 4),
    (513, 128, 9000, 8800, 8, 2.0, 0.0, "bf16", 2),       # three token tiles
    (5, 96, 3000, 2999, 128, 1.0, 0.0, "bf16", 4),        # K at its maximum; hidden below one stage
    (9, 136, 1100, 1000, 16, 1.0, 10.0, "f32", None),
    (2100, 128, 9000, 8990, 24, 1.0, 30.0, "bf16", 4),   # nine token tiles over the CTA pairs
    (1800, 136, 4000, 4000, 8, 0.7, 0.0, "bf16", 2),     # pilot of 8 of 16 units
    (300, 136, 1500, 1450, 16, 1.0, 30.0, "bf16", 3),    # under 8 units: the pilot covers the vocab
    (96, 256, 20000, 19990, 16, -0.5, 0.0, "bf16", 4),   # negative multiplier: order reversed
    (40, 128, 12000, 12000, 8, -1.0, 30.0, "bf16", 4),   # negative multiplier with the soft cap
    # fused launch: 2432 rows = two rows for each of the 1216 select warps
    # (76 CTA pairs x 16 epilogue warps), ten token tiles
    (2432, 128, 10240, 10240, 16, 1.0, 30.0, "bf16", 2),
    (1000, 200, 30000, 29990, 16, 0.7, 0.0, "bf16", 2),  # fused, ragged hidden and vocab
    (300, 136, 70000, 69990, 32, 1.0, 30.0, "bf16", 2),  # fused with K = 32 (18 pilot units)
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"m{c[0]}-h{c[1]}-v{c[2]}-k{c[4]}-{c[7]}")
def test_unary_topk_small(cuda, case):
    rows, hidden, vd, vt, k, mult, cap, dtype, launches = case
    if launches is not None and _gb300():
        assert _launches(rows, vd, k, mult, dtype) == launches
    w = synth.BY_NAME["tiny-fp32"].scaled(batch=rows, block_size=2, hidden=hidden, draft_vocab=vd,
                                target_vocab=vt, top_k=k, mult=mult, cap=cap, dtype=dtype, seed=91)
    inp = synth.make(w, parts=("h", "lm_head"))
    ids, vals, err = _run(cuda, inp["h"], inp["lm_head"], vt, mult, cap, k)
    assert err & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    ties = _check(inp["h"], inp["lm_head"], vt, mult, cap, k, ids, vals, list(range(rows)))
    print(f"near-ties accepted: {ties}")


def _sample_rows(w, n_min=64):
    """At least n_min rows: the first and last row of every bf16 token tile (rows
    in near-equal tiles of at most 256), then seeded random rows."""
    n_tiles = (w.rows + 255) // 256
    bn = ((w.rows + n_tiles - 1) // n_tiles + 15) // 16 * 16
    rows = set()
    for t in range(0, w.rows, bn):
        rows.update((t, min(t + bn, w.rows) - 1))
    rng = np.random.default_rng(5)
    while len(rows) < n_min:
        rows.add(int(rng.integers(0, w.rows)))
    return sorted(rows)


# all rows where the oracle finishes in seconds; otherwise every token tile's
# first and last row plus random rows, 64 at least
ALL_ROWS = {"tiny-fp32", "qwen3-8b-bf16", "reduced-vocab-bs12-bf16"}


@pytest.mark.parametrize("name", [c.name for c in synth.CONFIGS])
def test_unary_topk_named_workloads(cuda, name):
    w = synth.BY_NAME[name]
    inp = synth.make(w, parts=("h", "lm_head"))
    ids, vals, err = _run(cuda, inp["h"], inp["lm_head"], w.target_vocab, w.mult, w.cap, w.top_k)
    assert err == 0, hex(err)
    rows = list(range(w.rows)) if name in ALL_ROWS else _sample_rows(w)
    ties = _check(inp["h"], inp["lm_head"], w.target_vocab, w.mult, w.cap, w.top_k, ids, vals, rows)
    # properties that hold for every row
    assert np.all(ids >= 0) and np.all(ids < w.target_vocab)
    assert np.all(np.diff(vals, axis=1) <= 0)
    assert all(len(set(r)) == w.top_k for r in ids.tolist())
    print(f"{name}: {len(rows)} rows compared, near-ties accepted {ties}")


def test_overflowing_candidate_lists_fall_back_exactly(cuda):
    # the minimum workspace leaves room for K candidates per row: every row
    # that meets a filter-pass survivor overflows and is recomputed exactly
    rows, hidden, vd, vt, k = 24, 128, 20000, 19900, 16
    w = synth.BY_NAME["tiny-fp32"].scaled(batch=rows, block_size=2, hidden=hidden, draft_vocab=vd,
                                target_vocab=vt, top_k=k, dtype="bf16", seed=92)
    inp = synth.make(w, parts=("h", "lm_head"))
    ws = dflash2.unary_topk_workspace_min(rows, vd, k, dflash2.BF16)
    ids, vals, err = _run(cuda, inp["h"], inp["lm_head"], vt, 1.0, 0.0, k, ws_bytes=ws)
    assert err & dflash2.DEVINFO_TOPK_FALLBACK
    assert err & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    _check(inp["h"], inp["lm_head"], vt, 1.0, 0.0, k, ids, vals, list(range(rows)))


def test_logits_rising_with_id_defeat_the_pilot_but_stay_exact(cuda):
    # lm_head rows aligned with h and scaled up with the vocab id: the pilot
    # tiles see small logits, the threshold is weak and the lists overflow
    rows, hidden, vd, k = 6, 64, 30000, 32
    rng = np.random.default_rng(93)
    h = rng.standard_normal((rows, hidden)).astype(np.float32)
    direction = h.mean(0)
    W = (np.linspace(0.0, 1.0, vd)[:, None] * direction[None, :] +
         0.01 * rng.standard_normal((vd, hidden))).astype(np.float32)
    h16, W16 = synth.to_bf16_bits(h), synth.to_bf16_bits(W)
    ids, vals, err = _run(cuda, h16, W16, vd, 1.0, 0.0, k)
    assert err & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    _check(h16, W16, vd, 1.0, 0.0, k, ids, vals, list(range(rows)))


def test_high_padded_logits_are_never_chosen(cuda):
    rows, hidden, vd, vt, k = 16, 128, 6000, 5500, 32
    rng = np.random.default_rng(94)
    h = (np.abs(rng.standard_normal((rows, hidden))) + 0.1).astype(np.float32)
    W = (0.02 * rng.standard_normal((vd, hidden))).astype(np.float32)
    W[vt:] = 1.0                                   # padded rows carry the largest logits
    h16, W16 = synth.to_bf16_bits(h), synth.to_bf16_bits(W)
    ids, vals, err = _run(cuda, h16, W16, vt, 1.0, 0.0, k)
    assert err == 0
    assert ids.max() < vt and np.all(np.isfinite(vals))
    _check(h16, W16, vt, 1.0, 0.0, k, ids, vals, list(range(rows)))


def test_k_equal_to_target_vocab_returns_every_valid_id(cuda):
    rows, hidden, vd, vt = 4, 64, 130, 100
    w = synth.BY_NAME["tiny-fp32"].scaled(batch=rows, block_size=2, hidden=hidden, draft_vocab=vd,
                                target_vocab=vt, top_k=vt, dtype="bf16", seed=95)
    inp = synth.make(w, parts=("h", "lm_head"))
    ids, vals, err = _run(cuda, inp["h"], inp["lm_head"], vt, 1.0, 0.0, vt)
    assert err == 0
    for r in range(rows):
        assert sorted(ids[r].tolist()) == list(range(vt))
    _check(inp["h"], inp["lm_head"], vt, 1.0, 0.0, vt, ids, vals, list(range(rows)))


def test_zero_multiplier_ties_resolve_to_smallest_ids(cuda):
    rows, hidden, vd, k = 3, 64, 9000, 20
    w = synth.BY_NAME["tiny-fp32"].scaled(batch=rows, block_size=2, hidden=hidden, draft_vocab=vd,
                                target_vocab=vd, top_k=k, dtype="bf16", seed=96)
    inp = synth.make(w, parts=("h", "lm_head"))
    ids, vals, err = _run(cuda, inp["h"], inp["lm_head"], vd, 0.0, 0.0, k)
    assert err == 0
    for r in range(rows):
        np.testing.assert_array_equal(ids[r], np.arange(k))
        assert np.all(vals[r] == 0)


def test_zero_rows_is_a_no_op(cuda):
    h = torch.empty((0, 64), dtype=torch.bfloat16, device=cuda)
    W = torch.zeros((256, 64), dtype=torch.bfloat16, device=cuda)
    ids, vals, err = dflash2.unary_topk(h, W, 256, 1.0, 0.0, 8)
    assert ids.shape == (0, 8)


def test_launch_plan_of_the_named_workloads(cuda):
    """Which bf16 path each workload takes on a 152-SM GB300, so that both
    the fused launch and the split passes stay covered by the parity tests
    above: the Qwen3-8B-shaped workload is fused; the padded vocab (two more
    tile rounds) and the stress size (16 rows per epilogue warp) are split;
    the 7-row fp32 workload splits its vocab over CTAs."""
    lib = dflash2.library()
    plan = {c.name: lib.dflash2_unary_topk_launches(c.rows, c.draft_vocab, c.top_k, c.mult,
                                                    dflash2.BF16 if c.dtype == "bf16"
                                                    else dflash2.F32)
            for c in synth.CONFIGS}
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the plan depends on the SM count")
    assert plan["qwen3-8b-bf16"] == 2
    assert plan["padded-vocab-bf16"] == 4
    assert plan["stress-bf16"] == 4
    assert plan["tiny-fp32"] == 2   # vocab chunks, then the merge

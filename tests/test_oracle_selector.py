"""Pins for the oracle's projection, selector lattice and walk.

Pins: a hand-worked example (tests/golden/selector_tiny.txt), closed-form
softmax draws, numpy matmul/einsum special cases, exhaustive per-slot
enumeration for greedy rows, invariants (one-hot greedy q, q sums to 1, K = 1,
temperature clamp, mixed-batch independence) and a chi-square test of the
sampled draw against q.
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "selector_tiny.txt")


def _read_golden(path):
    vals = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, rhs = (s.strip() for s in line.split("=", 1))
        rows = [[float(t) for t in r.split()] for r in rhs.split(";")]
        vals[key] = np.array(rows if len(rows) > 1 else rows[0])
    return vals


def test_hand_worked_selector_example(ora):
    gd = _read_golden(GOLDEN)
    f = np.float32
    A, B = gd["A"].astype(f), gd["B"].astype(f)
    proj, h = gd["proj"].astype(f), gd["h"].astype(f)
    cand = gd["cand"].astype(np.int64)[None]
    cand_u = gd["cand_u"].astype(f)[None]
    anchors = np.atleast_1d(gd["anchor"]).astype(np.int64)
    g = ora.project(h, proj)
    np.testing.assert_array_equal(g, h)
    scores, errors = ora.lattice(g, A, B, anchors, cand, cand_u)
    assert errors == 0
    np.testing.assert_array_equal(scores[0, 0], gd["lattice_slot0"].astype(f))
    np.testing.assert_array_equal(scores[0, 1], gd["lattice_slot1"].astype(f))
    tokens, q, chosen = ora.walk(scores, cand, np.zeros((1, 2), f), np.ones(1, f), np.ones(1, np.uint8))
    np.testing.assert_array_equal(chosen[0], gd["greedy_index"].astype(np.int32))
    np.testing.assert_array_equal(tokens[0], gd["greedy_tokens"].astype(np.int64))
    np.testing.assert_array_equal(q[0], np.eye(2, dtype=f)[[1, 1]])


def _one_slot(scores_row, uniform, temperature):
    k = len(scores_row)
    scores = np.zeros((1, 1, k, k), np.float32)
    scores[0, 0, 0] = scores_row
    cand = np.arange(100, 100 + k, dtype=np.int64)[None, None]
    return scores, cand, np.array([[uniform]], np.float32), np.array([temperature], np.float32)


@pytest.mark.parametrize("temperature,uniform,index,q_ref", [
    # scores (ln1, ln2, ln5): softmax (1, 2, 5)/8, cdf (1/8, 3/8, 1)
    (1.0, 0.3, 1, (1 / 8, 2 / 8, 5 / 8)),
    (1.0, 0.1, 0, (1 / 8, 2 / 8, 5 / 8)),
    (1.0, 0.5, 2, (1 / 8, 2 / 8, 5 / 8)),
    (1.0, 0.999999, 2, (1 / 8, 2 / 8, 5 / 8)),
    # T = 1/2 squares the weights: (1, 4, 25)/30, cdf (1/30, 5/30, 1)
    (0.5, 0.1, 1, (1 / 30, 4 / 30, 25 / 30)),
    (0.5, 0.01, 0, (1 / 30, 4 / 30, 25 / 30)),
    (0.5, 0.2, 2, (1 / 30, 4 / 30, 25 / 30)),
])
def test_sampled_draw_closed_forms(ora, temperature, uniform, index, q_ref):
    row = np.array([0.0, math.log(2.0), math.log(5.0)], np.float32)
    scores, cand, uni, temps = _one_slot(row, uniform, temperature)
    tokens, q, chosen = ora.walk(scores, cand, uni, temps, np.zeros(1, np.uint8))
    assert chosen[0, 0] == index and tokens[0, 0] == 100 + index
    np.testing.assert_allclose(q[0, 0], q_ref, rtol=1e-6)


def test_inverse_cdf_boundary_and_cap(ora):
    # equal scores: p = 1/4 each, cdf (0.25, 0.5, 0.75, 1.0) exactly in fp32
    row = np.zeros(4, np.float32)
    for u, idx in [(0.0, 0), (0.25, 1), (0.2499999, 0), (0.75, 3), (0.99999994, 3)]:
        scores, cand, uni, temps = _one_slot(row, u, 1.0)
        _, _, chosen = ora.walk(scores, cand, uni, temps, np.zeros(1, np.uint8))
        assert chosen[0, 0] == idx, u
    # a uniform of 1.0 counts all K entries; the index is capped at K - 1
    scores, cand, uni, temps = _one_slot(row, 1.0, 1.0)
    _, _, chosen = ora.walk(scores, cand, uni, temps, np.zeros(1, np.uint8))
    assert chosen[0, 0] == 3


def test_greedy_tie_takes_lowest_index(ora):
    row = np.array([1.0, 3.0, 3.0, 2.0], np.float32)
    scores, cand, uni, temps = _one_slot(row, 0.9, 1.0)
    tokens, q, chosen = ora.walk(scores, cand, uni, temps, np.ones(1, np.uint8))
    assert chosen[0, 0] == 1
    np.testing.assert_array_equal(q[0, 0], [0, 1, 0, 0])


def _random_selector(seed, batch=4, slots=7, k=8, rank=16, hidden=32, vocab=200, scale=1.0):
    rng = np.random.default_rng(seed)
    f = np.float32
    A = (rng.standard_normal((vocab, rank)) * scale).astype(f)
    B = (rng.standard_normal((vocab, rank)) * scale).astype(f)
    proj = (rng.standard_normal((rank, hidden)) * 0.2).astype(f)
    h = rng.standard_normal((batch * slots, hidden)).astype(f)
    cand = np.stack([rng.choice(vocab, size=k, replace=False) for _ in range(batch * slots)]).reshape(batch, slots, k)
    cand_u = np.sort(rng.standard_normal((batch, slots, k)).astype(f), axis=-1)[..., ::-1].copy()
    anchors = rng.integers(0, vocab, size=batch).astype(np.int64)
    return A, B, proj, h, cand.astype(np.int64), cand_u, anchors


def test_projection_matches_numpy_matmul(ora):
    A, B, proj, h, cand, cand_u, anchors = _random_selector(20, hidden=48, rank=12)
    g = ora.project(h, proj)
    np.testing.assert_allclose(g, h.astype(np.float64) @ proj.astype(np.float64).T, rtol=1e-12, atol=1e-12)


def test_lattice_matches_einsum(ora):
    A, B, proj, h, cand, cand_u, anchors = _random_selector(21)
    batch, slots, k = cand.shape
    g = ora.project(h, proj)
    scores, errors = ora.lattice(g, A, B, anchors, cand, cand_u)
    assert errors == 0
    gg = g.reshape(batch, slots, -1)
    A64, B64 = A.astype(np.float64), B.astype(np.float64)
    for b in range(batch):
        for s in range(slots):
            prev_ids = np.full(k, anchors[b]) if s == 0 else cand[b, s - 1]
            ref = np.einsum("pj,j,cj->pc", A64[prev_ids], gg[b, s], B64[cand[b, s]]) + cand_u[b, s][None, :]
            np.testing.assert_allclose(scores[b, s], ref.astype(np.float32), rtol=1e-6, atol=1e-6)


def test_out_of_range_ids_are_counted_and_zeroed(ora):
    A, B, proj, h, cand, cand_u, anchors = _random_selector(22, batch=2, slots=3)
    cand = cand.copy()
    cand[1, 2, 3] = 10_000
    anchors = anchors.copy()
    anchors[0] = -1
    g = ora.project(h, proj)
    scores, errors = ora.lattice(g, A, B, anchors, cand, cand_u)
    assert errors >= 2
    np.testing.assert_array_equal(scores[0, 0], np.broadcast_to(cand_u[0, 0], (cand.shape[2],) * 2))
    np.testing.assert_array_equal(scores[1, 2, :, 3], np.full(cand.shape[2], cand_u[1, 2, 3]))


def test_greedy_walk_is_the_per_slot_argmax_by_enumeration(ora):
    A, B, proj, h, cand, cand_u, anchors = _random_selector(23, scale=2.0)
    batch, slots, k = cand.shape
    g = ora.project(h, proj).reshape(batch, slots, -1)
    res = ora.selector(h, proj, A, B, anchors, cand, cand_u, np.zeros((batch, slots), np.float32),
                       np.ones(batch, np.float32), np.ones(batch, np.uint8))
    for b in range(batch):
        prev_id = anchors[b]
        for s in range(slots):
            # enumerate every candidate edge from the chosen predecessor
            edges = [np.float32(sum(float(A[prev_id, j]) * g[b, s, j] * float(B[cand[b, s, c], j])
                                    for j in range(A.shape[1])) + float(cand_u[b, s, c]))
                     for c in range(k)]
            best = max(edges)
            assert res["chosen"][b, s] == min(c for c in range(k) if edges[c] == best)
            prev_id = cand[b, s, res["chosen"][b, s]]
        np.testing.assert_array_equal(res["q"][b], np.eye(k, dtype=np.float32)[res["chosen"][b]])


def test_sampled_q_is_a_distribution_and_k1_is_trivial(ora):
    A, B, proj, h, cand, cand_u, anchors = _random_selector(24)
    batch, slots, k = cand.shape
    uni = np.random.default_rng(1).random((batch, slots), dtype=np.float32)
    res = ora.selector(h, proj, A, B, anchors, cand, cand_u, uni, np.full(batch, 0.7, np.float32),
                       np.zeros(batch, np.uint8))
    assert np.all(np.abs(res["q"].sum(-1) - 1.0) <= 1e-6 * k)
    assert np.all(res["q"] >= 0)
    res1 = ora.selector(h, proj, A, B, anchors, cand[..., :1].copy(), cand_u[..., :1].copy(), uni,
                        np.full(batch, 0.7, np.float32), np.zeros(batch, np.uint8))
    np.testing.assert_array_equal(res1["tokens"], cand[..., 0])
    np.testing.assert_array_equal(res1["q"], np.ones((batch, slots, 1), np.float32))


def test_temperature_clamp_reduces_to_greedy(ora):
    A, B, proj, h, cand, cand_u, anchors = _random_selector(25, scale=2.0)
    batch, slots, _ = cand.shape
    uni = np.random.default_rng(2).random((batch, slots), dtype=np.float32)
    greedy = ora.selector(h, proj, A, B, anchors, cand, cand_u, uni, np.ones(batch, np.float32),
                          np.ones(batch, np.uint8))
    # T = 0 is clamped to 1e-5: the softmax is a point mass on the argmax
    cold = ora.selector(h, proj, A, B, anchors, cand, cand_u, uni * np.float32(0.999),
                        np.zeros(batch, np.float32), np.zeros(batch, np.uint8))
    np.testing.assert_array_equal(cold["tokens"], greedy["tokens"])


def test_greedy_rows_ignore_other_rows(ora):
    # mixed-batch determinism: a greedy row's output does not depend on the
    # temperatures or uniforms of any row
    A, B, proj, h, cand, cand_u, anchors = _random_selector(26)
    batch, slots, _ = cand.shape
    mask = np.array([1, 0, 1, 0], np.uint8)
    r = np.random.default_rng(3)
    outs = [ora.selector(h, proj, A, B, anchors, cand, cand_u, r.random((batch, slots), dtype=np.float32),
                         r.uniform(0.2, 2.0, batch).astype(np.float32), mask) for _ in range(3)]
    for o in outs[1:]:
        np.testing.assert_array_equal(o["tokens"][mask == 1], outs[0]["tokens"][mask == 1])
        np.testing.assert_array_equal(o["q"][mask == 1], outs[0]["q"][mask == 1])


def test_draw_frequencies_follow_q(ora):
    # 100k independent draws on one fixed slot: the empirical index counts
    # must agree with q (chi-square, 7 degrees of freedom).
    n, k = 100_000, 8
    row = np.random.default_rng(4).standard_normal(k).astype(np.float32)
    scores = np.zeros((n, 1, k, k), np.float32)
    scores[:, 0, 0] = row
    cand = np.tile(np.arange(k, dtype=np.int64), (n, 1, 1))
    uni = np.random.default_rng(5).random((n, 1), dtype=np.float32)
    _, q, chosen = ora.walk(scores, cand, uni, np.full(n, 0.8, np.float32), np.zeros(n, np.uint8))
    counts = np.bincount(chosen[:, 0], minlength=k)
    expect = q[0, 0].astype(np.float64) * n
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert chi2 < 29.9   # 7 dof: P(chi2 > 29.9) ~ 1e-4

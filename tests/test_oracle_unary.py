"""Pins for the oracle's unary logits, padded-vocab mask and top-K.

u = cap * tanh(mult * z / cap) (or mult * z when cap = 0) with
z = h . lm_head^T; padded rows [target_vocab, draft_vocab) are -inf; the top-K
is ordered by u descending, equal u by smaller id.  Checks use numpy's matmul
and lexsort as independent library routines, closed forms of tanh, and
constructed worst cases.
"""
import math

import numpy as np

from block_draft_proposal_gb300 import synth


def _f32(rng, *shape, std=1.0):
    return (rng.standard_normal(shape) * std).astype(np.float32)


def test_logits_match_numpy_matmul(ora):
    rng = np.random.default_rng(10)
    m, h, v = 5, 96, 300          # not square: a transposed operand cannot pass
    hs, w = _f32(rng, m, h), _f32(rng, v, h, std=0.1)
    u = ora.unary_rows(hs, w, target_vocab=v, mult=1.0, cap=0.0)
    ref = hs.astype(np.float64) @ w.astype(np.float64).T
    np.testing.assert_allclose(u, ref, rtol=1e-12, atol=1e-12)


def test_bf16_inputs_widen_exactly(ora):
    rng = np.random.default_rng(11)
    hs = synth.to_bf16_bits(_f32(rng, 3, 64))
    w = synth.to_bf16_bits(_f32(rng, 50, 64, std=0.1))
    u = ora.unary_rows(hs, w, target_vocab=50, mult=1.0, cap=0.0)
    ref = synth.bf16_bits_to_f32(hs).astype(np.float64) @ synth.bf16_bits_to_f32(w).astype(np.float64).T
    np.testing.assert_allclose(u, ref, rtol=1e-13, atol=1e-13)


def test_row_selection(ora):
    rng = np.random.default_rng(12)
    hs, w = _f32(rng, 7, 32), _f32(rng, 40, 32)
    full = ora.unary_rows(hs, w, 40, 1.0, 0.0)
    part = ora.unary_rows(hs, w, 40, 1.0, 0.0, rows=[6, 2])
    np.testing.assert_array_equal(part, full[[6, 2]])


def test_multiplier_without_cap_is_linear(ora):
    rng = np.random.default_rng(13)
    hs, w = _f32(rng, 4, 32), _f32(rng, 60, 32)
    z = ora.unary_rows(hs, w, 60, 1.0, 0.0)
    np.testing.assert_array_equal(ora.unary_rows(hs, w, 60, 0.5, 0.0), 0.5 * z)
    np.testing.assert_array_equal(ora.unary_rows(hs, w, 60, -3.0, 0.0), -3.0 * z)


def test_softcap_closed_forms(ora):
    # hidden = 1 and lm_head = [[1]] make z equal to h exactly.
    cap, mult = 30.0, 0.5
    a = np.float32(math.atanh(0.5) * cap / mult)          # tanh(mult*z/cap) = 1/2
    u = ora.unary_rows(np.array([[a]], np.float32), np.ones((1, 1), np.float32), 1, mult, cap)
    assert abs(u[0, 0] - cap / 2) < 1e-5
    neg = ora.unary_rows(np.array([[-a]], np.float32), np.ones((1, 1), np.float32), 1, mult, cap)
    assert neg[0, 0] == -u[0, 0]                           # odd function
    big = ora.unary_rows(np.array([[1e6]], np.float32), np.ones((1, 1), np.float32), 1, mult, cap)
    assert 0 <= cap - big[0, 0] < 1e-9                    # saturates at cap
    tiny = ora.unary_rows(np.array([[1e-3]], np.float32), np.ones((1, 1), np.float32), 1, mult, cap)
    assert abs(tiny[0, 0] - mult * np.float32(1e-3)) < 1e-12  # linear near zero
    rng = np.random.default_rng(14)
    u = ora.unary_rows(_f32(rng, 3, 16, std=50.0), _f32(rng, 20, 16), 20, 1.0, cap)
    assert np.all(np.abs(u) < cap)


def test_padded_rows_are_masked(ora):
    rng = np.random.default_rng(15)
    hs, w = _f32(rng, 3, 16), _f32(rng, 50, 16)
    u = ora.unary_rows(hs, w, target_vocab=41, mult=1.0, cap=0.0)
    assert np.all(u[:, 41:] == -np.inf) and np.all(np.isfinite(u[:, :41]))


def _lexsort_topk(u, k):
    uf = u.astype(np.float32)
    ids = np.empty((u.shape[0], k), np.int64)
    for r in range(u.shape[0]):
        order = np.lexsort((np.arange(u.shape[1]), -uf[r].astype(np.float64)))
        ids[r] = order[:k]
    return ids, np.take_along_axis(uf, ids, axis=1)


def test_topk_matches_lexsort(ora):
    rng = np.random.default_rng(16)
    u = rng.standard_normal((6, 1000))
    ids, vals = ora.topk(u, 17)
    ref_ids, ref_vals = _lexsort_topk(u, 17)
    np.testing.assert_array_equal(ids, ref_ids)
    np.testing.assert_array_equal(vals, ref_vals)
    assert np.all(np.diff(vals, axis=1) <= 0)


def test_topk_ties_go_to_smaller_id(ora):
    # integer-valued u with many exact ties; also ties created by fp32 rounding
    rng = np.random.default_rng(17)
    u = rng.integers(-3, 4, size=(4, 200)).astype(np.float64)
    u[1] = 1.0 + rng.integers(0, 2, size=200) * 2.0 ** -40   # equal once rounded to fp32
    ids, _ = ora.topk(u, 9)
    ref_ids, _ = _lexsort_topk(u, 9)
    np.testing.assert_array_equal(ids, ref_ids)
    np.testing.assert_array_equal(ids[1], np.arange(9))


def test_high_padded_logits_never_chosen(ora):
    # Padded lm_head rows built to carry the largest logits must still lose:
    # the regression the DSpark padded-vocab review asks for.
    rng = np.random.default_rng(18)
    vd, vt, h, k = 300, 257, 32, 20
    hs = np.abs(_f32(rng, 4, h)) + 0.1
    w = _f32(rng, vd, h, std=0.01)
    w[vt:] = 10.0
    u = ora.unary_rows(hs, w, target_vocab=vt, mult=1.0, cap=0.0)
    ids, vals = ora.topk(u, k)
    assert ids.max() < vt and np.all(np.isfinite(vals))
    # K equal to the logical vocab returns every valid id and no padded one
    ids_all, _ = ora.topk(u, vt)
    assert sorted(ids_all[0].tolist()) == list(range(vt))


def test_oracle_results_do_not_depend_on_the_thread_count():
    """The OpenMP loops split independent rows only: one thread and all give
    the same bits (the CPU baseline times both)."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(77)
    h = rng.normal(0, 1, (9, 64)).astype(np.float32)
    w = rng.normal(0, 0.1, (300, 64)).astype(np.float32)
    threads = oracle.set_threads(0)
    try:
        oracle.set_threads(1)
        one = oracle.unary_rows(h, w, 290, 1.0, 30.0)
        oracle.set_threads(max(2, threads))
        many = oracle.unary_rows(h, w, 290, 1.0, 30.0)
    finally:
        oracle.set_threads(threads)
    assert np.array_equal(one, many)

"""Pins of the oracle's speculative-sampling verification.

The rule (Leviathan et al. 2023; Chen et al. 2023) is lossless: whatever the
draft distribution q, each emitted token is distributed as the target's p.
These tests check that theorem statistically, the acceptance rate
sum_y min(p(y), qt(y)), a hand-worked example, and the greedy and
degenerate cases."""
import numpy as np
import pytest

import oracle


def _logits_of(p):
    return np.log(np.asarray(p, dtype=np.float64)).astype(np.float32)


def test_hand_worked_example():
    # V = 4, T = 1, p = (0.1, 0.2, 0.3, 0.4); candidates (3, 1) with q = (0.75, 0.25);
    # draft x = 3: accept iff r * 0.75 < 0.4, i.e. r < 0.5333.  On rejection the
    # residual is max(0, p - qt) = (0.1, 0, 0.3, 0), total 0.4: u = 0.3 -> target
    # 0.12, first cumulative above it at y = 2; u = 0.2 -> target 0.08 -> y = 0.
    lg = np.stack([_logits_of([0.1, 0.2, 0.3, 0.4])] * 2)[None]      # [1, 2, 4]
    args = dict(temperatures=np.ones(1, np.float32), greedy=np.zeros(1, np.uint8),
                draft=np.array([[3]]), cand=np.array([[[3, 1]]]),
                q=np.array([[[0.75, 0.25]]], np.float32))
    for r0, u, want_len, want in [(0.6, 0.3, 0, [2, -1]), (0.6, 0.2, 0, [0, -1]),
                                  (0.5, 0.95, 1, [3, 3])]:
        acc, out, err = oracle.verify(lg, r=np.array([[r0, u]], np.float32), **args)
        assert err == 0 and acc[0] == want_len and out[0].tolist() == want, (r0, u, out)
    # accepted at r = 0.5; the bonus token from position 1 with u = 0.95: cumulative
    # p = 0.1, 0.3, 0.6, 1.0 first exceeds 0.95 at y = 3


@pytest.mark.parametrize("temp", [1.0, 0.6])
def test_emitted_tokens_follow_p(temp):
    # S = 1, V = 7: draft x ~ q over K = 3 candidates; the first emitted token must
    # be distributed as p_0, and the acceptance rate must be sum min(p, qt)
    rng = np.random.default_rng(12)
    V, K, n = 7, 3, 200000
    lg0 = rng.standard_normal(V).astype(np.float32)
    lg1 = rng.standard_normal(V).astype(np.float32)
    p0 = np.exp(lg0.astype(np.float64) / np.float32(temp))
    p0 /= p0.sum()
    cand = np.array([5, 0, 2])
    qv = np.array([0.5, 0.3, 0.2], np.float32)
    pick = rng.choice(K, size=n, p=qv.astype(np.float64) / qv.sum())
    logits = np.broadcast_to(np.stack([lg0, lg1])[None], (n, 2, V)).copy()
    acc, out, err = oracle.verify(
        logits, np.full(n, temp, np.float32), np.zeros(n, np.uint8), cand[pick][:, None],
        np.broadcast_to(cand, (n, 1, K)).copy(), np.broadcast_to(qv, (n, 1, K)).copy(),
        rng.random((n, 2), dtype=np.float32))
    assert err == 0
    first = out[:, 0]
    freq = np.bincount(first, minlength=V)
    chi2 = ((freq - n * p0) ** 2 / (n * p0)).sum()
    assert chi2 < 22.5, (chi2, freq / n, p0)               # 6 dof, p ~ 0.001
    qt = np.zeros(V)
    qt[cand] = qv
    rate = np.minimum(p0, qt).sum()
    assert abs(acc.mean() - rate) < 5 * np.sqrt(rate * (1 - rate) / n)


def test_greedy_rows():
    lg = np.array([[[0.0, 3.0, 1.0, 3.0], [2.0, 0.0, 5.0, 1.0], [9.0, 0.0, 0.0, 0.0]]],
                  np.float32)                               # argmax 1 (tie: smallest), 2, 0
    base = dict(temperatures=np.full(1, 0.7, np.float32), greedy=np.ones(1, np.uint8),
                cand=np.array([[[1, 3], [2, 0]]]), q=np.array([[[1, 0], [1, 0]]], np.float32),
                r=np.full((1, 3), 0.999, np.float32))
    acc, out, _ = oracle.verify(lg, draft=np.array([[1, 2]]), **base)
    assert acc[0] == 2 and out[0].tolist() == [1, 2, 0]     # both accepted, bonus argmax
    acc, out, _ = oracle.verify(lg, draft=np.array([[3, 2]]), **base)
    assert acc[0] == 0 and out[0].tolist() == [1, -1, -1]   # rejected: the argmax


def test_q_equal_to_p_always_accepts():
    # p supported on the candidates and q = p there: min(1, p/q) = 1 for every draft
    p = np.array([0.0, 0.5, 0.0, 0.3, 0.2])
    lg = np.where(p > 0, np.log(np.maximum(p, 1e-300)), -1e30).astype(np.float32)
    n = 1000
    rng = np.random.default_rng(13)
    cand = np.array([1, 3, 4])
    qv = p[cand].astype(np.float32)
    pick = rng.choice(3, size=n, p=p[cand] / p[cand].sum())
    acc, out, err = oracle.verify(
        np.broadcast_to(np.stack([lg, lg])[None], (n, 2, 5)).copy(), np.ones(n, np.float32),
        np.zeros(n, np.uint8), cand[pick][:, None], np.broadcast_to(cand, (n, 1, 3)).copy(),
        np.broadcast_to(qv, (n, 1, 3)).copy(), rng.random((n, 2), dtype=np.float32))
    assert err == 0 and np.all(acc == 1)
    assert set(out[:, 1].tolist()) <= {1, 3, 4}


def test_draft_outside_candidates_is_an_error():
    lg = np.zeros((1, 2, 4), np.float32)
    acc, out, err = oracle.verify(lg, np.ones(1, np.float32), np.zeros(1, np.uint8),
                                  np.array([[2]]), np.array([[[0, 1]]]),
                                  np.array([[[0.5, 0.5]]], np.float32),
                                  np.full((1, 2), 0.5, np.float32))
    assert err == 1 and acc[0] == 0 and out[0].tolist() == [-1, -1]

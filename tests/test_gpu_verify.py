"""GPU parity of dflash2_verify against the oracle.

accept_len and out_tokens must equal the oracle's, except at a documented
near-tie: the acceptance test r*q < p(x) or the inverse-CDF boundary
u*Z' vs the cumulative residual within the fp32 error bound of the GPU's
softmax (relative 4e-5 here: ~150-term lane sums, a warp tree and 32 chunk
partials, each step a few roundings).  After an accepted near-tie the
request is not compared further."""
import numpy as np
import pytest
import torch

import oracle
from block_draft_proposal_gb300 import dflash2, synth

pytestmark = pytest.mark.gpu
REL = 4e-5


def make_case(B, S, K, V, dtype, seed, boost=6.0):
    rng = np.random.default_rng(seed)
    cand = np.zeros((B, S, K), dtype=np.int64)
    for i in range(B * S):
        cand.reshape(-1, K)[i] = rng.choice(V, size=K, replace=False)
    greedy = (np.arange(B) % 2 == 0).astype(np.uint8)
    qraw = rng.random((B, S, K)) + 0.05
    q = (qraw / qraw.sum(-1, keepdims=True)).astype(np.float32)
    q64 = q.astype(np.float64)
    pick = np.zeros((B, S), dtype=np.int64)
    for b in range(B):
        for s in range(S):
            pick[b, s] = rng.choice(K, p=q64[b, s] / q64[b, s].sum())
    q[greedy == 1] = 0.0
    for b in np.nonzero(greedy)[0]:
        q[b, np.arange(S), pick[b]] = 1.0                    # greedy rows: one-hot q
    draft = np.take_along_axis(cand, pick[..., None], -1)[..., 0]
    logits = rng.standard_normal((B, S + 1, V)).astype(np.float32)
    for b in range(B):
        for s in range(S):
            logits[b, s, cand[b, s]] += boost                # candidates carry much of p
        if greedy[b]:                                        # greedy: accept a prefix
            L = rng.integers(0, S + 1)
            for s in range(L):
                logits[b, s, draft[b, s]] += 40.0
    temps = np.where(greedy == 1, 1.0, 0.8).astype(np.float32)
    r = rng.random((B, S + 1), dtype=np.float32)
    if dtype == "bf16":
        logits = synth.to_bf16_bits(logits)
    return dict(logits=logits, temps=temps, greedy=greedy, draft=draft.astype(np.int64),
                cand=cand.astype(np.int64), q=q, r=r)


def _p(row, temp):
    z = row.astype(np.float64) / float(max(np.float32(temp), np.float32(1e-5)))
    e = np.exp(z - z.max())
    return e / e.sum()


def run_gpu(c, dev):
    f = lambda a: dflash2.to_device(a, dev)
    acc, out, err = dflash2.verify(f(c["logits"]), f(c["temps"]), f(c["greedy"]), f(c["draft"]),
                                   f(c["cand"]), f(c["q"]), f(c["r"]))
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy(), int(err.item())


def compare(c, acc_g, out_g):
    acc_o, out_o, errs = oracle.verify(c["logits"], c["temps"], c["greedy"], c["draft"], c["cand"],
                                       c["q"], c["r"])
    assert errs == 0
    logits = c["logits"]
    lf = synth.bf16_bits_to_f32(logits) if logits.dtype == np.uint16 else logits
    B, S1, V = lf.shape
    S = S1 - 1
    ties = 0
    for b in range(B):
        if acc_g[b] == acc_o[b] and np.array_equal(out_g[b], out_o[b]):
            continue
        assert not c["greedy"][b], f"greedy request {b} differs"
        # first divergence: an acceptance decision or the emitted token
        s = min(acc_g[b], acc_o[b])
        p = _p(lf[b, s], c["temps"][b])
        if acc_g[b] != acc_o[b]:
            k = int(np.nonzero(c["cand"][b, s] == c["draft"][b, s])[0][0])
            lhs = float(c["r"][b, s]) * float(c["q"][b, s, k])
            px = p[c["draft"][b, s]]
            assert abs(lhs - px) <= REL * px + 1e-12, (b, s, lhs, px)
        else:
            res = p.copy()
            if s < S:
                for k in range(c["cand"].shape[-1]):
                    y = c["cand"][b, s, k]
                    res[y] = max(0.0, res[y] - float(c["q"][b, s, k]))
            cum = np.cumsum(res)
            target = float(c["r"][b, S]) * cum[-1]
            lo = min(out_g[b, s], out_o[b, s])
            assert abs(cum[lo] - target) <= REL * cum[-1] + 1e-12, (b, s, cum[lo], target)
        ties += 1
    return ties


@pytest.mark.parametrize("B,S,K,V,dtype", [
    (64, 7, 8, 1000, "f32"), (48, 15, 16, 20000, "bf16"),
    (16, 5, 4, 1001, "f32"), (16, 5, 4, 999, "bf16"),         # vocab off the vector grid
    (8, 0, 4, 500, "f32"), (12, 3, 128, 4096, "bf16"),        # no slots; K at its maximum
])
def test_verify_matches_oracle(cuda, B, S, K, V, dtype):
    c = make_case(B, S, K, V, dtype, seed=B * 31 + V)
    acc, out, err = run_gpu(c, cuda)
    assert err == 0
    ties = compare(c, acc, out)
    print(f"near-ties accepted: {ties}; mean accept {acc.mean():.2f}")


def test_verify_full_size_bench_workload(cuda):
    w = synth.BY_NAME["qwen3-8b-bf16"]
    c = make_case(w.batch, w.slots, w.top_k, w.target_vocab, "bf16", seed=77)
    acc, out, err = run_gpu(c, cuda)
    assert err == 0
    ties = compare(c, acc, out)
    print(f"full size: near-ties {ties}; mean accept {acc.mean():.2f}")


def test_all_accepted_draws_the_bonus(cuda):
    c = make_case(32, 4, 8, 3000, "f32", seed=5, boost=0.0)
    c["greedy"][:] = 0
    for b in range(32):                    # p concentrated on the draft: always accepted
        for s in range(4):
            c["logits"][b, s, c["draft"][b, s]] += 60.0
    acc, out, err = run_gpu(c, cuda)
    assert err == 0 and np.all(acc == 4)
    assert compare(c, acc, out) == 0


def test_emitted_tokens_follow_p(cuda):
    # the lossless theorem on the GPU: the first emitted token is distributed as p_0
    rng = np.random.default_rng(21)
    V, K, n = 7, 3, 40000
    lg0 = rng.standard_normal(V).astype(np.float32)
    p0 = _p(lg0, 1.0)
    cand = np.array([5, 0, 2])
    qv = np.array([0.5, 0.3, 0.2], np.float32)
    pick = rng.choice(K, size=n, p=qv.astype(np.float64) / qv.sum())
    c = dict(logits=np.broadcast_to(np.stack([lg0, lg0])[None], (n, 2, V)).copy(),
             temps=np.ones(n, np.float32), greedy=np.zeros(n, np.uint8),
             draft=cand[pick][:, None].astype(np.int64),
             cand=np.broadcast_to(cand, (n, 1, K)).astype(np.int64).copy(),
             q=np.broadcast_to(qv, (n, 1, K)).copy(), r=rng.random((n, 2), dtype=np.float32))
    acc, out, err = run_gpu(c, cuda)
    assert err == 0
    freq = np.bincount(out[:, 0], minlength=V)
    chi2 = ((freq - n * p0) ** 2 / (n * p0)).sum()
    assert chi2 < 22.5, (chi2, freq / n, p0)


def test_draft_outside_candidates(cuda):
    c = make_case(4, 3, 4, 200, "f32", seed=3)
    c["draft"][1, 1] = 199 if 199 not in c["cand"][1, 1] else 198
    acc, out, err = run_gpu(c, cuda)
    assert err & dflash2.DEVERR_ID_RANGE
    assert acc[1] == 0 and np.all(out[1] == -1)

"""Parity bookkeeping shared by the GPU tests and the smoke run: tolerances,
the near-tie rule and the element-by-element comparators.

Tolerances (floating point):
  conv: fp32  |gpu - oracle| <= 1e-5 * sum_t |c_t| |x_{i-t}| + 1e-30 (componentwise
        relative), bf16  <= 2e-2 absolute;
  q:    fp32  <= 1e-5 (relative to the row max of 1), bf16 configs <= 2e-2 absolute;
  u:    the forward-error bound below.
Ids (top-K membership and order, walk tokens) must be equal; a mismatch is
accepted only as a documented near-tie, i.e. when the exact (double) values of
the two competing items are closer than the fp32 forward-error bound of the
arithmetic that produced them:

  |u_gpu(v) - u(v)| <= |mult| * (H + 2) * 2^-24 * sum_j |h_j W_vj| + 8 * 2^-24 * |u(v)|

(recursive fp32 summation of H exact bf16 products, Higham's gamma_n; plus the
rounding of the transform).  For a sampled draw the boundary test
`uniform >= cdf[k]` is accepted as a near-tie when |uniform - cdf[k]| is within
K * 2^-23 plus the propagated edge error.  After an accepted near-tie the
request's later tokens and q are not compared with the oracle's (its path may
legitimately differ from there on).  Accepted near-ties are counted and
reported.
"""
from __future__ import annotations

import numpy as np

EPS32 = 2.0 ** -24


def f64(a: np.ndarray) -> np.ndarray:
    """float32 or bf16 bit patterns (uint16) -> float64."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def u_error_bound(h_row64: np.ndarray, W64: np.ndarray, ids, u_exact: np.ndarray, mult: float):
    """Per-id bound on |u_gpu - u| for the given vocab ids of one row."""
    ids = np.asarray(ids)
    s = np.abs(W64[ids]) @ np.abs(h_row64)
    hidden = h_row64.shape[0]
    return abs(mult) * (hidden + 2) * EPS32 * s + 8 * EPS32 * np.abs(u_exact[ids]) + 1e-30


def check_topk_row(gpu_ids, gpu_u, ora_ids, u_exact, bound_fn, k):
    """Compare one row's GPU top-K with the oracle's.  Returns the number of
    accepted near-ties; raises AssertionError on any other difference."""
    gpu_ids = np.asarray(gpu_ids)
    ora_ids = np.asarray(ora_ids)
    assert len(set(gpu_ids.tolist())) == k, "duplicate ids in a GPU top-K row"
    b_gpu = bound_fn(gpu_ids)
    err = np.abs(gpu_u.astype(np.float64) - u_exact[gpu_ids])
    assert np.all(err <= b_gpu), f"cand_u off by {err.max()} > bound {b_gpu[np.argmax(err - b_gpu)]}"
    ties = 0
    for i in range(k):
        a, b = int(gpu_ids[i]), int(ora_ids[i])
        if a == b:
            continue
        gap = abs(u_exact[a] - u_exact[b])
        tol = bound_fn([a])[0] + bound_fn([b])[0]
        assert gap <= tol, f"position {i}: gpu id {a} vs oracle id {b}, gap {gap} > {tol}"
        ties += 1
    return ties


def compare_topk_rows(h, W, u, ora_ids, mult, k, ids, vals, rows, target_vocab):
    """Every listed row of the GPU top-K (ids [*, K], vals [*, K], indexed by
    the row numbers in `rows`) against the oracle's u (one row of u and
    ora_ids per entry of `rows`).  Returns (accepted near-ties, the rows whose
    id lists differ from the oracle's anywhere)."""
    ties, differing = 0, []
    for r, m in enumerate(rows):
        h64 = f64(h[m])

        def bound(sel, h64=h64, r=r):
            sel = np.asarray(sel)
            return u_error_bound(h64, f64(W[sel]), np.arange(len(sel)), u[r][sel], mult)

        t = check_topk_row(ids[m], vals[m], ora_ids[r], u[r], bound, k)
        ties += t
        if t:
            differing.append(m)
        assert np.all(ids[m] < target_vocab)
        assert np.all(np.diff(vals[m]) <= 0)
    return ties, differing


def walk_edge_bound(inp, cand, anchors, hidden):
    """Per-edge forward-error bound [B, S, K(prev), K(cur)] of the fp32 edges
    (the projection's hidden-length sums and the rank-length edge sums)."""
    batch, slots, k = cand.shape
    A, B = f64(inp["A"]), f64(inp["B"])
    r = A.shape[1]
    habs = np.abs(f64(inp["h"]))
    gabs = habs @ np.abs(f64(inp["proj"])).T                   # sum_i |h_i P_ji|
    g = f64(inp["h"]) @ f64(inp["proj"]).T
    gerr = (hidden + 2) * EPS32 * gabs                         # |g_gpu - g|
    out = np.empty((batch, slots, k, k))
    for b in range(batch):
        for s in range(slots):
            prev = np.full(k, anchors[b]) if s == 0 else cand[b, s - 1]
            prev = np.clip(prev, 0, A.shape[0] - 1)
            pa = np.abs(A[prev])                               # [k, r]
            cb = np.abs(B[np.clip(cand[b, s], 0, B.shape[0] - 1)])
            row = b * slots + s
            lat = (pa * np.abs(g[row])[None, :]) @ cb.T        # sum |A g B|
            lat_g = (pa * gerr[row][None, :]) @ cb.T
            out[b, s] = (r + 4) * EPS32 * lat + lat_g
    return out


def compare_walk(inp, ora, cand, cand_u, tokens, q, ps, dtype, hidden, stop=None,
                 u_err=None):
    """Compare a GPU walk (tokens [B, S], q [B, S, K], and the edges it read,
    ps [B, S, K], or None) with the oracle's walk `ora` over the candidates
    `cand` / `cand_u` [B, S, K].

    Tokens must be equal up to an accepted near-tie; q must match within the
    tolerance; greedy q is exactly one-hot and sampled q sums to one.  After an
    accepted near-tie the request's later slots are checked for their edges
    (against the oracle lattice row of the GPU's own predecessor) and the form
    of q only.  Request b is compared on slots s < stop[b] (all slots by
    default).  u_err [B, S, K]
    is added to the edge tolerance when the GPU's unary values are its own (the
    end-to-end chain), not the ones the oracle walked.  Returns the number of
    accepted near-ties."""
    batch, slots, k = cand.shape
    bound = walk_edge_bound(inp, cand, inp["anchors"], hidden) + np.abs(cand_u)[:, :, None, :] * EPS32
    if u_err is not None:
        bound = bound + u_err[:, :, None, :]
    scores = ora["scores"]
    q_tol = 1e-5 if dtype == "f32" else 2e-2
    ties = 0
    for b in range(batch):
        greedy = bool(inp["greedy"][b])
        prev = 0
        diverged = False
        end = slots if stop is None else int(stop[b])
        for s in range(end):
            row = cand[b, s]
            hit = np.nonzero(row == tokens[b, s])[0]
            assert hit.size == 1, (b, s, "token is not one of the slot's candidates")
            gi = int(hit[0])                                   # GPU index (ids are distinct)
            # edges the GPU read: the oracle lattice row of the GPU's predecessor
            e_ref = scores[b, s, prev].astype(np.float64)
            tol = bound[b, s, prev] + np.abs(e_ref) * EPS32
            if ps is not None:
                assert np.all(np.abs(ps[b, s].astype(np.float64) - e_ref) <= tol), (b, s)
            if greedy:
                np.testing.assert_array_equal(q[b, s], np.eye(k, dtype=np.float32)[gi])
            else:
                assert abs(q[b, s].astype(np.float64).sum() - 1.0) <= 1e-6 * k
            oi = int(ora["chosen"][b, s])
            if diverged:
                pass          # after an accepted near-tie only the edges and q's form are checked
            elif gi != oi:
                if greedy:
                    gap = abs(float(e_ref[gi]) - float(e_ref[oi]))
                    assert gap <= tol[gi] + tol[oi], (b, s, gi, oi, gap)
                else:
                    t = max(float(inp["temperatures"][b]), 1e-5)
                    p = ora["q"][b, s].astype(np.float64)
                    cdf = np.cumsum(p)
                    lo, hi = min(gi, oi), max(gi, oi)
                    slack = k * 2.0 ** -23 + 4 * float(tol.max()) / t
                    assert np.all(np.abs(inp["uniforms"][b, s] - cdf[lo:hi]) <= slack), (b, s)
                ties += 1
                diverged = True
            else:
                assert abs(q[b, s] - ora["q"][b, s]).max() <= q_tol, (b, s)
            prev = gi
    return ties


def check_step_against_oracle(w, inp, out):
    """The whole step against the chained oracle, element by element: every
    top-K row (ids exact up to accepted near-ties, u within its bound), the
    walk of every request (tokens exact up to accepted near-ties, q within
    tolerance) on the slots before its first top-K row that differs from the
    oracle's, and the remap of the GPU's tokens bit for bit.  Returns the
    accepted near-ties (top-K, walk).  `out` holds the step's output tensors
    (dflash2.proposal_step), `inp` the host inputs it was given."""
    import oracle
    u = oracle.unary_rows(inp["h"], inp["lm_head"], w.target_vocab, w.mult, w.cap)
    ora_ids, ora_u = oracle.topk(u, w.top_k)
    ids = out["cand_ids"].cpu().numpy()
    vals = out["cand_u"].cpu().numpy()
    rows = list(range(w.rows))
    topk_ties, differing = compare_topk_rows(inp["h"], inp["lm_head"], u, ora_ids, w.mult,
                                             w.top_k, ids, vals, rows, w.target_vocab)
    # a request is walked on the oracle's candidates up to its first top-K row
    # that differs (an accepted near-tie may change the path from there on)
    stop = np.full(w.batch, w.slots)
    for m in differing:
        b, s = divmod(m, w.slots)
        stop[b] = min(stop[b], s)
    cand = ora_ids.reshape(w.batch, w.slots, w.top_k)
    cand_u = ora_u.reshape(w.batch, w.slots, w.top_k)
    ora = oracle.selector(inp["h"], inp["proj"], inp["A"], inp["B"], inp["anchors"], cand, cand_u,
                          inp["uniforms"], inp["temperatures"], inp["greedy"])
    assert ora["errors"] == 0
    # the GPU walked its own unary values: their bound joins the edge tolerance
    u_err = np.zeros((w.rows, w.top_k))
    for m in rows:
        h64 = f64(inp["h"][m])
        u_err[m] = u_error_bound(h64, f64(inp["lm_head"][ora_ids[m]]), np.arange(w.top_k),
                                 u[m][ora_ids[m]], w.mult)
    walk_ties = compare_walk(inp, ora, cand, cand_u, out["tokens"].cpu().numpy(),
                             out["q"].cpu().numpy(), None, w.dtype, w.hidden, stop=stop,
                             u_err=u_err.reshape(w.batch, w.slots, w.top_k))
    # the remap of the GPU's own tokens is exact
    ref_tgt, errors = oracle.d2t(out["tokens"].cpu().numpy().reshape(-1), inp["d2t"],
                                 w.draft_vocab, w.target_vocab)
    assert errors == 0
    np.testing.assert_array_equal(out["target_ids"].cpu().numpy().reshape(-1), ref_tgt)
    return topk_ties, walk_ties


def conv_tolerance(dtype: str, abs_conv: np.ndarray | None):
    if dtype == "bf16":
        return 2e-2
    return 1e-5 * abs_conv + 1e-30

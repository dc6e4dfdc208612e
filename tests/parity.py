"""Parity bookkeeping shared by the GPU tests: tolerances and the near-tie rule.

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
K * 2^-23 plus the propagated edge error.  Accepted near-ties are counted and
reported.
"""
from __future__ import annotations

import numpy as np

EPS32 = 2.0 ** -24


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


def conv_tolerance(dtype: str, abs_conv: np.ndarray | None):
    if dtype == "bf16":
        return 2e-2
    return 1e-5 * abs_conv + 1e-30

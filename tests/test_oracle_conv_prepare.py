"""Pins of the oracle's kernel projection and DFlashGroupedConv prepare/finish.

sglang DFlash2 PR, DFlashGroupedConv: one bias-free Linear(hidden, 2*taps*groups)
gives each token's coefficients of both sides, laid out [2, taps, groups];
prepare() convolves the input with side 0 (and base_kernel[0]), finish()
convolves the sublayer output with side 1 (and base_kernel[1]).
"""
import numpy as np
import pytest

import oracle
from block_draft_proposal_gb300 import synth


def _bf16(a):
    return synth.to_bf16_bits(np.asarray(a, dtype=np.float32))


def _f(a):
    return synth.bf16_bits_to_f32(a) if a.dtype == np.uint16 else a


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_hot_rows_pick_channels(dtype):
    rng = np.random.default_rng(3)
    n, hidden, r = 9, 48, 40
    x = rng.standard_normal((n, hidden)).astype(np.float32)
    pick = rng.integers(0, hidden, size=r)
    w = np.zeros((r, hidden), dtype=np.float32)
    w[np.arange(r), pick] = 1.0
    if dtype == "bf16":
        x, w = _bf16(x), _bf16(w)
    coef = oracle.kernel_projection(x, w)
    np.testing.assert_array_equal(coef, x[:, pick])      # coef[i, r] = x[i, pick[r]]


def test_exact_on_integer_inputs():
    # small integers: every product and partial sum is exact, so the result is
    # the plain matrix product, rounded once to bf16
    rng = np.random.default_rng(4)
    n, hidden, r = 17, 300, 64
    x = rng.integers(-3, 4, size=(n, hidden)).astype(np.float32)
    w = rng.integers(-3, 4, size=(r, hidden)).astype(np.float32)
    exact = x.astype(np.int64) @ w.astype(np.int64).T
    np.testing.assert_array_equal(oracle.kernel_projection(x, w), exact.astype(np.float32))
    np.testing.assert_array_equal(oracle.kernel_projection(_bf16(x), _bf16(w)),
                                  _bf16(exact.astype(np.float32)))


def test_matches_numpy_float64_product():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((13, 200)).astype(np.float32)
    w = (rng.standard_normal((56, 200)) * 0.02).astype(np.float32)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    got = oracle.kernel_projection(x, w).astype(np.float64)
    # both round a double sum once to fp32; the sums differ only in order
    assert np.max(np.abs(got - ref) / (np.abs(ref) + 1e-30)) < 2 ** -23


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prepare_is_identity_at_module_init(dtype):
    # base_kernel[:, 0] = 1 and a zero projection: both convolutions pass x through
    w = synth.BY_NAME["tiny-fp32"].scaled(dtype=dtype)
    d = synth.make(w, parts=("x",))
    x = d["x"]
    base2 = np.zeros((2, w.taps, w.hidden), dtype=np.float32)
    base2[:, 0] = 1.0
    wkp = np.zeros((2 * w.taps * w.groups, w.hidden), dtype=np.float32)
    if dtype == "bf16":
        base2, wkp = _bf16(base2), _bf16(wkp)
    out, coef = oracle.conv_prepare(x, wkp, base2, w.block_size, w.group_size, w.taps)
    np.testing.assert_array_equal(out, x)
    assert not np.any(_f(coef))
    np.testing.assert_array_equal(oracle.conv_finish(x, coef, base2, w.block_size, w.group_size,
                                                     w.taps), x)


def test_sides_taps_and_groups_by_brute_force():
    # random fp32 case against explicit loops over (token, channel, tap); side 0
    # and side 1 use different bases so a swapped side or tap order fails
    rng = np.random.default_rng(6)
    n, hidden, gs, taps, bs = 11, 16, 4, 3, 5
    groups = hidden // gs
    x = rng.standard_normal((n, hidden)).astype(np.float32)
    y = rng.standard_normal((n, hidden)).astype(np.float32)
    wkp = rng.standard_normal((2 * taps * groups, hidden)).astype(np.float32) * 0.1
    base2 = rng.standard_normal((2, taps, hidden)).astype(np.float32)
    out, coef = oracle.conv_prepare(x, wkp, base2, bs, gs, taps)
    fin = oracle.conv_finish(y, coef, base2, bs, gs, taps)
    c = x.astype(np.float64) @ wkp.astype(np.float64).T          # [n, 2*taps*groups]
    c = c.astype(np.float32).astype(np.float64).reshape(n, 2, taps, groups)
    for side, src, got in ((0, x, out), (1, y, fin)):
        want = np.zeros((n, hidden))
        for i in range(n):
            for ch in range(hidden):
                for t in range(taps):
                    if i % bs >= t:
                        want[i, ch] += (float(base2[side, t, ch]) + c[i, side, t, ch // gs]) \
                            * float(src[i - t, ch])
        np.testing.assert_allclose(got, want.astype(np.float32), rtol=2e-6, atol=1e-6)

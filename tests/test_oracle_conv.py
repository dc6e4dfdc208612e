"""Pins for the oracle's grouped dynamic conv and its bf16 rounding.

The conv is the block-causal grouped dynamic depthwise convolution of the
sglang DFlash2 PR (_grouped_conv): out[i,c] = sum over taps t with
pos(i) >= t of (base[t,c] + delta[i,t,c//gs]) * x[i-t,c], pos(i) = i mod bs.
Nothing here re-types that loop: each test checks the oracle against a
library routine on a special case (np.convolve, shift matrices), a closed
form, or an invariant.
"""
import numpy as np
import pytest

from block_draft_proposal_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _f32(rng, *shape, std=1.0):
    return (rng.standard_normal(shape) * std).astype(np.float32)


def _ref_depthwise(x, kernel, bs):
    """Causal depthwise conv restarted at every block start, via np.convolve.

    kernel[t, c] multiplies x[i - t, c].  np.convolve(a, k)[i] = sum_t k[t] a[i-t],
    so truncating to the block length gives exactly the taps that stay inside
    the block."""
    n, h = x.shape
    out = np.zeros((n, h), dtype=np.float64)
    for start in range(0, n, bs):
        blk = x[start:start + bs].astype(np.float64)
        for c in range(h):
            out[start:start + len(blk), c] = np.convolve(blk[:, c], kernel[:, c].astype(np.float64))[:len(blk)]
    return out


@pytest.mark.parametrize("n,bs,taps", [(32, 8, 4), (30, 8, 4), (36, 12, 6), (10, 1, 3), (21, 4, 7)])
def test_token_independent_coefficients_match_numpy_convolve(ora, n, bs, taps):
    # delta[i, t, g] = d[t, g] for every token: the conv is a plain depthwise
    # causal convolution with kernel base[t, c] + d[t, c // gs] inside each block.
    rng = np.random.default_rng(1)
    h, gs = 48, 8
    x = _f32(rng, n, h)
    base = _f32(rng, taps, h, std=0.5)
    d = _f32(rng, taps, h // gs, std=0.5)
    delta = np.broadcast_to(d, (n, taps, h // gs)).copy()
    kernel = base.astype(np.float64) + np.repeat(d.astype(np.float64), gs, axis=1)
    ref = _ref_depthwise(x, kernel, bs)
    out = ora.conv(x, base, delta, block_size=bs, group_size=gs, taps=taps)
    np.testing.assert_allclose(out, ref, rtol=2e-7, atol=1e-30)


def test_group_index_is_channel_div_group_size(ora):
    # One group carries a large coefficient; only its gs contiguous channels
    # may see it (a c % groups mix-up would spread it across the row).
    n, h, gs, taps, bs = 8, 32, 8, 1, 8
    x = np.ones((n, h), dtype=np.float32)
    base = np.zeros((taps, h), dtype=np.float32)
    delta = np.zeros((n, taps, h // gs), dtype=np.float32)
    delta[:, 0, 2] = 5.0
    out = ora.conv(x, base, delta, block_size=bs, group_size=gs, taps=taps)
    expect = np.zeros((n, h), dtype=np.float32)
    expect[:, 16:24] = 5.0
    np.testing.assert_array_equal(out, expect)


def test_token_dependent_delta_matches_shift_matrices(ora):
    # Brute force on a tiny case by linear algebra: tap t is the lower shift
    # matrix S_t (x[i-t] -> row i) masked by [pos(i) >= t], times per-token
    # per-channel coefficients.
    rng = np.random.default_rng(2)
    n, h, gs, taps, bs = 14, 16, 4, 3, 5
    x = _f32(rng, n, h)
    base = _f32(rng, taps, h)
    delta = _f32(rng, n, taps, h // gs)
    pos = np.arange(n) % bs
    ref = np.zeros((n, h))
    for t in range(taps):
        shift = np.eye(n, k=-t) * (pos >= t)[:, None]
        coef = base[t][None, :].astype(np.float64) + np.repeat(delta[:, t, :].astype(np.float64), gs, axis=1)
        ref += coef * (shift @ x.astype(np.float64))
    out = ora.conv(x, base, delta, block_size=bs, group_size=gs, taps=taps)
    np.testing.assert_allclose(out, ref, rtol=2e-7, atol=1e-30)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_identity_initialisation_is_exact(ora, dtype):
    # The module initialises base with tap 0 = 1 and the rest 0; with zero
    # delta the conv is the identity, bit for bit.
    rng = np.random.default_rng(3)
    n, h, gs, taps, bs = 24, 64, 8, 4, 8
    x = _f32(rng, n, h)
    base = np.zeros((taps, h), dtype=np.float32)
    base[0] = 1.0
    delta = np.zeros((n, taps, h // gs), dtype=np.float32)
    if dtype == "bf16":
        x, base, delta = (synth.to_bf16_bits(a) for a in (x, base, delta))
    out = ora.conv(x, base, delta, block_size=bs, group_size=gs, taps=taps)
    np.testing.assert_array_equal(out, x)


def test_block_size_one_keeps_only_tap_zero(ora):
    rng = np.random.default_rng(4)
    n, h, gs, taps = 9, 16, 8, 4
    x, base = _f32(rng, n, h), _f32(rng, taps, h)
    delta = _f32(rng, n, taps, h // gs)
    out = ora.conv(x, base, delta, block_size=1, group_size=gs, taps=taps)
    coef0 = base[0][None, :].astype(np.float64) + np.repeat(delta[:, 0, :].astype(np.float64), gs, axis=1)
    np.testing.assert_allclose(out, (coef0 * x).astype(np.float32), rtol=0, atol=0)


def test_block_locality_and_linearity(ora):
    rng = np.random.default_rng(5)
    n, h, gs, taps, bs = 40, 32, 8, 4, 10
    x, y = _f32(rng, n, h), _f32(rng, n, h)
    base = _f32(rng, taps, h)
    delta = _f32(rng, n, taps, h // gs)
    out = ora.conv(x, base, delta, block_size=bs, group_size=gs, taps=taps)
    x2 = x.copy()
    x2[10:20] += 3.0                       # perturb block 1 only
    out2 = ora.conv(x2, base, delta, block_size=bs, group_size=gs, taps=taps)
    np.testing.assert_array_equal(out2[:10], out[:10])
    np.testing.assert_array_equal(out2[20:], out[20:])
    assert np.any(out2[10:20] != out[10:20])
    a, b = np.float32(0.75), np.float32(-2.0)
    lhs = ora.conv((a * x + b * y).astype(np.float32), base, delta, block_size=bs, group_size=gs, taps=taps)
    rhs = a * out.astype(np.float64) + b * ora.conv(y, base, delta, block_size=bs, group_size=gs, taps=taps).astype(np.float64)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-5, atol=1e-5)


def test_taps_beyond_block_are_masked(ora):
    rng = np.random.default_rng(6)
    n, h, gs, bs = 16, 16, 8, 4
    x = _f32(rng, n, h)
    base6, delta6 = _f32(rng, 6, h), _f32(rng, n, 6, h // gs)
    out6 = ora.conv(x, base6, delta6, block_size=bs, group_size=gs, taps=6)
    out4 = ora.conv(x, base6[:4].copy(), delta6[:, :4].copy(), block_size=bs, group_size=gs, taps=4)
    np.testing.assert_array_equal(out6, out4)


def test_delta_row_stride_reads_side_zero_of_a_two_sided_projection(ora):
    # The kernel projection yields [n, 2, taps, groups]; side 0 is read in
    # place with a row stride of 2 * taps * groups.
    rng = np.random.default_rng(7)
    n, h, gs, taps, bs = 12, 32, 8, 3, 6
    x, base = _f32(rng, n, h), _f32(rng, taps, h)
    both = _f32(rng, n, 2, taps, h // gs)
    strided = ora.conv(x, base, both, block_size=bs, group_size=gs, taps=taps,
                       delta_row_stride=2 * taps * (h // gs))
    packed = ora.conv(x, base, both[:, 0].copy(), block_size=bs, group_size=gs, taps=taps)
    np.testing.assert_array_equal(strided, packed)


def test_bf16_output_rounding_matches_torch_cast(ora):
    # taps=1 with delta=0: out = round_bf16(base * x).  A bf16 x bf16 product is
    # exact in fp32, so torch's fp32 -> bf16 cast (nearest-even) is the single
    # rounding the oracle must reproduce.
    import torch
    rng = np.random.default_rng(8)
    n, h = 64, 64
    x = synth.to_bf16_bits(_f32(rng, n, h, std=3.0))
    base = synth.to_bf16_bits(_f32(rng, 1, h, std=3.0))
    delta = synth.to_bf16_bits(np.zeros((n, 1, h // 8), dtype=np.float32))
    out = ora.conv(x, base, delta, block_size=4, group_size=8, taps=1)
    prod = synth.bf16_bits_to_f32(base)[0][None, :] * synth.bf16_bits_to_f32(x)
    ref = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(out, ref)


def test_round_bf16_special_values(ora):
    import torch
    vals = [0.0, -0.0, 1.0, 1.00390625, 1.01171875, -1.00390625, 3.0e38, 3.4e38, -3.4e38,
            1e-40, -1e-40, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 65504.0, 0.1, -7.77]
    for v in vals:
        want = int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0])
        assert ora.round_bf16(v) == want, v
    # a double just above a bf16 halfway point must round up, which a
    # double -> float -> bf16 path would miss (float would round it to the tie)
    v = 1.00390625 + 2.0 ** -40
    assert ora.round_bf16(v) == 0x3F81

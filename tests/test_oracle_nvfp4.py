"""Pins of the oracle's NVFP4 (E2M1 codes, E4M3 block scales, fp32
second-level scales) lm_head path: the element table of the format (a golden
fixture, cited in the file), a brute-force nearest-value encoder written here,
invariants every block quantization must satisfy whatever its rounding, and a
plain numpy matmul of the values decoded by the table."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_values.txt")


def _table():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].split()
            if line:
                vals[int(line[0])] = float(line[1])
    assert sorted(vals) == list(range(16))
    return np.array([vals[c] for c in range(16)])


TABLE = _table()


def _brute_encode(x):
    """Nearest E2M1 magnitude by search over the table; an exact tie goes to
    the even code; magnitudes beyond 6 saturate."""
    out = np.empty(len(x), dtype=np.uint8)
    mags = TABLE[:8]
    for i, v in enumerate(np.asarray(x, dtype=np.float64)):
        a = abs(v)
        if a > 6.0:
            out[i] = 7 | (8 if np.signbit(v) else 0)
            continue
        d = np.abs(mags - a)
        best = np.flatnonzero(d == d.min())
        c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
        out[i] = c | (8 if np.signbit(v) else 0)
    return out


def _unpack(q, cols):
    q = np.asarray(q, dtype=np.uint8)
    c = np.empty(q.shape[:-1] + (cols,), dtype=np.uint8)
    c[..., 0::2] = q & 15
    c[..., 1::2] = q >> 4
    return c


def test_every_code_decodes_to_the_format_table():
    codes = np.arange(16, dtype=np.uint8)
    ours = oracle.e2m1_decode(codes)
    np.testing.assert_array_equal(ours, TABLE)
    assert np.array_equal(np.signbit(ours), np.signbit(TABLE))   # code 8 is -0


def test_encode_is_the_nearest_value_ties_to_even():
    # every value, every midpoint between neighbours, and points just around them
    mags = TABLE[:8]
    mids = (mags[:-1] + mags[1:]) / 2
    pts = np.concatenate([mags, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                          np.nextafter(mids.astype(np.float32), np.float32(10))])
    rng = np.random.default_rng(404)
    pts = np.concatenate([pts, rng.uniform(0, 8, 5000), rng.exponential(1.0, 5000),
                          [6.5, 6.99, 7.0, 7.01, 1e3, 1e30]]).astype(np.float32)
    x = np.concatenate([pts, -pts])
    np.testing.assert_array_equal(oracle.e2m1_encode(x), _brute_encode(x))
    # the midpoints themselves: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    np.testing.assert_array_equal(oracle.e2m1_encode(mids.astype(np.float32)),
                                  np.array([0, 2, 2, 4, 4, 6, 6], dtype=np.uint8))


@pytest.mark.parametrize("per_tensor", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_block_quantization_invariants(per_tensor, dtype):
    rng = np.random.default_rng(7 + per_tensor)
    rows, cols = 9, 96
    x = rng.standard_normal((rows, cols)).astype(np.float32) * rng.uniform(0.01, 5, (rows, 1)) \
        .astype(np.float32)
    x[2, 16:32] = 0.0            # an all-zero block
    x[3] = 0.0                   # an all-zero row
    x[4, 5] = 40.0               # a block dominated by one value
    x[5, 40:48] = 1e-30          # a block below the smallest scale
    if dtype == "bf16":
        import torch
        x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
        xin = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        xin = x
    q, s, g = oracle.quantize_nvfp4(xin, per_tensor=per_tensor)
    assert q.shape == (rows, cols // 2) and s.shape == (rows, cols // 16)
    codes = _unpack(q, cols)
    vals = TABLE[codes]
    sdec = oracle.e4m3_decode(s)
    assert np.all(s < 0x80)                                  # scales are non-negative
    gg = np.full(rows, g) if per_tensor else np.asarray(g, np.float64)
    amax_rows = np.abs(x).max(axis=1)
    amax = np.full(rows, np.abs(x).max()) if per_tensor else amax_rows
    for m in range(rows):
        if amax[m] == 0:
            assert gg[m] == 1.0 and np.all(codes[m] == 0)
            continue
        assert gg[m] == pytest.approx(amax[m] / 2688.0, rel=1e-6)
        for b in range(cols // 16):
            blk = x[m, 16 * b:16 * b + 16].astype(np.float64)
            deq = gg[m] * sdec[m, b] * vals[m, 16 * b:16 * b + 16]
            ab = np.abs(blk).max()
            if sdec[m, b] == 0:
                assert np.all(codes[m, 16 * b:16 * b + 16] & 7 == 0)
                assert ab * 2688.0 / amax[m] / 6 < 2.0 ** -9   # below half the smallest scale
                continue
            # the block scale is the E4M3 value nearest to amax_b / 6 in encoded units
            assert sdec[m, b] == pytest.approx(ab / 6 * 2688.0 / amax[m], rel=2 ** -3.9)
            # the block's largest element is coded +-6 (scale rounding stays within 6%)
            j = int(np.argmax(np.abs(blk)))
            assert codes[m, 16 * b + j] & 7 == 7
            assert np.sign(vals[m, 16 * b + j]) == np.sign(blk[j])
            # every element within half the widest E2M1 gap (1 of 6), in units of the block max
            assert np.all(np.abs(deq - blk) <= ab * (1.0 / 6.0) * 1.07 + 1e-30)
            # signs are kept (zero codes aside)
            nz = (codes[m, 16 * b:16 * b + 16] & 7) != 0
            assert np.all(np.sign(deq[nz]) == np.sign(blk[nz]))
    # packing: element 2i in the low nibble
    assert np.array_equal(q & 15, codes[:, 0::2]) and np.array_equal(q >> 4, codes[:, 1::2])


def test_nvfp4_logits_are_the_decoded_matmul():
    rng = np.random.default_rng(11)
    rows, vocab, hidden = 6, 40, 64
    h = rng.standard_normal((rows, hidden)).astype(np.float32)
    w = (rng.standard_normal((vocab, hidden)) * 0.05).astype(np.float32)
    qh, sh, gh = oracle.quantize_nvfp4(h)
    qw, sw, gw = oracle.quantize_nvfp4(w, per_tensor=True)
    dh = gh[:, None] * np.repeat(oracle.e4m3_decode(sh), 16, axis=1) * TABLE[_unpack(qh, hidden)]
    dw = np.float64(gw) * np.repeat(oracle.e4m3_decode(sw), 16, axis=1) \
        * TABLE[_unpack(qw, hidden)]
    z = dh @ dw.T
    u = oracle.unary_rows_nvfp4(qh, sh, gh, qw, sw, gw, vocab, 1.0, 0.0)
    np.testing.assert_allclose(u, z, rtol=1e-12, atol=1e-300)
    # the transform, the padded mask and a row subset on top of the same logits
    u2 = oracle.unary_rows_nvfp4(qh, sh, gh, qw, sw, gw, 33, 0.7, 30.0, rows=[5, 0])
    np.testing.assert_allclose(u2[:, :33], 30.0 * np.tanh(0.7 * z[[5, 0], :33] / 30.0),
                               rtol=1e-12)
    assert np.all(np.isneginf(u2[:, 33:]))
    # dequantized values approximate the inputs (NVFP4's error: about 6% of a block max)
    assert np.abs(dh - h).max() <= np.abs(h).max() * 0.2

"""Pins of the oracle's FP8 (E4M3) lm_head path against torch's float8_e4m3fn
conversions (a library routine written independently of the oracle), closed
forms of the format, and a plain matmul of the decoded values."""
import numpy as np
import pytest
import torch

import oracle


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn) \
        .float().numpy().astype(np.float64)


def _torch_encode(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_every_code_decodes_like_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = oracle.e4m3_decode(codes), _torch_decode(codes)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert set(np.nonzero(np.isnan(ours))[0].tolist()) == {0x7F, 0xFF}
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])
    assert oracle.e4m3_decode(np.array([0x7E]))[0] == 448.0
    assert oracle.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9


def test_encode_rounds_to_nearest_even_like_torch():
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(finite).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(vals), finite)   # -0 keeps its sign
    # every midpoint between neighbouring codes goes to the even code
    pos = np.sort(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    mids = np.concatenate([mids, -mids])
    np.testing.assert_array_equal(oracle.e4m3_encode(mids), _torch_encode(mids))
    rng = np.random.default_rng(81)
    x = np.concatenate([rng.uniform(-460, 460, 20000), rng.normal(0, 1, 20000),
                        rng.uniform(-2.0 ** -6, 2.0 ** -6, 20000)]).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(x), _torch_encode(x))


def test_encode_saturates_at_448():
    big = np.array([464.0, 480.0, 1e6, np.inf], dtype=np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(big), np.full(4, 0x7E, np.uint8))
    np.testing.assert_array_equal(oracle.e4m3_encode(-big), np.full(4, 0xFE, np.uint8))
    assert oracle.e4m3_encode(np.array([463.99], np.float32))[0] == 0x7E
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def _bf16(a):
    b = np.asarray(a, dtype=np.float32).view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _bf16_to_f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_row_quantization(dtype):
    rng = np.random.default_rng(82)
    h = rng.normal(0, 1, (9, 200)).astype(np.float32)
    h[3] = 0.0
    h[5] *= 1e-3
    h[6, 17] = 40.0            # one dominant entry
    hin = _bf16(h) if dtype == "bf16" else h
    hf = _bf16_to_f32(hin) if dtype == "bf16" else h
    q, d = oracle.quantize_rows_e4m3(hin)
    assert q.dtype == np.uint8 and d.dtype == np.float32
    # zero row: every code 0, scale 1
    assert (q[3] == 0).all() and d[3] == 1.0
    for m in (0, 1, 2, 4, 5, 6, 7, 8):
        amax = np.abs(hf[m]).max()
        inv = np.float32(448.0) / np.float32(amax)
        assert d[m] == np.float32(amax) / np.float32(448.0)
        # codes are torch's rounding of the fp32 product h * (448 / amax)
        np.testing.assert_array_equal(q[m], _torch_encode(hf[m] * inv))
        # the largest magnitude lands on +-448
        j = int(np.abs(hf[m]).argmax())
        assert q[m, j] & 0x7F == 0x7E
        # dequantization error: 2^-4 relative for normals, half a subnormal step below
        deq = oracle.e4m3_decode(q[m]) * np.float64(d[m])
        err = np.abs(deq - hf[m])
        assert (err <= np.maximum(np.abs(hf[m]) * 2.0 ** -4, float(d[m]) * 2.0 ** -10)).all()
    # scaling a row by a power of two scales d and leaves the codes
    q2, d2 = oracle.quantize_rows_e4m3((hf * np.float32(8.0)).astype(np.float32))
    keep = [0, 1, 2, 4, 5, 6, 7, 8]
    np.testing.assert_array_equal(q2[keep], q[keep])
    np.testing.assert_array_equal(d2[keep], d[keep] * np.float32(8.0))


def test_fp8_logits_are_the_decoded_matmul():
    rng = np.random.default_rng(83)
    rows, hidden, vd, vt = 5, 96, 70, 61
    qh = rng.integers(0, 256, (rows, hidden), dtype=np.uint8)
    qw = rng.integers(0, 256, (vd, hidden), dtype=np.uint8)
    qh[(qh & 0x7F) == 0x7F] = 0x10       # no NaN codes
    qw[(qw & 0x7F) == 0x7F] = 0x21
    dh = rng.uniform(0.001, 0.01, rows).astype(np.float32)
    sw = rng.uniform(0.001, 0.01, vd).astype(np.float32)
    z = (_torch_decode(qh) @ _torch_decode(qw).T) * dh[:, None].astype(np.float64) \
        * sw[None, :].astype(np.float64)
    for mult, cap in ((1.0, 0.0), (0.5, 30.0), (-1.0, 0.0)):
        u = oracle.unary_rows_fp8(qh, dh, qw, sw, vt, mult, cap)
        ref = cap * np.tanh(mult * z / cap) if cap > 0 else mult * z
        np.testing.assert_allclose(u[:, :vt], ref[:, :vt], rtol=1e-14, atol=0)
        assert np.isneginf(u[:, vt:]).all()
    sel = np.array([4, 0])
    np.testing.assert_array_equal(oracle.unary_rows_fp8(qh, dh, qw, sw, vt, 1.0, 0.0, rows=sel),
                                  oracle.unary_rows_fp8(qh, dh, qw, sw, vt, 1.0, 0.0)[sel])

"""GPU parity of dflash2_conv_prepare / dflash2_conv_finish against the oracle.

coef: bf16 results are the bf16 rounding of an fp32 sum within the accumulation
bound of the exact product (mostly equal to the oracle's), fp32 results within
that bound.  The convolutions are checked staged (the oracle
convolves with the GPU's own coefficients) under the conv tolerance, and on
integer-valued inputs, where every step is exact, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from block_draft_proposal_gb300 import dflash2, synth
from parity import conv_tolerance

pytestmark = pytest.mark.gpu


def _f64(a):
    return (synth.bf16_bits_to_f32(a) if a.dtype == np.uint16 else a).astype(np.float64)


def _check_coef(gpu, ref, x, wkp):
    exact = _f64(x) @ _f64(wkp).T
    hidden = x.shape[1]
    acc_bound = (hidden + 2) * 2.0 ** -24 * (np.abs(_f64(x)) @ np.abs(_f64(wkp)).T) + 1e-30
    g, r = _f64(gpu), _f64(ref)
    if gpu.dtype == np.uint16:
        # the GPU value is the bf16 rounding (half a step, at most 2^-8 relative) of
        # an fp32 sum within acc_bound of the exact product; the oracle rounds the
        # exact product itself, so the two differ only where that sum straddles a
        # rounding boundary (or cancellation makes acc_bound exceed the step)
        err = np.abs(g - exact)
        lim = (np.abs(exact) + acc_bound) * 2.0 ** -8 + acc_bound
        assert np.all(err <= lim), (err - lim).max()
        bad = g != r
        assert bad.mean() < 0.02, bad.mean()
        return int(bad.sum())
    assert np.all(np.abs(g - exact) <= acc_bound + 2.0 ** -24 * np.abs(exact))
    return 0


def _conv_ok(gpu, ref, dtype, abs_conv):
    g, r = _f64(gpu), _f64(ref)
    if dtype == "bf16":
        # 2e-2 absolute, or one bf16 step of the oracle value where that is larger:
        # with projected coefficients of order one the outputs reach magnitudes
        # where rounding the same value to bf16 already differs by one step
        lim = np.maximum(conv_tolerance("bf16", None), np.abs(r) * 2.0 ** -7)
        diff = np.abs(g - r)
        assert np.all(diff <= lim), (diff - lim).max()
        assert (diff > 0).mean() < 0.02
    else:
        assert np.all(np.abs(g - r) <= conv_tolerance("f32", abs_conv))


def _abs_conv(src, base, coef_side, w):
    f = lambda a: np.abs(_f64(a)).astype(np.float32)
    return oracle.conv(f(src), f(base), f(coef_side), w.block_size, w.group_size,
                       w.taps).astype(np.float64)


CASES = [("tiny-fp32", {}), ("qwen3-8b-bf16", dict(batch=4)), ("padded-vocab-bf16", dict(batch=2)),
         ("reduced-vocab-bs12-bf16", dict(batch=3)), ("stress-bf16", dict(batch=1)),
         # ragged: hidden not a multiple of the 128-element stage, tokens not of a tile
         ("qwen3-8b-bf16", dict(batch=3, block_size=7, hidden=200, group_size=8, taps=3)),
         ("qwen3-8b-bf16", dict(batch=5, block_size=2, hidden=1032, group_size=8, taps=4))]


@pytest.mark.parametrize("name,scale", CASES, ids=lambda c: str(c))
def test_prepare_and_finish(cuda, name, scale):
    w = synth.BY_NAME[name].scaled(**scale)
    d = synth.make(w, parts=("x", "w_kp", "base2", "h"))
    x, wkp, base2 = d["x"], d["w_kp"], d["base2"]
    tx, tw, tb = (dflash2.to_device(a, cuda) for a in (x, wkp, base2))
    out, coef, err = dflash2.conv_prepare(tx, tw, tb, w.block_size, w.group_size, w.taps)
    # finish on another input of the same shape (the sublayer output)
    y = np.ascontiguousarray(np.resize(d["h"], x.shape))
    ty = dflash2.to_device(y, cuda)
    fin = dflash2.conv_finish(ty, coef, tb, w.block_size, w.group_size, w.taps)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    g_coef = dflash2.to_host_bits(coef).reshape(w.n_tokens, -1)
    ref_coef = oracle.kernel_projection(x, wkp)
    mism = _check_coef(g_coef, ref_coef, x, wkp)
    print(f"{name} {scale}: coef rounding-boundary mismatches {mism}")
    # staged: the oracle's convolutions on the GPU's own coefficients
    gr = w.groups
    side0 = np.ascontiguousarray(g_coef[:, : w.taps * gr])
    side1 = np.ascontiguousarray(g_coef[:, w.taps * gr:])
    ref_out = oracle.conv(x, np.ascontiguousarray(base2[0]), side0, w.block_size, w.group_size,
                          w.taps)
    ref_fin = oracle.conv_finish(y, g_coef, base2, w.block_size, w.group_size, w.taps)
    _conv_ok(dflash2.to_host_bits(out), ref_out, w.dtype,
             None if w.dtype == "bf16" else _abs_conv(x, base2[0], side0, w))
    _conv_ok(dflash2.to_host_bits(fin), ref_fin, w.dtype,
             None if w.dtype == "bf16" else _abs_conv(y, base2[1], side1, w))


def test_integer_inputs_are_bit_exact(cuda):
    # small integers: the projection, its bf16 rounding and the conv are exact
    w = synth.BY_NAME["qwen3-8b-bf16"].scaled(batch=3, hidden=512, block_size=5)
    rng = np.random.default_rng(8)
    to = lambda a: synth.to_bf16_bits(a.astype(np.float32))
    x = to(rng.integers(-2, 3, size=(w.n_tokens, w.hidden)))
    wkp = to(rng.integers(-1, 2, size=(2 * w.taps * w.groups, w.hidden)) *
             (rng.random((2 * w.taps * w.groups, w.hidden)) < 0.05))
    base2 = to(rng.integers(-2, 3, size=(2, w.taps, w.hidden)))
    tx, tw, tb = (dflash2.to_device(a, cuda) for a in (x, wkp, base2))
    out, coef, err = dflash2.conv_prepare(tx, tw, tb, w.block_size, w.group_size, w.taps)
    fin = dflash2.conv_finish(tx, coef, tb, w.block_size, w.group_size, w.taps)
    torch.cuda.synchronize()
    ref_out, ref_coef = oracle.conv_prepare(x, wkp, base2, w.block_size, w.group_size, w.taps)
    np.testing.assert_array_equal(dflash2.to_host_bits(coef).reshape(w.n_tokens, -1), ref_coef)
    np.testing.assert_array_equal(dflash2.to_host_bits(out), ref_out)
    np.testing.assert_array_equal(dflash2.to_host_bits(fin),
                                  oracle.conv_finish(x, ref_coef, base2, w.block_size,
                                                     w.group_size, w.taps))


def test_argument_errors(cuda):
    lib = dflash2.library()
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device=cuda)
    wk = torch.zeros((2 * 4 * 8, 64), dtype=torch.bfloat16, device=cuda)
    b2 = torch.zeros((2, 4, 64), dtype=torch.bfloat16, device=cuda)
    coef = torch.zeros((4, 2, 4, 8), dtype=torch.bfloat16, device=cuda)
    out = torch.empty_like(x)
    p = lambda t: t.data_ptr()
    # hidden % group_size, taps < 1, block_size < 1, dtype, empty
    assert lib.dflash2_conv_prepare(p(x), p(wk), p(b2), 4, 64, 7, 4, 16, 1, p(out), p(coef), None, None) == 1
    assert lib.dflash2_conv_prepare(p(x), p(wk), p(b2), 4, 64, 8, 0, 16, 1, p(out), p(coef), None, None) == 1
    assert lib.dflash2_conv_prepare(p(x), p(wk), p(b2), 4, 64, 8, 4, 0, 1, p(out), p(coef), None, None) == 1
    assert lib.dflash2_conv_prepare(p(x), p(wk), p(b2), 4, 64, 8, 4, 16, 7, p(out), p(coef), None, None) == 2
    assert lib.dflash2_conv_prepare(p(x), p(wk), p(b2), 0, 64, 8, 4, 16, 1, p(out), p(coef), None, None) == 0
    # bf16 projection wants a 16-byte aligned x
    assert lib.dflash2_conv_prepare(p(x) + 2, p(wk), p(b2), 3, 64, 8, 4, 16, 1, p(out), p(coef), None, None) == 3
    assert lib.dflash2_conv_finish(p(x), p(b2), p(coef), 4, 64, 8, 4, 16, 1, p(out), None) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["qwen3-8b-bf16", "stress-bf16"])
def test_full_size_sampled_blocks(cuda, name):
    # full-size launch; the oracle recomputes a sample of whole blocks (the conv
    # of a token needs its block's earlier rows)
    w = synth.BY_NAME[name]
    d = synth.make(w, parts=("x", "w_kp", "base2"))
    x, wkp, base2 = d["x"], d["w_kp"], d["base2"]
    tx, tw, tb = (dflash2.to_device(a, cuda) for a in (x, wkp, base2))
    out, coef, err = dflash2.conv_prepare(tx, tw, tb, w.block_size, w.group_size, w.taps)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    g_coef = dflash2.to_host_bits(coef).reshape(w.n_tokens, -1)
    g_out = dflash2.to_host_bits(out)
    blocks = np.random.default_rng(9).choice(w.batch, size=2, replace=False)
    rows = np.concatenate([np.arange(b * w.block_size, (b + 1) * w.block_size) for b in blocks])
    xs = np.ascontiguousarray(x[rows])
    _check_coef(g_coef[rows], oracle.kernel_projection(xs, wkp), xs, wkp)
    side0 = np.ascontiguousarray(g_coef[rows, : w.taps * w.groups])
    ref = oracle.conv(xs, np.ascontiguousarray(base2[0]), side0, w.block_size, w.group_size,
                      w.taps)
    _conv_ok(g_out[rows], ref, w.dtype, None)

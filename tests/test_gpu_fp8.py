"""GPU parity of the FP8 (E4M3) lm_head path: dflash2_quantize_rows_e4m3 and
dflash2_unary_topk_fp8 against the oracle's W8A8 definition.

The activation codes decide integers, so they must equal the oracle's bit for
bit (both sides work in fp32).  The logits are exact products of codes summed
in fp32 by the tensor cores: each returned u must lie within the fp32
accumulation bound of the oracle's exact (double) value, and the ids must be
the oracle's top-K up to accepted near-ties (tests/parity.py)."""
import numpy as np
import pytest
import torch

import oracle
from block_draft_proposal_gb300 import dflash2, synth
from parity import check_topk_row

pytestmark = pytest.mark.gpu
EPS32 = 2.0 ** -24
DEC = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))   # code -> value (NaN codes unused)


def _case(rows, hidden, vd, seed, h_dtype):
    rng = np.random.default_rng(seed)
    h = rng.normal(0, 1, (rows, hidden)).astype(np.float32)
    if rows > 3:
        h[1] = 0.0                               # a zero row: codes 0, scale 1
        h[2, :] *= 1e-30                         # tiny values: subnormal codes
        h[3, 5] = 75.0                           # one dominant entry
    hin = synth.to_bf16_bits(h) if h_dtype == "bf16" else h
    qw = synth.fp8_codes(rng.normal(0, 64, (vd, hidden)).astype(np.float32))
    sw = (rng.uniform(0.5, 1.5, vd) * (0.02 / 64)).astype(np.float32)
    return hin, qw, sw


def _dev(a, dev):
    return dflash2.to_device(a, dev)


@pytest.mark.parametrize("rows,cols,h_dtype", [(5, 256, "bf16"), (33, 4096, "bf16"),
                                               (7, 144, "f32"), (300, 96, "bf16")])
def test_quantize_rows_matches_the_oracle_bit_for_bit(cuda, rows, cols, h_dtype):
    hin, _, _ = _case(rows, cols, 1, 90 + rows, h_dtype)
    if h_dtype == "f32":
        hin[0, :4] = [-0.0, 448.0, -1e-40, 3.0e38]   # -0, a subnormal float, a huge value
    q, d = dflash2.quantize_rows_e4m3(_dev(hin, cuda))
    torch.cuda.synchronize()
    q_ref, d_ref = oracle.quantize_rows_e4m3(hin)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    np.testing.assert_array_equal(d.cpu().numpy(), d_ref)


def _check_fp8(hin, qw, sw, vt, mult, cap, k, ids, vals, rows):
    qh, dh = oracle.quantize_rows_e4m3(hin)
    u = oracle.unary_rows_fp8(qh, dh, qw, sw, vt, mult, cap, rows=rows)
    ora_ids, _ = oracle.topk(u, k)
    hidden = qh.shape[1]
    ties = 0
    for r, m in enumerate(rows):
        a = np.abs(DEC[qh[m]])

        def bound(sel, r=r, m=m, a=a):
            sel = np.asarray(sel)
            s = (np.abs(DEC[qw[sel]]) @ a) * float(dh[m]) * sw[sel].astype(np.float64)
            return abs(mult) * (hidden + 4) * EPS32 * s + 8 * EPS32 * np.abs(u[r][sel]) + 1e-30

        ties += check_topk_row(ids[m], vals[m], ora_ids[r], u[r], bound, k)
        assert np.all(ids[m] < vt)
        assert np.all(np.diff(vals[m]) <= 0)
    return ties


CASES = [
    # rows, hidden, draft_vocab, target_vocab, k, mult, cap, h dtype
    (37, 256, 5000, 4900, 16, 0.5, 30.0, "bf16"),     # pilot-only vocab, padded tail
    (300, 272, 40000, 39990, 32, 1.0, 0.0, "bf16"),   # hidden one stage and a 16-element tail
    (7, 512, 70000, 70000, 64, 1.0, 30.0, "f32"),
    (513, 128, 9000, 8800, 8, 2.0, 0.0, "bf16"),      # three token tiles, hidden below a stage
    (5, 96, 3000, 2999, 128, 1.0, 0.0, "bf16"),       # K at its maximum
    (1800, 144, 4000, 4000, 8, 0.7, 0.0, "bf16"),
    (40, 256, 9000, 9000, 16, -1.0, 0.0, "bf16"),     # negative multiplier: the split passes
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"r{c[0]}-h{c[1]}-v{c[2]}-k{c[4]}")
def test_fp8_topk_matches_the_oracle(cuda, case):
    rows, hidden, vd, vt, k, mult, cap, h_dtype = case
    hin, qw, sw = _case(rows, hidden, vd, 7 * rows + hidden, h_dtype)
    ids, vals, err = dflash2.unary_topk_fp8(_dev(hin, cuda), _dev(qw, cuda), _dev(sw, cuda), vt,
                                            mult, cap, k)
    torch.cuda.synchronize()
    assert int(err.item()) & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    plan = dflash2.library().dflash2_unary_topk_launches(rows, vd, k, mult, dflash2.BF16)
    check = sorted(set([0, 1, 2, 3, rows - 1] + list(range(0, rows, max(1, rows // 12)))))
    ties = _check_fp8(hin, qw, sw, vt, mult, cap, k, ids.cpu().numpy(), vals.cpu().numpy(),
                      np.asarray(check))
    print(f"{case}: {'fused' if plan == 2 else 'split'} path, near-ties {ties}")


def test_fp8_topk_at_the_qwen3_size_on_sampled_rows(cuda):
    w = synth.BY_NAME["qwen3-8b-bf16"]
    inp = synth.make(w, parts=("h", "lm_head_fp8", "w_scale"))
    ids, vals, err = dflash2.unary_topk_fp8(_dev(inp["h"], cuda), _dev(inp["lm_head_fp8"], cuda),
                                            _dev(inp["w_scale"], cuda), w.target_vocab, w.mult,
                                            w.cap, w.top_k)
    torch.cuda.synchronize()
    assert int(err.item()) & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    rows = np.array([0, 1, 239, 240, 479])
    _check_fp8(inp["h"], inp["lm_head_fp8"], inp["w_scale"], w.target_vocab, w.mult, w.cap,
               w.top_k, ids.cpu().numpy(), vals.cpu().numpy(), rows)


def test_fp8_matches_bf16_candidates_closely(cuda):
    """The FP8 head is a quantization of nothing here, but on a head whose
    codes decode exactly to bf16 values, the FP8 and bf16 paths see the same
    weights: their candidates must agree up to the activation rounding."""
    rng = np.random.default_rng(95)
    rows, hidden, vd, k = 24, 256, 6000, 16
    qw = synth.fp8_codes(rng.normal(0, 64, (vd, hidden)).astype(np.float32))
    sw = np.full(vd, 2.0 ** -12, dtype=np.float32)           # a power of two: exact in bf16
    wf = (DEC[qw] * sw[:, None]).astype(np.float32)           # exact in bf16 (4 significant bits)
    h = rng.normal(0, 1, (rows, hidden)).astype(np.float32)
    i8, _, _ = dflash2.unary_topk_fp8(_dev(synth.to_bf16_bits(h), cuda), _dev(qw, cuda),
                                      _dev(sw, cuda), vd, 1.0, 0.0, k)
    i16, _, _ = dflash2.unary_topk(_dev(synth.to_bf16_bits(h), cuda),
                                   _dev(synth.to_bf16_bits(wf), cuda), vd, 1.0, 0.0, k)
    torch.cuda.synchronize()
    overlap = np.mean([len(set(a) & set(b)) / k for a, b in zip(i8.cpu().numpy(),
                                                                i16.cpu().numpy())])
    assert overlap > 0.6


@pytest.mark.parametrize("case", [(1, 16, 300, 300, 8, 1.0, 0.0, "bf16"),
                                  (2, 32, 200, 150, 4, 1.0, 30.0, "f32"),
                                  (3, 4096, 257, 257, 16, 1.0, 0.0, "bf16")],
                         ids=lambda c: f"r{c[0]}-h{c[1]}-v{c[2]}")
def test_fp8_topk_minimum_sizes(cuda, case):
    """One or two rows, hidden of one 16-code row, a vocab inside one unit or
    one row past it."""
    rows, hidden, vd, vt, k, mult, cap, h_dtype = case
    hin, qw, sw = _case(rows, hidden, vd, 500 + hidden, h_dtype)
    ids, vals, err = dflash2.unary_topk_fp8(_dev(hin, cuda), _dev(qw, cuda), _dev(sw, cuda), vt,
                                            mult, cap, k)
    torch.cuda.synchronize()
    assert int(err.item()) & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    _check_fp8(hin, qw, sw, vt, mult, cap, k, ids.cpu().numpy(), vals.cpu().numpy(),
               np.arange(rows))

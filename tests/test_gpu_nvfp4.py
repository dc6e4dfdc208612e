"""GPU parity of the NVFP4 lm_head path: dflash2_quantize_rows_nvfp4 and
dflash2_unary_topk_nvfp4 against the oracle's W4A4 definition.

The activation codes, block scales and second-level scales decide integers
(or are fixed by one IEEE operation), so they must equal the oracle's bit for
bit.  The head checkpoint (codes, block scales, tensor scale) is quantized by
the oracle.  The logits are exact block sums of code products, scaled by the
two block scales and summed in fp32 by the tensor cores: each returned u must
lie within the fp32 accumulation bound of the oracle's exact (double) value,
and the ids must be the oracle's top-K up to accepted near-ties
(tests/parity.py)."""
import numpy as np
import pytest
import torch

import oracle
from block_draft_proposal_gb300 import dflash2, synth
from parity import check_topk_row

pytestmark = pytest.mark.gpu
EPS32 = 2.0 ** -24
E2M1 = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
E4M3 = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))


def _unpack(q, cols):
    c = np.empty(q.shape[:-1] + (cols,), dtype=np.uint8)
    c[..., 0::2] = q & 15
    c[..., 1::2] = q >> 4
    return c


def _case(rows, hidden, vd, seed, h_dtype):
    rng = np.random.default_rng(seed)
    h = rng.normal(0, 1, (rows, hidden)).astype(np.float32)
    if rows > 4:
        h[1] = 0.0                               # a zero row: codes 0, scales 1
        h[2, :] *= 1e-30                         # tiny values
        h[3, 5] = 75.0                           # one dominant entry
        h[4, :16] = 0.0                          # one zero block
    hin = synth.to_bf16_bits(h) if h_dtype == "bf16" else h
    w = (rng.normal(0, 0.02, (vd, hidden)) * rng.uniform(0.2, 3.0, (vd, 1))).astype(np.float32)
    qw, sw, gw = oracle.quantize_nvfp4(w, per_tensor=True)
    return hin, qw, sw, float(gw)


def _dev(a, dev):
    return dflash2.to_device(a, dev)


@pytest.mark.parametrize("rows,cols,h_dtype", [(5, 256, "bf16"), (33, 4096, "bf16"),
                                               (7, 144, "f32"), (300, 96, "bf16"),
                                               (2, 7168, "f32")])
def test_quantize_rows_matches_the_oracle_bit_for_bit(cuda, rows, cols, h_dtype):
    hin, _, _, _ = _case(rows, cols, 1, 90 + rows, h_dtype)
    if h_dtype == "f32":
        hin[0, :4] = [-0.0, 6.0, -1e-40, -0.01]   # -0, a subnormal float, a value rounding to -0
    q, s, g = dflash2.quantize_rows_nvfp4(_dev(hin, cuda))
    torch.cuda.synchronize()
    q_ref, s_ref, g_ref = oracle.quantize_nvfp4(hin)
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(g.cpu().numpy(), g_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)


def _check_nvfp4(hin, qw, sw, gw, vt, mult, cap, k, ids, vals, rows):
    qh, sh, gh = oracle.quantize_nvfp4(hin)
    u = oracle.unary_rows_nvfp4(qh, sh, gh, qw, sw, gw, vt, mult, cap, rows=rows)
    ora_ids, _ = oracle.topk(u, k)
    hidden = qh.shape[1] * 2
    ties = 0
    for r, m in enumerate(rows):
        a = np.abs(E2M1[_unpack(qh[m], hidden)]) * np.repeat(E4M3[sh[m]], 16)

        def bound(sel, r=r, m=m, a=a):
            sel = np.asarray(sel)
            wv = np.abs(E2M1[_unpack(qw[sel], hidden)]) * np.repeat(E4M3[sw[sel]], 16, axis=1)
            s = (wv @ a) * float(gh[m]) * gw
            return abs(mult) * (hidden + 4) * EPS32 * s + 8 * EPS32 * np.abs(u[r][sel]) + 1e-30

        ties += check_topk_row(ids[m], vals[m], ora_ids[r], u[r], bound, k)
        assert np.all(ids[m] < vt)
        assert np.all(np.diff(vals[m]) <= 0)
    return ties


CASES = [
    # rows, hidden, draft_vocab, target_vocab, k, mult, cap, h dtype
    (37, 256, 5000, 4900, 16, 0.5, 30.0, "bf16"),     # pilot-only vocab, padded tail
    (300, 320, 40000, 39990, 32, 1.0, 0.0, "bf16"),   # hidden one stage and a 64-element tail
    (7, 512, 70000, 70000, 64, 1.0, 30.0, "f32"),
    (513, 128, 9000, 8800, 8, 2.0, 0.0, "bf16"),      # five token tiles, hidden below a stage
    (5, 192, 3000, 2999, 128, 1.0, 0.0, "bf16"),      # K at its maximum
    (1800, 192, 4000, 4000, 8, 0.7, 0.0, "bf16"),
    (40, 256, 9000, 9000, 16, -1.0, 0.0, "bf16"),     # negative multiplier: the split passes
    (130, 1024, 20000, 20000, 24, 1.0, 30.0, "bf16"), # two token tiles of 65
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"r{c[0]}-h{c[1]}-v{c[2]}-k{c[4]}")
def test_nvfp4_topk_matches_the_oracle(cuda, case):
    rows, hidden, vd, vt, k, mult, cap, h_dtype = case
    hin, qw, sw, gw = _case(rows, hidden, vd, 7 * rows + hidden, h_dtype)
    tiles = dflash2.nvfp4_tile_scales(_dev(sw, cuda), hidden)
    ids, vals, err = dflash2.unary_topk_nvfp4(_dev(hin, cuda), _dev(qw, cuda), tiles, gw,
                                              vt, mult, cap, k)
    torch.cuda.synchronize()
    assert int(err.item()) & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    check = sorted(set([0, 1, 2, 3, 4, rows - 1] + list(range(0, rows, max(1, rows // 12)))))
    check = [c for c in check if c < rows]
    ties = _check_nvfp4(hin, qw, sw, gw, vt, mult, cap, k, ids.cpu().numpy(), vals.cpu().numpy(),
                        np.asarray(check))
    print(f"{case}: near-ties {ties}")


def test_nvfp4_topk_at_the_qwen3_size_on_sampled_rows(cuda):
    w = synth.BY_NAME["qwen3-8b-bf16"].scaled(draft_vocab=60000, target_vocab=60000)
    rng = np.random.default_rng(606)
    h = synth.make(w, parts=("h",))["h"]
    wf = rng.normal(0, 0.02, (w.draft_vocab, w.hidden)).astype(np.float32)
    qw, sw, gw = oracle.quantize_nvfp4(wf, per_tensor=True)
    tiles = dflash2.nvfp4_tile_scales(_dev(sw, cuda), w.hidden)
    ids, vals, err = dflash2.unary_topk_nvfp4(_dev(h, cuda), _dev(qw, cuda), tiles, float(gw),
                                              w.target_vocab, w.mult, w.cap, w.top_k)
    torch.cuda.synchronize()
    assert int(err.item()) & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    rows = np.array([0, 1, 127, 128, 239, 240, 479])
    ties = _check_nvfp4(h, qw, sw, float(gw), w.target_vocab, w.mult, w.cap, w.top_k,
                        ids.cpu().numpy(), vals.cpu().numpy(), rows)
    print(f"qwen3 shape, vocab 60000: near-ties {ties}")


def test_nvfp4_topk_at_the_stress_hidden_on_sampled_rows(cuda):
    """hidden 7168 (14 stages of 512 elements), 960 rows (8 token tiles of
    128), K 64, mult 0.5 with cap: the stress draft's shapes with a smaller
    vocab."""
    w = synth.BY_NAME["stress-bf16"].scaled(batch=64, draft_vocab=24000, target_vocab=24000)
    rng = np.random.default_rng(707)
    h = synth.make(w, parts=("h",))["h"]
    wf = rng.normal(0, 0.02, (w.draft_vocab, w.hidden)).astype(np.float32)
    qw, sw, gw = oracle.quantize_nvfp4(wf, per_tensor=True)
    tiles = dflash2.nvfp4_tile_scales(_dev(sw, cuda), w.hidden)
    ids, vals, err = dflash2.unary_topk_nvfp4(_dev(h, cuda), _dev(qw, cuda), tiles, float(gw),
                                              w.target_vocab, w.mult, w.cap, w.top_k)
    torch.cuda.synchronize()
    assert int(err.item()) & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    rows = np.array([0, 1, 127, 128, 511, 512, 895, 959])
    ties = _check_nvfp4(h, qw, sw, float(gw), w.target_vocab, w.mult, w.cap, w.top_k,
                        ids.cpu().numpy(), vals.cpu().numpy(), rows)
    print(f"stress hidden, vocab 24000: near-ties {ties}")


def test_nvfp4_overflowing_candidate_lists_fall_back_exactly(cuda):
    """The minimum workspace leaves room for K candidates per row: rows whose
    lists overflow are recomputed exactly on CUDA cores from the codes and
    block scales (flagged DEVINFO_TOPK_FALLBACK) and still match the oracle."""
    rows, hidden, vd, vt, k = 24, 128, 20000, 19900, 16
    hin, qw, sw, gw = _case(rows, hidden, vd, 92, "bf16")
    min_ws = dflash2.unary_topk_workspace_min(rows, vd, k, dflash2.BF16)
    prefix = (dflash2.unary_topk_nvfp4_workspace_size(rows, hidden, vd, k)
              - dflash2.unary_topk_workspace_size(rows, vd, k, dflash2.BF16))
    ws = torch.empty(prefix + min_ws, dtype=torch.uint8, device=cuda)
    tiles = dflash2.nvfp4_tile_scales(_dev(sw, cuda), hidden)
    ids, vals, err = dflash2.unary_topk_nvfp4(_dev(hin, cuda), _dev(qw, cuda), tiles, gw,
                                              vt, 1.0, 0.0, k, workspace=ws)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & dflash2.DEVINFO_TOPK_FALLBACK
    assert e & ~dflash2.DEVINFO_TOPK_FALLBACK == 0
    _check_nvfp4(hin, qw, sw, gw, vt, 1.0, 0.0, k, ids.cpu().numpy(), vals.cpu().numpy(),
                 np.arange(rows))


def test_nvfp4_rejects_bad_arguments(cuda):
    lib = dflash2.library()
    h = torch.zeros((4, 96), dtype=torch.bfloat16, device=cuda)   # hidden not a multiple of 64
    q = torch.zeros((100, 48), dtype=torch.uint8, device=cuda)
    s = torch.zeros((100, 6), dtype=torch.uint8, device=cuda)
    with pytest.raises(dflash2.Dflash2Error):
        dflash2.unary_topk_nvfp4(h, q, s, 1.0, 100, 1.0, 0.0, 4)
    h = torch.zeros((4, 128), dtype=torch.bfloat16, device=cuda)
    q = torch.zeros((100, 64), dtype=torch.uint8, device=cuda)
    s = torch.zeros(int(lib.dflash2_nvfp4_scale_tiles_size(100, 128)), dtype=torch.uint8,
                    device=cuda)
    for g in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(dflash2.Dflash2Error):
            dflash2.unary_topk_nvfp4(h, q, s, g, 100, 1.0, 0.0, 4)
    # cols not a multiple of 16
    assert lib.dflash2_quantize_rows_nvfp4(dflash2._ptr(h), 4, 120, dflash2.BF16, None, None,
                                           None, None) == 1


@pytest.mark.parametrize("rows,hidden", [(5, 64), (300, 576), (128, 4096), (129, 1024)])
def test_scale_tiles_follow_the_documented_layout(cuda, rows, hidden):
    """dflash2_nvfp4_tile_scales against the layout of include/dflash2.h written
    out with numpy: rows in blocks of 128, cells of 4 scales, nw8 cells per
    row, tile (rb, w) of 512 bytes with row rb*128 + l + 32 j's cell at
    l*16 + j*4; zeros elsewhere."""
    rng = np.random.default_rng(rows + hidden)
    nsf = hidden // 16
    sc = rng.integers(1, 255, size=(rows, nsf), dtype=np.uint8)
    tiles = dflash2.nvfp4_tile_scales(_dev(sc, cuda), hidden).cpu().numpy()
    nw = nsf // 4
    nw8 = (nw + 7) // 8 * 8
    nrb = (rows + 127) // 128
    ref = np.zeros(nrb * nw8 * 512, dtype=np.uint8)
    for r in range(rows):
        rb, rl = divmod(r, 128)
        l, j = rl % 32, rl // 32
        for w in range(nw):
            o = (rb * nw8 + w) * 512 + l * 16 + j * 4
            ref[o:o + 4] = sc[r, 4 * w:4 * w + 4]
    np.testing.assert_array_equal(tiles, ref)

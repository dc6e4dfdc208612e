"""GPU parity of dflash2_grouped_conv against the CPU oracle, element by element.

Every named workload at full size, plus edge cases: ragged token counts, taps
beyond the block, block size 1, non-power-of-two blocks, a strided two-sided
coefficient projection, the scalar (unaligned / narrow-group) path, and empty
input."""
import numpy as np
import pytest
import torch

import oracle
from block_draft_proposal_gb300 import dflash2, synth
from parity import conv_tolerance

pytestmark = pytest.mark.gpu


def _abs_conv(x, base, delta, w, stride=None):
    f = synth.bf16_bits_to_f32 if x.dtype == np.uint16 else (lambda a: a)
    ax, ab, ad = (np.abs(f(a)).astype(np.float32) for a in (x, base, delta))
    return oracle.conv(ax, ab, ad, w.block_size, w.group_size, w.taps,
                       delta_row_stride=stride).astype(np.float64)


def _compare(gpu, ref, w, x, base, delta, stride=None):
    if w.dtype == "bf16":
        diff = np.abs(synth.bf16_bits_to_f32(gpu).astype(np.float64) - synth.bf16_bits_to_f32(ref))
        assert diff.max() <= conv_tolerance("bf16", None), diff.max()
        # rounding the same double to bf16 differs by at most one bf16 step
        ulp = np.abs(synth.bf16_bits_to_f32(ref)).astype(np.float64) * 2.0 ** -7 + 1e-38
        assert np.all(diff <= ulp + 1e-6), (diff - ulp).max()
    else:
        tol = conv_tolerance("f32", _abs_conv(x, base, delta, w, stride))
        diff = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
        assert np.all(diff <= tol), (diff - tol).max()


def _run(w, dev, x, base, delta, stride=None, offset_elems=0):
    tx, tb, td = (dflash2.to_device(a, dev) for a in (x, base, delta))
    if offset_elems:
        # a view that starts off the 16-byte grid forces the scalar path
        big = torch.empty(tx.numel() + offset_elems, dtype=tx.dtype, device=dev)
        big[offset_elems:] = tx.reshape(-1)
        tx = big[offset_elems:].view(tx.shape)
    out = dflash2.grouped_conv(tx, tb, td, w.block_size, w.group_size, w.taps,
                               delta_row_stride=stride)
    torch.cuda.synchronize()
    return dflash2.to_host_bits(out)


@pytest.mark.parametrize("name", [c.name for c in synth.CONFIGS])
def test_conv_matches_oracle_on_named_workloads(cuda, name):
    w = synth.BY_NAME[name]
    inp = synth.make(w, parts=("x", "base", "delta"))
    gpu = _run(w, cuda, inp["x"], inp["base"], inp["delta"])
    ref = oracle.conv(inp["x"], inp["base"], inp["delta"], w.block_size, w.group_size, w.taps)
    _compare(gpu, ref, w, inp["x"], inp["base"], inp["delta"])


EDGE = [
    # (batch, block, hidden, group, taps, dtype)   n = batch * block, then trimmed
    dict(batch=3, block_size=8, hidden=256, group_size=8, taps=4, dtype="bf16", trim=5),
    dict(batch=5, block_size=12, hidden=320, group_size=8, taps=6, dtype="bf16", trim=7),
    dict(batch=4, block_size=3, hidden=64, group_size=8, taps=6, dtype="bf16", trim=0),
    dict(batch=9, block_size=1, hidden=128, group_size=8, taps=4, dtype="f32", trim=0),
    dict(batch=2, block_size=7, hidden=96, group_size=16, taps=3, dtype="f32", trim=3),
    dict(batch=3, block_size=16, hidden=72, group_size=4, taps=4, dtype="bf16", trim=0),   # scalar path
    dict(batch=3, block_size=16, hidden=60, group_size=6, taps=2, dtype="f32", trim=1),    # scalar path
    dict(batch=40, block_size=16, hidden=1024, group_size=8, taps=70, dtype="bf16", trim=9),  # taps > 64 clipped by block
    dict(batch=2, block_size=100, hidden=64, group_size=8, taps=70, dtype="bf16", trim=13),  # > 64 live taps: scalar path
    # pipelined path: a block of 40 (halo rows before each 16-token tile) with 8
    # taps over three 64-vector strips, the last one vector wide; fp32 with five
    # taps and no halo; group size 16 with blocks of 32 (halo, 32 groups per strip)
    dict(batch=3, block_size=40, hidden=1032, group_size=8, taps=8, dtype="bf16", trim=11),
    dict(batch=6, block_size=16, hidden=512, group_size=8, taps=5, dtype="f32", trim=2),
    dict(batch=7, block_size=32, hidden=2048, group_size=16, taps=4, dtype="bf16", trim=0),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"b{c['block_size']}-h{c['hidden']}-g{c['group_size']}-t{c['taps']}-{c['dtype']}")
def test_conv_edge_cases(cuda, case):
    c = dict(case)
    trim = c.pop("trim")
    w = synth.BY_NAME["tiny-fp32"].scaled(**c, x_std=1.0, seed=77)
    inp = synth.make(w, parts=("x", "base", "delta"))
    n = w.n_tokens - trim
    x, delta = inp["x"][:n].copy(), inp["delta"][:n].copy()
    gpu = _run(w, cuda, x, inp["base"], delta)
    ref = oracle.conv(x, inp["base"], delta, w.block_size, w.group_size, w.taps)
    _compare(gpu, ref, w, x, inp["base"], delta)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_conv_misaligned_input_takes_scalar_path(cuda, dtype):
    w = synth.BY_NAME["tiny-fp32"].scaled(batch=4, dtype=dtype, x_std=1.0, seed=78)
    inp = synth.make(w, parts=("x", "base", "delta"))
    gpu = _run(w, cuda, inp["x"], inp["base"], inp["delta"], offset_elems=1)
    ref = oracle.conv(inp["x"], inp["base"], inp["delta"], w.block_size, w.group_size, w.taps)
    _compare(gpu, ref, w, inp["x"], inp["base"], inp["delta"])


def test_conv_reads_side_zero_of_two_sided_projection(cuda):
    w = synth.BY_NAME["qwen3-8b-bf16"].scaled(batch=6, seed=79)
    inp = synth.make(w, parts=("x", "base"))
    both = synth.normal(w.seed, "delta", (w.n_tokens, 2, w.taps, w.groups), 0.02, "bf16")
    stride = 2 * w.taps * w.groups
    gpu = _run(w, cuda, inp["x"], inp["base"], both, stride=stride)
    ref = oracle.conv(inp["x"], inp["base"], both, w.block_size, w.group_size, w.taps,
                      delta_row_stride=stride)
    _compare(gpu, ref, w, inp["x"], inp["base"], both, stride)


def test_conv_empty_input_is_a_no_op(cuda):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=cuda)
    base = torch.zeros((4, 256), dtype=torch.bfloat16, device=cuda)
    delta = torch.zeros((0, 4, 32), dtype=torch.bfloat16, device=cuda)
    out = dflash2.grouped_conv(x, base, delta, 8, 8, 4)
    assert out.shape == (0, 256)


def test_conv_identity_init_is_bit_exact(cuda):
    w = synth.BY_NAME["stress-bf16"].scaled(batch=8, seed=80)
    inp = synth.make(w, parts=("x",))
    base = np.zeros((w.taps, w.hidden), np.float32)
    base[0] = 1.0
    gpu = _run(w, cuda, inp["x"], synth.to_bf16_bits(base),
               synth.to_bf16_bits(np.zeros((w.n_tokens, w.taps, w.groups), np.float32)))
    np.testing.assert_array_equal(gpu, inp["x"])

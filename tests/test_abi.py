"""The C ABI: libdflash2.so loads on a machine without a GPU, exports every
entry point include/dflash2.h declares, and rejects bad arguments on the host
before touching CUDA.  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash2.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build_library()
    from block_draft_proposal_gb300 import dflash2
    return dflash2.library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash2_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    from block_draft_proposal_gb300 import dflash2
    assert _declared() == sorted(dflash2.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (dflash2_\w+)", out))
    for name in _declared():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings_and_version(lib):
    assert lib.dflash2_abi_version() == 9
    assert lib.dflash2_status_string(0) == b"ok"
    for s in range(1, 7):
        assert lib.dflash2_status_string(s) not in (b"ok", b"unknown status")
    assert lib.dflash2_status_string(99) == b"unknown status"


def test_host_validation_rejects_before_any_launch(lib):
    null = None
    # conv: bad dtype, hidden not divisible by group size, short delta stride, empty input
    assert lib.dflash2_grouped_conv(null, null, null, 0, null, 8, 64, 8, 4, 8, 7, null) == 2
    assert lib.dflash2_grouped_conv(null, null, null, 32, null, 8, 60, 8, 4, 8, 1, null) == 1
    assert lib.dflash2_grouped_conv(null, null, null, 31, null, 8, 64, 8, 4, 8, 1, null) == 1
    assert lib.dflash2_grouped_conv(null, null, null, 32, null, 0, 64, 8, 4, 8, 1, null) == 0
    assert lib.dflash2_grouped_conv(null, null, null, 32, null, 8, 64, 8, 0, 8, 1, null) == 1
    # unary top-k: K out of range, K above the target vocab, a quantised dtype
    args = (null, null, 7, 256, 4096, 4096, 1.0, 0.0)
    assert lib.dflash2_unary_topk(*args, 0, 1, null, null, null, 0, null, null) == 1
    assert lib.dflash2_unary_topk(*args, 129, 1, null, null, null, 0, null, null) == 1
    assert lib.dflash2_unary_topk(null, null, 7, 256, 4096, 4, 1.0, 0.0, 8, 1, null, null, null, 0,
                                  null, null) == 1
    assert lib.dflash2_unary_topk(*args, 8, 3, null, null, null, 0, null, null) == 2
    assert lib.dflash2_unary_topk(null, null, 0, 256, 4096, 4096, 1.0, 0.0, 8, 1, null, null, null,
                                  0, null, null) == 0
    # selector walk: rank not a multiple of 8 (bf16), K too large
    w = (null,) * 4
    assert lib.dflash2_selector_walk(*w, 10, *(null,) * 6, 2, 3, 64, 12, 8, 1, null, null, null,
                                     null, 0, null, null) == 1
    assert lib.dflash2_selector_walk(*w, 10, *(null,) * 6, 2, 3, 64, 16, 200, 1, null, null, null,
                                     null, 0, null, null) == 1
    # the split walk: the same shape checks, and a missing workspace, before any launch
    assert lib.dflash2_selector_project(null, null, 2, 3, 64, 12, 8, 1, null, 0, null,
                                        null) == 1
    assert lib.dflash2_selector_project(null, null, 2, 3, 64, 16, 8, 4, null, 0, null,
                                        null) == 2
    assert lib.dflash2_selector_project(ctypes.c_void_p(256), ctypes.c_void_p(256), 2, 3, 64, 16,
                                        8, 1, null, 0, null, null) == 4
    assert lib.dflash2_selector_project(null, null, 0, 3, 64, 16, 8, 1, null, 0, null,
                                        null) == 0
    assert lib.dflash2_selector_walk_projected(null, null, 10, *(null,) * 6, 2, 3, 64, 16, 200, 1,
                                               null, null, null, null, 0, null, null) == 1
    assert lib.dflash2_selector_walk_projected(null, null, 0, *(null,) * 6, 2, 3, 64, 16, 8, 1,
                                               null, null, null, null, 0, null, null) == 1
    # FP8 head: dtype, shapes, hidden % 16 and the workspace are checked before any launch
    p16 = ctypes.c_void_p(256)
    fp8 = (p16, 1, p16, p16)
    assert lib.dflash2_unary_topk_fp8(p16, 3, p16, p16, 7, 256, 4096, 4096, ctypes.c_float(1.0),
                                      ctypes.c_float(0.0), 8, p16, p16, p16, 1 << 30, null,
                                      null) == 2
    assert lib.dflash2_unary_topk_fp8(*fp8, 7, 256, 4096, 4096, ctypes.c_float(1.0),
                                      ctypes.c_float(0.0), 129, p16, p16, p16, 1 << 30, null,
                                      null) == 1
    assert lib.dflash2_unary_topk_fp8(*fp8, 7, 264, 4096, 4096, ctypes.c_float(1.0),
                                      ctypes.c_float(0.0), 8, p16, p16, p16, 1 << 30, null,
                                      null) == 3
    assert lib.dflash2_unary_topk_fp8(*fp8, 7, 256, 4096, 4096, ctypes.c_float(1.0),
                                      ctypes.c_float(0.0), 8, p16, p16, null, 0, null, null) == 4
    assert lib.dflash2_unary_topk_fp8(*fp8, 0, 256, 4096, 4096, ctypes.c_float(1.0),
                                      ctypes.c_float(0.0), 8, p16, p16, null, 0, null, null) == 0
    assert lib.dflash2_quantize_rows_e4m3(p16, 4, 64, 5, p16, p16, null) == 2
    assert lib.dflash2_quantize_rows_e4m3(p16, 4, 0, 1, p16, p16, null) == 1
    assert lib.dflash2_quantize_rows_e4m3(null, 0, 64, 1, null, null, null) == 0
    assert lib.dflash2_unary_topk_fp8_workspace_size(480, 4096, 151936, 16) > \
        lib.dflash2_unary_topk_workspace_size(480, 151936, 16, 1) + 480 * 4096
    # top-K merge: shard count, list sizes and offsets are checked before any launch
    offs = (ctypes.c_int64 * 2)(0, 100)
    assert lib.dflash2_topk_merge(null, null, offs, 0, 4, 8, 8, null, null, null, null) == 1
    assert lib.dflash2_topk_merge(null, null, offs, 2, 4, 2049, 8, null, null, null, null) == 1
    assert lib.dflash2_topk_merge(null, null, offs, 2, 4, 8, 129, null, null, null, null) == 1
    assert lib.dflash2_topk_merge(null, null, offs, 2, 0, 8, 8, null, null, null, null) == 0
    assert lib.dflash2_topk_merge(null, null, offs, 2, 4, 8, 8, null, null, null, null) == 1
    bad = (ctypes.c_int64 * 2)(0, -1)
    p8 = ctypes.c_void_p(64)
    assert lib.dflash2_topk_merge(p8, p8, bad, 2, 4, 8, 8, p8, p8, null, null) == 1
    # d2t: a table exists exactly when the draft vocab is smaller than the target
    assert lib.dflash2_d2t_remap(null, null, 4, 100, 200, null, null, null) == 1
    assert lib.dflash2_d2t_remap(null, ctypes.c_void_p(64), 4, 200, 100, null, null, null) == 1
    assert lib.dflash2_d2t_remap(null, null, 0, 201, 200, null, null, null) == 0


def test_workspace_sizes_are_host_arithmetic(lib):
    rec = lib.dflash2_unary_topk_workspace_size(480, 151936, 16, 1)
    mn = lib.dflash2_unary_topk_workspace_min(480, 151936, 16, 1)
    assert rec > mn > 0
    # fp32: no workspace needed; the recommended one splits the vocab over CTAs
    assert lib.dflash2_unary_topk_workspace_min(7, 4096, 8, 0) == 0
    assert lib.dflash2_unary_topk_workspace_size(7, 4096, 8, 0) == 16 * 7 * 8 * 12
    assert lib.dflash2_unary_topk_workspace_size(480, 4096, 8, 0) == 0  # one chunk per row
    # launch counts: fp32 is one kernel on any device, zero rows queue nothing,
    # a rejected dtype answers -1 (bf16 needs the device's SM count)
    assert lib.dflash2_unary_topk_launches(7, 4096, 8, ctypes.c_float(1.0), 0) == 2  # chunks
    assert lib.dflash2_unary_topk_launches(480, 4096, 8, ctypes.c_float(1.0), 0) == 1
    assert lib.dflash2_unary_topk_launches(0, 4096, 8, ctypes.c_float(1.0), 1) == 0
    assert lib.dflash2_unary_topk_launches(7, 4096, 8, ctypes.c_float(1.0), 3) == -1
    assert lib.dflash2_unary_topk_launches(7, 4096, 129, ctypes.c_float(1.0), 0) == -1
    walk = lib.dflash2_selector_walk_workspace_size(32, 15, 4096, 64, 16, 1)
    assert walk >= 32 * 15 * 64 * 4 + 32 * 15 * 16 * (16 + 3) * 4   # partials + the lattice
    # top_k above the lattice mode's 32 needs the partials only
    assert lib.dflash2_selector_walk_workspace_size(32, 15, 4096, 64, 64, 1) < walk


def test_noalloc_walk_checks_arguments_before_its_scratch(lib):
    """dflash2_selector_walk_noalloc gives an invalid shape the status the
    workspace walk gives it, before comparing the shape's scratch need with
    its fixed array; an empty batch touches no device state."""
    null = None

    def call(batch, slots, hidden, rank, top_k, dtype, table_rows=1000):
        return lib.dflash2_selector_walk_noalloc(
            null, null, null, null, table_rows, null, null, null, null, null, null, batch, slots,
            hidden, rank, top_k, dtype, null, null, null, null, null)

    assert call(4096, 15, 4096, 512, 16, 1) == 1      # rank above 256: INVALID_ARG, not WORKSPACE
    assert call(4096, 15, 4096, 64, 200, 1) == 1      # top_k above 128
    assert call(4096, 15, 4096, 60, 16, 1) == 1       # bf16 rank not a multiple of 8
    assert call(8, 15, 4096, 64, 16, 7) == 2          # dtype
    assert call(8, 15, 4096, 64, 16, 1, table_rows=0) == 1
    assert call(0, 15, 4096, 64, 16, 1) == 0          # nothing to do
    assert call(1024, 15, 4096, 256, 16, 1) == 4      # beyond the 4 MiB array: WORKSPACE

"""Thin ctypes binding of libdflash2.so (declared in include/dflash2.h).

Argument marshalling only: each function checks shapes and dtypes of torch
CUDA tensors, passes their data pointers and the current CUDA stream to the
C entry point of the same name, and raises :class:`Dflash2Error` on a
non-OK status.  Every step of the hot path runs in the library's kernels;
there is no fallback.  If the shared library is missing the first call
raises: build it with ``python -c "import __graft_entry__ as g; g.build()"``.

PyTorch provides device memory and streams only.  Workspaces are caller-owned
device buffers; the helpers here allocate them with torch when not given.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdflash2.so")
_lock = threading.Lock()
_lib = None

OK = 0
F32, BF16 = 0, 1
DEVERR_ID_RANGE = 0x1
DEVERR_TIMEOUT = 0x2
DEVERR_SHORT = 0x4
DEVINFO_TOPK_FALLBACK = 0x100
ABI_VERSION = 9

# Every symbol include/dflash2.h declares.
EXPORTS = (
    "dflash2_status_string", "dflash2_abi_version", "dflash2_grouped_conv",
    "dflash2_unary_topk_workspace_size", "dflash2_unary_topk_workspace_min",
    "dflash2_unary_topk", "dflash2_selector_walk_workspace_size", "dflash2_selector_walk",
    "dflash2_d2t_remap", "dflash2_selector_walk_noalloc", "dflash2_philox_uniforms",
    "dflash2_conv_prepare", "dflash2_conv_finish", "dflash2_verify_workspace_size",
    "dflash2_verify", "dflash2_selector_project", "dflash2_selector_walk_projected",
    "dflash2_unary_topk_launches", "dflash2_topk_merge", "dflash2_quantize_rows_e4m3",
    "dflash2_unary_topk_fp8_workspace_size", "dflash2_unary_topk_fp8",
    "dflash2_quantize_rows_nvfp4", "dflash2_unary_topk_nvfp4_workspace_size",
    "dflash2_unary_topk_nvfp4", "dflash2_nvfp4_scale_tiles_size", "dflash2_nvfp4_tile_scales",
)
NOALLOC_SCRATCH_BYTES = 4 << 20


class Dflash2Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = library().dflash2_status_string(status).decode()
        super().__init__(f"{fn}: {msg} (status {status})")


def library():
    """Load libdflash2.so once and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: the CUDA extension is not built "
                "(run `python -c \"import __graft_entry__ as g; g.build()\"`)")
        lib = ctypes.CDLL(_LIB_PATH)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                ctypes.c_float, ctypes.c_size_t)
        lib.dflash2_status_string.argtypes = [i32]
        lib.dflash2_status_string.restype = ctypes.c_char_p
        lib.dflash2_abi_version.argtypes = []
        lib.dflash2_abi_version.restype = i32
        lib.dflash2_grouped_conv.argtypes = [P, P, P, i64, P, i64, i32, i32, i32, i32, i32, P]
        lib.dflash2_grouped_conv.restype = i32
        lib.dflash2_unary_topk_workspace_size.argtypes = [i64, i64, i32, i32]
        lib.dflash2_unary_topk_workspace_size.restype = sz
        lib.dflash2_unary_topk_workspace_min.argtypes = [i64, i64, i32, i32]
        lib.dflash2_unary_topk_workspace_min.restype = sz
        lib.dflash2_unary_topk.argtypes = [P, P, i64, i32, i64, i64, f32, f32, i32, i32, P, P, P,
                                           sz, P, P]
        lib.dflash2_unary_topk.restype = i32
        lib.dflash2_selector_walk_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.dflash2_selector_walk_workspace_size.restype = sz
        lib.dflash2_selector_walk.argtypes = [P, P, P, P, i64, P, P, P, P, P, P, i32, i32, i32,
                                              i32, i32, i32, P, P, P, P, sz, P, P]
        lib.dflash2_selector_walk.restype = i32
        lib.dflash2_d2t_remap.argtypes = [P, P, i64, i64, i64, P, P, P]
        lib.dflash2_d2t_remap.restype = i32
        lib.dflash2_selector_walk_noalloc.argtypes = [P, P, P, P, i64, P, P, P, P, P, P, i32, i32,
                                                      i32, i32, i32, i32, P, P, P, P, P]
        lib.dflash2_selector_walk_noalloc.restype = i32
        lib.dflash2_philox_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint64, P, i64, P, P]
        lib.dflash2_philox_uniforms.restype = i32
        lib.dflash2_conv_prepare.argtypes = [P, P, P, i64, i32, i32, i32, i32, i32, P, P, P, P]
        lib.dflash2_conv_prepare.restype = i32
        lib.dflash2_conv_finish.argtypes = [P, P, P, i64, i32, i32, i32, i32, i32, P, P]
        lib.dflash2_conv_finish.restype = i32
        lib.dflash2_verify_workspace_size.argtypes = [i32, i32, i64]
        lib.dflash2_verify_workspace_size.restype = sz
        lib.dflash2_verify.argtypes = [P, i64, P, P, P, P, P, P, i32, i32, i32, i32, P, P, P, sz,
                                       P, P]
        lib.dflash2_verify.restype = i32
        lib.dflash2_selector_project.argtypes = [P, P, i32, i32, i32, i32, i32, i32, P, sz, P, P]
        lib.dflash2_selector_project.restype = i32
        lib.dflash2_selector_walk_projected.argtypes = [P, P, i64, P, P, P, P, P, P, i32, i32, i32,
                                                        i32, i32, i32, P, P, P, P, sz, P, P]
        lib.dflash2_selector_walk_projected.restype = i32
        lib.dflash2_quantize_rows_e4m3.argtypes = [P, i64, i32, i32, P, P, P]
        lib.dflash2_quantize_rows_e4m3.restype = i32
        lib.dflash2_unary_topk_fp8_workspace_size.argtypes = [i64, i32, i64, i32]
        lib.dflash2_unary_topk_fp8_workspace_size.restype = sz
        lib.dflash2_unary_topk_fp8.argtypes = [P, i32, P, P, i64, i32, i64, i64, f32, f32, i32, P,
                                               P, P, sz, P, P]
        lib.dflash2_unary_topk_fp8.restype = i32
        lib.dflash2_quantize_rows_nvfp4.argtypes = [P, i64, i32, i32, P, P, P, P]
        lib.dflash2_quantize_rows_nvfp4.restype = i32
        lib.dflash2_unary_topk_nvfp4_workspace_size.argtypes = [i64, i32, i64, i32]
        lib.dflash2_unary_topk_nvfp4_workspace_size.restype = sz
        lib.dflash2_unary_topk_nvfp4.argtypes = [P, i32, P, P, f32, i64, i32, i64, i64, f32, f32,
                                                 i32, P, P, P, sz, P, P]
        lib.dflash2_unary_topk_nvfp4.restype = i32
        lib.dflash2_nvfp4_scale_tiles_size.argtypes = [i64, i32]
        lib.dflash2_nvfp4_scale_tiles_size.restype = sz
        lib.dflash2_nvfp4_tile_scales.argtypes = [P, i64, i32, P, P]
        lib.dflash2_nvfp4_tile_scales.restype = i32
        lib.dflash2_topk_merge.argtypes = [P, P, P, i32, i64, i32, i32, P, P, P, P]
        lib.dflash2_topk_merge.restype = i32
        lib.dflash2_unary_topk_launches.argtypes = [i64, i64, i32, f32, i32]
        lib.dflash2_unary_topk_launches.restype = i32
        if lib.dflash2_abi_version() != ABI_VERSION:
            raise RuntimeError("libdflash2.so ABI version mismatch; rebuild it")
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != OK:
        raise Dflash2Error(fn, status)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}: fp32 or bf16 only")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# ---- entry points -----------------------------------------------------------------

def grouped_conv(x, base, delta, block_size: int, group_size: int, taps: int, out=None,
                 delta_row_stride: int | None = None, stream=None):
    """dflash2_grouped_conv: x [n, hidden], base [taps, hidden], delta rows of
    [taps, hidden/group_size] (row stride delta_row_stride elements)."""
    n, hidden = x.shape
    for t, nm in ((x, "x"), (base, "base"), (delta, "delta")):
        _need(t, nm, x.dtype)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", x.dtype, x.shape)
    groups = hidden // group_size
    if delta_row_stride is None:
        delta_row_stride = taps * groups
    if delta.numel() < (n - 1) * delta_row_stride + taps * groups if n else False:
        raise ValueError("delta is too small for n rows at this row stride")
    _check("dflash2_grouped_conv", library().dflash2_grouped_conv(
        _ptr(x), _ptr(base), _ptr(delta), delta_row_stride, _ptr(out), n, hidden, group_size,
        taps, block_size, _dtype_code(x), _stream(stream)))
    return out


def unary_topk_workspace_size(rows: int, draft_vocab: int, top_k: int, dtype_code: int) -> int:
    return int(library().dflash2_unary_topk_workspace_size(rows, draft_vocab, top_k, dtype_code))


def unary_topk_workspace_min(rows: int, draft_vocab: int, top_k: int, dtype_code: int) -> int:
    return int(library().dflash2_unary_topk_workspace_min(rows, draft_vocab, top_k, dtype_code))


def unary_topk(h, lm_head, target_vocab: int, mult: float, cap: float, top_k: int,
               cand_ids=None, cand_u=None, workspace=None, err=None, stream=None):
    """dflash2_unary_topk: top_k (ids, u) per row of h against lm_head."""
    rows, hidden = h.shape
    draft_vocab = lm_head.shape[0]
    _need(h, "h")
    _need(lm_head, "lm_head", h.dtype)
    code = _dtype_code(h)
    dev = h.device
    if cand_ids is None:
        cand_ids = torch.empty((rows, top_k), dtype=torch.int64, device=dev)
    if cand_u is None:
        cand_u = torch.empty((rows, top_k), dtype=torch.float32, device=dev)
    _need(cand_ids, "cand_ids", torch.int64)
    _need(cand_u, "cand_u", torch.float32)
    if workspace is None:
        workspace = torch.empty(max(1, unary_topk_workspace_size(rows, draft_vocab, top_k, code)),
                                dtype=torch.uint8, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    _check("dflash2_unary_topk", library().dflash2_unary_topk(
        _ptr(h), _ptr(lm_head), rows, hidden, draft_vocab, target_vocab, float(mult),
        float(cap), top_k, code, _ptr(cand_ids), _ptr(cand_u), _ptr(workspace),
        workspace.numel(), _ptr(err), _stream(stream)))
    return cand_ids, cand_u, err


def quantize_rows_e4m3(x, q=None, scale=None, stream=None):
    """dflash2_quantize_rows_e4m3: per-row E4M3 codes (uint8) and scales of x."""
    rows, cols = x.shape
    _need(x, "x")
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check("dflash2_quantize_rows_e4m3", library().dflash2_quantize_rows_e4m3(
        _ptr(x), rows, cols, _dtype_code(x), _ptr(q), _ptr(scale), _stream(stream)))
    return q, scale


def unary_topk_fp8_workspace_size(rows: int, hidden: int, draft_vocab: int, top_k: int) -> int:
    return int(library().dflash2_unary_topk_fp8_workspace_size(rows, hidden, draft_vocab, top_k))


def unary_topk_fp8(h, lm_head_q, w_scale, target_vocab: int, mult: float, cap: float, top_k: int,
                   cand_ids=None, cand_u=None, workspace=None, err=None, stream=None):
    """dflash2_unary_topk_fp8: top_k (ids, u) per row of h against an E4M3 head
    (lm_head_q uint8 codes [draft_vocab, hidden], w_scale float [draft_vocab])."""
    rows, hidden = h.shape
    draft_vocab = lm_head_q.shape[0]
    _need(h, "h")
    _need(lm_head_q, "lm_head_q", torch.uint8, (draft_vocab, hidden))
    _need(w_scale, "w_scale", torch.float32, (draft_vocab,))
    dev = h.device
    if cand_ids is None:
        cand_ids = torch.empty((rows, top_k), dtype=torch.int64, device=dev)
    if cand_u is None:
        cand_u = torch.empty((rows, top_k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, unary_topk_fp8_workspace_size(rows, hidden, draft_vocab,
                                                                     top_k)),
                                dtype=torch.uint8, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    _check("dflash2_unary_topk_fp8", library().dflash2_unary_topk_fp8(
        _ptr(h), _dtype_code(h), _ptr(lm_head_q), _ptr(w_scale), rows, hidden, draft_vocab,
        target_vocab, float(mult), float(cap), top_k, _ptr(cand_ids), _ptr(cand_u),
        _ptr(workspace), workspace.numel(), _ptr(err), _stream(stream)))
    return cand_ids, cand_u, err


def quantize_rows_nvfp4(x, codes=None, scales=None, g=None, stream=None):
    """dflash2_quantize_rows_nvfp4: per-row NVFP4 codes (uint8, two per byte),
    E4M3 block scales (uint8, one per 16 elements) and fp32 second-level
    scales of x."""
    rows, cols = x.shape
    _need(x, "x")
    dev = x.device
    if codes is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev)
    if g is None:
        g = torch.empty(rows, dtype=torch.float32, device=dev)
    _check("dflash2_quantize_rows_nvfp4", library().dflash2_quantize_rows_nvfp4(
        _ptr(x), rows, cols, _dtype_code(x), _ptr(codes), _ptr(scales), _ptr(g),
        _stream(stream)))
    return codes, scales, g


def nvfp4_tile_scales(scales, hidden: int, tiles=None, stream=None):
    """dflash2_nvfp4_tile_scales: the scale tiles of row-major E4M3 block
    scales [rows, hidden / 16] (uint8), as the NVFP4 GEMM reads them."""
    rows = scales.shape[0]
    _need(scales, "scales", torch.uint8, (rows, hidden // 16))
    if tiles is None:
        tiles = torch.empty(max(1, int(library().dflash2_nvfp4_scale_tiles_size(rows, hidden))),
                            dtype=torch.uint8, device=scales.device)
    _check("dflash2_nvfp4_tile_scales", library().dflash2_nvfp4_tile_scales(
        _ptr(scales), rows, hidden, _ptr(tiles), _stream(stream)))
    return tiles


def unary_topk_nvfp4_workspace_size(rows: int, hidden: int, draft_vocab: int, top_k: int) -> int:
    return int(library().dflash2_unary_topk_nvfp4_workspace_size(rows, hidden, draft_vocab,
                                                                 top_k))


def unary_topk_nvfp4(h, lm_head_q, w_scale_tiles, w_global: float, target_vocab: int, mult: float,
                     cap: float, top_k: int, cand_ids=None, cand_u=None, workspace=None, err=None,
                     stream=None):
    """dflash2_unary_topk_nvfp4: top_k (ids, u) per row of h against an NVFP4
    head (lm_head_q uint8 [draft_vocab, hidden / 2] codes, w_scale_tiles its
    E4M3 block scales as nvfp4_tile_scales returns them, w_global its fp32
    scale)."""
    rows, hidden = h.shape
    draft_vocab = lm_head_q.shape[0]
    _need(h, "h")
    _need(lm_head_q, "lm_head_q", torch.uint8, (draft_vocab, hidden // 2))
    _need(w_scale_tiles, "w_scale_tiles", torch.uint8)
    need = int(library().dflash2_nvfp4_scale_tiles_size(draft_vocab, hidden))
    if w_scale_tiles.numel() < need:
        raise ValueError(f"w_scale_tiles: uint8 scale tiles of {need} bytes expected")
    dev = h.device
    if cand_ids is None:
        cand_ids = torch.empty((rows, top_k), dtype=torch.int64, device=dev)
    if cand_u is None:
        cand_u = torch.empty((rows, top_k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, unary_topk_nvfp4_workspace_size(rows, hidden, draft_vocab,
                                                                       top_k)),
                                dtype=torch.uint8, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    _check("dflash2_unary_topk_nvfp4", library().dflash2_unary_topk_nvfp4(
        _ptr(h), _dtype_code(h), _ptr(lm_head_q), _ptr(w_scale_tiles), float(w_global), rows, hidden,
        draft_vocab, target_vocab, float(mult), float(cap), top_k, _ptr(cand_ids), _ptr(cand_u),
        _ptr(workspace), workspace.numel(), _ptr(err), _stream(stream)))
    return cand_ids, cand_u, err


def topk_merge(ids, u, id_offsets, k_out: int, out_ids=None, out_u=None, err=None, stream=None):
    """dflash2_topk_merge: the k_out best (u, global id) per row over shard
    lists ids / u [shards, rows, k_in] (shard-local ids; u = -inf absent)."""
    shards, rows, k_in = ids.shape
    _need(ids, "ids", torch.int64)
    _need(u, "u", torch.float32, tuple(ids.shape))
    offs = [int(o) for o in id_offsets]
    if len(offs) != shards:
        raise ValueError("one id offset per shard")
    dev = ids.device
    if out_ids is None:
        out_ids = torch.empty((rows, k_out), dtype=torch.int64, device=dev)
    if out_u is None:
        out_u = torch.empty((rows, k_out), dtype=torch.float32, device=dev)
    _need(out_ids, "out_ids", torch.int64, (rows, k_out))
    _need(out_u, "out_u", torch.float32, (rows, k_out))
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    host_offs = (ctypes.c_int64 * shards)(*offs)
    _check("dflash2_topk_merge", library().dflash2_topk_merge(
        _ptr(ids), _ptr(u), ctypes.cast(host_offs, ctypes.c_void_p), shards, rows, k_in, k_out,
        _ptr(out_ids), _ptr(out_u), _ptr(err), _stream(stream)))
    return out_ids, out_u, err


def vocab_shard(draft_vocab: int, target_vocab: int, shards: int, s: int):
    """Shard s of `shards` near-equal slices of the lm_head rows: (first id,
    rows in the slice, ids of the slice below target_vocab)."""
    if not 0 <= s < shards:
        raise ValueError("shard index out of range")
    per = -(-draft_vocab // shards)
    first = min(s * per, draft_vocab)
    n = min(per, draft_vocab - first)
    return first, n, max(0, min(n, target_vocab - first))


def shard_topk(h, lm_head_slice, first: int, target_vocab: int, mult: float, cap: float,
               top_k: int, workspace=None, err=None, stream=None):
    """This shard's part of a vocab-sharded unary top-K: dflash2_unary_topk over
    its lm_head rows, as a [rows, top_k] list with shard-local ids.  A slice
    with fewer than top_k ids below target_vocab pads its list with u = -inf
    (absent for the merge)."""
    rows = h.shape[0]
    n = lm_head_slice.shape[0]
    local_target = max(0, min(n, target_vocab - first))
    k_here = min(top_k, local_target)
    if k_here == top_k:
        ids, u, _ = unary_topk(h, lm_head_slice, local_target, mult, cap, top_k,
                               workspace=workspace, err=err, stream=stream)
        return ids, u
    s = torch.cuda.current_stream(h.device) if stream is None else stream
    with torch.cuda.stream(s):
        ids = torch.zeros((rows, top_k), dtype=torch.int64, device=h.device)
        u = torch.full((rows, top_k), float("-inf"), dtype=torch.float32, device=h.device)
        if k_here > 0 and rows > 0:
            i2, u2, _ = unary_topk(h, lm_head_slice, local_target, mult, cap, k_here,
                                   workspace=workspace, err=err, stream=s)
            ids[:, :k_here] = i2
            u[:, :k_here] = u2
    return ids, u


def gather_shard_lists(ids, u, group=None):
    """The exchange of a vocab-sharded top-K: every rank's [rows, K] list,
    all-gathered into [world, rows, K] (rank order = shard order)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    all_ids = [torch.empty_like(ids) for _ in range(world)]
    all_u = [torch.empty_like(u) for _ in range(world)]
    dist.all_gather(all_ids, ids.contiguous(), group=group)
    dist.all_gather(all_u, u.contiguous(), group=group)
    return torch.stack(all_ids), torch.stack(all_u)


def unary_topk_vocab_sharded(h, lm_head_slice, draft_vocab: int, target_vocab: int, mult: float,
                             cap: float, top_k: int, group=None, err=None, stream=None):
    """Vocab-sharded unary top-K over a process group: this rank holds lm_head
    rows vocab_shard(draft_vocab, target_vocab, world, rank); the shard's
    list, one all-gather and dflash2_topk_merge give every rank the unsharded
    result (the same ids and u as dflash2_unary_topk over the whole lm_head)."""
    import torch.distributed as dist
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    first, n, _ = vocab_shard(draft_vocab, target_vocab, world, rank)
    if lm_head_slice.shape[0] != n:
        raise ValueError(f"rank {rank} holds {lm_head_slice.shape[0]} lm_head rows, expected {n}")
    ids, u = shard_topk(h, lm_head_slice, first, target_vocab, mult, cap, top_k, err=err,
                        stream=stream)
    all_ids, all_u = gather_shard_lists(ids, u, group)
    offsets = [vocab_shard(draft_vocab, target_vocab, world, s)[0] for s in range(world)]
    return topk_merge(all_ids, all_u, offsets, top_k, err=err, stream=stream)


def selector_walk_workspace_size(batch: int, slots: int, hidden: int, rank: int, top_k: int,
                                 dtype_code: int) -> int:
    return int(library().dflash2_selector_walk_workspace_size(batch, slots, hidden, rank, top_k,
                                                              dtype_code))


def selector_walk(h, proj, A, B, anchor_ids, cand_ids, cand_u, temperatures, greedy, uniforms,
                  tokens=None, q=None, path_scores=None, workspace=None, err=None,
                  with_path_scores: bool = False, stream=None):
    """dflash2_selector_walk over [batch, slots, top_k] candidates."""
    batch, slots, top_k = cand_ids.shape
    hidden = h.shape[-1]
    rank = proj.shape[0]
    code = _dtype_code(h)
    dev = h.device
    for t, nm in ((h, "h"), (proj, "proj"), (A, "A"), (B, "B")):
        _need(t, nm, h.dtype)
    _need(anchor_ids, "anchor_ids", torch.int64, (batch,))
    _need(cand_ids, "cand_ids", torch.int64)
    _need(cand_u, "cand_u", torch.float32, (batch, slots, top_k))
    _need(temperatures, "temperatures", torch.float32, (batch,))
    _need(greedy, "greedy", torch.uint8, (batch,))
    _need(uniforms, "uniforms", torch.float32, (batch, slots))
    if A.shape != B.shape or A.shape[1] != rank:
        raise ValueError("A and B must both be [table_rows, rank]")
    if tokens is None:
        tokens = torch.empty((batch, slots), dtype=torch.int64, device=dev)
    if q is None:
        q = torch.empty((batch, slots, top_k), dtype=torch.float32, device=dev)
    if path_scores is None and with_path_scores:
        path_scores = torch.empty((batch, slots, top_k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(
            max(1, selector_walk_workspace_size(batch, slots, hidden, rank, top_k, code)),
            dtype=torch.uint8, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    _check("dflash2_selector_walk", library().dflash2_selector_walk(
        _ptr(h), _ptr(proj), _ptr(A), _ptr(B), A.shape[0], _ptr(anchor_ids), _ptr(cand_ids),
        _ptr(cand_u), _ptr(temperatures), _ptr(greedy), _ptr(uniforms), batch, slots, hidden,
        rank, top_k, code, _ptr(tokens), _ptr(q), _ptr(path_scores), _ptr(workspace),
        workspace.numel(), _ptr(err), _stream(stream)))
    return tokens, q, path_scores, err


def selector_project(h, proj, batch: int, slots: int, top_k: int, workspace, err=None,
                     stream=None):
    """dflash2_selector_project: the projection partials of g = h . proj^T into
    `workspace` (a selector_walk workspace for the same shapes), for a later
    selector_walk_projected call ordered after it."""
    hidden = h.shape[-1]
    rank = proj.shape[0]
    code = _dtype_code(h)
    for t, nm in ((h, "h"), (proj, "proj")):
        _need(t, nm, h.dtype)
    if h.numel() != batch * slots * hidden:
        raise ValueError("h must hold batch * slots rows of hidden")
    _need(workspace, "workspace", torch.uint8)
    _check("dflash2_selector_project", library().dflash2_selector_project(
        _ptr(h), _ptr(proj), batch, slots, hidden, rank, top_k, code, _ptr(workspace),
        workspace.numel(), _ptr(err), _stream(stream)))
    return workspace


def selector_walk_projected(A, B, anchor_ids, cand_ids, cand_u, temperatures, greedy, uniforms,
                            hidden: int, workspace, tokens=None, q=None, path_scores=None,
                            err=None, with_path_scores: bool = False, stream=None):
    """dflash2_selector_walk_projected: the edges and the walk from the
    projection a selector_project call left in `workspace`."""
    batch, slots, top_k = cand_ids.shape
    rank = A.shape[1]
    code = _dtype_code(A)
    dev = A.device
    _need(A, "A")
    _need(B, "B", A.dtype)
    _need(anchor_ids, "anchor_ids", torch.int64, (batch,))
    _need(cand_ids, "cand_ids", torch.int64)
    _need(cand_u, "cand_u", torch.float32, (batch, slots, top_k))
    _need(temperatures, "temperatures", torch.float32, (batch,))
    _need(greedy, "greedy", torch.uint8, (batch,))
    _need(uniforms, "uniforms", torch.float32, (batch, slots))
    _need(workspace, "workspace", torch.uint8)
    if A.shape != B.shape:
        raise ValueError("A and B must both be [table_rows, rank]")
    if tokens is None:
        tokens = torch.empty((batch, slots), dtype=torch.int64, device=dev)
    if q is None:
        q = torch.empty((batch, slots, top_k), dtype=torch.float32, device=dev)
    if path_scores is None and with_path_scores:
        path_scores = torch.empty((batch, slots, top_k), dtype=torch.float32, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    _check("dflash2_selector_walk_projected", library().dflash2_selector_walk_projected(
        _ptr(A), _ptr(B), A.shape[0], _ptr(anchor_ids), _ptr(cand_ids), _ptr(cand_u),
        _ptr(temperatures), _ptr(greedy), _ptr(uniforms), batch, slots, hidden, rank, top_k, code,
        _ptr(tokens), _ptr(q), _ptr(path_scores), _ptr(workspace), workspace.numel(), _ptr(err),
        _stream(stream)))
    return tokens, q, path_scores, err


def selector_walk_noalloc(h, proj, A, B, anchor_ids, cand_ids, cand_u, temperatures, greedy,
                          uniforms, tokens=None, q=None, path_scores=None, err=None,
                          with_path_scores: bool = False, stream=None):
    """dflash2_selector_walk_noalloc: the selector walk with the library's own
    fixed 4 MiB scratch instead of a workspace, for callers that cannot hand
    over device memory at call time.  Calls that overlap on the GPU share that
    scratch and race; shapes needing more scratch raise Dflash2Error."""
    batch, slots, top_k = cand_ids.shape
    for t, nm in ((h, "h"), (proj, "proj"), (A, "A"), (B, "B")):
        _need(t, nm, h.dtype)
    _need(anchor_ids, "anchor_ids", torch.int64, (batch,))
    _need(cand_ids, "cand_ids", torch.int64)
    _need(cand_u, "cand_u", torch.float32, (batch, slots, top_k))
    _need(temperatures, "temperatures", torch.float32, (batch,))
    _need(greedy, "greedy", torch.uint8, (batch,))
    _need(uniforms, "uniforms", torch.float32, (batch, slots))
    dev = h.device
    if tokens is None:
        tokens = torch.empty((batch, slots), dtype=torch.int64, device=dev)
    if q is None:
        q = torch.empty((batch, slots, top_k), dtype=torch.float32, device=dev)
    if path_scores is None and with_path_scores:
        path_scores = torch.empty((batch, slots, top_k), dtype=torch.float32, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    _check("dflash2_selector_walk_noalloc", library().dflash2_selector_walk_noalloc(
        _ptr(h), _ptr(proj), _ptr(A), _ptr(B), A.shape[0], _ptr(anchor_ids), _ptr(cand_ids),
        _ptr(cand_u), _ptr(temperatures), _ptr(greedy), _ptr(uniforms), batch, slots,
        h.shape[-1], proj.shape[0], top_k, _dtype_code(h), _ptr(tokens), _ptr(q),
        _ptr(path_scores), _ptr(err), _stream(stream)))
    return tokens, q, path_scores, err


def d2t_remap(draft_ids, d2t, draft_vocab: int, target_vocab: int, out=None, err=None,
              stream=None):
    """dflash2_d2t_remap: target = draft + d2t[draft] (identity when d2t is None)."""
    _need(draft_ids, "draft_ids", torch.int64)
    if d2t is not None:
        _need(d2t, "d2t", torch.int64, (draft_vocab,))
    if out is None:
        out = torch.empty_like(draft_ids)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=draft_ids.device)
    _check("dflash2_d2t_remap", library().dflash2_d2t_remap(
        _ptr(draft_ids), _ptr(d2t), draft_ids.numel(), draft_vocab, target_vocab, _ptr(out),
        _ptr(err), _stream(stream)))
    return out, err


def conv_prepare(x, w_kp, base2, block_size: int, group_size: int, taps: int, out=None,
                 coef=None, err=None, stream=None):
    """dflash2_conv_prepare: (conv of x with coefficient side 0, coef [n, 2, taps, groups])."""
    n, hidden = x.shape
    groups = hidden // group_size
    code = _dtype_code(x)
    _need(x, "x", x.dtype)
    _need(w_kp, "w_kp", x.dtype, (2 * taps * groups, hidden))
    _need(base2, "base2", x.dtype, (2, taps, hidden))
    if out is None:
        out = torch.empty_like(x)
    if coef is None:
        coef = torch.empty((n, 2, taps, groups), dtype=x.dtype, device=x.device)
    _need(coef, "coef", x.dtype, (n, 2, taps, groups))
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=x.device)
    _check("dflash2_conv_prepare", library().dflash2_conv_prepare(
        _ptr(x), _ptr(w_kp), _ptr(base2), n, hidden, group_size, taps, block_size, code,
        _ptr(out), _ptr(coef), _ptr(err), _stream(stream)))
    return out, coef, err


def conv_finish(y, coef, base2, block_size: int, group_size: int, taps: int, out=None,
                stream=None):
    """dflash2_conv_finish: conv of y with coefficient side 1 and base side 1."""
    n, hidden = y.shape
    groups = hidden // group_size
    code = _dtype_code(y)
    _need(y, "y", y.dtype)
    _need(coef, "coef", y.dtype, (n, 2, taps, groups))
    _need(base2, "base2", y.dtype, (2, taps, hidden))
    if out is None:
        out = torch.empty_like(y)
    _check("dflash2_conv_finish", library().dflash2_conv_finish(
        _ptr(y), _ptr(base2), _ptr(coef), n, hidden, group_size, taps, block_size, code,
        _ptr(out), _stream(stream)))
    return out


def verify(target_logits, temperatures, greedy, draft, cand, q, uniforms, accept_len=None,
           out_tokens=None, workspace=None, err=None, stream=None):
    """dflash2_verify: speculative-sampling verification of a proposed block.

    target_logits [B, S+1, V]; draft [B, S] and cand [B, S, K] are target ids."""
    b, s1, vocab = target_logits.shape
    slots = s1 - 1
    k = cand.shape[-1]
    code = _dtype_code(target_logits)
    _need(target_logits, "target_logits", target_logits.dtype)
    _need(temperatures, "temperatures", torch.float32, (b,))
    _need(greedy, "greedy", torch.uint8, (b,))
    _need(draft, "draft", torch.int64, (b, slots))
    _need(cand, "cand", torch.int64, (b, slots, k))
    _need(q, "q", torch.float32, (b, slots, k))
    _need(uniforms, "uniforms", torch.float32, (b, s1))
    dev = target_logits.device
    if accept_len is None:
        accept_len = torch.empty(b, dtype=torch.int64, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((b, s1), dtype=torch.int64, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, verify_workspace_size(b, slots, vocab)),
                                dtype=torch.uint8, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    _check("dflash2_verify", library().dflash2_verify(
        _ptr(target_logits), vocab, _ptr(temperatures), _ptr(greedy), _ptr(draft), _ptr(cand),
        _ptr(q), _ptr(uniforms), b, slots, k, code, _ptr(accept_len), _ptr(out_tokens),
        _ptr(workspace), workspace.numel(), _ptr(err), _stream(stream)))
    return accept_len, out_tokens, err


def verify_workspace_size(batch: int, slots: int, vocab: int) -> int:
    return int(library().dflash2_verify_workspace_size(batch, slots, vocab))


def philox_uniforms(seed: int, n: int, out=None, offset: int = 0, counter=None, device=None,
                    stream=None):
    """dflash2_philox_uniforms: n float32 uniforms in [0, 1) from Philox4x64-10.

    With ``counter`` (a 1-element int64 device tensor holding the uint64 bits),
    the base is read and advanced on the device, so a captured graph draws a
    fresh sequence at every replay."""
    if counter is not None:
        _need(counter, "counter", torch.int64, (1,))
        device = counter.device
    if out is None:
        if device is None:
            raise ValueError("philox_uniforms needs `out`, `counter` or `device`")
        out = torch.empty(int(n), dtype=torch.float32, device=device)
    else:
        _need(out, "out", torch.float32)
        if out.numel() < n:
            raise ValueError("out holds fewer than n elements")
    _check("dflash2_philox_uniforms", library().dflash2_philox_uniforms(
        int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _ptr(counter), int(n), _ptr(out),
        _stream(stream)))
    return out


# ---- host <-> device helpers (plumbing) ----------------------------------------------

def to_device(a: np.ndarray, device) -> torch.Tensor:
    """numpy -> torch on `device`; uint16 arrays are bf16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    """torch -> numpy; bf16 comes back as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


class ProposalBuffers:
    """Caller-owned outputs and workspaces of one proposal step (allocated once)."""

    def __init__(self, w, device):
        code = F32 if w.dtype == "f32" else BF16
        fdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        self.conv_out = torch.empty((w.n_tokens, w.hidden), dtype=fdt, device=device)
        self.cand_ids = torch.empty((w.rows, w.top_k), dtype=torch.int64, device=device)
        self.cand_u = torch.empty((w.rows, w.top_k), dtype=torch.float32, device=device)
        self.tokens = torch.empty((w.batch, w.slots), dtype=torch.int64, device=device)
        self.q = torch.empty((w.batch, w.slots, w.top_k), dtype=torch.float32, device=device)
        self.target_ids = torch.empty((w.batch, w.slots), dtype=torch.int64, device=device)
        self.uniforms = torch.empty((w.batch, w.slots), dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws_topk = torch.empty(max(1, unary_topk_workspace_size(w.rows, w.draft_vocab, w.top_k, code)),
                                   dtype=torch.uint8, device=device)
        self.ws_walk = torch.empty(max(1, selector_walk_workspace_size(w.batch, w.slots, w.hidden,
                                                                       w.rank, w.top_k, code)),
                                   dtype=torch.uint8, device=device)
        # the second stream of an overlapped step and the events that fork it
        # from, and join it back into, the caller's stream
        self.side_stream = torch.cuda.Stream(device=device)
        self.fork = torch.cuda.Event()
        self.join = torch.cuda.Event()


def proposal_step(w, t: dict, bufs: ProposalBuffers | None = None, stream=None,
                  rng=None, overlap: bool = True) -> dict:
    """One pass of the hot path: conv, unary candidates, selector walk, d2t remap.

    `t` holds the device tensors of synth.make(w) (bf16 tensors as torch.bfloat16).
    With ``rng = (seed, counter)`` the walk's uniforms are drawn on the device
    (dflash2_philox_uniforms, counter advanced on the device) instead of taken
    from ``t["uniforms"]``.  Returns the output tensors (no synchronisation).

    With ``overlap`` the work that needs only the step's inputs (the uniforms,
    the grouped conv and the selector projection) runs on a second stream,
    forked from and joined back into `stream` by events, beside the unary
    top-K; the walk waits for both.  The results are the same either way; the
    fork and join are captured into a CUDA graph like the launches."""
    dev = t["h"].device
    if bufs is None:
        bufs = ProposalBuffers(w, dev)
    main = torch.cuda.current_stream(dev) if stream is None else stream
    side = main
    if overlap:
        side = bufs.side_stream
        bufs.fork.record(main)
        side.wait_event(bufs.fork)
    uniforms = t.get("uniforms")
    if rng is not None:
        seed, counter = rng
        philox_uniforms(seed, w.rows, out=bufs.uniforms.view(-1), counter=counter, stream=side)
        uniforms = bufs.uniforms
    grouped_conv(t["x"], t["base"], t["delta"], w.block_size, w.group_size, w.taps,
                 out=bufs.conv_out, stream=side)
    selector_project(t["h"], t["proj"], w.batch, w.slots, w.top_k, bufs.ws_walk, err=bufs.err,
                     stream=side)
    unary_topk(t["h"], t["lm_head"], w.target_vocab, w.mult, w.cap, w.top_k,
               cand_ids=bufs.cand_ids, cand_u=bufs.cand_u, workspace=bufs.ws_topk, err=bufs.err,
               stream=main)
    if overlap:
        bufs.join.record(side)
        main.wait_event(bufs.join)
    selector_walk_projected(t["A"], t["B"], t["anchors"],
                            bufs.cand_ids.view(w.batch, w.slots, w.top_k),
                            bufs.cand_u.view(w.batch, w.slots, w.top_k), t["temperatures"],
                            t["greedy"], uniforms, w.hidden, bufs.ws_walk, tokens=bufs.tokens,
                            q=bufs.q, err=bufs.err, stream=main)
    d2t_remap(bufs.tokens, t.get("d2t"), w.draft_vocab, w.target_vocab, out=bufs.target_ids,
              err=bufs.err, stream=main)
    return dict(conv_out=bufs.conv_out, cand_ids=bufs.cand_ids, cand_u=bufs.cand_u,
                tokens=bufs.tokens, q=bufs.q, target_ids=bufs.target_ids, err=bufs.err,
                uniforms=uniforms)

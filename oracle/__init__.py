"""CPU oracle for the DFlash2 draft-proposal hot path — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
library never links, loads or calls it, and it imports nothing from the
product package: the two implementations share no code.

The arithmetic lives in ``oracle.c`` (plain C, double accumulation, one
rounding at each output).  This module compiles it with gcc on first use and
marshals numpy arrays through ctypes.  bf16 tensors travel as ``uint16`` bit
patterns.

Every function is pinned by ``tests/test_oracle_*.py`` against brute force,
closed forms, invariants or library special cases; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, no FP contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_round_bf16.argtypes = [f64]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_conv.argtypes = [P, P, P, i64, P, i64, i32, i32, i32, i32, i32]
            lib.oracle_conv.restype = ctypes.c_int
            lib.oracle_unary_rows.argtypes = [P, P, P, i64, i32, i64, i64, f64, f64, i32, P]
            lib.oracle_unary_rows.restype = None
            lib.oracle_topk.argtypes = [P, i64, i64, i32, P, P]
            lib.oracle_topk.restype = ctypes.c_int
            lib.oracle_project.argtypes = [P, P, i64, i32, i32, i32, P]
            lib.oracle_project.restype = None
            lib.oracle_lattice.argtypes = [P, P, P, i64, P, P, P, i32, i32, i32, i32, i32, P]
            lib.oracle_lattice.restype = i64
            lib.oracle_walk.argtypes = [P, P, P, P, P, i32, i32, i32, P, P, P]
            lib.oracle_walk.restype = None
            lib.oracle_d2t.argtypes = [P, P, i64, i64, i64, P]
            lib.oracle_d2t.restype = i64
            u64 = ctypes.c_uint64
            lib.oracle_philox4x64.argtypes = [P, P, P]
            lib.oracle_philox4x64.restype = None
            lib.oracle_philox_uniforms.argtypes = [u64, u64, i64, P]
            lib.oracle_philox_uniforms.restype = None
            lib.oracle_kernel_projection.argtypes = [P, P, i64, i32, i32, i32, P]
            lib.oracle_kernel_projection.restype = None
            lib.oracle_verify.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i64, i32, P, P]
            lib.oracle_verify.restype = i64
            lib.oracle_set_threads.argtypes = [i32]
            lib.oracle_set_threads.restype = i32
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = f64
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_quantize_rows_e4m3.argtypes = [P, i64, i32, i32, P, P]
            lib.oracle_quantize_rows_e4m3.restype = None
            lib.oracle_unary_rows_fp8.argtypes = [P, P, P, P, P, i64, i32, i64, i64, f64, f64, P]
            lib.oracle_unary_rows_fp8.restype = None
            lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_decode.restype = f64
            lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint8
            lib.oracle_quantize_nvfp4.argtypes = [P, i64, i32, i32, i32, P, P, P]
            lib.oracle_quantize_nvfp4.restype = None
            lib.oracle_unary_rows_nvfp4.argtypes = [P, P, P, P, P, ctypes.c_float, P, i64, i32,
                                                    i64, i64, f64, f64, P]
            lib.oracle_unary_rows_nvfp4.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _elem(a: np.ndarray):
    """Return (contiguous array, dtype code) for a float32 or bf16-bits array."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"oracle takes float32 or uint16 (bf16 bits), got {a.dtype}")


def _same(code, *arrays):
    for a in arrays:
        if _elem(a)[1] != code:
            raise TypeError("all floating inputs of one call must share a dtype")


def round_bf16(v: float) -> int:
    """Nearest bf16 bit pattern of a double, ties to even, one rounding."""
    return int(_load().oracle_round_bf16(float(v)))


def conv(x, base, delta, block_size: int, group_size: int, taps: int,
         delta_row_stride: int | None = None):
    """Grouped dynamic depthwise conv; returns out with x's dtype."""
    x, code = _elem(x)
    base, _ = _elem(base)
    delta, _ = _elem(delta)
    _same(code, base, delta)
    n, hidden = x.shape
    groups = hidden // group_size
    if delta_row_stride is None:
        delta_row_stride = taps * groups
    out = np.empty_like(x)
    rc = _load().oracle_conv(_ptr(x), _ptr(base), _ptr(delta), delta_row_stride,
                             _ptr(out), n, hidden, group_size, taps, block_size, code)
    if rc:
        raise ValueError("oracle_conv rejected its arguments")
    return out


def unary_rows(h, lm_head, target_vocab: int, mult: float, cap: float,
               rows=None) -> np.ndarray:
    """u (double) for the selected rows of h over the whole draft vocab."""
    h, code = _elem(h)
    lm_head, _ = _elem(lm_head)
    _same(code, lm_head)
    hidden = h.shape[1]
    vd = lm_head.shape[0]
    if rows is None:
        sel, n_sel = None, h.shape[0]
    else:
        sel = np.ascontiguousarray(rows, dtype=np.int64)
        n_sel = sel.shape[0]
    u = np.empty((n_sel, vd), dtype=np.float64)
    _load().oracle_unary_rows(_ptr(h), _ptr(lm_head), _ptr(sel), n_sel, hidden, vd,
                              target_vocab, float(mult), float(cap), code, _ptr(u))
    return u


def topk(u: np.ndarray, k: int):
    """Top-K (ids int64, values float32) per row of a double u matrix."""
    u = np.ascontiguousarray(u, dtype=np.float64)
    n, vd = u.shape
    ids = np.empty((n, k), dtype=np.int64)
    vals = np.empty((n, k), dtype=np.float32)
    if _load().oracle_topk(_ptr(u), n, vd, k, _ptr(ids), _ptr(vals)):
        raise ValueError("oracle_topk failed")
    return ids, vals


def project(h, proj) -> np.ndarray:
    """g = h . proj^T in double; proj is [rank, hidden]."""
    h, code = _elem(h)
    proj, _ = _elem(proj)
    _same(code, proj)
    rows, hidden = h.shape
    rank = proj.shape[0]
    g = np.empty((rows, rank), dtype=np.float64)
    _load().oracle_project(_ptr(h), _ptr(proj), rows, hidden, rank, code, _ptr(g))
    return g


def lattice(g, A, B, anchors, cand, cand_u):
    """Full [batch, slots, K, K] fp32 edge lattice and the out-of-range count."""
    g = np.ascontiguousarray(g, dtype=np.float64)
    A, code = _elem(A)
    B, _ = _elem(B)
    _same(code, B)
    cand = np.ascontiguousarray(cand, dtype=np.int64)
    batch, slots, k = cand.shape
    anchors = np.ascontiguousarray(anchors, dtype=np.int64)
    cand_u = np.ascontiguousarray(cand_u, dtype=np.float32)
    rank = A.shape[1]
    scores = np.empty((batch, slots, k, k), dtype=np.float32)
    errors = _load().oracle_lattice(_ptr(g), _ptr(A), _ptr(B), A.shape[0], _ptr(anchors),
                                    _ptr(cand), _ptr(cand_u), batch, slots, rank, k,
                                    code, _ptr(scores))
    return scores, int(errors)


def walk(scores, cand, uniforms, temperatures, greedy):
    """Walk a lattice; returns (tokens int64 [B,S], q float32 [B,S,K], index int32 [B,S])."""
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    cand = np.ascontiguousarray(cand, dtype=np.int64)
    batch, slots, k = cand.shape
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    temperatures = np.ascontiguousarray(temperatures, dtype=np.float32)
    greedy = np.ascontiguousarray(greedy, dtype=np.uint8)
    tokens = np.empty((batch, slots), dtype=np.int64)
    q = np.empty((batch, slots, k), dtype=np.float32)
    chosen = np.empty((batch, slots), dtype=np.int32)
    _load().oracle_walk(_ptr(scores), _ptr(cand), _ptr(uniforms), _ptr(temperatures),
                        _ptr(greedy), batch, slots, k, _ptr(tokens), _ptr(q), _ptr(chosen))
    return tokens, q, chosen


def d2t(draft_ids, table, draft_vocab: int, target_vocab: int):
    """Draft-to-target remap; returns (target ids, error count)."""
    ids = np.ascontiguousarray(draft_ids, dtype=np.int64)
    tbl = None if table is None else np.ascontiguousarray(table, dtype=np.int64)
    out = np.empty_like(ids)
    errors = _load().oracle_d2t(_ptr(ids), _ptr(tbl), ids.size, draft_vocab,
                                target_vocab, _ptr(out))
    return out, int(errors)


def selector(h, proj, A, B, anchors, cand, cand_u, uniforms, temperatures, greedy):
    """Projection, lattice and walk chained: the selector stage end to end."""
    batch, slots, _ = np.shape(cand)
    g = project(np.asarray(h).reshape(batch * slots, -1), proj)
    scores, errors = lattice(g, A, B, anchors, cand, cand_u)
    tokens, q, chosen = walk(scores, cand, uniforms, temperatures, greedy)
    return dict(g=g, scores=scores, errors=errors, tokens=tokens, q=q, chosen=chosen)


def philox4x64(counter, key) -> np.ndarray:
    """One Philox4x64-10 block: 4 counter words, 2 key words -> 4 uint64 words."""
    c = np.ascontiguousarray(counter, dtype=np.uint64)
    k = np.ascontiguousarray(key, dtype=np.uint64)
    if c.shape != (4,) or k.shape != (2,):
        raise ValueError("counter has 4 words, key 2")
    out = np.zeros(4, dtype=np.uint64)
    _load().oracle_philox4x64(_ptr(c), _ptr(k), _ptr(out))
    return out


def philox_uniforms(seed: int, base: int, n: int) -> np.ndarray:
    """n float32 uniforms in [0, 1): word i % 4 of the block at counter base + i // 4."""
    out = np.zeros(int(n), dtype=np.float32)
    if n:
        _load().oracle_philox_uniforms(int(seed) & (2**64 - 1), int(base) & (2**64 - 1), int(n),
                                       _ptr(out))
    return out


def kernel_projection(x, w_kp) -> np.ndarray:
    """coef[i, r] = sum_j x[i, j] w_kp[r, j], rounded once to x's dtype."""
    x, code = _elem(x)
    w_kp, _ = _elem(w_kp)
    _same(code, w_kp)
    n, hidden = x.shape
    r, h2 = w_kp.shape
    if h2 != hidden:
        raise ValueError("w_kp must be [out_features, hidden]")
    coef = np.empty((n, r), dtype=x.dtype)
    _load().oracle_kernel_projection(_ptr(x), _ptr(w_kp), n, hidden, r, code, _ptr(coef))
    return coef


def conv_prepare(x, w_kp, base2, block_size: int, group_size: int, taps: int):
    """DFlashGroupedConv.prepare: (conv of x with coefficient side 0, coef).

    base2 is base_kernel [2, taps, hidden]; coef is [n, 2, taps, groups] flat
    per token ([n, 2 * taps * groups])."""
    coef = kernel_projection(x, w_kp)
    groups = x.shape[1] // group_size
    out = conv(x, np.ascontiguousarray(base2[0]), coef, block_size, group_size, taps,
               delta_row_stride=2 * taps * groups)
    return out, coef


def conv_finish(y, coef, base2, block_size: int, group_size: int, taps: int):
    """DFlashGroupedConv.finish: conv of y with coefficient side 1 and base side 1."""
    groups = y.shape[1] // group_size
    side1 = np.ascontiguousarray(coef.reshape(coef.shape[0], -1)[:, taps * groups:])
    return conv(y, np.ascontiguousarray(base2[1]), side1, block_size, group_size, taps,
                delta_row_stride=taps * groups)


def verify(logits, temperatures, greedy, draft, cand, q, r):
    """Speculative-sampling verification of a proposed block.

    logits [B, S+1, V] (float32 or bf16 bits); temperatures [B] f32; greedy [B] u8;
    draft [B, S] and cand [B, S, K] target ids (int64); q [B, S, K] f32;
    r [B, S+1] f32 (r[:, s] accepts slot s, r[:, S] draws the emitted token).
    Returns (accept_len [B] int64, out_tokens [B, S+1] int64, errors)."""
    logits, code = _elem(logits)
    b, s1, vocab = logits.shape
    slots = s1 - 1
    draft = np.ascontiguousarray(draft, dtype=np.int64).reshape(b, slots)
    cand = np.ascontiguousarray(cand, dtype=np.int64)
    k = cand.shape[-1]
    cand = cand.reshape(b, slots, k)
    q = np.ascontiguousarray(q, dtype=np.float32).reshape(b, slots, k)
    r = np.ascontiguousarray(r, dtype=np.float32).reshape(b, s1)
    temperatures = np.ascontiguousarray(temperatures, dtype=np.float32)
    greedy = np.ascontiguousarray(greedy, dtype=np.uint8)
    acc = np.zeros(b, dtype=np.int64)
    out = np.zeros((b, s1), dtype=np.int64)
    errors = _load().oracle_verify(_ptr(logits), _ptr(temperatures), _ptr(greedy), _ptr(draft),
                                   _ptr(cand), _ptr(q), _ptr(r), b, slots, k, vocab, code,
                                   _ptr(acc), _ptr(out))
    return acc, out, int(errors)


def e4m3_decode(codes) -> np.ndarray:
    """Values (double) of E4M3 codes (uint8 array)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    lib = _load()
    return np.array([lib.oracle_e4m3_decode(int(b)) for b in c.reshape(-1)],
                    dtype=np.float64).reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (round to nearest even, saturating) of float32 values."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    lib = _load()
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in a.reshape(-1)],
                    dtype=np.uint8).reshape(a.shape)


def quantize_rows_e4m3(h):
    """Per-row E4M3 codes and dequantization scales (uint8 [rows, hidden],
    float32 [rows]) of a float32 or bf16-bits matrix."""
    h, code = _elem(h)
    rows, hidden = h.shape
    q = np.empty((rows, hidden), dtype=np.uint8)
    d = np.empty(rows, dtype=np.float32)
    _load().oracle_quantize_rows_e4m3(_ptr(h), rows, hidden, code, _ptr(q), _ptr(d))
    return q, d


def unary_rows_fp8(qh, dh, qw, sw, target_vocab: int, mult: float, cap: float,
                   rows=None) -> np.ndarray:
    """u (double) of the W8A8 logits for the selected rows over the whole vocab."""
    qh = np.ascontiguousarray(qh, dtype=np.uint8)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    dh = np.ascontiguousarray(dh, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    hidden = qh.shape[1]
    vd = qw.shape[0]
    if rows is None:
        sel, n_sel = None, qh.shape[0]
    else:
        sel = np.ascontiguousarray(rows, dtype=np.int64)
        n_sel = sel.shape[0]
    u = np.empty((n_sel, vd), dtype=np.float64)
    _load().oracle_unary_rows_fp8(_ptr(qh), _ptr(dh), _ptr(qw), _ptr(sw), _ptr(sel), n_sel,
                                  hidden, vd, target_vocab, float(mult), float(cap), _ptr(u))
    return u


def e2m1_decode(codes) -> np.ndarray:
    """Values (double) of E2M1 codes (the low 4 bits of a uint8 array)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    lib = _load()
    return np.array([lib.oracle_e2m1_decode(int(b) & 15) for b in c.reshape(-1)],
                    dtype=np.float64).reshape(c.shape)


def e2m1_encode(x) -> np.ndarray:
    """E2M1 codes (round to nearest even, saturating at 6) of float32 values."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    lib = _load()
    return np.array([lib.oracle_e2m1_encode(float(v)) for v in a.reshape(-1)],
                    dtype=np.uint8).reshape(a.shape)


def quantize_nvfp4(x, per_tensor: bool = False):
    """NVFP4 quantization of a float32 or bf16-bits matrix [rows, cols]
    (cols a multiple of 16): packed codes uint8 [rows, cols/2], E4M3 block
    scales uint8 [rows, cols/16], and the fp32 second-level scales (one per
    row, or one for the tensor)."""
    x, code = _elem(x)
    rows, cols = x.shape
    if cols % 16:
        raise ValueError("cols must be a multiple of 16")
    q = np.empty((rows, cols // 2), dtype=np.uint8)
    s = np.empty((rows, cols // 16), dtype=np.uint8)
    g = np.empty(1 if per_tensor else rows, dtype=np.float32)
    _load().oracle_quantize_nvfp4(_ptr(x), rows, cols, code, int(per_tensor), _ptr(q), _ptr(s),
                                  _ptr(g))
    return q, s, (g[0] if per_tensor else g)


def unary_rows_nvfp4(qh, sh, gh, qw, sw, gw: float, target_vocab: int, mult: float, cap: float,
                     rows=None) -> np.ndarray:
    """u (double) of the NVFP4 (W4A4) logits for the selected rows over the whole vocab."""
    qh = np.ascontiguousarray(qh, dtype=np.uint8)
    sh = np.ascontiguousarray(sh, dtype=np.uint8)
    gh = np.ascontiguousarray(gh, dtype=np.float32)
    qw = np.ascontiguousarray(qw, dtype=np.uint8)
    sw = np.ascontiguousarray(sw, dtype=np.uint8)
    hidden = qh.shape[1] * 2
    vd = qw.shape[0]
    if rows is None:
        sel, n_sel = None, qh.shape[0]
    else:
        sel = np.ascontiguousarray(rows, dtype=np.int64)
        n_sel = sel.shape[0]
    u = np.empty((n_sel, vd), dtype=np.float64)
    _load().oracle_unary_rows_nvfp4(_ptr(qh), _ptr(sh), _ptr(gh), _ptr(qw), _ptr(sw), float(gw),
                                    _ptr(sel), n_sel, hidden, vd, target_vocab, float(mult),
                                    float(cap), _ptr(u))
    return u


def set_threads(n: int = 0) -> int:
    """Set (n > 0) or ask (n <= 0) the oracle's OpenMP thread count; returns it."""
    return int(_load().oracle_set_threads(int(n)))

"""Seeded synthetic inputs for the DFlash2 draft-proposal hot path.

This module is the ONE thing the CUDA path and the CPU oracle share: it draws
random inputs and holds none of the method's arithmetic.  It imports neither
the CUDA binding nor the oracle.

Inputs are drawn with numpy's PCG64.  Each named part has its own stream,
``default_rng([seed, part_index])``, so a test can draw one part without
drawing (or changing) the others.  bf16 tensors are the fp32 draws rounded to
nearest-even; the oracle reads the same bf16 values as uint16 bit patterns.

The five named workloads restate the configurations the method is exercised
on (sizes in the docstring of :data:`CONFIGS`).  Weights are N(0, 0.02); the
conv input x is N(0, 0.02) for the tiny fp32 case and N(0, 1) for the bf16
cases; the proposal hidden states h are N(0, 1).  Sampling uses the even
batch rows as greedy rows and the odd rows as sampled rows for the "mixed"
workloads.  Synthetic draws stand in for the GSM8K runs that the DFlash2 PR
quotes for acceptance and speed-up: no dataset item is used.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

PARTS = ("x", "base", "delta", "h", "lm_head", "A", "B", "proj", "uniforms",
         "d2t", "anchors", "w_kp", "base2", "lm_head_fp8", "w_scale", "lm_head_nvfp4",
         "w_scales_nvfp4")


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    block_size: int
    hidden: int
    group_size: int
    taps: int
    draft_vocab: int
    target_vocab: int
    rank: int
    top_k: int
    dtype: str            # "f32" or "bf16"
    mult: float
    cap: float
    sampling: str         # "greedy", "mixed" (even rows greedy) or "sampled"
    temperature: float    # temperature of the sampled rows
    x_std: float = 1.0
    h_std: float = 1.0
    w_std: float = 0.02
    seed: int = 0x5EED

    @property
    def slots(self) -> int:           # proposals per request (block_size - 1)
        return self.block_size - 1

    @property
    def n_tokens(self) -> int:        # conv rows: every position of every block
        return self.batch * self.block_size

    @property
    def rows(self) -> int:            # proposal rows entering the lm_head
        return self.batch * self.slots

    @property
    def groups(self) -> int:
        return self.hidden // self.group_size

    @property
    def uses_d2t(self) -> bool:       # only a pruned draft vocab needs the table
        return self.draft_vocab < self.target_vocab

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


# 1 tiny fp32 | 2 Qwen3-8B-shaped bf16 | 3 padded vocab | 4 reduced vocab with a
# 12-position block | 5 large-batch, large-K stress.  Unstated fields of 3 and 4
# take taps 4 (3), group size 8 and the "not enabled" mult 1 / cap 0.
CONFIGS = [
    Workload("tiny-fp32", 1, 8, 256, 8, 4, 4096, 4096, 16, 8, "f32", 1.0, 0.0,
             "greedy", 1.0, x_std=0.02, seed=0x5EED + 0),
    Workload("qwen3-8b-bf16", 32, 16, 4096, 8, 4, 151936, 151936, 64, 16, "bf16",
             1.0, 30.0, "mixed", 0.7, seed=0x5EED + 1),
    Workload("padded-vocab-bf16", 64, 16, 4096, 8, 4, 201024, 200058, 64, 32,
             "bf16", 1.0, 0.0, "sampled", 1.0, seed=0x5EED + 2),
    Workload("reduced-vocab-bs12-bf16", 128, 12, 5120, 8, 6, 32768, 151936, 64, 16,
             "bf16", 1.0, 0.0, "mixed", 0.8, seed=0x5EED + 3),
    Workload("stress-bf16", 512, 16, 7168, 8, 4, 163840, 163840, 128, 64, "bf16",
             0.5, 30.0, "sampled", 0.6, seed=0x5EED + 4),
]
BY_NAME = {w.name: w for w in CONFIGS}


def rng(seed: int, part: str) -> np.random.Generator:
    return np.random.default_rng([int(seed), PARTS.index(part)])


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even); return the uint16 bits."""
    import torch  # torch's fp32 -> bf16 cast rounds to nearest-even
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def fp8_codes(a: np.ndarray) -> np.ndarray:
    """E4M3 (float8_e4m3fn) codes of float32 values within +-448, as uint8."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def normal(seed: int, part: str, shape, std: float, dtype: str) -> np.ndarray:
    a = rng(seed, part).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return to_bf16_bits(a) if dtype == "bf16" else a


def sampling_params(w: Workload):
    """Temperatures (f32 [B]) and greedy mask (u8 [B]).  Greedy rows get T=1."""
    greedy = np.zeros(w.batch, dtype=np.uint8)
    if w.sampling == "greedy":
        greedy[:] = 1
    elif w.sampling == "mixed":
        greedy[0::2] = 1
    elif w.sampling != "sampled":
        raise ValueError(w.sampling)
    temps = np.where(greedy == 1, np.float32(1.0), np.float32(w.temperature))
    return temps.astype(np.float32), greedy


def d2t_table(w: Workload, seed: int | None = None):
    """Offsets for a pruned draft vocab: a sorted random subset S of the target
    vocab with |S| = draft_vocab, stored as d2t[i] = S[i] - i (the offset form
    of vLLM's draft_id_to_target_id).  None when no table is needed."""
    if not w.uses_d2t:
        return None
    g = rng(w.seed if seed is None else seed, "d2t")
    subset = np.sort(g.choice(w.target_vocab, size=w.draft_vocab, replace=False))
    return (subset - np.arange(w.draft_vocab)).astype(np.int64)


DEFAULT_PARTS = PARTS[:11]  # the proposal step's inputs; w_kp / base2 feed the conv prepare,
                            # lm_head_fp8 / w_scale the FP8 head


def nvfp4_w_global(w: Workload) -> float:
    """The tensor scale of the synthetic NVFP4 head: uniform codes have an rms
    of about 3.2 and the block scales about 1, so the weights' rms is about
    w_std."""
    return float(w.w_std / 3.2)


def make(w: Workload, parts=DEFAULT_PARTS) -> dict:
    """Draw the requested parts of a workload.  Floating parts are float32 for
    "f32" workloads and uint16 bf16 bits for "bf16" workloads."""
    s, dt = w.seed, w.dtype
    out = {}
    for p in parts:
        if p == "x":
            out[p] = normal(s, p, (w.n_tokens, w.hidden), w.x_std, dt)
        elif p == "base":
            out[p] = normal(s, p, (w.taps, w.hidden), w.w_std, dt)
        elif p == "delta":
            out[p] = normal(s, p, (w.n_tokens, w.taps, w.groups), w.w_std, dt)
        elif p == "h":
            out[p] = normal(s, p, (w.rows, w.hidden), w.h_std, dt)
        elif p == "lm_head":
            out[p] = normal(s, p, (w.draft_vocab, w.hidden), w.w_std, dt)
        elif p in ("A", "B"):
            out[p] = normal(s, p, (w.draft_vocab, w.rank), w.w_std, dt)
        elif p == "proj":
            out[p] = normal(s, p, (w.rank, w.hidden), w.w_std, dt)
        elif p == "uniforms":
            out[p] = rng(s, p).random(size=(w.batch, w.slots), dtype=np.float32)
        elif p == "d2t":
            out[p] = d2t_table(w)
        elif p == "w_kp":     # kernel_projection weight [2 * taps * groups, hidden]
            out[p] = normal(s, p, (2 * w.taps * w.groups, w.hidden), w.w_std, dt)
        elif p == "base2":    # base_kernel of both conv sides [2, taps, hidden]
            out[p] = normal(s, p, (2, w.taps, w.hidden), w.w_std, dt)
        elif p == "lm_head_fp8":
            # an FP8 (E4M3) checkpoint of the head: codes of N(0, 64^2) draws
            # (torch's float8_e4m3fn conversion), about 3 sigma inside +-448
            out[p] = fp8_codes(rng(s, p).standard_normal(size=(w.draft_vocab, w.hidden),
                                                         dtype=np.float32) * np.float32(64.0))
        elif p == "w_scale":
            # per-row dequantization scales: scale * code ~ N(0, w_std^2)
            out[p] = (rng(s, p).uniform(0.5, 1.5, size=w.draft_vocab)
                      * (w.w_std / 64.0)).astype(np.float32)
        elif p == "lm_head_nvfp4":
            # an NVFP4 checkpoint of the head: uniformly drawn E2M1 code bytes
            # (two codes each) [draft_vocab, hidden / 2] ...
            out[p] = rng(s, p).integers(0, 256, size=(w.draft_vocab, w.hidden // 2),
                                        dtype=np.uint8)
        elif p == "w_scales_nvfp4":
            # ... and their E4M3 block scales, one per 16 elements, in [0.5, 1.5]
            out[p] = fp8_codes(rng(s, p).uniform(0.5, 1.5, size=(w.draft_vocab, w.hidden // 16))
                               .astype(np.float32))
        elif p == "anchors":
            hi = min(w.draft_vocab, w.target_vocab)
            out[p] = rng(s, p).integers(0, hi, size=w.batch, dtype=np.int64)
        else:
            raise KeyError(p)
    if "uniforms" in parts:
        out["temperatures"], out["greedy"] = sampling_params(w)
    return out

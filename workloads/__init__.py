"""Seeded synthetic inputs for the QSA indexer, shared by tests and bench.

This module holds none of the indexer's arithmetic: it draws random numbers
(numpy PCG64 ``default_rng(seed)``), rounds them to the activation type with
torch's own casts, and builds the caller-supplied cos/sin table.  Both the CUDA
path and the CPU oracle receive the bit patterns it returns.

Workloads follow the shapes, distributions and structure the "Qsa Indexer
Kernels" page describes for indexQk [B, S, 640], the raw gammas wQ/wK [128],
contextLengths [B] with padding rows, and the FP32 cos/sin table
[maxPositions, 64] (cos in columns 0..31, sin in 32..63).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

ROW_WIDTH = 640
HEAD_DIM = 128
NUM_Q_HEADS = 4
ROPE_THETA = 1.0e6
RMS_EPS = 1.0e-6
GAMMA_STD = 0.1

TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}
NAN_BITS = {"bf16": 0x7FC0, "fp16": 0x7E00}


def round_to_t(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 samples to T with torch's cast; returns uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(TORCH_DTYPES[dtype])
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def cos_sin_table(max_positions: int, theta: float = ROPE_THETA) -> np.ndarray:
    """FP32 [max_positions, 64]: angle(p, i) = p * theta^(-2i/64) for i < 32, built in float64."""
    inv_freq = theta ** (-np.arange(0, 64, 2, dtype=np.float64) / 64.0)
    ang = np.arange(max_positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def gamma(rng: np.random.Generator, dtype: str, std: float = GAMMA_STD) -> np.ndarray:
    """Raw checkpoint gamma [128] ~ N(0, std^2) (the kernels add the +1)."""
    return round_to_t(rng.normal(0.0, std, HEAD_DIM), dtype)


def index_qk(rng: np.random.Generator, B: int, S: int, dtype: str,
             outlier_frac: float = 0.0, outlier_scale: float = 50.0,
             context_lengths: np.ndarray | None = None, nan_padding: bool = False) -> np.ndarray:
    """indexQk [B, S, 640] ~ N(0, 1) as T bits.

    ``outlier_frac``: each row is scaled by ``outlier_scale`` with this Bernoulli
    probability (all 640 columns).  ``nan_padding``: rows t >= contextLengths[b]
    are filled with NaN in every column.
    """
    x = rng.standard_normal((B, S, ROW_WIDTH), dtype=np.float32)
    if outlier_frac > 0.0:
        pick = rng.random((B, S)) < outlier_frac
        x[pick] *= np.float32(outlier_scale)
    bits = round_to_t(x, dtype)
    if nan_padding:
        assert context_lengths is not None
        t = np.arange(S)[None, :]
        pad = t >= np.asarray(context_lengths)[:, None]
        bits[pad] = NAN_BITS[dtype]
    return bits


@dataclass
class Workload:
    """One synthetic problem instance (all arrays on the host)."""
    name: str
    dtype: str
    B: int
    S: int
    index_qk: np.ndarray          # uint16 [B, S, 640]
    w_q: np.ndarray               # uint16 [128]
    w_k: np.ndarray               # uint16 [128]
    cos_sin: np.ndarray           # float32 [maxPositions, 64]
    context_lengths: np.ndarray   # int32 [B]
    eps: float = RMS_EPS
    meta: dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return (self.S + 3) // 4


def tiny(dtype: str = "bf16", seed: int = 0) -> Workload:
    """B=1, S=64, ctx=[50]; wQ/wK ~ N(0, 0.1^2); cos/sin [64, 64], theta 1e6."""
    rng = np.random.default_rng(seed)
    B, S = 1, 64
    ctx = np.array([50], np.int32)
    iq = index_qk(rng, B, S, dtype)
    return Workload("tiny B=1 S=64", dtype, B, S, iq, gamma(rng, dtype), gamma(rng, dtype),
                    cos_sin_table(S), ctx)


def batched(dtype: str = "bf16", seed: int = 1) -> Workload:
    """B=4, S=2048; 1% outlier rows x50; ctx ~ U{1..2048}; NaN padding rows."""
    rng = np.random.default_rng(seed)
    B, S = 4, 2048
    ctx = rng.integers(1, S + 1, size=B).astype(np.int32)
    iq = index_qk(rng, B, S, dtype, outlier_frac=0.01, context_lengths=ctx, nan_padding=True)
    return Workload(f"batched prefill B=4 S=2048 {dtype}", dtype, B, S, iq, gamma(rng, dtype),
                    gamma(rng, dtype), cos_sin_table(S), ctx)


def long_prefill(dtype: str = "bf16", seed: int = 2) -> Workload:
    """B=1, S=32768, ctx=[32765] (the last block is incomplete)."""
    rng = np.random.default_rng(seed)
    B, S = 1, 32768
    ctx = np.array([32765], np.int32)
    iq = index_qk(rng, B, S, dtype)
    return Workload("long prefill B=1 S=32768", dtype, B, S, iq, gamma(rng, dtype),
                    gamma(rng, dtype), cos_sin_table(S), ctx)


def decode_parity(dtype: str = "bf16", seed: int = 3) -> Workload:
    """B=16, S=8192, ctx ~ U{4..8192}; sub-range tiles are drawn by ``subrange_tiles``."""
    rng = np.random.default_rng(seed)
    B, S = 16, 8192
    ctx = rng.integers(4, S + 1, size=B).astype(np.int32)
    iq = index_qk(rng, B, S, dtype, context_lengths=ctx, nan_padding=True)
    wl = Workload("decode-parity B=16 S=8192", dtype, B, S, iq, gamma(rng, dtype),
                  gamma(rng, dtype), cos_sin_table(S), ctx)
    wl.meta["rng_state"] = rng.bit_generator.state
    return wl


def subrange_tiles(seed: int, past_len: int, num_blocks: int, max_tile: int = 64):
    """[blockBegin, blockEnd) tiles of U{1..max_tile} blocks covering
    [max(past_len/4 - 2, 0), num_blocks) in order."""
    rng = np.random.default_rng([seed, past_len])
    g = max(past_len // 4 - 2, 0)
    tiles = []
    while g < num_blocks:
        n = int(rng.integers(1, max_tile + 1))
        tiles.append((g, min(g + n, num_blocks)))
        g += n
    return tiles


def scoring(dtype: str = "bf16", seed: int = 4, B: int = 8, S: int = 16384,
            full_context: bool = True) -> Workload:
    """B=8, S=16384, indexQk ~ N(0,1).  ctx = S for every sequence (full_context), or
    ctx ~ U{1..S} for the padded correctness variant."""
    rng = np.random.default_rng(seed)
    if full_context:
        ctx = np.full(B, S, np.int32)
    else:
        ctx = rng.integers(1, S + 1, size=B).astype(np.int32)
    iq = index_qk(rng, B, S, dtype, context_lengths=ctx, nan_padding=not full_context)
    tag = "full context" if full_context else "padded"
    return Workload(f"scoring B={B} S={S} {dtype} {tag}", dtype, B, S, iq, gamma(rng, dtype),
                    gamma(rng, dtype), cos_sin_table(S), ctx)


def custom(B: int, S: int, ctx, dtype: str = "bf16", seed: int = 0,
           nan_padding: bool = True, outlier_frac: float = 0.0,
           max_positions: int | None = None) -> Workload:
    """Arbitrary shapes for edge-case tests."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, np.int32).reshape(B)
    iq = index_qk(rng, B, S, dtype, outlier_frac=outlier_frac, context_lengths=ctx,
                  nan_padding=nan_padding)
    return Workload(f"custom B={B} S={S}", dtype, B, S, iq, gamma(rng, dtype), gamma(rng, dtype),
                    cos_sin_table(max_positions or max(S, 4)), ctx)

"""Seeded synthetic inputs for video-DiT attention.

This module only draws numbers: it holds none of the attention, RoPE or merge arithmetic.
Both the CUDA path (through the binding) and the fp64 CPU oracle are fed from it, so the
two sides always see the same bf16 bits.

Recipe: numpy ``Generator(PCG64(seed))``; standard normal fp32 values rounded to bf16
(round to nearest even); token rows beyond the valid length ("pad rows") hold N(0, 10^2)
garbage, also rounded to bf16, which a correct kernel must never let into a result.
Everything is returned as fp32 arrays whose values are exactly representable in bf16, in
the contiguous BSHD layout [batch, sequence, heads, head_dim].
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np

TILE = 128          # rows per attention tile; sequences are padded to a multiple of it
PAD_SIGMA = 10.0    # standard deviation of the garbage written into pad rows


def padded_len(n: int, multiple: int = TILE) -> int:
    """Smallest multiple of `multiple` that is >= n."""
    return ((n + multiple - 1) // multiple) * multiple


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 value (ties to even), returned as fp32. Inputs must be finite
    (then the 32-bit integer sums below cannot overflow)."""
    x = np.array(x, dtype=np.float32, copy=True, order="C")
    u = x.view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    u += np.uint32(0x7FFF)
    u += lsb
    u &= np.uint32(0xFFFF0000)
    return x


def _normal(rng: np.random.Generator, shape, sigma: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return bf16_round(x)


def _fill_pad_rows(rng, x: np.ndarray, valid) -> None:
    """Overwrites rows >= valid[b] of x [B, S, H, D] with N(0, PAD_SIGMA^2) garbage."""
    B, S = x.shape[:2]
    vals = [int(valid)] * B if np.ndim(valid) == 0 else [int(v) for v in valid]
    for b in range(B):
        if vals[b] < S:
            x[b, vals[b]:] = _normal(rng, x[b, vals[b]:].shape, PAD_SIGMA)


@dataclass
class AttnCase:
    """One attention problem: shapes, valid lengths and rotary geometry.

    rope: None, "1d" (positions pos_offset + row) or "3d" (grid (T, Hh, W), row-major).
    kv_valid may be an int or one int per batch (cross-attention).
    """
    name: str
    B: int
    H: int
    D: int
    Sq: int
    Skv: int
    q_valid: int
    kv_valid: object
    rope: Optional[str] = None
    grid: Optional[Tuple[int, int, int]] = None
    q_pos_offset: int = 0
    k_pos_offset: int = 0
    seed: int = 0
    theta: float = 10000.0
    axis_dims: Tuple[int, int, int] = (44, 42, 42)

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))


def make_qkv(case: AttnCase):
    """Draws q [B, Sq, H, D], k and v [B, Skv, H, D] for `case` (pad rows hold garbage)."""
    rng = np.random.Generator(np.random.PCG64(case.seed))
    q = _normal(rng, (case.B, case.Sq, case.H, case.D))
    k = _normal(rng, (case.B, case.Skv, case.H, case.D))
    v = _normal(rng, (case.B, case.Skv, case.H, case.D))
    _fill_pad_rows(rng, q, case.q_valid)
    _fill_pad_rows(rng, k, case.kv_valid)
    _fill_pad_rows(rng, v, case.kv_valid)
    return q, k, v


def draw_kv_lengths(seed: int, B: int, max_len: int) -> List[int]:
    """Per-batch valid text lengths, uniform on [1, max_len] inclusive."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in rng.integers(1, max_len + 1, size=B)]


# ---------------------------------------------------------------------------
# The five workloads (video token grids shaped like the pages' Wan / LTX runs)
# ---------------------------------------------------------------------------
def tiny_case() -> AttnCase:
    """B=1, H=2, D=64; 300 valid tokens padded to 384; 1-D positions 0..299."""
    return AttnCase("tiny", B=1, H=2, D=64, Sq=384, Skv=384, q_valid=300, kv_valid=300,
                    rope="1d", seed=1000)


def wan480_case() -> AttnCase:
    """Wan 480x832x9: latent grid 3 x 30 x 52 = 4680 tokens padded to 4736; H=40, D=128."""
    return AttnCase("wan480x832x9", B=1, H=40, D=128, Sq=4736, Skv=4736, q_valid=4680,
                    kv_valid=4680, rope="3d", grid=(3, 30, 52), seed=1001)


def cross_case() -> AttnCase:
    """Short-KV cross-attention: B=2, H=40, D=128; 4680 video queries (padded to 4736)
    against 512 text slots with per-batch valid lengths uniform on [1, 512]; no RoPE."""
    kv = draw_kv_lengths(1002 + 7919, 2, 512)
    return AttnCase("cross_shortkv", B=2, H=40, D=128, Sq=4736, Skv=512, q_valid=4680,
                    kv_valid=kv, rope=None, seed=1002)


def wan720_case() -> AttnCase:
    """Wan 720p 81 frames: grid 21 x 45 x 80 = 75,600 tokens padded to 75,648; H=40, D=128."""
    return AttnCase("wan720p81f", B=1, H=40, D=128, Sq=75648, Skv=75648, q_valid=75600,
                    kv_valid=75600, rope="3d", grid=(21, 45, 80), seed=1004)


@dataclass
class ShardedCase:
    """Queries attending key shards: shard s holds keys at global positions
    offsets[s] .. offsets[s] + valid[s] - 1, padded to a whole number of tiles."""
    name: str
    B: int
    H: int
    D: int
    Sq: int
    q_valid: int
    shard_valid: Tuple[int, ...]
    seed: int
    theta: float = 10000.0
    shard_pad: List[int] = field(default_factory=list)

    def __post_init__(self):
        self.shard_pad = [padded_len(n) for n in self.shard_valid]

    @property
    def offsets(self) -> List[int]:
        out, acc = [], 0
        for n in self.shard_valid:
            out.append(acc)
            acc += n
        return out

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))


def sharded_case() -> ShardedCase:
    """B=1, H=32, D=128; 1024 queries over 37,800 keys in 4 contiguous shards
    (9472 / 9472 / 9472 / 9384 valid); 1-D RoPE at global positions."""
    return ShardedCase("sharded_keys", B=1, H=32, D=128, Sq=1024, q_valid=1024,
                       shard_valid=(9472, 9472, 9472, 9384), seed=1003)


def make_sharded(case: ShardedCase):
    """Returns q [B, Sq, H, D] and a list of (k_s, v_s) [B, shard_pad[s], H, D]."""
    rng = np.random.Generator(np.random.PCG64(case.seed))
    q = _normal(rng, (case.B, case.Sq, case.H, case.D))
    _fill_pad_rows(rng, q, case.q_valid)
    shards = []
    for n, n_pad in zip(case.shard_valid, case.shard_pad):
        k = _normal(rng, (case.B, n_pad, case.H, case.D))
        v = _normal(rng, (case.B, n_pad, case.H, case.D))
        _fill_pad_rows(rng, k, n)
        _fill_pad_rows(rng, v, n)
        shards.append((k, v))
    return q, shards


def sample_rows(n_valid: int, n_total: int, count: int, seed: int) -> np.ndarray:
    """Query rows for sampled checks: the first and last valid rows, rows on both sides of
    every 128-row tile boundary near the ends, the first pad row, and `count` random rows."""
    rng = np.random.Generator(np.random.PCG64(seed))
    fixed = {0, 1, TILE - 1, TILE, TILE + 1, n_valid - 1, min(n_valid, n_total - 1),
             n_total - 1, (n_valid // TILE) * TILE - 1, (n_valid // TILE) * TILE}
    picks = set(int(x) for x in rng.integers(0, n_valid, size=count))
    rows = sorted(r for r in fixed | picks if 0 <= r < n_total)
    return np.asarray(rows, dtype=np.int64)


def make_norm_weights(D: int, seed: int) -> np.ndarray:
    """Synthetic per-head RMSNorm weights [D] fp32: 1 + 0.1 * N(0, 1) (no trained weights)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)

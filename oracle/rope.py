"""Split-halves rotary position embedding, fp64 (oracle; test infrastructure only).

Sources (the web pages this method is taken from):

* Difflet PR #153, "Wan padding + split RoPE" commit notes: the rotary embedding is applied
  to channel pairs (i, i + D/2) of each head -- "a slice and a concat" -- after one channel
  permutation [0, 2, ..., 1, 3, ...] of q and k, which leaves q . k unchanged. Pad rows get
  the identity rotation (angle 0).
* Wan-style 3-D positions: head_dim split 44/42/42 channels for (t, h, w), theta = 10000 per
  axis; tokens of a T x H x W latent grid in row-major order (t slowest).

Readings taken where the pages are silent:

* rotation sign: x'[i] = x[i] cos a - x[i+D/2] sin a, x'[i+D/2] = x[i] sin a + x[i+D/2] cos a,
  i.e. (x[i] + j x[i+D/2]) * exp(+j a).
* 3-D: pair i (channels i and i + D/2) for i < 22 rotates with the t coordinate using
  frequency theta^(-2 i / 44); pairs 22..42 with h using theta^(-2 (i-22) / 42); pairs 43..63
  with w using theta^(-2 (i-43) / 42). This is what the whole-head permutation does to an
  interleaved layout whose complex pairs are ordered (t, h, w).
"""
from __future__ import annotations

import numpy as np


def rope_angles_1d(positions, head_dim: int, theta: float = 10000.0) -> np.ndarray:
    """Angles [n, D/2]: a[p, i] = position_p * theta^(-2 i / D)."""
    half = head_dim // 2
    pos = np.asarray(positions, dtype=np.float64).reshape(-1, 1)
    i = np.arange(half, dtype=np.float64).reshape(1, -1)
    freq = np.power(float(theta), -2.0 * i / head_dim)
    return pos * freq


def grid_positions(T: int, Hh: int, W: int) -> np.ndarray:
    """(t, h, w) of each token of a T x Hh x W grid in row-major order (t slowest): [T*Hh*W, 3]."""
    t, h, w = np.meshgrid(np.arange(T), np.arange(Hh), np.arange(W), indexing="ij")
    return np.stack([t.ravel(), h.ravel(), w.ravel()], axis=1)


def rope_angles_3d(T: int, Hh: int, W: int, head_dim: int = 128,
                   axis_dims=(44, 42, 42), theta: float = 10000.0) -> np.ndarray:
    """Angles [T*Hh*W, D/2] for 3-D split-halves RoPE.

    The D/2 pairs are cut into consecutive blocks of axis_dims[a] / 2 pairs, one block per
    axis (t, h, w); pair j of axis a's block has frequency theta^(-2 j / axis_dims[a]).
    """
    assert sum(axis_dims) == head_dim and all(d % 2 == 0 for d in axis_dims)
    pos = grid_positions(T, Hh, W).astype(np.float64)
    blocks = []
    for a, d_axis in enumerate(axis_dims):
        j = np.arange(d_axis // 2, dtype=np.float64).reshape(1, -1)
        freq = np.power(float(theta), -2.0 * j / d_axis)
        blocks.append(pos[:, a:a + 1] * freq)
    return np.concatenate(blocks, axis=1)


def pad_angles(angles: np.ndarray, total_rows: int) -> np.ndarray:
    """Appends zero angles (identity rotation) for pad rows up to total_rows."""
    n, half = angles.shape
    assert total_rows >= n
    out = np.zeros((total_rows, half), dtype=np.float64)
    out[:n] = angles
    return out


def rope_split_halves(x: np.ndarray, angles: np.ndarray) -> np.ndarray:
    """Rotates x [B, S, H, D] (any float dtype, computed in fp64) by angles [S, D/2].

    Channel i is paired with channel i + D/2:
      y[i]       = x[i] cos a_i - x[i+D/2] sin a_i
      y[i + D/2] = x[i] sin a_i + x[i+D/2] cos a_i
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    assert angles.shape == (x.shape[1], half)
    c = np.cos(angles)[None, :, None, :]
    s = np.sin(angles)[None, :, None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)

"""Pure-Python per-query attention (oracle pin; test infrastructure only).

An independent restatement of the same definition as ``oracle.attention`` -- split-halves
rotary embedding, scores over the valid keys only, natural-log LSE -- written with Python
floats, ``math`` and ``math.fsum`` and no numpy, so that a slip in the vectorised oracle
(a transposed operand, a wrong pairing, a dropped term) shows up as a disagreement on tiny
inputs. Sources: Difflet PR #153 (split-halves rotation, pad keys dropped), maxdiffusion
PR #491 (real KV length as the ragged tail), mstar PR #376 (natural-log LSE).
"""
from __future__ import annotations

import math


def frequencies_1d(head_dim, theta=10000.0):
    return [theta ** (-(2.0 * i) / head_dim) for i in range(head_dim // 2)]


def angles_1d(position, head_dim, theta=10000.0):
    return [position * f for f in frequencies_1d(head_dim, theta)]


def angles_3d(t, h, w, head_dim=128, axis_dims=(44, 42, 42), theta=10000.0):
    out = []
    for coord, d_axis in zip((t, h, w), axis_dims):
        for j in range(d_axis // 2):
            out.append(coord * theta ** (-(2.0 * j) / d_axis))
    assert len(out) == head_dim // 2
    return out


def token_to_thw(n, Hh, W):
    """Row-major (t slowest) token index -> (t, h, w)."""
    return n // (Hh * W), (n // W) % Hh, n % W


def rotate(x, angles):
    half = len(x) // 2
    first = [x[i] * math.cos(angles[i]) - x[i + half] * math.sin(angles[i]) for i in range(half)]
    second = [x[i] * math.sin(angles[i]) + x[i + half] * math.cos(angles[i]) for i in range(half)]
    return first + second


def attend_one(q_row, keys, values, scale, q_angles=None, key_angles=None):
    """q_row: list[D]; keys, values: list of list[D] (valid keys only).

    Returns (o: list[D], lse: float); with no keys, ([0.0]*D, -inf).
    """
    D = len(q_row)
    if not keys:
        return [0.0] * D, float("-inf")
    q = rotate(q_row, q_angles) if q_angles is not None else list(q_row)
    scores = []
    for j, key in enumerate(keys):
        kk = rotate(key, key_angles[j]) if key_angles is not None else list(key)
        scores.append(scale * math.fsum(q[d] * kk[d] for d in range(D)))
    m = max(scores)
    lse = m + math.log(math.fsum(math.exp(s - m) for s in scores))
    weights = [math.exp(s - lse) for s in scores]
    o = [math.fsum(weights[j] * values[j][d] for j in range(len(keys))) for d in range(D)]
    return o, lse

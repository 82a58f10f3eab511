"""Pins for the oracle's per-head q/k RMSNorm (CPU only).

Checked against what the definition fixes rather than against the oracle's own formula:
hand-derived values, closed forms for constant rows, unit RMS of the output, scale
invariance, per-head independence, a pure-Python restatement, the composition with RoPE and
attention in the pages' order (norm, then rotation), and planted mistakes that each fail one
of these checks.
"""
import math

import numpy as np
import pytest

from oracle.attention import attention
from oracle.qknorm import rms_norm_heads
from oracle.rope import rope_angles_1d, rope_split_halves


def _rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def test_hand_derived_values():
    # x = (3, 4): mean of squares 12.5; w = (1, 2).
    y = rms_norm_heads(np.array([3.0, 4.0]), np.array([1.0, 2.0]), eps=0.0)
    assert np.allclose(y, [3.0 / math.sqrt(12.5), 8.0 / math.sqrt(12.5)], rtol=0, atol=1e-15)
    # eps adds to the mean of squares: 12.5 + 0.5 = 13.
    y = rms_norm_heads(np.array([3.0, 4.0]), np.array([1.0, 2.0]), eps=0.5)
    assert np.allclose(y, [3.0 / math.sqrt(13.0), 8.0 / math.sqrt(13.0)], rtol=0, atol=1e-15)


@pytest.mark.parametrize("c", [-2.0, 0.25, 7.0])
def test_constant_row_closed_form(c):
    D, eps = 64, 1e-6
    w = 1.0 + 0.1 * _rand((D,), 3)
    y = rms_norm_heads(np.full((2, 5, 3, D), c), w, eps)
    expect = c / math.sqrt(c * c + eps) * w
    assert np.max(np.abs(y - expect)) < 1e-14


def test_unit_rms_of_output():
    x = _rand((2, 9, 4, 128), 4) * 3.7
    y = rms_norm_heads(x, np.ones(128), eps=0.0)
    assert np.max(np.abs(np.mean(y * y, axis=-1) - 1.0)) < 1e-12


def test_weight_applied_after_normalisation():
    x = _rand((3, 7, 2, 64), 5)
    w = 0.5 + _rand((64,), 6) ** 2
    y = rms_norm_heads(x, w, eps=0.0)
    assert np.max(np.abs(np.mean((y / w) ** 2, axis=-1) - 1.0)) < 1e-12


def test_scale_invariance():
    x = _rand((2, 6, 3, 64), 7)
    w = 1.0 + 0.2 * _rand((64,), 8)
    y = rms_norm_heads(x, w, eps=0.0)
    assert np.max(np.abs(rms_norm_heads(5.5 * x, w, eps=0.0) - y)) < 1e-13
    assert np.max(np.abs(rms_norm_heads(-0.25 * x, w, eps=0.0) + y)) < 1e-13


def test_norm_is_per_head():
    x = _rand((1, 4, 3, 32), 9)
    w = np.ones(32)
    y = rms_norm_heads(x, w)
    x2 = x.copy()
    x2[:, :, 1, 5] += 10.0           # one channel of head 1
    y2 = rms_norm_heads(x2, w)
    assert np.array_equal(y2[:, :, 0], y[:, :, 0]) and np.array_equal(y2[:, :, 2], y[:, :, 2])
    assert np.all(np.abs(y2[:, :, 1] - y[:, :, 1]) > 0)   # every channel of head 1 moves


def test_pure_python_restatement():
    x = _rand((2, 3, 2, 16), 10)
    w = 1.0 + 0.3 * _rand((16,), 11)
    eps = 1e-6
    y = rms_norm_heads(x, w, eps)
    for b in range(2):
        for s in range(3):
            for h in range(2):
                row = [float(v) for v in x[b, s, h]]
                r = math.sqrt(math.fsum(v * v for v in row) / len(row) + eps)
                ref = [row[d] / r * float(w[d]) for d in range(16)]
                assert max(abs(a - c) for a, c in zip(y[b, s, h], ref)) < 1e-14


def test_attention_with_norm_is_attention_on_normalised_inputs():
    B, S, H, D = 1, 40, 2, 32
    q, k, v = _rand((B, S, H, D), 12), _rand((B, S, H, D), 13), _rand((B, S, H, D), 14)
    wq, wk = 1.0 + 0.2 * _rand((D,), 15), 1.0 + 0.2 * _rand((D,), 16)
    ang = rope_angles_1d(np.arange(S), D)
    O1, L1 = attention(q, k, v, 33, 37, 0.2, ang, ang, norm_q=wq, norm_k=wk)
    O2, L2 = attention(rms_norm_heads(q, wq), rms_norm_heads(k, wk), v, 33, 37, 0.2, ang, ang)
    assert np.max(np.abs(O1 - O2)) < 1e-12 and np.max(np.abs(L1[:, :33] - L2[:, :33])) < 1e-12


def test_norm_then_rotation_differs_from_rotation_then_norm():
    # With a non-uniform weight the order matters; the pages normalise before rotating.
    x = _rand((1, 16, 1, 32), 17)
    w = 0.3 + _rand((32,), 18) ** 2
    ang = rope_angles_1d(np.arange(16) + 50, 32)
    a = rope_split_halves(rms_norm_heads(x, w), ang)
    b = rms_norm_heads(rope_split_halves(x, ang), w)
    assert np.max(np.abs(a - b)) > 1e-2


# --- planted mistakes: each must fail one of the pins above ---------------------------------
def _over_heads(x, w, eps=1e-6):          # norm over the head axis instead of the channels
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-2, keepdims=True) + eps) * w


def _weight_inside(x, w, eps=1e-6):       # weight applied before the RMS
    xw = np.asarray(x, dtype=np.float64) * w
    return xw / np.sqrt(np.mean(xw * xw, axis=-1, keepdims=True) + eps)


def _no_eps(x, w, eps=1e-6):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) * w


def test_planted_mistakes_are_caught():
    # per-head independence catches the wrong axis
    x = _rand((1, 4, 3, 32), 9)
    x2 = x.copy()
    x2[:, :, 1, 5] += 10.0
    assert not np.array_equal(_over_heads(x2, np.ones(32))[:, :, 0], _over_heads(x, np.ones(32))[:, :, 0])
    # the weight-after-normalisation pin catches the weight inside the RMS
    x = _rand((3, 7, 2, 64), 5)
    w = 0.5 + _rand((64,), 6) ** 2
    assert np.max(np.abs(np.mean((_weight_inside(x, w, 0.0) / w) ** 2, axis=-1) - 1.0)) > 1e-3
    # the hand-derived eps value catches a dropped eps
    y = _no_eps(np.array([3.0, 4.0]), np.array([1.0, 2.0]), eps=0.5)
    assert not np.allclose(y, [3.0 / math.sqrt(13.0), 8.0 / math.sqrt(13.0)], rtol=0, atol=1e-6)

"""Pins for the oracle's split-halves RoPE (CPU only).

Each check is something the pages or the mathematics fix independently of the oracle's
own formula: the complex-multiply form, norm preservation, the identity at position 0 (and
for pad rows), the relative-position property, the Difflet page's statement that one channel
permutation [0, 2, ..., 1, 3, ...] of q and k turns interleaved rotary into split halves
without changing q . k, an independent pure-Python restatement, and hand-derived values.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import brute
from oracle.rope import (grid_positions, pad_angles, rope_angles_1d, rope_angles_3d,
                         rope_split_halves)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def complex_form_error(rope_fn, seed=1, D=64, S=37):
    """max |rope(x) - (x_i + j x_{i+D/2}) e^{j a}| over random x and angles."""
    x = _rand((2, S, 3, D), seed)
    ang = _rand((S, D // 2), seed + 1) * 7.0
    y = rope_fn(x, ang)
    z = (x[..., : D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * ang)[None, :, None, :]
    return max(np.abs(y[..., : D // 2] - z.real).max(), np.abs(y[..., D // 2:] - z.imag).max())


def test_complex_multiply_form():
    assert complex_form_error(rope_split_halves) < 1e-13


def test_pair_norms_preserved():
    x = _rand((1, 50, 4, 128), 3)
    ang = rope_angles_1d(np.arange(50) * 97, 128)
    y = rope_split_halves(x, ang)
    n0 = x[..., :64] ** 2 + x[..., 64:] ** 2
    n1 = y[..., :64] ** 2 + y[..., 64:] ** 2
    assert np.max(np.abs(n1 - n0) / n0) < 1e-12


def test_position_zero_and_pad_rows_are_identity():
    x = _rand((1, 20, 2, 64), 4)
    ang = pad_angles(rope_angles_1d(np.arange(10), 64), 20)
    y = rope_split_halves(x, ang)
    assert np.array_equal(y[:, 0], x[:, 0])          # position 0
    assert np.array_equal(y[:, 10:], x[:, 10:])      # pad rows: angle 0
    a3 = pad_angles(rope_angles_3d(2, 3, 4), 30)
    assert np.all(a3[0] == 0) and np.all(a3[24:] == 0)


@pytest.mark.parametrize("D", [64, 128])
def test_relative_position_property_1d(D):
    q = _rand((1, 1, 1, D), 5)
    k = _rand((1, 1, 1, D), 6)
    for m, n in [(0, 0), (3, 1), (1000, 37), (37, 1000), (37799, 12)]:
        lhs = np.sum(rope_split_halves(q, rope_angles_1d([m], D)) *
                     rope_split_halves(k, rope_angles_1d([n], D)))
        rhs = np.sum(rope_split_halves(q, rope_angles_1d([m - n], D)) * k)
        assert abs(lhs - rhs) < 1e-9 * max(1.0, abs(lhs))


def test_relative_position_property_3d():
    """q~ . k~ depends on the (t, h, w) difference only (each pair's angle is linear in one
    grid coordinate)."""
    T, Hh, W = 4, 5, 6
    ang = rope_angles_3d(T, Hh, W)
    pos = grid_positions(T, Hh, W)
    index = {tuple(p): n for n, p in enumerate(pos)}
    q = _rand((1, 1, 1, 128), 7)
    k = _rand((1, 1, 1, 128), 8)

    def dot(a, b):
        return np.sum(rope_split_halves(q, ang[[index[a]]]) * rope_split_halves(k, ang[[index[b]]]))

    assert abs(dot((1, 2, 3), (0, 1, 1)) - dot((3, 4, 5), (2, 3, 3))) < 1e-10
    assert abs(dot((2, 0, 5), (1, 4, 0)) - dot((3, 0, 5), (2, 4, 0))) < 1e-10
    assert abs(dot((0, 0, 0), (0, 0, 0)) - np.sum(q * k)) < 1e-12


def _interleaved_rope(x, ang):
    """Rotary in the interleaved layout: channel pairs (2i, 2i+1) rotated by ang[:, i]."""
    c = np.cos(ang)[None, :, None, :]
    s = np.sin(ang)[None, :, None, :]
    xe, xo = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = xe * c - xo * s
    y[..., 1::2] = xe * s + xo * c
    return y


@pytest.mark.parametrize("D", [64, 128])
def test_interleaved_equivalence_under_channel_permutation(D):
    """Difflet PR #153: permuting each head's channels to [0, 2, ..., 1, 3, ...] turns the
    interleaved rotary into split halves and leaves q . k unchanged."""
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])
    q = _rand((1, 9, 2, D), 9)
    k = _rand((1, 9, 2, D), 10)
    ang = rope_angles_1d(np.arange(9) * 13, D)
    qi, ki = _interleaved_rope(q, ang), _interleaved_rope(k, ang)
    qs, ks = rope_split_halves(q[..., perm], ang), rope_split_halves(k[..., perm], ang)
    assert np.max(np.abs(qi[..., perm] - qs)) < 1e-12
    s_inter = np.einsum("bqhd,bkhd->bhqk", qi, ki)
    s_split = np.einsum("bqhd,bkhd->bhqk", qs, ks)
    assert np.max(np.abs(s_inter - s_split)) < 1e-10


def test_matches_pure_python_restatement_1d_and_3d():
    x = _rand((1, 24, 1, 128), 11)
    a1 = rope_angles_1d(np.arange(24) + 500, 128)
    y1 = rope_split_halves(x, a1)
    a3 = rope_angles_3d(2, 3, 4)
    y3 = rope_split_halves(x, a3)
    for n in range(24):
        row = list(x[0, n, 0])
        r1 = brute.rotate(row, brute.angles_1d(n + 500, 128))
        t, h, w = brute.token_to_thw(n, 3, 4)
        r3 = brute.rotate(row, brute.angles_3d(t, h, w))
        assert np.max(np.abs(np.array(r1) - y1[0, n, 0])) < 1e-10
        assert np.max(np.abs(np.array(r3) - y3[0, n, 0])) < 1e-12


def test_golden_closed_forms():
    with open(os.path.join(GOLDEN, "rope_closed_form.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        D = len(c["x"])
        if c["kind"] == "1d":
            ang = rope_angles_1d([c["position"]], D, c.get("theta", 10000.0))
        else:
            T, Hh, W = c["grid"]
            ang = rope_angles_3d(T, Hh, W)[[c["token"]]]
        x = np.asarray(c["x"], dtype=np.float64).reshape(1, 1, 1, D)
        y = rope_split_halves(x, ang).ravel()
        for idx, val in c["expect"].items():
            assert abs(y[int(idx)] - val) < 1e-12, (c["name"], idx, y[int(idx)], val)


def test_mutants_fail_the_pins():
    """Negative controls: plausible mistakes in a rotation each fail a pin above."""
    def wrong_sign(x, ang):
        y = rope_split_halves(x, -ang)
        return y

    def wrong_pairing(x, ang):   # rotates (2i, 2i+1) instead of (i, i + D/2)
        return _interleaved_rope(np.asarray(x, dtype=np.float64), ang)

    def dropped_term(x, ang):
        D = x.shape[-1]
        c, s = np.cos(ang)[None, :, None, :], np.sin(ang)[None, :, None, :]
        x1, x2 = x[..., : D // 2], x[..., D // 2:]
        return np.concatenate([x1 * c, x1 * s + x2 * c], axis=-1)

    for bad in (wrong_sign, wrong_pairing, dropped_term):
        assert complex_form_error(bad) > 1e-3, bad.__name__
    # a wrong frequency exponent changes the golden values
    x = np.zeros((1, 1, 1, 4))
    x[..., 1] = 1.0
    ang_bad = np.array([[1.0, 1.0 * 10000.0 ** (-1.0 / 4)]])   # -i/D instead of -2i/D
    y = rope_split_halves(x, ang_bad).ravel()
    assert abs(y[3] - math.sin(0.01)) > 1e-3

"""Pins for the oracle's fixed-m softmax metadata and softmax (CPU only).

Checked against what the definition and the mathematics fix, not against the oracle's own
formula: the bound holds for every valid score (brute force) and is reached when a key points
along the query; the rotation leaves it unchanged; pad rows change neither bounds nor
decisions; a hand-derived decision on either side of the threshold; the fixed-m softmax
against scipy's softmax / logsumexp for m far from the row maximum; attention at the fixed m
against the plain oracle attention; and planted mistakes that each fail one of these pins.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle.attention import attention
from oracle.fixed_m import (BLOCK_ROWS, FIXED_M_SPAN_LN, attention_fixed_m, fixed_path_blocks,
                            row_bounds, softmax_fixed_m)
from oracle.rope import rope_angles_1d, rope_angles_3d, rope_split_halves


def _rand(shape, seed, sd=1.0):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape) * sd


def _scores(q, k, scale):
    B, Sq, H, _ = q.shape
    Skv = k.shape[1]
    s = np.zeros((B, H, Sq, Skv))
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                for j in range(Skv):
                    s[b, h, i, j] = scale * math.fsum(float(x) * float(y) for x, y in zip(q[b, i, h], k[b, j, h]))
    return s


def test_bound_holds_for_every_valid_score():
    q, k = _rand((2, 9, 3, 16), 1), _rand((2, 11, 3, 16), 2, sd=2.0)
    scale, qv, kv = 0.3, 7, 8
    m = row_bounds(q, k, qv, kv, scale)
    s = _scores(q, k, scale)
    for b in range(2):
        for h in range(3):
            for i in range(qv):
                assert np.all(np.abs(s[b, h, i, :kv]) <= m[b, i, h] * (1 + 1e-12))


def test_bound_is_reached_by_a_key_along_the_query():
    q = _rand((1, 4, 2, 8), 3)
    k = _rand((1, 6, 2, 8), 4)
    scale = 0.25
    # key 5 of head 1 points along query 2 and has the largest norm of the valid keys
    k[0, 5, 1] = q[0, 2, 1] / np.linalg.norm(q[0, 2, 1]) * (np.max(np.linalg.norm(k[0, :, 1], axis=-1)) + 1.0)
    m = row_bounds(q, k, 4, 6, scale)
    s = _scores(q, k, scale)
    assert abs(np.max(s[0, 1, 2]) - m[0, 2, 1]) <= 1e-12 * m[0, 2, 1]


@pytest.mark.parametrize("rope", ["1d", "3d"])
def test_rotation_leaves_the_bounds_unchanged(rope):
    B, S, H, D = 1, 24, 2, 128
    q, k = _rand((B, S, H, D), 5), _rand((B, S, H, D), 6)
    ang = rope_angles_1d(np.arange(S) + 7, D) if rope == "1d" else rope_angles_3d(2, 3, 4, D)
    m_raw = row_bounds(q, k, 20, 22, 0.125)
    m_rot = row_bounds(rope_split_halves(q, ang), rope_split_halves(k, ang), 20, 22, 0.125)
    assert np.max(np.abs(m_raw - m_rot)) <= 1e-12 * np.max(m_raw)


def test_pad_rows_change_neither_bounds_nor_decisions():
    q, k = _rand((1, 64, 2, 16), 7), _rand((1, 48, 2, 16), 8)
    qv, kv, scale = 40, 30, 0.25
    m0 = row_bounds(q, k, qv, kv, scale)
    q2, k2 = q.copy(), k.copy()
    q2[:, qv:] = 1e6          # pad query rows with huge values
    k2[:, kv:] = -1e6         # pad key rows with huge values
    m1 = row_bounds(q2, k2, qv, kv, scale)
    assert np.array_equal(m0, m1)
    assert np.all(m1[:, qv:] == 0)
    assert np.array_equal(fixed_path_blocks(m0, qv), fixed_path_blocks(m1, qv))
    # a block holding only pad rows, or a mix, is decided by its valid rows alone
    m_pad_huge = m1.copy()
    m_pad_huge[:, qv:] = 1e9
    assert np.array_equal(fixed_path_blocks(m_pad_huge, qv), fixed_path_blocks(m1, qv))


def test_hand_derived_decision_on_either_side_of_the_threshold():
    # B1 H1 D2: q row 0 = (a, 0), key rows of norms 1 and b (max b); scale 1 -> m_0 = a * b.
    # The fixed path needs 2 * a * b <= 64 ln 2 = 44.3614...
    b = 2.0
    for a, expect in ((11.0, True), (11.2, False)):   # 2ab = 44.0 / 44.8
        q = np.zeros((1, BLOCK_ROWS, 1, 2))
        q[0, 0, 0] = (a, 0.0)
        k = np.zeros((1, 2, 1, 2))
        k[0, 0, 0] = (0.0, 1.0)
        k[0, 1, 0] = (b * 0.6, b * 0.8)
        m = row_bounds(q, k, 1, 2, 1.0)
        assert m[0, 0, 0] == pytest.approx(a * b, rel=1e-15)
        assert bool(fixed_path_blocks(m, 1)[0, 0, 0]) is expect
    assert FIXED_M_SPAN_LN == pytest.approx(44.3614195558365, rel=1e-12)


@pytest.mark.parametrize("shift", [-40.0, -3.0, 0.0, 5.0, 40.0])
def test_fixed_m_softmax_is_the_plain_softmax(shift):
    s = _rand((37,), 9, sd=3.0)
    m = float(np.max(s)) + shift
    p, lse = softmax_fixed_m(s, m)
    assert np.max(np.abs(p - softmax(s))) <= 1e-14
    assert abs(lse - logsumexp(s)) <= 1e-12 * max(1.0, abs(lse))


def test_attention_at_fixed_m_is_the_plain_attention():
    B, S, H, D = 1, 40, 2, 32
    q, k, v = _rand((B, S, H, D), 10), _rand((B, S, H, D), 11), _rand((B, S, H, D), 12)
    ang = rope_angles_1d(np.arange(S), D)
    qr, kr = rope_split_halves(q, ang), rope_split_halves(k, ang)
    scale, qv, kv = 1 / math.sqrt(D), 33, 37
    m = row_bounds(qr, kr, qv, kv, scale)
    O1, L1 = attention_fixed_m(qr, kr, v, qv, kv, scale, m)
    O2, L2 = attention(q, k, v, qv, kv, scale, ang, ang)
    assert np.max(np.abs(O1 - O2)) <= 1e-12
    assert np.max(np.abs(L1[:, :qv] - L2[:, :qv])) <= 1e-12
    assert np.all(L1[:, qv:] == -np.inf) and np.all(O1[:, qv:] == 0)


# --- planted mistakes: each must fail one of the pins above ---------------------------------
def _bound_squared_norms(q, k, qv, kv, scale):          # ||q||^2 ||k||^2 instead of norms
    m = row_bounds(q, k, qv, kv, scale)
    return m * m / scale


def _bound_with_pads(q, k, qv, kv, scale):              # maximum taken over every key row
    return row_bounds(q, k, qv, k.shape[1], scale)


def _lse_without_m(s, m):                               # m not added back
    p, lse = softmax_fixed_m(s, m)
    return p, lse - float(m)


def test_planted_mistakes_are_caught():
    # squared norms: the tightness pin fails
    q = _rand((1, 4, 2, 8), 3)
    k = _rand((1, 6, 2, 8), 4)
    k[0, 5, 1] = q[0, 2, 1] / np.linalg.norm(q[0, 2, 1]) * (np.max(np.linalg.norm(k[0, :, 1], axis=-1)) + 1.0)
    s = _scores(q, k, 0.25)
    assert abs(np.max(s[0, 1, 2]) - _bound_squared_norms(q, k, 4, 6, 0.25)[0, 2, 1]) > 1e-3
    # pads in the maximum: the pad pin fails
    q, k = _rand((1, 64, 2, 16), 7), _rand((1, 48, 2, 16), 8)
    k2 = k.copy()
    k2[:, 30:] = -1e6
    assert not np.array_equal(_bound_with_pads(q, k, 40, 30, 0.25), _bound_with_pads(q, k2, 40, 30, 0.25))
    # m not added back to the LSE: the softmax pin fails
    s = _rand((37,), 9, sd=3.0)
    _, lse = _lse_without_m(s, float(np.max(s)) + 5.0)
    assert abs(lse - logsumexp(s)) > 1.0

"""Pins for the oracle's FP8 (e4m3) attention (CPU only).

The e4m3 rounding is checked against an independent bit-level decoder of the OCP format
(every code, ties to the even code, saturation, hand-derived values), not against its own
formula. The attention steps are checked with the rounding replaced by the identity, which
must give the plain fp64 attention whatever the tile order and lazy maximum do; with the
rounding in place the result stays within the error the format allows; planted mistakes
fail one of these pins.
"""
import math

import numpy as np
import pytest

from oracle.attention import attention
from oracle.fp8 import (E4M3_MAX, attention_fp8, e4m3_round, e4m3_values, quantize_per_head,
                        quantize_q_tiles)
from oracle.rope import rope_angles_1d, rope_split_halves


def _decode(code: int) -> float:
    """e4m3 bit pattern -> value (independent of e4m3_round): S EEEE MMM, bias 7."""
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 15 and m == 7:
        return math.nan
    return s * ((m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))


def _codes():
    return {c: _decode(c) for c in range(256) if not math.isnan(_decode(c))}


def test_value_set_matches_the_bit_level_decoder():
    dec = sorted(set(_codes().values()))
    assert np.array_equal(np.array(dec), e4m3_values())
    assert len(dec) == 253                       # 254 finite codes, +0 and -0 equal
    assert max(dec) == 448.0 and min(v for v in dec if v > 0) == 2.0 ** -9


def test_every_value_rounds_to_itself():
    v = e4m3_values()
    assert np.array_equal(e4m3_round(v), v)


def test_midpoints_round_to_the_even_code():
    codes = _codes()
    pos = sorted((val, c) for c, val in codes.items() if val > 0 or c == 0)
    for (a, ca), (b, cb) in zip(pos, pos[1:]):
        even = a if ca % 2 == 0 else b
        assert e4m3_round((a + b) / 2) == even, (a, b)
        assert e4m3_round(-(a + b) / 2) == -even


def test_hand_derived_values_and_saturation():
    # 0.1 = 1.6 * 2^-4 -> mantissa 0.6 * 8 = 4.8 -> 5 -> 1.625 * 2^-4
    assert e4m3_round(0.1) == 0.1015625
    assert e4m3_round(1.0) == 1.0 and e4m3_round(3.0) == 3.0
    assert e4m3_round(1.0625) == 1.0              # tie between 1.0 (m=0) and 1.125 (m=1)
    assert e4m3_round(1.1875) == 1.25             # tie between 1.125 (m=1) and 1.25 (m=2)
    assert e4m3_round(2.0 ** -10) == 0.0          # half the smallest subnormal: ties to 0
    assert e4m3_round(3 * 2.0 ** -10) == 2.0 ** -8  # tie between 1 and 2 subnormal steps
    assert e4m3_round(470.0) == 448.0 and e4m3_round(1e6) == 448.0 and e4m3_round(-1e6) == -448.0
    assert np.isnan(e4m3_round(np.nan))


def test_relative_error_in_the_normal_range():
    x = np.exp(np.random.Generator(np.random.PCG64(1)).uniform(np.log(2.0 ** -6), np.log(448.0), 20000))
    assert np.max(np.abs(e4m3_round(x) - x) / x) <= 2.0 ** -4


def test_quantisation_scales():
    rng = np.random.Generator(np.random.PCG64(2))
    x = rng.standard_normal((1, 300, 2, 16))
    x[:, 250:] = 1e6                               # pad rows: never in a scale
    q8, sq = quantize_q_tiles(x, 250)
    assert sq.shape == (1, 2, 3)
    for t in range(2):
        r0, r1 = 128 * t, min(128 * t + 128, 250)
        for h in range(2):
            assert sq[0, h, t] == pytest.approx(np.max(np.abs(x[0, r0:r1, h])) / E4M3_MAX, rel=1e-15)
            assert np.max(np.abs(q8[0, r0:r1, h])) == E4M3_MAX     # the amax maps to 448
    assert np.all(q8[:, 250:] == 0)
    k8, sk = quantize_per_head(x, 250)
    assert sk[0, 1] == pytest.approx(np.max(np.abs(x[0, :250, 1])) / E4M3_MAX, rel=1e-15)
    assert np.all(k8[:, 250:] == 0)


def _case(seed, S=300, H=2, D=32, qv=280, kv=290):
    rng = np.random.Generator(np.random.PCG64(seed))
    q, k, v = (rng.standard_normal((1, S, H, D)) for _ in range(3))
    ang = rope_angles_1d(np.arange(S), D)
    return q, k, v, ang, qv, kv


def test_without_rounding_the_steps_are_the_plain_attention():
    q, k, v, ang, qv, kv = _case(3)
    scale = 1 / math.sqrt(32)
    # scores spread wide, so that the lazy maximum moves during a row
    q = q * 4.0
    O1, L1 = attention_fp8(rope_split_halves(q, ang), rope_split_halves(k, ang), v, qv, kv, scale,
                           round_fn=lambda x: x)
    O2, L2 = attention(q, k, v, qv, kv, scale, ang, ang)
    assert np.max(np.abs(O1 - O2)) <= 1e-12
    assert np.max(np.abs(L1[:, :qv] - L2[:, :qv])) <= 1e-12
    assert np.all(L1[:, qv:] == -np.inf) and np.all(O1[:, qv:] == 0)


def test_with_rounding_the_error_stays_within_what_the_format_allows():
    q, k, v, ang, qv, kv = _case(4, D=64)
    scale = 1 / 8.0
    qr, kr = rope_split_halves(q, ang), rope_split_halves(k, ang)
    O1, L1 = attention_fp8(qr, kr, v, qv, kv, scale)
    O2, L2 = attention(q, k, v, qv, kv, scale, ang, ang)
    # e4m3 keeps 3 mantissa bits (relative rounding <= 2^-4 per operand)
    assert 1e-3 < np.max(np.abs(O1 - O2)) <= 0.1
    assert np.max(np.abs(L1[:, :qv] - L2[:, :qv])) <= 0.1


# --- planted mistakes: each must fail one of the pins above ---------------------------------
def test_planted_mistakes_are_caught():
    q, k, v, ang, qv, kv = _case(3)
    scale = 1 / math.sqrt(32)
    q = q * 4.0
    qr, kr = rope_split_halves(q, ang), rope_split_halves(k, ang)
    O2, L2 = attention(q, k, v, qv, kv, scale, ang, ang)
    import oracle.fp8 as F
    # the rescale threshold changes nothing in exact arithmetic (m may lag) ...
    orig = F.RESCALE_THRESHOLD_LOG2
    try:
        F.RESCALE_THRESHOLD_LOG2 = -1e9            # m moves on every tile ...
        O1, _ = attention_fp8(qr, kr, v, qv, kv, scale, round_fn=lambda x: x)
        assert np.max(np.abs(O1 - O2)) <= 1e-12   # ... and the result is the same
        # ... but with e4m3 rounding and P still scaled by 112 (for p <= 4), letting m lag
        # by 8 saturates 112 p: the error pin fails
        F.RESCALE_THRESHOLD_LOG2 = 8.0
        O8, _ = attention_fp8(qr, kr, v, qv, kv, scale)
        assert np.max(np.abs(O8 - O2)) > 0.1
    finally:
        F.RESCALE_THRESHOLD_LOG2 = orig
    # a midpoint rounded away from even fails the tie pin
    assert np.round(1.0625 * 8) / 8 == 1.0 and math.floor(1.0625 * 8 + 0.5) / 8 != 1.0
    # a q scale taken from the wrong tile moves the LSE
    q8, sq = quantize_q_tiles(qr, qv)
    assert not np.allclose(sq[:, :, 0], sq[:, :, 1])

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


# ---------------------------------------------------------------------------------------
# The format-derived bounds (oracle.fp8_bound), which the GPU's FP8 result is held to
# against exact attention of the dequantised operands.
# ---------------------------------------------------------------------------------------
from oracle import fp8_bound as FB   # noqa: E402


def _rand_case(seed, B=1, S=256, H=2, D=128):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, S, H, D)), rng.standard_normal((B, S, H, D)),
            rng.standard_normal((B, S, H, D)))


def _sim_p_rounding(q, k, v, L, scale, rows, heads, lag, sigma=FB.SIGMA, round_fn=e4m3_round):
    """An FP8 result whose only error is the rounding of sigma p (p relative to a maximum that
    lags by `lag` in log2 units), computed in fp64 from the dequantised operands."""
    qd, kd, vd, _ = FB.dequantized_operands(q, k, v, q.shape[1], L)
    out = np.zeros((q.shape[0], len(rows), len(heads), q.shape[3]))
    for hi, h in enumerate(heads):
        for ri, i in enumerate(rows):
            s = scale * (kd[0, :L, h] @ qd[0, i, h])
            x = s / math.log(2.0)
            p = np.exp2(x - (np.max(x) - lag))
            out[0, ri, hi] = (round_fn(sigma * p) @ vd[0, :L, h]) / (sigma * np.sum(p))
    return out


def test_dequantized_operands_keep_each_tiles_amax_and_the_grid():
    q, k, v = _rand_case(11, S=300)
    qd, kd, vd, (sq, sk, sv) = FB.dequantized_operands(q, k, v, 300, 290)
    for t in range(3):
        r0, r1 = t * 128, min(300, (t + 1) * 128)
        for h in range(2):
            # the tile's amax maps to 448 exactly (up to the fp64 rounding of amax / 448 * 448)
            assert math.isclose(np.max(np.abs(qd[0, r0:r1, h])), np.max(np.abs(q[0, r0:r1, h])), rel_tol=1e-15)
            codes = qd[0, r0:r1, h] / sq[0, h, t]
            assert np.allclose(codes, e4m3_round(codes), rtol=1e-14, atol=0)   # on the e4m3 grid
    assert np.all(kd[0, 290:] == 0) and np.all(vd[0, 290:] == 0)
    for h in range(2):
        assert math.isclose(np.max(np.abs(kd[0, :290, h])), np.max(np.abs(k[0, :290, h])), rel_tol=1e-15)


def test_exact_quantized_equals_plain_attention_on_grid_inputs():
    """Inputs already on the e4m3 grid with power-of-two scales are not moved by the
    quantisation: the result is plain attention."""
    rng = np.random.default_rng(12)
    S, D = 256, 128

    def grid(shape, tiles):
        x = e4m3_round(rng.standard_normal(shape) * 100.0)
        for r0 in tiles:
            x[0, r0, :, 0] = 448.0
        return x * 2.0 ** -7
    q = grid((1, S, 2, D), [0, 128])
    k = grid((1, S, 2, D), [0])
    v = grid((1, S, 2, D), [0])
    Oq, Lq = FB.exact_quantized(q, k, v, S, S, 1 / math.sqrt(D))
    Oe, Le = attention(q, k, v, S, S, 1 / math.sqrt(D))
    assert np.array_equal(Oq, Oe) and np.array_equal(Lq, Le)


@pytest.mark.parametrize("lag", [0.0, 0.7, 2.0])
def test_p_rounding_bound_covers_the_rounding_of_p_at_any_lag(lag):
    q, k, v = _rand_case(13)
    scale, rows, heads = 1 / math.sqrt(128), [0, 3, 77, 128, 255], [0, 1]
    Oq, _ = FB.exact_quantized(q, k, v, 256, 256, scale, rows=rows, heads=heads)
    # the simulation quantises with this module's own rounding: no ambiguous elements
    bO, bL = FB.p_rounding_bound(q, k, v, 256, 256, scale, rows, heads, abs_window=0.0, rel_window=0.0)
    sim = _sim_p_rounding(q, k, v, 256, scale, rows, heads, lag)
    err = np.abs(sim - Oq)
    assert np.all(err <= bO)
    assert np.all(bL < 1e-3) and np.all(bL > 0)
    bO2, bL2 = FB.p_rounding_bound(q, k, v, 256, 256, scale, rows, heads)   # the windows only widen it
    assert np.all(bO2 >= bO) and np.all(bL2 >= bL)
    # the bound is not vacuous: it is far below what dropping P entirely would cost
    assert np.max(bO) < 0.25 * np.max(np.abs(Oq))


def test_p_rounding_bound_catches_planted_mistakes():
    """A much coarser P format (one mantissa bit instead of three), a lost key or a wrong P
    scale in the normalisation moves the result past the bound."""
    q, k, v = _rand_case(14, S=128)
    scale, rows, heads = 1 / math.sqrt(128), [0, 50, 127], [0]
    Oq, _ = FB.exact_quantized(q, k, v, 128, 128, scale, rows=rows, heads=heads)
    bO, _ = FB.p_rounding_bound(q, k, v, 128, 128, scale, rows, heads)

    def coarse(x):
        x = np.asarray(x, dtype=np.float64)
        _, e = np.frexp(np.where(x == 0, 1.0, x))
        step = np.exp2(e.astype(np.float64) - 1.0)   # one mantissa bit
        return np.round(x / step) * step
    bad = _sim_p_rounding(q, k, v, 128, scale, rows, heads, 0.0, round_fn=coarse)
    assert np.any(np.abs(bad - Oq) > bO)

    def drop_max(x):
        y = e4m3_round(x)
        y[np.argmax(x)] = 0.0
        return y
    bad = _sim_p_rounding(q, k, v, 128, scale, rows, heads, 0.0, round_fn=drop_max)
    assert np.all(np.any(np.abs(bad - Oq) > bO, axis=-1))
    bad = _sim_p_rounding(q, k, v, 128, scale, rows, heads, 0.0, round_fn=lambda x: e4m3_round(x) * 1.25)
    assert np.any(np.abs(bad - Oq) > bO)


def test_ambiguous_steps_marks_codes_next_to_a_midpoint():
    s = 0.5
    # codes (x / s): on the grid, at a midpoint, just off a midpoint, far from one
    x = np.array([1.25, 1.3125, 1.3125 + 2.0 ** -24, 1.29, 300.0, 304.0, 2.0 ** -8]) * s
    st = FB.ambiguous_steps(x, s)
    spacing = np.array([0.125, 0.125, 0.125, 0.125, 32.0, 32.0, 2.0 ** -9]) * s
    assert list(st > 0) == [False, True, True, False, False, True, False]
    assert np.all(st[st > 0] == spacing[st > 0])
    assert np.all(FB.ambiguous_steps(x, s, 0.0, 0.0)[[0, 2, 3, 4, 6]] == 0)


def test_operand_bound_covers_the_quantisation_of_the_operands():
    q, k, v = _rand_case(15)
    scale, rows, heads = 1 / math.sqrt(128), [0, 9, 200, 255], [0, 1]
    Oq, _ = FB.exact_quantized(q, k, v, 256, 256, scale, rows=rows, heads=heads)
    Oe, _ = attention(q, k, v, 256, 256, scale, rows=rows, heads=heads)
    ob = FB.operand_bound(q, k, v, 256, 256, scale, rows, heads)
    assert np.all(np.abs(Oq - Oe) <= ob)
    assert np.max(np.abs(Oq - Oe)) > 1e-3   # the quantisation does move the result


def test_the_same_steps_program_lies_within_the_format_bound():
    """The fp64 program that takes the kernel's steps (lazy maximum, P = e4m3(112 p)) is one
    valid FP8 implementation: it must lie within the bound, with margin."""
    rng = np.random.default_rng(16)
    B, S, H, D = 1, 384, 2, 128
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    ang = rope_angles_1d(np.arange(S), D)
    qr, kr = rope_split_halves(q, ang), rope_split_halves(k, ang)
    rows, heads, scale = [0, 1, 127, 128, 200, 299], [0, 1], 1 / math.sqrt(D)
    Of, Lf = attention_fp8(qr, kr, v, 300, 333, scale, rows=rows, heads=heads)
    Of, Lf = Of[:, rows][:, :, heads], Lf[:, rows][:, :, heads]
    Oq, Lq = FB.exact_quantized(qr, kr, v, 300, 333, scale, rows=rows, heads=heads)
    bO, bL = FB.p_rounding_bound(qr, kr, v, 300, 333, scale, rows, heads)
    assert np.all(np.abs(Of - Oq) <= 0.6 * bO)
    assert np.all(np.abs(Lf - Lq) <= bL)

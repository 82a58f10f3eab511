"""FP8 (e4m3) attention, emulated in fp64 (oracle; test infrastructure only -- nothing in the
package imports it).

Motivation: mstar PR #376 (LTX-2.5 TP/SP) reports a sizing experiment in which rowwise FP8
linears cut the SP2 step by about a quarter. The pages do not apply FP8 to attention; this
is that number format carried over to the attention hot path, with the steps below.

Number format: e4m3 as in the OCP 8-bit floating point definition -- 1 sign bit, 4 exponent
bits with bias 7, 3 mantissa bits; normal values (1 + m/8) * 2^(e-7) for e = 1..15 (the code
S.1111.111 is NaN, so the largest finite value is 1.75 * 2^8 = 448); subnormals m/8 * 2^-6;
no infinities. Conversion here rounds to nearest, ties to even, and saturates to +-448.

Steps (readings of this repository; the pages fix none of them):

1. Rotation as in the split-halves RoPE, then quantisation. q~ is scaled per 128-row tile
   of one head: s_q = amax / 448 over the tile's valid rows (1 when the amax is 0),
   q8 = e4m3(q~ / s_q). k~ and v are scaled once per (b, h) over the valid rows, the same
   way. Pad rows quantise to 0.
2. Scores s_ij = scale * s_q * s_k * (q8_i . k8_j), exact products of e4m3 values summed.
3. Softmax over key tiles of 128 in order, with a running maximum m in log2 units that may
   lag by up to 2: m is replaced by a tile's maximum x only when x > m + 2 (the first tile
   sets it), so every p = 2^(x_ij - m) <= 4 (x_ij = s_ij * log2(e)) and P8 = e4m3(112 p)
   fits e4m3 without saturating. (The bf16 path lets m lag by up to 8, p <= 2^8, which
   448-based scaling could not hold; an exact maximum would rescale O far more often.)
   l accumulates p; O accumulates P8 . v8. When m moves, l and O are multiplied by
   2^(m_old - m_new).
4. Output O = O * s_v / (112 * l), LSE = (m + log2 l) * ln 2; pad rows O = 0, LSE = -inf.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
RESCALE_THRESHOLD_LOG2 = 2.0
P_SCALE = E4M3_MAX / 2.0 ** RESCALE_THRESHOLD_LOG2   # 112: 448 over the largest p (4)
TILE = 128


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even), saturating to +-448. NaN stays NaN."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    nan = np.isnan(x)
    # The grid spacing at magnitude a: 2^(e - 3) for a in [2^e, 2^(e+1)), e >= -6;
    # 2^-9 below 2^-6 (subnormals). frexp gives e exactly: a = f * 2^k with f in [0.5, 1).
    _, k = np.frexp(np.where(nan | (a == 0), 1.0, a))
    e = np.maximum(k.astype(np.float64) - 1.0, -6.0)
    step = np.exp2(e - 3.0)
    q = a / step
    r = np.round(q)            # numpy rounds halves to even
    y = r * step
    y = np.minimum(y, E4M3_MAX)
    return np.where(nan, np.nan, np.sign(x) * y)


def e4m3_values() -> np.ndarray:
    """All finite e4m3 values (254 codes: both zeros collapse, NaN codes excluded), sorted."""
    vals = set()
    for s in (1.0, -1.0):
        for e in range(16):
            for m in range(8):
                if e == 15 and m == 7:
                    continue            # NaN
                v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
                vals.add(s * v)
    return np.array(sorted(vals))


def _scale(amax: float) -> float:
    return amax / E4M3_MAX if amax > 0 else 1.0


def quantize_q_tiles(qr, q_valid: int):
    """q~ [B, S, H, D] -> (q8 values, scales [B, H, S / 128]) with one scale per 128-row tile."""
    qr = np.asarray(qr, dtype=np.float64)
    B, S, H, D = qr.shape
    nt = (S + TILE - 1) // TILE
    q8 = np.zeros_like(qr)
    sc = np.ones((B, H, nt))
    for b in range(B):
        for h in range(H):
            for t in range(nt):
                r0, r1 = t * TILE, min((t + 1) * TILE, q_valid)
                if r1 <= r0:
                    continue
                s = _scale(float(np.max(np.abs(qr[b, r0:r1, h]))))
                sc[b, h, t] = s
                q8[b, r0:r1, h] = e4m3_round(qr[b, r0:r1, h] / s)
    return q8, sc


def quantize_per_head(x, valid: int):
    """x [B, S, H, D] -> (x8 values, scales [B, H]) with one scale per (b, h) over valid rows."""
    x = np.asarray(x, dtype=np.float64)
    B, S, H, D = x.shape
    x8 = np.zeros_like(x)
    sc = np.ones((B, H))
    for b in range(B):
        for h in range(H):
            if valid == 0:
                continue
            s = _scale(float(np.max(np.abs(x[b, :valid, h]))))
            sc[b, h] = s
            x8[b, :valid, h] = e4m3_round(x[b, :valid, h] / s)
    return x8, sc


def attention_fp8(qr, kr, v, q_valid: int, kv_valid: int, scale: float, rows=None, heads=None,
                  round_fn=e4m3_round):
    """FP8 attention of the steps above on rotated q~, k~ (or raw ones without RoPE) and v.

    Returns O [B, Sq, H, D] and LSE [B, Sq, H] on the selected rows / heads. round_fn is the
    e4m3 rounding; passing the identity gives the same algorithm without quantisation.
    """
    qr = np.asarray(qr, dtype=np.float64)
    kr = np.asarray(kr, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, H, D = qr.shape
    if round_fn is e4m3_round:
        q8, sq = quantize_q_tiles(qr, q_valid)
        k8, sk = quantize_per_head(kr, kv_valid)
        v8, sv = quantize_per_head(v, kv_valid)
    else:
        q8, k8, v8 = qr, kr, v
        sq, sk, sv = np.ones((B, H, (Sq + TILE - 1) // TILE)), np.ones((B, H)), np.ones((B, H))
    rows = range(q_valid) if rows is None else [r for r in rows if r < q_valid]
    heads = range(H) if heads is None else heads
    O = np.zeros((B, Sq, H, D))
    L = np.full((B, Sq, H), -np.inf)
    if kv_valid == 0:
        return O, L
    log2e = 1.0 / math.log(2.0)
    pscale = P_SCALE if round_fn is e4m3_round else 1.0
    for b in range(B):
        for h in heads:
            for i in rows:
                c = scale * sq[b, h, i // TILE] * sk[b, h] * log2e
                m, l = -np.inf, 0.0
                acc = np.zeros(D)
                for j0 in range(0, kv_valid, TILE):
                    j1 = min(j0 + TILE, kv_valid)
                    x = c * (k8[b, j0:j1, h] @ q8[b, i, h])
                    mt = float(np.max(x))
                    if m == -np.inf or mt > m + RESCALE_THRESHOLD_LOG2:
                        if m != -np.inf:
                            f = 2.0 ** (m - mt)
                            l *= f
                            acc *= f
                        m = mt
                    p = np.exp2(x - m)
                    l += float(np.sum(p))
                    acc += round_fn(pscale * p) @ v8[b, j0:j1, h]
                O[b, i, h] = acc * sv[b, h] / (pscale * l)
                L[b, i, h] = (m + math.log2(l)) * math.log(2.0)
    return O, L

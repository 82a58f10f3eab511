"""Error bounds of FP8 (e4m3) attention against exact attention, derived from the number
format (oracle; test infrastructure only -- nothing in the package imports it).

The FP8 attention of this repository is defined (its header, and mstar PR #376 for the
motivation: rowwise FP8 linears) by two things a caller can see:

1. Operand quantisation. q~ (rotated q) is scaled per 128-row tile of a head, k~ and v per
   (b, h), with scale = amax / 448 over the valid rows, and each element is rounded to the
   nearest e4m3 value (OCP 8-bit floating point: 3 mantissa bits; largest value 448;
   subnormal spacing 2^-9).
2. The probabilities of the softmax enter P.V as e4m3 values P = e4m3(sigma p), where p is
   the softmax numerator relative to a maximum that lags the true one by at most 2 (log2), so
   1 <= max_j p_j <= 4, and sigma = 112 keeps sigma p <= 448; the row sum l is taken over the
   unrounded p.

Everything else (scores and products accumulated in fp32, ex2 and log2 in fp32) is plain
floating point. This module bounds the distance of such an FP8 result from

    O_q, LSE_q = exact attention (fp64) of the dequantised operands (q8 s_q, k8 s_k, v8 s_v),

which the tests compute with the plain oracle (oracle.attention) -- not with a program that
takes the kernel's steps. Step 1 is the format's own effect and is computed exactly, so
|O_fp8 - O_exact| <= |O_q - O_exact| + bound_O holds with both terms known.

bound_O (per row and channel d) comes from step 2 and the fp32 arithmetic:
  * P rounding. Round to nearest moves sigma p_j by at most half the e4m3 spacing there:
    2^-4 sigma p_j in the normal range (sigma p_j >= 2^-6), 2^-10 below it. In units of the
    normalised weight w_j = p_j / l (l >= max_j p_j >= 1) that is c_j = 2^-4 w_j + 2^-10 / sigma.
    Values below half the smallest subnormal (sigma p_j < 2^-10) are flushed to zero, a
    one-sided error of w_j that is added in full. The other errors are bounded and,
    rounding independent values, centred; Hoeffding's inequality bounds their sum
    sum_j e_j v_jd by sqrt(2 ln(2 / delta) sum_j (c_j v_jd)^2) except with probability delta,
    and the worst case sum_j c_j |v_jd| bounds it always (the smaller of the two is used).
  * fp32 scores. The products of two e4m3 values are exact in fp32 and a sum of D of them
    is within gamma_D = D 2^-23 / (1 - D 2^-23) of its exact value relative to the sum of
    magnitudes (one ulp per addition, so truncating adders are covered too); scaling by
    the fp32 constant and ex2.approx add a few 2^-22. A perturbation
    of at most eps on every score moves every softmax weight by a factor within
    exp(+-2 eps), so the weighted sum moves by at most (exp(2 eps) - 1) sum_j w_j |v_jd|.
  * fp32 accumulation of the P.V products over the L keys (gamma_L relative to the sum of
    magnitudes) and the fp32 rescales of O when the maximum moves.
  * The output is rounded to bf16 (half an ulp: 2^-9 relative).
  * An operand whose scaled value lies next to a rounding midpoint may be rounded to the
    other neighbour by a program that rotates or divides in fp32 (ambiguous_steps): each
    such element adds one e4m3 step to the score bound (q~, k~) or to the output (v).
bound_LSE: eps (the scores) plus the fp32 rounding of m + log2 l and of the final product
(a few ulps of |LSE|).

A format-only bound on |O_q - O_exact| (how far the operand quantisation can move the
result) is `operand_bound`: every operand element moves by at most half the e4m3 spacing
at its scaled value; by Hoeffding over the D channels each score moves by at most t_j,
and to first order the output moves by at most 2 max_j t_j sum_j w_j |v_jd| plus the
rounding of v itself (Hoeffding again over the keys). It is loose (several times the
measured error) and is reported as a sanity bound, not the parity tolerance.
"""
from __future__ import annotations

import math

import numpy as np

from .attention import attention
from .fp8 import E4M3_MAX, quantize_per_head, quantize_q_tiles

U = 2.0 ** -4              # e4m3 unit roundoff (3 mantissa bits), normal range
SUB_HALF = 2.0 ** -10      # half the e4m3 subnormal spacing (2^-9)
SIGMA = 112.0              # P scale: 448 over the largest p (4)
P_NORMAL_MIN = 2.0 ** -6   # smallest normal e4m3 value


def dequantized_operands(qr, kr, v, q_valid: int, kv_valid: int):
    """The operands the FP8 products see, back in fp64: e4m3 codes times their scales
    (q~ per 128-row tile, k~ and v per (b, h); pad rows 0)."""
    q8, sq = quantize_q_tiles(qr, q_valid)
    k8, sk = quantize_per_head(kr, kv_valid)
    v8, sv = quantize_per_head(v, kv_valid)
    B, S, H, D = q8.shape
    tile = np.minimum(np.arange(S) // 128, sq.shape[2] - 1)
    qd = q8 * np.transpose(sq[:, :, tile], (0, 2, 1))[..., None]
    kd = k8 * sk[:, None, :, None]
    vd = v8 * sv[:, None, :, None]
    return qd, kd, vd, (sq, sk, sv)


def exact_quantized(qr, kr, v, q_valid: int, kv_valid: int, scale: float, rows=None, heads=None):
    """O_q, LSE_q: plain fp64 attention of the dequantised operands (no RoPE applied here:
    pass rotated q~, k~)."""
    qd, kd, vd, _ = dequantized_operands(qr, kr, v, q_valid, kv_valid)
    return attention(qd, kd, vd, q_valid, kv_valid, scale, rows=rows, heads=heads)


def ambiguous_steps(x, scale, abs_window: float = 2.0 ** -16, rel_window: float = 2.0 ** -20):
    """For each element of x (scaled by `scale` into e4m3 code units): the full e4m3 spacing
    at its code if the code lies within the window of a rounding midpoint (so that another
    program computing the same code in fp32 -- a rotation, a division by the scale -- may round
    it to the other neighbour), else 0. Used to widen the bounds by one step on such elements."""
    y = np.abs(np.asarray(x, dtype=np.float64) / scale)
    _, k = np.frexp(np.where(y == 0, 1.0, y))
    ex = np.maximum(k.astype(np.float64) - 1.0, -6.0)
    step = np.exp2(ex - 3.0)
    frac = y / step - np.floor(y / step)             # position between two grid values
    dist = np.abs(frac - 0.5) * step                  # distance to the midpoint, code units
    amb = dist <= abs_window + rel_window * y
    # just above a power of two the grid below is finer: a value within the window of 2^e
    # can also round across the binade edge; one (coarser) step covers both
    return np.where(amb, step * scale, 0.0)


def _hoeffding(c2_sum, delta):
    return np.sqrt(2.0 * math.log(2.0 / delta) * c2_sum)


def p_rounding_bound(qr, kr, v, q_valid: int, kv_valid: int, scale: float, rows, heads,
                     delta: float = 1e-9, sigma: float = SIGMA, abs_window: float = 2.0 ** -16,
                     rel_window: float = 2.0 ** -20):
    """bound_O [B, len(rows), len(heads), D] and bound_LSE [B, len(rows), len(heads)] of an
    FP8 result against exact_quantized (see the module docstring). The windows are those of
    ambiguous_steps (0 and 0: the result was quantised by this module's own rounding)."""
    qd, kd, vd, (sq, sk, sv) = dequantized_operands(qr, kr, v, q_valid, kv_valid)
    B, Sq, H, D = qd.shape
    rows = np.asarray(list(rows), dtype=np.int64)
    heads = list(heads)
    qr = np.asarray(qr, dtype=np.float64)
    kr = np.asarray(kr, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    bO = np.zeros((B, len(rows), len(heads), D))
    bL = np.zeros((B, len(rows), len(heads)))
    L = int(kv_valid)
    if L == 0:
        return bO, bL
    # fp32 sums of exact products; the tensor core may truncate, so one ulp (2^-23) per add
    gamma = D * 2.0 ** -23 / (1.0 - D * 2.0 ** -23)
    gamma_l = L * 2.0 ** -23 / (1.0 - L * 2.0 ** -23)
    for b in range(B):
        for hi, h in enumerate(heads):
            k = kd[b, :L, h]                   # [L, D]
            vv = vd[b, :L, h]                  # [L, D]
            ak = ambiguous_steps(kr[b, :L, h], sk[b, h], abs_window, rel_window)   # may round the other way
            av = ambiguous_steps(v[b, :L, h], sv[b, h], abs_window, rel_window)
            for ri, i in enumerate(rows):
                if i >= q_valid:
                    continue
                q = qd[b, i, h]
                aq = ambiguous_steps(qr[b, i, h], sq[b, h, min(i // 128, sq.shape[2] - 1)], abs_window, rel_window)
                s = scale * (k @ q)            # exact scores of the dequantised operands
                mag = scale * (np.abs(k) @ np.abs(q))
                flip = scale * (np.abs(k) @ aq + ak @ np.abs(q) + ak @ aq)   # one-step flips
                eps = float(np.max(gamma * mag + 4.0 * 2.0 ** -24 * np.abs(s) + flip)) + 4.0 * 2.0 ** -22
                m = float(np.max(s))
                e = np.exp(s - m)
                w = e / np.sum(e)
                # kernel-unit probabilities p = w * l with max p in [1, 4]: sigma p_j >= sigma w_j / w_max
                # is the smallest it can be, so the flush test uses the lag that makes p smallest
                p_low = w / np.max(w)
                flushed = sigma * p_low < SUB_HALF
                c = (U * w + SUB_HALF / sigma)[:, None] * np.abs(vv)          # [L, D]
                c[flushed] = 0.0
                # Hoeffding, or the worst case sum_j c_j when that is smaller (few dominant keys)
                stat = np.minimum(_hoeffding(np.sum(c * c, axis=0), delta), np.sum(c, axis=0))
                flush = np.sum((w[flushed])[:, None] * np.abs(vv[flushed]), axis=0)
                wv = np.sum(w[:, None] * np.abs(vv), axis=0)
                score = (math.exp(2.0 * eps) - 1.0) * wv
                # fp32 accumulation of the P.V products over the L keys, and the rescales of O
                acc = gamma_l * np.sum(((1.0 + U) * w + SUB_HALF / sigma)[:, None] * np.abs(vv), axis=0) \
                    + 16.0 * 2.0 ** -24 * wv
                o_q = w @ vv
                vflip = (w * 1.0)[None, :] @ av     # one-step flips of v elements
                core = stat + flush + score + acc + vflip[0]
                out_round = 2.0 ** -8 * (np.abs(o_q) + core)   # bf16 output rounding (with slack)
                bO[b, ri, hi] = core + out_round + 1e-7
                lse = m + math.log(float(np.sum(e)))
                bL[b, ri, hi] = eps + 8.0 * 2.0 ** -24 * (abs(lse) + 1.0) + 2.0 ** -21
    return bO, bL


def operand_bound(qr, kr, v, q_valid: int, kv_valid: int, scale: float, rows, heads, delta: float = 1e-9):
    """Format-only bound on |O_q - O_exact| per row and channel (first order in the score
    perturbation; see the module docstring). qr, kr: rotated q~, k~ (fp64), v raw."""
    qr = np.asarray(qr, dtype=np.float64)
    kr = np.asarray(kr, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    _, _, _, (sq, sk, sv) = dequantized_operands(qr, kr, v, q_valid, kv_valid)
    B, Sq, H, D = qr.shape
    rows = np.asarray(list(rows), dtype=np.int64)
    heads = list(heads)
    out = np.zeros((B, len(rows), len(heads), D))
    L = int(kv_valid)
    if L == 0:
        return out

    def half_spacing(x, s):
        # half the e4m3 spacing at |x / s|, in units of x
        a = np.abs(x / s)
        _, kexp = np.frexp(np.where(a == 0, 1.0, a))
        ex = np.maximum(kexp.astype(np.float64) - 1.0, -6.0)
        return 0.5 * np.exp2(ex - 3.0) * s

    for b in range(B):
        for hi, h in enumerate(heads):
            k = kr[b, :L, h]
            vv = v[b, :L, h]
            hk = half_spacing(k, sk[b, h])
            hv = half_spacing(vv, sv[b, h])
            for ri, i in enumerate(rows):
                if i >= q_valid:
                    continue
                q = qr[b, i, h]
                hq = half_spacing(q, sq[b, h, min(i // 128, sq.shape[2] - 1)])
                s = scale * (k @ q)
                w = np.exp(s - np.max(s))
                w /= np.sum(w)
                c = scale * (hq[None, :] * np.abs(k) + hk * np.abs(q)[None, :] + hq[None, :] * hk)  # [L, D]
                t = _hoeffding(np.sum(c * c, axis=1), delta)                                           # [L]
                wv = np.sum(w[:, None] * np.abs(vv), axis=0)
                tv = _hoeffding(np.sum((w[:, None] * hv) ** 2, axis=0), delta)
                tmax = float(np.max(t))
                out[b, ri, hi] = (math.exp(2.0 * tmax) - 1.0) * wv + tv
    return out

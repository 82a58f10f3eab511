"""Fixed-m softmax for attention rows, fp64 (oracle; test infrastructure only -- nothing in
the package imports it).

Source: maxdiffusion PR #491 (Wan fast inference), lane-padding commit and its test list. A
"fixed-m per Q block" attention kernel takes per-Q-block metadata from norm reductions over q
and k; a block whose metadata allows it skips the online softmax (no running maximum, no
rescaling of the accumulator), other blocks take the online-softmax path. The reductions
exclude the pad Q/K/V rows, so pad values cannot push a block onto the online path.

The pages give no formula for the metadata. Readings taken here:

* the bound of row i is m_i = scale * ||q~_i|| * max_{j < L} ||k~_j||, with L the valid key
  count. By Cauchy-Schwarz no valid score s_ij = scale * q~_i . k~_j exceeds it, and
  |s_ij| <= m_i. The rotation is an isometry per channel pair, so the norms of the rotated
  rows equal those of the raw rows, and the raw rows serve.
* the pages also name a key mean; this reading does not centre the keys (no k mean), so
  the metadata is one maximum per (b, h) and one norm per query row;
* a block is 32 consecutive query rows of one (b, h) (rows 32c .. 32c + 31 of the padded
  sequence). It takes the fixed path when every valid row in it has 2 * m_i <= 64 ln 2,
  i.e. the largest score of the row is at least 2^-64 of exp(m_i) (all its scores lie in
  [-m_i, m_i]). Pad rows (i >= q_valid) do not take part in the decision;
* on the fixed path a row's softmax uses m_i in place of the running maximum:
  p_j = exp(s_ij - m_i), O_i = sum_j p_j v_j / sum_j p_j, LSE_i = m_i + ln sum_j p_j. In
  exact arithmetic this is the plain softmax and its log-sum-exp, whatever m_i is.
"""
from __future__ import annotations

import math

import numpy as np

# A block takes the fixed path when 2 * m_i <= FIXED_M_SPAN_LN for all its valid rows.
FIXED_M_SPAN_LN = 64.0 * math.log(2.0)
BLOCK_ROWS = 32


def row_bounds(q, k, q_valid: int, kv_valid: int, scale: float) -> np.ndarray:
    """Per-row score bounds m [B, Sq, H] (natural-log units): scale * ||q_i|| * max_{j<L} ||k_j||.

    q [B, Sq, H, D], k [B, Skv, H, D] (raw or rotated: the norms are the same). Pad query rows
    (i >= q_valid) get 0; only key rows j < kv_valid enter the maximum.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    B, Sq, H, _ = q.shape
    m = np.zeros((B, Sq, H))
    if q_valid == 0 or kv_valid == 0:
        return m
    qn = np.sqrt(np.sum(q[:, :q_valid] ** 2, axis=-1))            # [B, q_valid, H]
    kmax = np.sqrt(np.max(np.sum(k[:, :kv_valid] ** 2, axis=-1), axis=1))   # [B, H]
    m[:, :q_valid] = scale * qn * kmax[:, None, :]
    return m


def fixed_path_blocks(m, q_valid: int, block: int = BLOCK_ROWS,
                      span: float = FIXED_M_SPAN_LN) -> np.ndarray:
    """Per-block decision [B, ceil(Sq / block), H]: True where every valid row of the block
    has 2 * m_i <= span (the fixed path), False where some valid row does not (online)."""
    m = np.asarray(m, dtype=np.float64)
    B, Sq, H = m.shape
    nb = (Sq + block - 1) // block
    out = np.ones((B, nb, H), dtype=bool)
    for c in range(nb):
        r0, r1 = c * block, min((c + 1) * block, Sq, q_valid)
        if r1 > r0:
            out[:, c, :] = np.all(2.0 * m[:, r0:r1, :] <= span, axis=1)
    return out


def softmax_fixed_m(s, m: float):
    """One row's softmax weights and LSE with a fixed m: p = exp(s - m) / sum exp(s - m),
    lse = m + ln sum exp(s - m). s: the row's valid scores (1-D, at least one)."""
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - float(m))
    tot = float(np.sum(e))
    return e / tot, float(m) + math.log(tot)


def attention_fixed_m(q, k, v, q_valid: int, kv_valid: int, scale: float, m_rows,
                      rows=None, heads=None):
    """Attention with each valid row's softmax taken at its fixed m (m_rows [B, Sq, H]).

    q, k [B, S, H, D] already rotated (or without RoPE); v [B, Skv, H, D]. Returns O
    [B, Sq, H, D] and LSE [B, Sq, H] for the selected rows / heads (all by default), with
    O = 0 and LSE = -inf on pad rows. Equal to the plain attention in exact arithmetic.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, H, D = q.shape
    rows = range(q_valid) if rows is None else [r for r in rows if r < q_valid]
    heads = range(H) if heads is None else heads
    O = np.zeros((B, Sq, H, D))
    L = np.full((B, Sq, H), -np.inf)
    if kv_valid == 0:
        return O, L
    for b in range(B):
        for h in heads:
            kk = k[b, :kv_valid, h]
            vv = v[b, :kv_valid, h]
            for i in rows:
                s = scale * (kk @ q[b, i, h])
                p, lse = softmax_fixed_m(s, m_rows[b, i, h])
                O[b, i, h] = p @ vv
                L[b, i, h] = lse
    return O, L

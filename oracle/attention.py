"""Softmax attention with pad-key masking, natural-log LSE and the LSE merge, in fp64
(oracle; test infrastructure only).

Sources (the web pages this method is taken from):

* Difflet PR #153, Wan padding commit: the sequence is padded to whole tiles, self-attention
  drops the pad keys exactly, and the last block cuts the pad rows.
* maxdiffusion PR #491: pad keys are masked by giving the kernels the real KV length as a
  ragged tail; zero pad keys must not reach the softmax; the fused short-KV cross-attention
  of video queries against a text sequence.
* mstar PR #376: ragged attention that also returns the log-sum-exp as fp32 in natural log,
  and attention over key shards whose per-shard outputs and log-sum-exps are merged.

What is computed (the plain definition; flash attention reaches the same result exactly,
up to rounding order), for each batch b, head h and valid query row i:

    q~_i = R(pos_q(i)) q_i,  k~_j = R(pos_k(j)) k_j        (split-halves RoPE, optional)
    s_j  = scale * (q~_i . k~_j)            for j < L_kv(b) (pad keys never enter)
    LSE_i = m + ln sum_j exp(s_j - m),      m = max_j s_j
    O_i  = sum_j exp(s_j - LSE_i) v_j

Readings taken where the pages are silent: pad query rows (i >= q_valid) are defined as
O = 0 and LSE = -inf so they can be checked exactly; a row with no valid key (L_kv = 0)
gives the same; the merge of rows whose partial LSEs are all -inf gives O = 0, LSE = -inf.
"""
from __future__ import annotations

import numpy as np

from .qknorm import rms_norm_heads
from .rope import rope_split_halves


def _per_batch(value, B):
    if np.ndim(value) == 0:
        return [int(value)] * B
    vals = [int(x) for x in value]
    assert len(vals) == B
    return vals


def _rows_attention(qt: np.ndarray, kt: np.ndarray, vt: np.ndarray, scale: float):
    """qt [n, D], kt [L, D], vt [L, D] fp64 -> (O [n, D], LSE [n])."""
    n, D = qt.shape
    L = kt.shape[0]
    if L == 0:
        return np.zeros((n, vt.shape[1])), np.full(n, -np.inf)
    s = scale * (qt @ kt.T)                      # [n, L]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    lse = m[:, 0] + np.log(e.sum(axis=1))
    p = np.exp(s - lse[:, None])                 # softmax weights
    return p @ vt, lse


def attention(q, k, v, q_valid, kv_valid, scale, angles_q=None, angles_k=None,
              rows=None, heads=None, norm_q=None, norm_k=None, eps=1e-6):
    """Masked softmax attention over BSHD tensors.

    q: [B, Sq, H, D]; k, v: [B, Skv, H, D] (any float dtype; upcast to fp64).
    q_valid: int, queries i >= q_valid are pad rows.
    kv_valid: int or one int per batch; keys j >= kv_valid[b] are never read.
    angles_q [Sq, D/2], angles_k [Skv, D/2]: RoPE angles per row, or None for no RoPE.
    rows: optional iterable of query rows to evaluate (default: all Sq rows).
    heads: optional iterable of heads to evaluate (default: all).
    norm_q / norm_k [D]: per-head RMSNorm weights applied to q / k before the rotation
    (oracle.qknorm), or None for no norm; eps is the norm's epsilon.

    Returns (O [B, len(rows), len(heads), D] fp64, LSE [B, len(rows), len(heads)] fp64).
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    assert k.shape == (B, Skv, H, D) and v.shape == (B, Skv, H, D)
    kv_list = _per_batch(kv_valid, B)
    assert 0 <= q_valid <= Sq and all(0 <= L <= Skv for L in kv_list)
    rows = np.arange(Sq) if rows is None else np.asarray(list(rows), dtype=np.int64)
    heads = list(range(H)) if heads is None else list(heads)
    O = np.zeros((B, len(rows), len(heads), D))
    LSE = np.full((B, len(rows), len(heads)), -np.inf)
    valid_sel = rows < q_valid
    qrows = rows[valid_sel]
    for b in range(B):
        L = kv_list[b]
        # Only the valid prefix of k and v is ever touched: pad keys cannot contribute.
        kb = k[b:b + 1, :L][:, :, heads].astype(np.float64)
        vb = v[b, :L][:, heads].astype(np.float64)
        qb = q[b:b + 1, qrows][:, :, heads].astype(np.float64)
        if norm_k is not None:
            kb = rms_norm_heads(kb, norm_k, eps)
        if norm_q is not None:
            qb = rms_norm_heads(qb, norm_q, eps)
        if angles_k is not None:
            kb = rope_split_halves(kb, angles_k[:L])
        if angles_q is not None:
            qb = rope_split_halves(qb, angles_q[qrows])
        for hi in range(len(heads)):
            o, lse = _rows_attention(qb[0, :, hi, :], kb[0, :, hi, :], vb[:, hi, :], float(scale))
            O[b, valid_sel, hi, :] = o
            LSE[b, valid_sel, hi] = lse
    return O, LSE


def lse_merge(partial_o, partial_lse):
    """Merges partial attention results over key shards (mstar PR #376).

    partial_o [n, B, S, H, D], partial_lse [n, B, S, H]:
        lse = logsumexp_s lse_s,   out = sum_s exp(lse_s - lse) * O_s.
    Rows whose partial LSEs are all -inf give out = 0, lse = -inf.
    """
    po = np.asarray(partial_o, dtype=np.float64)
    pl = np.asarray(partial_lse, dtype=np.float64)
    n = pl.shape[0]
    m = pl.max(axis=0)                                   # [B, S, H]
    ok = m > -np.inf                                     # some shard saw a key for this row
    out = np.zeros(po.shape[1:])
    lse = np.full(pl.shape[1:], -np.inf)
    m_ok = m[ok]
    tot = np.zeros_like(m_ok)
    for s in range(n):                                   # log-sum-exp over shards
        tot += np.exp(pl[s][ok] - m_ok)
    lse[ok] = m_ok + np.log(tot)
    acc = np.zeros((m_ok.shape[0], po.shape[-1]))
    for s in range(n):                                   # out = sum_s exp(lse_s - lse) O_s
        acc += np.exp(pl[s][ok] - lse[ok])[:, None] * po[s][ok]
    out[ok] = acc
    return out, lse

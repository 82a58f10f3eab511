"""Pins for the oracle's masked softmax attention and natural-log LSE (CPU only).

What fixes the oracle from outside itself: an independent pure-Python per-query loop,
closed forms (q = 0 gives the mean of the valid values and LSE = ln L; one valid key gives
O = v_0 and LSE = its score), torch's fp64 scaled_dot_product_attention and scipy's
logsumexp for the no-RoPE case, invariance under permuting (key, value, position) triples,
and invariance of every result under arbitrary pad contents (the pages: pad keys are
dropped exactly; maxdiffusion PR #491's review: zero pad keys must not reach the softmax).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import brute
from oracle.attention import attention
from oracle.rope import grid_positions, pad_angles, rope_angles_1d, rope_angles_3d
from video_dit_attention_gb300.inputs import AttnCase, make_qkv, tiny_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _brute_case(q, k, v, q_valid, kv_valid, scale, ang_q, ang_k, rows, heads):
    B = q.shape[0]
    kvs = [kv_valid] * B if np.ndim(kv_valid) == 0 else list(kv_valid)
    O = np.zeros((B, len(rows), len(heads), q.shape[-1]))
    L = np.full((B, len(rows), len(heads)), -np.inf)
    for b in range(B):
        for ri, i in enumerate(rows):
            if i >= q_valid:
                continue
            for hi, h in enumerate(heads):
                keys = [list(map(float, k[b, j, h])) for j in range(kvs[b])]
                vals = [list(map(float, v[b, j, h])) for j in range(kvs[b])]
                o, lse = brute.attend_one(list(map(float, q[b, i, h])), keys, vals, scale,
                                          None if ang_q is None else list(ang_q[i]),
                                          None if ang_k is None else [list(ang_k[j]) for j in range(kvs[b])])
                O[b, ri, hi] = o
                L[b, ri, hi] = lse
    return O, L


@pytest.mark.parametrize("rope", [None, "1d", "3d"])
def test_matches_pure_python_brute_force(rope):
    D = 128 if rope == "3d" else 64
    case = AttnCase("t", B=2, H=2, D=D, Sq=24, Skv=30, q_valid=21, kv_valid=[17, 30], seed=5)
    q, k, v = make_qkv(case)
    if rope == "1d":
        ang_q = rope_angles_1d(np.arange(24) + 3, D)
        ang_k = rope_angles_1d(np.arange(30) + 40, D)
    elif rope == "3d":
        ang_q = pad_angles(rope_angles_3d(2, 3, 4), 24)
        ang_k = pad_angles(rope_angles_3d(2, 3, 5), 30)
    else:
        ang_q = ang_k = None
    rows = [0, 5, 16, 20, 21, 23]
    O, L = attention(q, k, v, 21, [17, 30], case.scale, ang_q, ang_k, rows=rows)
    Ob, Lb = _brute_case(q, k, v, 21, [17, 30], case.scale, ang_q, ang_k, rows, [0, 1])
    assert np.max(np.abs(O - Ob)) < 1e-12
    fin = np.isfinite(Lb)
    assert np.array_equal(fin, np.isfinite(L))
    assert np.max(np.abs(L[fin] - Lb[fin])) < 1e-12


def test_zero_query_gives_mean_of_valid_values_and_ln_L():
    case = AttnCase("t", B=1, H=3, D=64, Sq=8, Skv=50, q_valid=8, kv_valid=37, seed=6)
    q, k, v = make_qkv(case)
    q[:] = 0.0
    O, L = attention(q, k, v, 8, 37, case.scale)
    mean_v = v[0, :37].astype(np.float64).mean(axis=0)       # [H, D]
    assert np.max(np.abs(O[0] - mean_v[None])) < 1e-14
    assert np.max(np.abs(L - math.log(37))) < 1e-14


def test_single_valid_key():
    case = AttnCase("t", B=1, H=2, D=64, Sq=5, Skv=16, q_valid=5, kv_valid=1, seed=7)
    q, k, v = make_qkv(case)
    O, L = attention(q, k, v, 5, 1, case.scale)
    s0 = case.scale * np.einsum("qhd,hd->qh", q[0].astype(np.float64), k[0, 0].astype(np.float64))
    assert np.max(np.abs(O[0] - v[0, 0][None].astype(np.float64))) == 0.0
    assert np.max(np.abs(L[0] - s0)) < 1e-13


def test_matches_torch_sdpa_and_scipy_logsumexp_without_rope():
    case = AttnCase("t", B=2, H=3, D=64, Sq=40, Skv=50, q_valid=33, kv_valid=[29, 50], seed=8)
    q, k, v = make_qkv(case)
    O, L = attention(q, k, v, 33, [29, 50], case.scale)
    for b, Lk in enumerate([29, 50]):
        qt = torch.from_numpy(q[b, :33].astype(np.float64)).permute(1, 0, 2)   # [H, n, D]
        kt = torch.from_numpy(k[b, :Lk].astype(np.float64)).permute(1, 0, 2)
        vt = torch.from_numpy(v[b, :Lk].astype(np.float64)).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=case.scale)
        assert np.max(np.abs(O[b, :33] - ref.permute(1, 0, 2).numpy())) < 1e-12
        scores = torch.matmul(qt, kt.transpose(1, 2)).numpy() * case.scale  # [H, n, L]
        ref_lse = scipy.special.logsumexp(scores, axis=-1).T
        assert np.max(np.abs(L[b, :33] - ref_lse)) < 1e-12
    assert np.all(O[:, 33:] == 0.0) and np.all(L[:, 33:] == -np.inf)


def test_key_permutation_invariance_with_positions():
    D = 64
    case = AttnCase("t", B=1, H=2, D=D, Sq=16, Skv=40, q_valid=16, kv_valid=40, seed=9)
    q, k, v = make_qkv(case)
    ang_q = rope_angles_1d(np.arange(16), D)
    ang_k = rope_angles_1d(np.arange(40) * 3, D)
    perm = np.random.Generator(np.random.PCG64(1)).permutation(40)
    O1, L1 = attention(q, k, v, 16, 40, case.scale, ang_q, ang_k)
    O2, L2 = attention(q, k[:, perm], v[:, perm], 16, 40, case.scale, ang_q, ang_k[perm])
    assert np.max(np.abs(O1 - O2)) < 1e-13 and np.max(np.abs(L1 - L2)) < 1e-13


def test_pad_contents_change_nothing():
    case = tiny_case()
    q, k, v = make_qkv(case)
    ang = pad_angles(rope_angles_1d(np.arange(300), 64), 384)
    O1, L1 = attention(q, k, v, 300, 300, case.scale, ang, ang)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for x, fill in ((q2, np.nan), (k2, np.inf), (v2, -np.inf)):
        x[:, 300:] = fill
    O2, L2 = attention(q2, k2, v2, 300, 300, case.scale, ang, ang)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    # and equals attention over the unpadded tensors
    O3, L3 = attention(q[:, :300], k[:, :300], v[:, :300], 300, 300, case.scale,
                       ang[:300], ang[:300])
    assert np.array_equal(O1[:, :300], O3) and np.array_equal(L1[:, :300], L3)
    assert np.all(O1[:, 300:] == 0) and np.all(L1[:, 300:] == -np.inf)


def test_empty_key_set_gives_zero_and_minus_inf():
    case = AttnCase("t", B=2, H=1, D=64, Sq=4, Skv=8, q_valid=4, kv_valid=[0, 3], seed=10)
    q, k, v = make_qkv(case)
    O, L = attention(q, k, v, 4, [0, 3], case.scale)
    assert np.all(O[0] == 0) and np.all(L[0] == -np.inf) and np.all(np.isfinite(L[1]))


def test_sampled_rows_equal_full_rows():
    case = AttnCase("t", B=1, H=2, D=64, Sq=64, Skv=64, q_valid=50, kv_valid=45, seed=11)
    q, k, v = make_qkv(case)
    ang = rope_angles_1d(np.arange(64), 64)
    O, L = attention(q, k, v, 50, 45, case.scale, ang, ang)
    rows = [0, 7, 49, 50, 63]
    Os, Ls = attention(q, k, v, 50, 45, case.scale, ang, ang, rows=rows, heads=[1])
    # equal up to BLAS blocking order
    assert np.max(np.abs(O[:, rows][:, :, [1]] - Os)) < 1e-14
    Lf = L[:, rows][:, :, [1]]
    assert np.array_equal(np.isfinite(Lf), np.isfinite(Ls))
    assert np.max(np.abs(Lf[np.isfinite(Lf)] - Ls[np.isfinite(Ls)])) < 1e-13


def test_golden_closed_forms():
    with open(os.path.join(GOLDEN, "attention_closed_form.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = np.asarray(c["q"], dtype=np.float64)[None, :, None, :]
        k = np.asarray(c["k"], dtype=np.float64)[None, :, None, :]
        v = np.asarray(c["v"], dtype=np.float64)[None, :, None, :]
        O, L = attention(q, k, v, q.shape[1], c["kv_valid"], c["scale"])
        assert np.max(np.abs(O[0, :, 0] - np.asarray(c["expect_o"]))) < 1e-12, c["name"]
        assert np.max(np.abs(L[0, :, 0] - np.asarray(c["expect_lse"]))) < 1e-12, c["name"]


def test_mutants_fail_the_pins():
    """Negative controls: a pad key let into the softmax, a missing scale, or a transposed
    value operand each break a pin above."""
    case = AttnCase("t", B=1, H=1, D=64, Sq=6, Skv=10, q_valid=6, kv_valid=7, seed=12)
    q, k, v = make_qkv(case)
    Ob, Lb = _brute_case(q, k, v, 6, 7, case.scale, None, None, list(range(6)), [0])
    leak_O, leak_L = attention(q, k, v, 6, 8, case.scale)           # one pad key leaks in
    assert np.max(np.abs(leak_L - Lb)) > 1e-3
    noscale_O, noscale_L = attention(q, k, v, 6, 7, 1.0)
    assert np.max(np.abs(noscale_L - Lb)) > 1e-3
    vt = v.copy()
    vt[0, :7, 0, :7] = v[0, :7, 0, :7].T                             # transposed block of V
    t_O, _ = attention(q, k, vt, 6, 7, case.scale)
    assert np.max(np.abs(t_O - Ob)) > 1e-3

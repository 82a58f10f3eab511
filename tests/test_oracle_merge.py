"""Pins for the oracle's LSE merge of key-shard partials (CPU only).

mstar PR #376: queries attend each rank's key shard, the ragged attention returns the
natural-log LSE beside the output, and the partial (O, LSE) pairs are merged; its tests
check the sharded result against one rank and the LSE against torch.logsumexp. Here:
sharded-then-merged equals unsharded attention (RoPE at global positions), one shard is
the identity, an empty shard contributes nothing, and the merged LSE equals an independent
log-sum-exp.
"""
import numpy as np
import pytest
import scipy.special
import torch

from oracle.attention import attention, lse_merge
from oracle.rope import rope_angles_1d
from video_dit_attention_gb300.inputs import AttnCase, make_qkv


def _sharded(q, k, v, bounds, scale, ang_q, ang_k):
    po, pl = [], []
    for lo, hi in bounds:
        O, L = attention(q, k[:, lo:hi], v[:, lo:hi], q.shape[1], hi - lo, scale, ang_q,
                         None if ang_k is None else ang_k[lo:hi])
        po.append(O)
        pl.append(L)
    return np.stack(po), np.stack(pl)


@pytest.mark.parametrize("bounds", [[(0, 40), (40, 80), (80, 120), (120, 157)],
                                    [(0, 1), (1, 157)], [(0, 100), (100, 157)]])
def test_sharded_then_merged_equals_unsharded(bounds):
    D = 64
    case = AttnCase("t", B=1, H=3, D=D, Sq=20, Skv=157, q_valid=20, kv_valid=157, seed=21)
    q, k, v = make_qkv(case)
    ang_q = rope_angles_1d(np.arange(20), D)
    ang_k = rope_angles_1d(np.arange(157), D)     # global key positions
    O, L = attention(q, k, v, 20, 157, case.scale, ang_q, ang_k)
    po, pl = _sharded(q, k, v, bounds, case.scale, ang_q, ang_k)
    Om, Lm = lse_merge(po, pl)
    assert np.max(np.abs(Om - O)) < 1e-12
    assert np.max(np.abs(Lm - L)) < 1e-12


def test_single_shard_is_identity():
    rng = np.random.Generator(np.random.PCG64(3))
    po = rng.standard_normal((1, 2, 5, 3, 16))
    pl = rng.standard_normal((1, 2, 5, 3)) * 4
    Om, Lm = lse_merge(po, pl)
    assert np.max(np.abs(Om - po[0])) < 1e-15 and np.max(np.abs(Lm - pl[0])) < 1e-15


def test_empty_shard_contributes_nothing():
    rng = np.random.Generator(np.random.PCG64(4))
    po = rng.standard_normal((2, 1, 7, 2, 8))
    pl = rng.standard_normal((2, 1, 7, 2))
    Om, Lm = lse_merge(po, pl)
    po3 = np.concatenate([po, np.zeros((1, 1, 7, 2, 8))])
    pl3 = np.concatenate([pl, np.full((1, 1, 7, 2), -np.inf)])
    Om3, Lm3 = lse_merge(po3, pl3)
    assert np.array_equal(Om, Om3) and np.array_equal(Lm, Lm3)


def test_all_empty_rows_give_zero_and_minus_inf():
    po = np.ones((3, 1, 2, 1, 4))
    pl = np.full((3, 1, 2, 1), -np.inf)
    pl[1, 0, 1, 0] = 0.5
    Om, Lm = lse_merge(po, pl)
    assert np.all(Om[0, 0, 0] == 0) and Lm[0, 0, 0] == -np.inf
    assert np.allclose(Om[0, 1, 0], 1.0) and Lm[0, 1, 0] == 0.5


def test_lse_matches_independent_logsumexp():
    rng = np.random.Generator(np.random.PCG64(5))
    po = rng.standard_normal((4, 1, 9, 2, 8))
    pl = rng.standard_normal((4, 1, 9, 2)) * 30
    Om, Lm = lse_merge(po, pl)
    assert np.max(np.abs(Lm - scipy.special.logsumexp(pl, axis=0))) < 1e-12
    assert np.max(np.abs(Lm - torch.logsumexp(torch.from_numpy(pl), dim=0).numpy())) < 1e-12
    # the merge weights sum to one
    w = np.exp(pl - Lm[None])
    assert np.max(np.abs(w.sum(axis=0) - 1.0)) < 1e-12


def test_mutant_merges_fail_the_pins():
    """Negative controls: averaging partials, or weighting by exp(lse_s) without
    normalising, breaks sharded == unsharded."""
    D = 64
    case = AttnCase("t", B=1, H=1, D=D, Sq=6, Skv=30, q_valid=6, kv_valid=30, seed=22)
    q, k, v = make_qkv(case)
    O, L = attention(q, k, v, 6, 30, case.scale)
    po, pl = _sharded(q, k, v, [(0, 10), (10, 30)], case.scale, None, None)
    assert np.max(np.abs(po.mean(axis=0) - O)) > 1e-3
    unnorm = (np.exp(pl)[..., None] * po).sum(axis=0)
    assert np.max(np.abs(unnorm - O)) > 1e-3

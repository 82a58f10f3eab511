"""GPU parity of the FP8 (e4m3) attention (dit_attn_fwd_fp8) against the fp64 oracle that takes
the same steps (oracle.fp8.attention_fp8: same rotation, same per-tile / per-head scales, same
e4m3 rounding of q~, k~, v and of 112 p, same tiles and running maximum).

Tolerances, derived from what can still differ between the two: the GPU rotates and divides
by the scales in fp32, so an operand next to an e4m3 rounding boundary can land one step
(2^-4 relative) away from the oracle's; the same holds for 112 p, which the GPU forms with
ex2.approx in fp32. One step on one P element moves O by at most 2^-4 * p_j |v_j| / l, a few
1e-3 here; one step on a q~ or k~ element moves a score by about 2^-4 |q_d k_d| * scale. So
O is held to 2e-2 max-abs (as the bf16 path) and the LSE to 2e-3. Pad rows are exact.
"""
import math

import numpy as np
import pytest
import torch

from helpers import dev_bf16, gpu_tables_self, oracle_angles_self
from oracle.attention import attention
from oracle.fp8 import attention_fp8
from oracle.rope import rope_split_halves
from video_dit_attention_gb300.inputs import AttnCase, make_qkv, sample_rows, wan480_case

pytestmark = pytest.mark.gpu
O_TOL, LSE_TOL = 2e-2, 2e-3


def _run(lib, case, q, k, v):
    tabs = gpu_tables_self(lib, case) if case.rope else (None, None, None, None)
    out, lse = lib.dit_attn_fwd_fp8(dev_bf16(q), dev_bf16(k), dev_bf16(v), case.q_valid, int(case.kv_valid),
                                    *tabs, softmax_scale=case.scale)
    torch.cuda.synchronize()
    assert lib.dit_device_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _oracle(case, q, k, v, rows=None, heads=None):
    aq, ak = oracle_angles_self(case)
    qr = q if aq is None else rope_split_halves(q, aq)
    kr = k if ak is None else rope_split_halves(k, ak)
    return attention_fp8(qr, kr, v, case.q_valid, int(case.kv_valid), case.scale, rows=rows, heads=heads)


def _compare(O, L, Or, Lr, q_valid, rows=None, heads=None):
    Sq = O.shape[1]
    rows = np.arange(Sq) if rows is None else np.asarray(rows)
    heads = np.arange(O.shape[2]) if heads is None else np.asarray(heads)
    Og, Lg = O[:, rows][:, :, heads], L[:, rows][:, :, heads]
    valid = rows < q_valid
    assert np.all(Og[:, ~valid] == 0.0) and np.all(Lg[:, ~valid] == -np.inf)
    o_err = float(np.max(np.abs(Og[:, valid] - Or[:, rows[valid]][:, :, heads])))
    l_err = float(np.max(np.abs(Lg[:, valid] - Lr[:, rows[valid]][:, :, heads])))
    assert np.all(np.isfinite(Og[:, valid]))
    assert o_err <= O_TOL, f"O max-abs {o_err}"
    assert l_err <= LSE_TOL, f"LSE max-abs {l_err}"
    return o_err, l_err


CASES = [
    AttnCase("fp8-small", B=1, H=2, D=128, Sq=384, Skv=384, q_valid=300, kv_valid=300, rope="1d", seed=150),
    AttnCase("fp8-ragged", B=2, H=3, D=128, Sq=640, Skv=768, q_valid=601, kv_valid=700, rope="1d",
             seed=151, k_pos_offset=40),
    AttnCase("fp8-3d", B=1, H=4, D=128, Sq=512, Skv=512, q_valid=495, kv_valid=495, rope="3d",
             grid=(3, 5, 33), seed=152),
    AttnCase("fp8-norope", B=1, H=2, D=128, Sq=256, Skv=384, q_valid=250, kv_valid=333, rope=None, seed=153),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_fp8_matches_the_fp8_oracle(lib, case):
    q, k, v = make_qkv(case)
    O, L = _run(lib, case, q, k, v)
    Or, Lr = _oracle(case, q, k, v)
    _compare(O, L, Or, Lr, case.q_valid)
    # and it stays within the format's distance of exact attention
    aq, ak = oracle_angles_self(case)
    Oe, Le = attention(q, k, v, case.q_valid, case.kv_valid, case.scale, aq, ak)
    n = case.q_valid
    assert np.max(np.abs(O[:, :n] - Oe[:, :n])) <= 0.1
    assert np.max(np.abs(L[:, :n] - Le[:, :n])) <= 0.1


def test_fp8_pad_contents_do_not_reach_valid_rows(lib):
    case = AttnCase("fp8-pads", B=1, H=2, D=128, Sq=384, Skv=384, q_valid=290, kv_valid=301, rope="1d", seed=154)
    q, k, v = make_qkv(case)
    q0, k0, v0 = q.copy(), k.copy(), v.copy()
    for a, n in ((q0, case.q_valid), (k0, case.kv_valid), (v0, case.kv_valid)):
        a[:, n:] = 0.0
    q1, k1, v1 = q.copy(), k.copy(), v.copy()
    q1[:, case.q_valid:] = 3.0e4
    k1[:, case.kv_valid:] = np.inf
    v1[:, case.kv_valid:] = np.nan
    O0, L0 = _run(lib, case, q0, k0, v0)
    O1, L1 = _run(lib, case, q1, k1, v1)
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)


def test_fp8_wan480_sampled(lib):
    case = wan480_case()
    q, k, v = make_qkv(case)
    O, L = _run(lib, case, q, k, v)
    rows = sample_rows(case.q_valid, case.Sq, 16, seed=51)
    heads = [7, 33]
    Or, Lr = _oracle(case, q, k, v, rows=rows, heads=heads)
    _compare(O, L, Or, Lr, case.q_valid, rows=rows, heads=heads)
    assert np.all(O[:, case.q_valid:] == 0) and np.all(L[:, case.q_valid:] == -np.inf)


@pytest.mark.parametrize("qv,kv", [(1, 1), (129, 1), (1, 300), (200, 127), (128, 129)])
def test_fp8_ragged_and_degenerate_lengths(lib, qv, kv):
    case = AttnCase(f"fp8-edge-{qv}-{kv}", B=1, H=2, D=128, Sq=256, Skv=384, q_valid=qv, kv_valid=kv,
                    rope="1d", seed=155 + qv + kv)
    q, k, v = make_qkv(case)
    O, L = _run(lib, case, q, k, v)
    Or, Lr = _oracle(case, q, k, v)
    _compare(O, L, Or, Lr, case.q_valid)


@pytest.mark.parametrize("qv,kv", [(0, 300), (200, 0)])
def test_fp8_empty_inputs(lib, qv, kv):
    """No valid query row, or no valid key: O = 0 and LSE = -inf everywhere."""
    case = AttnCase("fp8-empty", B=1, H=2, D=128, Sq=256, Skv=384, q_valid=256, kv_valid=384, rope=None, seed=160)
    q, k, v = make_qkv(case)
    cq, sq = lib.dit_rope_table_1d(256, 256, 128, 10000.0, 0)
    ck, sk = lib.dit_rope_table_1d(384, 384, 128, 10000.0, 0)
    tabs = tuple(torch.from_numpy(t).cuda() for t in (cq, sq, ck, sk))
    out, lse = lib.dit_attn_fwd_fp8(dev_bf16(q), dev_bf16(k), dev_bf16(v), qv, kv, *tabs)
    torch.cuda.synchronize()
    assert lib.dit_device_status() == 0
    assert torch.all(out == 0) and torch.all(lse == -math.inf)

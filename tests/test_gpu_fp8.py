"""GPU parity of the FP8 (e4m3) attention (dit_attn_fwd_fp8).

Primary check, independent of how the kernel orders its steps: the GPU result against
exact fp64 attention of the dequantised operands (the plain oracle on e4m3 codes times the
documented per-tile / per-head scales), within a bound derived from the e4m3 format for
the rounding of the probabilities and the fp32 arithmetic (oracle.fp8_bound); then, by the
triangle inequality with that exactly computed operand effect, against exact attention of
the unquantised inputs. Inputs already on the e4m3 grid with power-of-two scales pin the
path to closed forms (q = 0 gives the mean of v and ln L; one key gives v_0 and its score).

Diagnostic check: the fp64 program that takes the same steps as the kernel
(oracle.fp8.attention_fp8: same rotation, same per-tile / per-head scales, same
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
from oracle import fp8_bound as FB
from oracle.fp8 import attention_fp8, e4m3_round
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


def _format_bound_check(case, q, k, v, O, L, rows, heads):
    """|O - O_q| <= bound_O and |LSE - LSE_q| <= bound_LSE on the valid rows (O_q, LSE_q: exact
    attention of the dequantised operands), hence |O - O_exact| <= |O_q - O_exact| + bound_O;
    the format-only bound covers |O_q - O_exact|. Returns the largest errors seen."""
    aq, ak = oracle_angles_self(case)
    qr = q if aq is None else rope_split_halves(q, aq)
    kr = k if ak is None else rope_split_halves(k, ak)
    rows = np.asarray([r for r in rows if r < case.q_valid])
    n_kv = int(case.kv_valid)
    Oq, Lq = FB.exact_quantized(qr, kr, v, case.q_valid, n_kv, case.scale, rows=rows, heads=heads)
    bO, bL = FB.p_rounding_bound(qr, kr, v, case.q_valid, n_kv, case.scale, rows, heads)
    Og = O[:, rows][:, :, heads]
    Lg = L[:, rows][:, :, heads]
    eO, eL = np.abs(Og - Oq), np.abs(Lg - Lq)
    assert np.all(eO <= bO), f"O off the dequantised-operand result by {np.max(eO - bO):.3e} beyond the bound"
    assert np.all(eL <= bL), f"LSE off by {np.max(eL - bL):.3e} beyond the bound"
    Oe, Le = attention(q, k, v, case.q_valid, n_kv, case.scale, aq, ak, rows=rows, heads=heads)
    assert np.all(np.abs(Og - Oe) <= np.abs(Oq - Oe) + bO)
    assert np.all(np.abs(Oq - Oe) <= FB.operand_bound(qr, kr, v, case.q_valid, n_kv, case.scale, rows, heads))
    return float(np.max(eO)), float(np.max(eL)), float(np.max(np.abs(Og - Oe)))


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_fp8_within_the_format_bound_of_exact_attention(lib, case):
    q, k, v = make_qkv(case)
    O, L = _run(lib, case, q, k, v)
    n = case.q_valid
    assert np.all(O[:, n:] == 0) and np.all(L[:, n:] == -np.inf)
    rows = sample_rows(case.q_valid, case.Sq, 40, seed=3)
    _format_bound_check(case, q, k, v, O, L, rows, list(range(case.H)))


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_fp8_matches_the_same_steps_oracle(lib, case):
    """Diagnostic: the fp64 program that takes the kernel's steps."""
    q, k, v = make_qkv(case)
    O, L = _run(lib, case, q, k, v)
    Or, Lr = _oracle(case, q, k, v)
    _compare(O, L, Or, Lr, case.q_valid)


def _grid_values(rng, shape, amax_pow2):
    """e4m3 values times 2^e (e = amax_pow2), with one element of magnitude 448 * 2^e in
    every 128-row tile of every head: each scale amax / 448 is then 2^e, a power of two, and
    quantising moves nothing. Such values are exact in bf16."""
    x = e4m3_round(rng.standard_normal(shape) * 60.0)
    x[:, ::128, :, 0] = 448.0
    return x * 2.0 ** amax_pow2


def test_fp8_on_grid_inputs_closed_forms(lib):
    """Inputs whose quantisation is exact (no RoPE): q = 0 gives O = mean of the valid v and
    LSE = ln L; a single key gives O = v_0 exactly and LSE = its score; and in general the
    result is within the P-rounding bound of exact attention itself."""
    rng = np.random.Generator(np.random.PCG64(171))
    B, H, D, S = 1, 2, 128, 384
    k = _grid_values(rng, (B, S, H, D), -7)
    v = _grid_values(rng, (B, S, H, D), -7)
    # q = 0: uniform weights
    case = AttnCase("fp8-grid-q0", B=B, H=H, D=D, Sq=S, Skv=S, q_valid=300, kv_valid=333, rope=None)
    q0 = np.zeros((B, S, H, D))
    O, L = _run(lib, case, q0, k, v)
    mean = v[:, :333].mean(axis=1)                      # [B, H, D]
    assert np.max(np.abs(O[:, :300] - mean[:, None])) <= 2.0 ** -8 * np.max(np.abs(mean)) + 1e-6
    assert np.max(np.abs(L[:, :300] - math.log(333))) <= 1e-5
    # one key: O = v_0 exactly (an e4m3 value times a power of two is exact in bf16)
    q = _grid_values(rng, (B, S, H, D), -7)
    case1 = AttnCase("fp8-grid-l1", B=B, H=H, D=D, Sq=S, Skv=S, q_valid=S, kv_valid=1, rope=None)
    O, L = _run(lib, case1, q, k, v)
    assert np.array_equal(O[0, :, 0], np.broadcast_to(v[0, 0, 0], (S, D)))
    assert np.array_equal(O[0, :, 1], np.broadcast_to(v[0, 0, 1], (S, D)))
    s0 = np.einsum("bshd,bhd->bsh", q, k[:, 0]) * case1.scale
    assert np.max(np.abs(L - s0)) <= 1e-5 * (1.0 + np.max(np.abs(s0)))
    # general: exact attention of the unquantised inputs, within the P-rounding bound
    case2 = AttnCase("fp8-grid", B=B, H=H, D=D, Sq=S, Skv=S, q_valid=S, kv_valid=S, rope=None)
    O, L = _run(lib, case2, q, k, v)
    rows = sample_rows(S, S, 40, seed=4)
    Oe, Le = attention(q, k, v, S, S, case2.scale, rows=rows, heads=[0, 1])
    Oq, Lq = FB.exact_quantized(q, k, v, S, S, case2.scale, rows=rows, heads=[0, 1])
    assert np.array_equal(Oq, Oe) and np.array_equal(Lq, Le)   # the quantisation is exact here
    bO, bL = FB.p_rounding_bound(q, k, v, S, S, case2.scale, rows, [0, 1])
    assert np.all(np.abs(O[:, rows] - Oe) <= bO) and np.all(np.abs(L[:, rows] - Le) <= bL)


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
    _format_bound_check(case, q, k, v, O, L, rows, heads)
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

"""GPU parity of dit_attn_fwd (self-attention, RoPE fused or not) against the fp64 oracle.

Covers: several 128-row tiles in every grid dimension with ragged tails; D = 64 and 128;
1-D and 3-D RoPE; valid lengths on and around tile boundaries; one valid key; q_valid = 0
and kv_valid = 0; pad contents (including NaN/Inf) changing nothing, bitwise; fused RoPE
equal to the standalone RoPE kernel followed by plain attention; the Wan 480x832x9
workload at full size on sampled rows.
"""
import numpy as np
import pytest
import torch

from helpers import compare, dev_bf16, gpu_tables_self, oracle_angles_self, oracle_self, run_self
from oracle.rope import rope_split_halves
from video_dit_attention_gb300.inputs import (AttnCase, make_qkv, sample_rows, tiny_case,
                                              wan480_case)

pytestmark = pytest.mark.gpu


def test_tiny_workload_full_parity(lib):
    case = tiny_case()
    q, k, v = make_qkv(case)
    O, L = run_self(lib, case, q, k, v)
    Or, Lr = oracle_self(case, q, k, v)
    compare(O, L, Or, Lr, case.q_valid)
    assert lib.dit_device_status() == 0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("rope", [None, "1d", "3d"])
def test_multi_tile_ragged(lib, D, rope):
    if rope == "3d" and D == 64:
        pytest.skip("3-D tables are defined for the 44/42/42 split of D = 128")
    if rope == "3d":   # 3 x 5 x 33 = 495 tokens on a 512-row padded grid
        case = AttnCase("mt3d", B=2, H=3, D=D, Sq=512, Skv=512, q_valid=495, kv_valid=495,
                        rope="3d", grid=(3, 5, 33), seed=31 + D)
    else:
        case = AttnCase("mt", B=2, H=3, D=D, Sq=512, Skv=640, q_valid=495, kv_valid=523,
                        rope=rope, seed=33 + D)
    q, k, v = make_qkv(case)
    O, L = run_self(lib, case, q, k, v)
    Or, Lr = oracle_self(case, q, k, v)
    compare(O, L, Or, Lr, case.q_valid)


@pytest.mark.parametrize("kv_valid", [1, 127, 128, 129, 383, 384])
@pytest.mark.parametrize("rope", [None, "1d"])
def test_kv_lengths_around_tile_boundaries(lib, kv_valid, rope):
    case = AttnCase("kv", B=1, H=2, D=128, Sq=256, Skv=384, q_valid=200, kv_valid=kv_valid,
                    rope=rope, seed=40 + kv_valid, k_pos_offset=1000)
    q, k, v = make_qkv(case)
    O, L = run_self(lib, case, q, k, v)
    Or, Lr = oracle_self(case, q, k, v)
    if kv_valid == 1 and rope is not None:
        # One key: LSE is a single score, with no averaging over keys. The fused path
        # rounds q~ and k~ to fp16 (relative 2^-11 each), so |dLSE| <= scale * 2^-10 *
        # sum_d |q~_d k~_d| (+ fp32 terms); check that bound and O = v_0 exactly.
        aq, ak = oracle_angles_self(case)
        qt = rope_split_halves(q[:, :200], aq[:200])
        kt = rope_split_halves(k[:, :1], ak[:1])
        bound = case.scale * 2.0 ** -10 * np.einsum("bqhd,bhd->bqh", np.abs(qt), np.abs(kt[:, 0])) + 1e-5
        assert np.all(np.abs(L[:, :200] - Lr[:, :200]) <= bound)
        assert np.array_equal(O[:, :200], np.broadcast_to(v[:, :1], O[:, :200].shape))
        assert np.all(O[:, 200:] == 0) and np.all(L[:, 200:] == -np.inf)
    else:
        compare(O, L, Or, Lr, case.q_valid)


@pytest.mark.parametrize("q_valid", [0, 1, 128, 129, 384])
def test_q_lengths(lib, q_valid):
    case = AttnCase("qv", B=1, H=2, D=64, Sq=384, Skv=256, q_valid=q_valid, kv_valid=250, seed=50 + q_valid)
    q, k, v = make_qkv(case)
    O, L = run_self(lib, case, q, k, v)
    Or, Lr = oracle_self(case, q, k, v)
    compare(O, L, Or, Lr, case.q_valid)


def test_no_keys_gives_zero_and_minus_inf(lib):
    case = AttnCase("nokv", B=1, H=2, D=128, Sq=256, Skv=128, q_valid=256, kv_valid=0, seed=60)
    q, k, v = make_qkv(case)
    O, L = run_self(lib, case, q, k, v)
    assert np.all(O == 0) and np.all(L == -np.inf)


def test_pad_contents_change_nothing_bitwise(lib):
    case = AttnCase("pad", B=2, H=2, D=128, Sq=384, Skv=384, q_valid=290, kv_valid=301,
                    rope="1d", seed=61)
    q, k, v = make_qkv(case)
    O1, L1 = run_self(lib, case, q, k, v)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:, 290:] = np.nan
    k2[:, 301:] = np.inf
    v2[:, 301:] = np.nan
    O2, L2 = run_self(lib, case, q2, k2, v2)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    assert np.all(O1[:, 290:] == 0) and np.all(L1[:, 290:] == -np.inf)


@pytest.mark.parametrize("D", [64, 128])
def test_fused_rope_against_standalone_rope_then_plain_attention(lib, D):
    """The unfused path (dit_rope_split_halves, bf16 output, then attention without RoPE)
    matches the oracle run on the same rotated bf16 tensors; the fused path, which keeps the
    rotated q/k in fp16, is at least as close to the exact oracle."""
    case = AttnCase("fuse", B=1, H=3, D=D, Sq=384, Skv=512, q_valid=350, kv_valid=470,
                    rope="1d", seed=62 + D, k_pos_offset=77)
    q, k, v = make_qkv(case)
    cq, sq, ck, sk = gpu_tables_self(lib, case)
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    O1, L1 = lib.dit_attn_fwd(qd, kd, vd, case.q_valid, case.kv_valid, cq, sq, ck, sk)
    qr = lib.dit_rope_split_halves(qd, cq, sq)
    kr = lib.dit_rope_split_halves(kd, ck, sk)
    O2, L2 = lib.dit_attn_fwd(qr, kr, vd, case.q_valid, case.kv_valid)
    torch.cuda.synchronize()
    from oracle.attention import attention
    qr_np, kr_np = qr.float().cpu().numpy(), kr.float().cpu().numpy()
    Or2, Lr2 = attention(qr_np, kr_np, v, case.q_valid, case.kv_valid, case.scale)
    compare(O2.float().cpu().numpy(), L2.cpu().numpy(), Or2, Lr2, case.q_valid)
    Or, Lr = oracle_self(case, q, k, v)
    e_fused = compare(O1.float().cpu().numpy(), L1.cpu().numpy(), Or, Lr, case.q_valid)
    n = case.q_valid
    e_unfused_lse = float(np.max(np.abs(L2.cpu().numpy()[:, :n] - Lr[:, :n])))
    assert e_fused[1] <= e_unfused_lse + 1e-6


def test_custom_softmax_scale(lib):
    case = AttnCase("scale", B=1, H=2, D=64, Sq=256, Skv=256, q_valid=256, kv_valid=256, seed=63)
    q, k, v = make_qkv(case)
    out, lse = lib.dit_attn_fwd(dev_bf16(q), dev_bf16(k), dev_bf16(v), 256, 256, softmax_scale=0.3)
    from oracle.attention import attention
    Or, Lr = attention(q, k, v, 256, 256, 0.3)
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), Or, Lr, 256)


def test_wan480_full_size_sampled_rows(lib):
    case = wan480_case()
    q, k, v = make_qkv(case)
    O, L = run_self(lib, case, q, k, v)
    rows = sample_rows(case.q_valid, case.Sq, 48, seed=7)
    heads = [0, 1, 17, 39]
    Or, Lr = oracle_self(case, q, k, v, rows=rows, heads=heads)
    compare(O, L, Or, Lr, case.q_valid, rows=rows, heads=heads)
    # every row of every head: pad rows exact, valid rows finite
    assert np.all(O[:, case.q_valid:] == 0) and np.all(L[:, case.q_valid:] == -np.inf)
    assert np.all(np.isfinite(L[:, :case.q_valid]))
    assert lib.dit_device_status() == 0


@pytest.mark.parametrize("D,rope", [(64, "1d"), (128, "1d"), (128, "3d")])
def test_workspace_rope_path_matches_fused_path_bitwise(lib, D, rope):
    """dit_attn_fwd_ws rotates each q/k row once into the workspace with the same arithmetic
    the fused path applies per tile, so the two give the same bits; both match the oracle."""
    if rope == "3d":
        case = AttnCase("ws3d", B=2, H=3, D=D, Sq=512, Skv=512, q_valid=495, kv_valid=495,
                        rope="3d", grid=(3, 5, 33), seed=81)
    else:
        case = AttnCase("ws1d", B=2, H=3, D=D, Sq=384, Skv=640, q_valid=300, kv_valid=601,
                        rope="1d", seed=82 + D, k_pos_offset=900)
    q, k, v = make_qkv(case)
    tabs = gpu_tables_self(lib, case)
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    O1, L1 = lib.dit_attn_fwd(qd, kd, vd, case.q_valid, case.kv_valid, *tabs)
    ws = torch.full((lib.dit_attn_workspace_bytes(case.B, case.Sq, case.Skv, case.H, case.D),), 0xAB,
                    dtype=torch.uint8, device="cuda")   # stale contents must not matter
    O2, L2 = lib.dit_attn_fwd_ws(qd, kd, vd, case.q_valid, case.kv_valid, *tabs, workspace=ws)
    O3, L3 = lib.dit_attn_fwd_ws(qd, kd, vd, case.q_valid, case.kv_valid, *tabs, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    assert torch.equal(O2, O3) and torch.equal(L2, L3)
    Or, Lr = oracle_self(case, q, k, v)
    compare(O2.float().cpu().numpy(), L2.cpu().numpy(), Or, Lr, case.q_valid)
    assert lib.dit_device_status() == 0


def test_workspace_rope_path_wan480_sampled(lib):
    case = wan480_case()
    q, k, v = make_qkv(case)
    tabs = gpu_tables_self(lib, case)
    out, lse = lib.dit_attn_fwd_ws(dev_bf16(q), dev_bf16(k), dev_bf16(v), case.q_valid, case.kv_valid, *tabs)
    torch.cuda.synchronize()
    O, L = out.float().cpu().numpy(), lse.cpu().numpy()
    rows = sample_rows(case.q_valid, case.Sq, 32, seed=17)
    heads = [3, 22, 38]
    Or, Lr = oracle_self(case, q, k, v, rows=rows, heads=heads)
    compare(O, L, Or, Lr, case.q_valid, rows=rows, heads=heads)
    assert np.all(O[:, case.q_valid:] == 0) and np.all(L[:, case.q_valid:] == -np.inf)
    assert lib.dit_device_status() == 0


@pytest.mark.parametrize("B,H,D,Sq,qv", [(1, 200, 64, 768, 300), (2, 90, 128, 768, 511)])
def test_workspace_rounds_with_skipped_items_bitwise(lib, B, H, D, Sq, qv):
    """More work items than CTAs, so the workspace path rotates in several rounds, and every
    third item (query rows past q_valid) has no work, so a CTA skips a round now and then and
    later uses heads that were rotated in the round it skipped. Bitwise equal to the per-tile
    path (which has no rounds), and parity with the oracle on sampled rows and heads."""
    case = AttnCase("wsrounds", B=B, H=H, D=D, Sq=Sq, Skv=Sq, q_valid=qv, kv_valid=Sq - 57,
                    rope="1d", seed=91 + D)
    q, k, v = make_qkv(case)
    tabs = gpu_tables_self(lib, case)
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    O1, L1 = lib.dit_attn_fwd(qd, kd, vd, case.q_valid, case.kv_valid, *tabs)
    O2, L2 = lib.dit_attn_fwd_ws(qd, kd, vd, case.q_valid, case.kv_valid, *tabs)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    rows = sample_rows(case.q_valid, case.Sq, 12, seed=23)
    heads = [0, H // 2, H - 1]
    Or, Lr = oracle_self(case, q, k, v, rows=rows, heads=heads)
    compare(O2.float().cpu().numpy(), L2.cpu().numpy(), Or, Lr, case.q_valid, rows=rows, heads=heads)
    assert lib.dit_device_status() == 0

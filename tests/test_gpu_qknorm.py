"""GPU parity of the per-head q/k RMSNorm + split-halves RoPE prologue: the standalone kernel
and the attention path that fuses it (dit_attn_fwd_ws_qknorm), against the fp64 oracle."""
import numpy as np
import pytest
import torch

from helpers import compare, dev_bf16, gpu_tables_self, oracle_angles_self
from oracle.attention import attention
from oracle.qknorm import rms_norm_heads
from oracle.rope import pad_angles, rope_angles_1d, rope_angles_3d, rope_split_halves
from video_dit_attention_gb300.inputs import (AttnCase, make_norm_weights, make_qkv, sample_rows,
                                              wan480_case)

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.mark.parametrize("D,rope", [(64, "1d"), (128, "1d"), (128, "3d")])
def test_standalone_rmsnorm_rope_kernel(lib, D, rope):
    B, S, H = 2, 300, 3
    rng = np.random.Generator(np.random.PCG64(120))
    x = torch.from_numpy(rng.standard_normal((B, S, H, D), dtype=np.float32) * 3.0).to(torch.bfloat16)
    w = make_norm_weights(D, seed=121)
    if rope == "1d":
        c, s = lib.dit_rope_table_1d(S, 280, D, 10000.0, 5)
        ang = pad_angles(rope_angles_1d(np.arange(280) + 5, D), S)
    else:
        c, s = lib.dit_rope_table_3d(S, (2, 10, 14), D)
        ang = pad_angles(rope_angles_3d(2, 10, 14), S)
    wd, cd, sd = torch.from_numpy(w).cuda(), torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()
    y = lib.dit_qk_rmsnorm_rope(x.cuda(), wd, cd, sd, eps=EPS)
    torch.cuda.synchronize()
    ref = rope_split_halves(rms_norm_heads(x.float().numpy(), w, EPS), ang)
    err = np.abs(y.float().cpu().numpy() - ref)
    # one bf16 rounding of the result (2^-8 relative) plus fp32 arithmetic
    assert np.all(err <= np.abs(ref) * 2.0 ** -8 + 1e-5)
    xi = x.cuda()
    lib.dit_qk_rmsnorm_rope(xi, wd, cd, sd, eps=EPS, out=xi)
    torch.cuda.synchronize()
    assert torch.equal(xi.cpu(), y.cpu())


def _run_fused(lib, case, q, k, v, wq, wk):
    tabs = gpu_tables_self(lib, case)
    out, lse = lib.dit_attn_fwd_ws_qknorm(dev_bf16(q), dev_bf16(k), dev_bf16(v), case.q_valid,
                                          int(case.kv_valid), torch.from_numpy(wq).cuda(),
                                          torch.from_numpy(wk).cuda(), *tabs, eps=EPS,
                                          softmax_scale=case.scale)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("case", [
    AttnCase("qkn-tiny", B=1, H=2, D=64, Sq=384, Skv=384, q_valid=300, kv_valid=300, rope="1d", seed=122),
    AttnCase("qkn-ragged", B=2, H=3, D=128, Sq=640, Skv=768, q_valid=601, kv_valid=700, rope="1d",
             seed=123, k_pos_offset=40),
    AttnCase("qkn-3d", B=1, H=4, D=128, Sq=512, Skv=512, q_valid=495, kv_valid=495, rope="3d",
             grid=(3, 5, 33), seed=124),
    AttnCase("qkn-rounds", B=1, H=200, D=64, Sq=768, Skv=768, q_valid=300, kv_valid=711, rope="1d", seed=125),
], ids=lambda c: c.name)
def test_fused_qknorm_attention_matches_oracle(lib, case):
    q, k, v = make_qkv(case)
    wq, wk = make_norm_weights(case.D, seed=126), make_norm_weights(case.D, seed=127)
    O, L = _run_fused(lib, case, q, k, v, wq, wk)
    aq, ak = oracle_angles_self(case)
    if case.H > 8:
        rows, heads = sample_rows(case.q_valid, case.Sq, 16, seed=31), [0, case.H // 2, case.H - 1]
    else:
        rows, heads = None, None
    Or, Lr = attention(q, k, v, case.q_valid, case.kv_valid, case.scale, aq, ak, rows=rows,
                       heads=heads, norm_q=wq, norm_k=wk, eps=EPS)
    compare(O, L, Or, Lr, case.q_valid, rows=rows, heads=heads)
    assert lib.dit_device_status() == 0


def test_fused_qknorm_is_scale_invariant(lib):
    """RMSNorm removes the scale of q and k: q and k scaled by 64 (exact in bf16) give the same
    attention up to eps, which does not scale with them (1e-6 against a mean square near 1)."""
    case = AttnCase("qkn-scale", B=1, H=2, D=128, Sq=256, Skv=384, q_valid=250, kv_valid=333, rope="1d", seed=128)
    q, k, v = make_qkv(case)
    wq, wk = make_norm_weights(128, seed=129), make_norm_weights(128, seed=130)
    O1, L1 = _run_fused(lib, case, q, k, v, wq, wk)
    O2, L2 = _run_fused(lib, case, q * 64.0, k * 64.0, v, wq, wk)
    n = case.q_valid
    assert np.max(np.abs(O1[:, :n] - O2[:, :n])) <= 1e-2
    assert np.max(np.abs(L1[:, :n] - L2[:, :n])) <= 1e-3


def test_fused_qknorm_wan480_sampled(lib):
    case = wan480_case()
    q, k, v = make_qkv(case)
    wq, wk = make_norm_weights(case.D, seed=131), make_norm_weights(case.D, seed=132)
    O, L = _run_fused(lib, case, q, k, v, wq, wk)
    rows = sample_rows(case.q_valid, case.Sq, 24, seed=33)
    heads = [5, 30]
    aq, ak = oracle_angles_self(case)
    Or, Lr = attention(q, k, v, case.q_valid, case.kv_valid, case.scale, aq, ak, rows=rows, heads=heads,
                       norm_q=wq, norm_k=wk, eps=EPS)
    compare(O, L, Or, Lr, case.q_valid, rows=rows, heads=heads)
    assert np.all(O[:, case.q_valid:] == 0) and np.all(L[:, case.q_valid:] == -np.inf)
    assert lib.dit_device_status() == 0

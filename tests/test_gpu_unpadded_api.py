"""GPU parity of the unpadded-tensor layer (attn_self, attn_cross, attn_sharded, rope): each
call pads on the device, runs the attention entry point and cuts the pad, so its results on
unpadded inputs must match the fp64 oracle on those inputs, and be bitwise those of the
padded entry point on the same valid rows (pad rows are never read)."""
import numpy as np
import pytest
import torch

from helpers import compare, dev_bf16
from oracle.attention import attention
from oracle.fp8 import attention_fp8
from oracle.rope import rope_angles_1d, rope_angles_3d, rope_split_halves
from video_dit_attention_gb300.inputs import AttnCase, make_norm_weights, make_qkv

pytestmark = pytest.mark.gpu


def _unpadded(case):
    """The case's valid rows only, as fp32 arrays of bf16 values and as CUDA tensors."""
    q, k, v = make_qkv(case)
    Lk = int(case.kv_valid)
    a = (q[:, :case.q_valid], k[:, :Lk], v[:, :Lk])
    return a, tuple(dev_bf16(x) for x in a)


def _np(out, lse):
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _angles_1d(L, off, D):
    return rope_angles_1d(np.arange(L) + off, D)


@pytest.mark.parametrize("D,Lq,Lk,qo,ko", [(128, 300, 333, 0, 0), (64, 129, 640, 7, 40), (128, 256, 128, 0, 5)])
def test_attn_self_1d_matches_oracle(lib, D, Lq, Lk, qo, ko):
    case = AttnCase("u1d", B=2, H=3, D=D, Sq=lib._tiles(Lq), Skv=lib._tiles(Lk), q_valid=Lq, kv_valid=Lk,
                    seed=170 + Lq)
    (q, k, v), (qd, kd, vd) = _unpadded(case)
    O, L = _np(*lib.attn_self(qd, kd, vd, "1d", q_pos_offset=qo, k_pos_offset=ko))
    assert O.shape == (2, Lq, 3, D) and L.shape == (2, Lq, 3)
    Or, Lr = attention(q, k, v, Lq, Lk, case.scale, _angles_1d(Lq, qo, D), _angles_1d(Lk, ko, D))
    compare(O, L, Or, Lr, Lq)


def test_attn_self_3d_and_the_padded_call_agree_bitwise(lib):
    grid = (3, 5, 33)
    n = 495
    case = AttnCase("u3d", B=1, H=4, D=128, Sq=512, Skv=512, q_valid=n, kv_valid=n, rope="3d", grid=grid, seed=175)
    qp, kp, vp = make_qkv(case)                      # padded, garbage pad rows
    O, L = _np(*lib.attn_self(dev_bf16(qp[:, :n]), dev_bf16(kp[:, :n]), dev_bf16(vp[:, :n]), grid))
    a = rope_angles_3d(*grid)
    Or, Lr = attention(qp[:, :n], kp[:, :n], vp[:, :n], n, n, case.scale, a, a)
    compare(O, L, Or, Lr, n)
    c, s = lib.dit_rope_table_3d(512, grid, 128)
    tabs = [torch.from_numpy(t).cuda() for t in (c, s, c, s)]
    Op, Lp = _np(*lib.dit_attn_fwd_ws(dev_bf16(qp), dev_bf16(kp), dev_bf16(vp), n, n, *tabs))
    assert np.array_equal(O, Op[:, :n]) and np.array_equal(L, Lp[:, :n])


def test_attn_self_without_rope_and_whole_tiles(lib):
    case = AttnCase("u-plain", B=1, H=2, D=64, Sq=384, Skv=256, q_valid=384, kv_valid=256, seed=176)
    (q, k, v), (qd, kd, vd) = _unpadded(case)
    O, L = _np(*lib.attn_self(qd, kd, vd))
    Or, Lr = attention(q, k, v, 384, 256, case.scale)
    compare(O, L, Or, Lr, 384)


def test_attn_self_modes(lib):
    Lq = Lk = 300
    case = AttnCase("u-modes", B=1, H=2, D=128, Sq=384, Skv=384, q_valid=Lq, kv_valid=Lk, seed=177)
    (q, k, v), (qd, kd, vd) = _unpadded(case)
    a = _angles_1d(Lq, 0, 128)
    Or, Lr = attention(q, k, v, Lq, Lk, case.scale, a, a)
    O, L = _np(*lib.attn_self(qd, kd, vd, "1d", mode="fixed_m"))
    compare(O, L, Or, Lr, Lq)
    wq, wk = make_norm_weights(128, seed=178), make_norm_weights(128, seed=179)
    O, L = _np(*lib.attn_self(qd, kd, vd, "1d", norm_q=torch.from_numpy(wq).cuda(),
                              norm_k=torch.from_numpy(wk).cuda()))
    Or2, Lr2 = attention(q, k, v, Lq, Lk, case.scale, a, a, norm_q=wq, norm_k=wk)
    compare(O, L, Or2, Lr2, Lq)
    O, L = _np(*lib.attn_self(qd, kd, vd, "1d", mode="fp8"))
    Of, Lf = attention_fp8(rope_split_halves(q, a), rope_split_halves(k, a), v, Lq, Lk, case.scale)
    assert np.max(np.abs(O - Of)) <= 2e-2 and np.max(np.abs(L - Lf)) <= 2e-3


def test_attn_self_empty_sequences(lib):
    q = torch.randn((1, 200, 2, 128), device="cuda").to(torch.bfloat16)
    e = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device="cuda")
    O, L = _np(*lib.attn_self(q, e, e, "1d"))
    assert O.shape == (1, 200, 2, 128) and np.all(O == 0) and np.all(L == -np.inf)
    O, L = _np(*lib.attn_self(e, q, q, "1d"))
    assert O.shape == (1, 0, 2, 128) and L.shape == (1, 0, 2)
    assert lib.dit_device_status() == 0


def test_attn_cross_matches_oracle(lib):
    lens = [249, 1]
    case = AttnCase("u-cross", B=2, H=3, D=128, Sq=640, Skv=384, q_valid=601, kv_valid=300, seed=180)
    q, k, v = make_qkv(case)
    q, k, v = q[:, :601], k[:, :300], v[:, :300]
    O, L = _np(*lib.attn_cross(dev_bf16(q), dev_bf16(k), dev_bf16(v), lens))
    Or, Lr = attention(q, k, v, 601, lens, case.scale)
    compare(O, L, Or, Lr, 601)


def test_attn_sharded_matches_unsharded_oracle(lib):
    sizes = [200, 128, 57]
    Lq, Lk = 300, sum(sizes)
    case = AttnCase("u-shards", B=1, H=2, D=128, Sq=384, Skv=512, q_valid=Lq, kv_valid=Lk, seed=181)
    (q, k, v), (qd, kd, vd) = _unpadded(case)
    offs = np.cumsum([0] + sizes)
    shards = [(kd[:, a:b].contiguous(), vd[:, a:b].contiguous()) for a, b in zip(offs[:-1], offs[1:])]
    O, L = _np(*lib.attn_sharded(qd, shards, "1d", q_pos_offset=11))
    Or, Lr = attention(q, k, v, Lq, Lk, case.scale, _angles_1d(Lq, 11, 128), _angles_1d(Lk, 0, 128))
    compare(O, L, Or, Lr, Lq)


@pytest.mark.parametrize("spec", ["1d", (2, 10, 14)])
def test_rope_matches_oracle(lib, spec):
    rng = np.random.Generator(np.random.PCG64(182))
    x = torch.from_numpy(rng.standard_normal((2, 280, 3, 128), dtype=np.float32)).to(torch.bfloat16)
    y = lib.rope(x.cuda(), spec, pos_offset=3)
    torch.cuda.synchronize()
    ang = _angles_1d(280, 3, 128) if spec == "1d" else rope_angles_3d(*spec)
    ref = rope_split_halves(x.float().numpy(), ang)
    err = np.abs(y.float().cpu().numpy() - ref)
    assert np.all(err <= np.abs(ref) * 2.0 ** -8 + 1e-5)     # one bf16 rounding of the result

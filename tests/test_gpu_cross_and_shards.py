"""GPU parity of short-KV cross-attention, the LSE merge, the sharded-keys flow, the
standalone RoPE kernel and the pad/unpad copies, against the fp64 oracle."""
import numpy as np
import pytest
import torch

from helpers import LSE_TOL, O_TOL, compare, dev_bf16
from oracle.attention import attention, lse_merge
from oracle.rope import pad_angles, rope_angles_1d, rope_angles_3d, rope_split_halves
from video_dit_attention_gb300.inputs import (AttnCase, ShardedCase, cross_case, make_qkv,
                                              make_sharded, sample_rows, sharded_case)

pytestmark = pytest.mark.gpu


def _run_cross(lib, case, q, k, v):
    kv = torch.tensor(case.kv_valid, dtype=torch.int32, device="cuda")
    out, lse = lib.dit_cross_attn_shortkv(dev_bf16(q), dev_bf16(k), dev_bf16(v), case.q_valid, kv,
                                          softmax_scale=case.scale)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("kv", [[1, 512], [128, 129], [300, 7], [511, 384], [0, 200]])
def test_cross_small(lib, kv):
    case = AttnCase("cross", B=2, H=3, D=128, Sq=384, Skv=512, q_valid=333, kv_valid=kv, seed=70)
    q, k, v = make_qkv(case)
    O, L = _run_cross(lib, case, q, k, v)
    Or, Lr = attention(q, k, v, case.q_valid, kv, case.scale)
    compare(O, L, Or, Lr, case.q_valid)


@pytest.mark.parametrize("D,kv", [(128, [300, 512]), (128, [129, 256]), (64, [511, 1]), (64, [385, 128])])
def test_cross_many_tiles_per_cta(lib, D, kv):
    """800 query tiles over the persistent grid (about five per CTA), so each CTA keeps a
    head's keys resident over several tiles, crosses head boundaries inside its range, and,
    for texts longer than 256 keys, alternates the order of the two key halves from tile to
    tile. Full comparison with the oracle."""
    case = AttnCase("crossmany", B=2, H=20, D=D, Sq=2560, Skv=512, q_valid=2500, kv_valid=kv, seed=74 + D)
    q, k, v = make_qkv(case)
    O, L = _run_cross(lib, case, q, k, v)
    Or, Lr = attention(q, k, v, case.q_valid, kv, case.scale)
    compare(O, L, Or, Lr, case.q_valid)
    assert lib.dit_device_status() == 0


@pytest.mark.parametrize("D,kv", [(128, [300, 200]), (64, [512, 129])])
def test_cross_one_tile_per_head(lib, D, kv):
    """One query tile per (batch, head) and 600 heads over the persistent grid, so every CTA
    range crosses several heads: each tile is a run of its own, with a fill of its own (two
    when the text is longer than 256 keys), and the ranges hold one to four tiles, so the Q
    loader's hand-over of the last buffer runs with every small tile count."""
    case = AttnCase("crossheads", B=2, H=300, D=D, Sq=128, Skv=512, q_valid=77, kv_valid=kv, seed=88 + D)
    q, k, v = make_qkv(case)
    O, L = _run_cross(lib, case, q, k, v)
    Or, Lr = attention(q, k, v, case.q_valid, kv, case.scale)
    compare(O, L, Or, Lr, case.q_valid)
    assert lib.dit_device_status() == 0


@pytest.mark.parametrize("D,kv,grow", [(128, [250, 256], 1), (128, [400, 512], 2), (64, [512, 300], 3)])
def test_cross_growing_maximum(lib, D, kv, grow):
    """Keys of one 128-key block scaled by 4 (exact in bf16), so that for many rows its scores
    exceed those of the block visited first by more than the softmax lets its reference trail
    (8 in log2 units, plus up to 1 for the reference's rounding up). With at most 256 keys
    one product covers both blocks and its maximum is taken before any exponential; with
    more, each key tile is a product of its own and O of the earlier products is rescaled.
    grow = the scaled block (1: keys 128-255, 2: 256-383, 3: 384-511). Odd query rows are
    scaled by 1/8, so that they see no such jump and the rescale runs on warps where only
    some rows need it. (Scaling by 8 takes the bf16 rounding of P alone past the O tolerance:
    a step-by-step simulation of the kernel's arithmetic gives 0.0234 there, 0.016 at 4.)"""
    case = AttnCase("crossgrow", B=2, H=4, D=D, Sq=768, Skv=512, q_valid=700, kv_valid=kv, seed=90 + grow)
    q, k, v = make_qkv(case)
    k[:, 128 * grow:128 * (grow + 1)] *= 4.0
    q[:, 1::2] *= 0.125
    s = np.einsum("qhd,khd->hqk", q[0, :700].astype(np.float64), k[0].astype(np.float64)) * case.scale / np.log(2)
    jump = s[:, :, 128 * grow:128 * (grow + 1)].max(-1) - s[:, :, :128].max(-1)
    assert np.mean(jump > 9.0) > 0.2 and np.mean(jump < 8.0) > 0.2
    O, L = _run_cross(lib, case, q, k, v)
    Or, Lr = attention(q, k, v, case.q_valid, kv, case.scale)
    compare(O, L, Or, Lr, case.q_valid)
    assert lib.dit_device_status() == 0


def test_cross_pad_garbage_is_nan_safe(lib):
    case = AttnCase("crossnan", B=2, H=2, D=64, Sq=256, Skv=256, q_valid=256, kv_valid=[77, 200], seed=71)
    q, k, v = make_qkv(case)
    O1, L1 = _run_cross(lib, case, q, k, v)
    k[0, 77:] = np.nan
    v[0, 77:] = np.inf
    v[1, 200:] = np.nan
    O2, L2 = _run_cross(lib, case, q, k, v)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    Or, Lr = attention(q, k, v, case.q_valid, case.kv_valid, case.scale)
    compare(O2, L2, Or, Lr, case.q_valid)


@pytest.mark.parametrize("bad", [513, -1, 2 ** 31 - 1])
def test_cross_out_of_range_length_fails_closed(lib, bad):
    """A device-side key length outside [0, Skv] is not clamped: that batch's rows get
    O = 0 / LSE = -inf and the status word reports DIT_STATUS_BAD_KV_LENGTH; the other batch
    is computed as usual, and the next call with good lengths leaves the status clear."""
    case = AttnCase("crossbad", B=2, H=3, D=128, Sq=256, Skv=512, q_valid=200, kv_valid=[300, 130], seed=73)
    q, k, v = make_qkv(case)
    assert lib.dit_device_status() == 0
    kv = torch.tensor([bad, 130], dtype=torch.int32, device="cuda")
    out, lse = lib.dit_cross_attn_shortkv(dev_bf16(q), dev_bf16(k), dev_bf16(v), case.q_valid, kv)
    torch.cuda.synchronize()
    assert lib.dit_device_status() == lib.DIT_STATUS_BAD_KV_LENGTH
    O, L = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(O[0] == 0) and np.all(L[0] == -np.inf)
    Or, Lr = attention(q[1:], k[1:], v[1:], case.q_valid, [130], case.scale)
    compare(O[1:], L[1:], Or, Lr, case.q_valid)
    O2, L2 = _run_cross(lib, case, q, k, v)
    assert lib.dit_device_status() == 0
    Or2, Lr2 = attention(q, k, v, case.q_valid, case.kv_valid, case.scale)
    compare(O2, L2, Or2, Lr2, case.q_valid)


def test_cross_workload_full(lib):
    case = cross_case()
    q, k, v = make_qkv(case)
    O, L = _run_cross(lib, case, q, k, v)
    rows = sample_rows(case.q_valid, case.Sq, 64, seed=8)
    Or, Lr = attention(q, k, v, case.q_valid, case.kv_valid, case.scale, rows=rows)
    compare(O, L, Or, Lr, case.q_valid, rows=rows)
    assert np.all(O[:, case.q_valid:] == 0) and np.all(L[:, case.q_valid:] == -np.inf)
    assert lib.dit_device_status() == 0


@pytest.mark.parametrize("n,D", [(4, 128), (1, 64), (8, 64), (9, 128)])
def test_lse_merge_kernel_against_oracle(lib, n, D):
    # n <= 8 runs the kernel unrolled for n partials, n = 9 the general loop
    rng = np.random.Generator(np.random.PCG64(72))
    B, S, H = 2, 130, 3
    po = torch.from_numpy(rng.standard_normal((n, B, S, H, D), dtype=np.float32)).to(torch.bfloat16)
    pl = rng.standard_normal((n, B, S, H)).astype(np.float32) * 5
    if n > 1:
        pl[1, 0, :10] = -np.inf        # an empty shard for some rows
    pl[:, 1, 5, 2] = -np.inf           # a row no shard saw
    out, lse = lib.dit_attn_lse_merge(po.cuda(), torch.from_numpy(pl).cuda())
    torch.cuda.synchronize()
    Or, Lr = lse_merge(po.float().numpy(), pl)
    og, lg = out.float().cpu().numpy(), lse.cpu().numpy()
    fin = np.isfinite(Lr)
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.max(np.abs(lg[fin] - Lr[fin])) <= LSE_TOL
    assert np.max(np.abs(og - Or)) <= O_TOL
    assert np.all(og[1, 5, 2] == 0)


def _sharded_gpu(lib, case, q, shards):
    """One dit_attn_fwd per key shard (RoPE at the shard's global positions), then the merge."""
    D = case.D
    cq, sq = lib.dit_rope_table_1d(case.Sq, case.q_valid, D, case.theta, 0)
    cq, sq = torch.from_numpy(cq).cuda(), torch.from_numpy(sq).cuda()
    qd = dev_bf16(q)
    n = len(shards)
    po = torch.empty((n,) + tuple(q.shape), dtype=torch.bfloat16, device="cuda")
    pl = torch.empty((n,) + tuple(q.shape[:3]), dtype=torch.float32, device="cuda")
    for s, ((k, v), off, nv, npad) in enumerate(zip(shards, case.offsets, case.shard_valid, case.shard_pad)):
        ck, sk = lib.dit_rope_table_1d(npad, nv, D, case.theta, off)
        lib.dit_attn_fwd(qd, dev_bf16(k), dev_bf16(v), case.q_valid, nv, cq, sq,
                         torch.from_numpy(ck).cuda(), torch.from_numpy(sk).cuda(),
                         out=po[s], lse=pl[s])
    out, lse = lib.dit_attn_lse_merge(po, pl)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _oracle_unsharded(case, q, shards, rows, heads):
    k = np.concatenate([kv[0][:, :n] for kv, n in zip(shards, case.shard_valid)], axis=1)
    v = np.concatenate([kv[1][:, :n] for kv, n in zip(shards, case.shard_valid)], axis=1)
    L = k.shape[1]
    aq = pad_angles(rope_angles_1d(np.arange(case.q_valid), case.D, case.theta), case.Sq)
    ak = rope_angles_1d(np.arange(L), case.D, case.theta)
    return attention(q, k, v, case.q_valid, L, case.scale, aq, ak, rows=rows, heads=heads)


def test_sharded_small_equals_unsharded(lib):
    case = ShardedCase("sh", B=1, H=2, D=128, Sq=256, q_valid=250, shard_valid=(300, 128, 1, 77), seed=73)
    q, shards = make_sharded(case)
    O, L = _sharded_gpu(lib, case, q, shards)
    Or, Lr = _oracle_unsharded(case, q, shards, None, None)
    compare(O, L, Or, Lr, case.q_valid)


def test_sharded_workload_full_size_sampled_rows(lib):
    case = sharded_case()
    q, shards = make_sharded(case)
    O, L = _sharded_gpu(lib, case, q, shards)
    rows = sample_rows(case.q_valid, case.Sq, 40, seed=9)
    heads = [0, 13, 31]
    Or, Lr = _oracle_unsharded(case, q, shards, rows, heads)
    compare(O, L, Or, Lr, case.q_valid, rows=rows, heads=heads)
    assert np.all(np.isfinite(L))
    assert lib.dit_device_status() == 0


def _sharded_one_call(lib, case, q, shards):
    """dit_attn_fwd_sharded: all shards in one launch (key chunks, RoPE at global positions),
    then the merge."""
    D = case.D
    cq, sq = lib.dit_rope_table_1d(case.Sq, case.q_valid, D, case.theta, 0)
    entries = []
    for (k, v), off, nv, npad in zip(shards, case.offsets, case.shard_valid, case.shard_pad):
        ck, sk = lib.dit_rope_table_1d(npad, nv, D, case.theta, off)
        entries.append((dev_bf16(k), dev_bf16(v), nv, torch.from_numpy(ck).cuda(), torch.from_numpy(sk).cuda()))
    ws = torch.full((lib.dit_attn_sharded_workspace_bytes(case.B, case.Sq, case.H, D, case.shard_pad,
                                                          case.shard_valid),), 0x7F, dtype=torch.uint8, device="cuda")
    out, lse = lib.dit_attn_fwd_sharded(dev_bf16(q), entries, case.q_valid, torch.from_numpy(cq).cuda(),
                                        torch.from_numpy(sq).cuda(), workspace=ws)
    torch.cuda.synchronize()
    assert lib.dit_device_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("D,B,valid", [(128, 1, (300, 128, 1, 77)), (64, 2, (1000, 0, 513)),
                                       (128, 2, (0, 0)), (128, 1, (2700,) * 5 + (129,))])
def test_sharded_one_call_equals_unsharded(lib, D, B, valid):
    """Shards of 1 key, of whole tiles, empty shards, all shards empty, and enough keys that
    shards are cut into several chunks: the one-call result equals unsharded attention."""
    case = ShardedCase("sh1", B=B, H=3, D=D, Sq=384, q_valid=333, shard_valid=valid, seed=75 + D + B)
    q, shards = make_sharded(case)
    O, L = _sharded_one_call(lib, case, q, shards)
    if sum(valid) == 0:
        assert np.all(O == 0) and np.all(L == -np.inf)
        return
    Or, Lr = _oracle_unsharded(case, q, shards, None, None)
    compare(O, L, Or, Lr, case.q_valid)


def test_sharded_one_call_workload_sampled_rows(lib):
    case = sharded_case()
    q, shards = make_sharded(case)
    O, L = _sharded_one_call(lib, case, q, shards)
    rows = sample_rows(case.q_valid, case.Sq, 40, seed=19)
    heads = [0, 7, 31]
    Or, Lr = _oracle_unsharded(case, q, shards, rows, heads)
    compare(O, L, Or, Lr, case.q_valid, rows=rows, heads=heads)
    assert np.all(np.isfinite(L))


@pytest.mark.parametrize("D,rope", [(64, "1d"), (128, "1d"), (128, "3d")])
def test_standalone_rope_kernel(lib, D, rope):
    B, S, H = 2, 300, 3
    rng = np.random.Generator(np.random.PCG64(74))
    x = torch.from_numpy(rng.standard_normal((B, S, H, D), dtype=np.float32)).to(torch.bfloat16)
    if rope == "1d":
        c, s = lib.dit_rope_table_1d(S, 280, D, 10000.0, 5)
        ang = pad_angles(rope_angles_1d(np.arange(280) + 5, D), S)
    else:
        c, s = lib.dit_rope_table_3d(S, (2, 10, 14), D)
        ang = pad_angles(rope_angles_3d(2, 10, 14), S)
    y = lib.dit_rope_split_halves(x.cuda(), torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda())
    torch.cuda.synchronize()
    ref = rope_split_halves(x.float().numpy(), ang)
    err = np.abs(y.float().cpu().numpy() - ref)
    # one bf16 rounding of the result (2^-8 relative) plus fp32 table/arithmetic error
    assert np.all(err <= np.abs(ref) * 2.0 ** -8 + 1e-5)
    # in place gives the same bits
    xi = x.cuda()
    lib.dit_rope_split_halves(xi, torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), out=xi)
    torch.cuda.synchronize()
    assert torch.equal(xi.cpu(), y.cpu())


def test_pad_and_unpad_copies(lib):
    rng = np.random.Generator(np.random.PCG64(75))
    x = torch.from_numpy(rng.standard_normal((2, 300, 5, 64), dtype=np.float32)).to(torch.bfloat16).cuda()
    xp = lib.dit_pad_tokens(x, 384)
    back = lib.dit_unpad_tokens(xp, 300)
    l = torch.from_numpy(rng.standard_normal((2, 300, 5), dtype=np.float32)).cuda()   # 20-byte rows
    lp = lib.dit_pad_tokens(l, 384)
    lb = lib.dit_unpad_tokens(lp, 300)
    torch.cuda.synchronize()
    assert torch.equal(back, x) and torch.equal(xp[:, :300], x)
    assert torch.equal(lb, l) and torch.equal(lp[:, :300], l)


def test_fma_exp2_against_exp2f_and_its_bound(lib):
    """The softmax's FMA-pipe exponential: within its stated 2.6e-6 relative error of the
    exact 2^x (fp64) over the range the kernel feeds it, and close to CUDA's exp2f."""
    x = torch.cat([torch.linspace(-125.0, 8.0, 1_000_001), torch.tensor([0.0, -0.5, 0.5, 1.0, -1.0, 7.99])])
    xd = x.cuda()
    y = lib.dit_exp2_fma_eval(xd)
    ref_cuda = torch.exp2(xd)
    torch.cuda.synchronize()
    exact = np.exp2(x.double().numpy())
    rel = np.abs(y.cpu().double().numpy() / exact - 1.0)
    assert rel.max() <= 3e-6, rel.max()
    assert torch.max(torch.abs(y / ref_cuda - 1.0)).item() <= 4e-6
    # below the clamp the result is 2^-125, never negative, NaN or a wrapped exponent
    z = lib.dit_exp2_fma_eval(torch.tensor([-126.0, -200.0, float("-inf")], device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(z > 0) and torch.all(z < 1e-37)

"""GPU parity of the fixed-m softmax path (dit_attn_fwd_ws_fixed_m) against the fp64 oracle:
outputs within the attention tolerances, the number of 32-row blocks that took the online
path equal to the oracle's decision (on inputs kept far from the threshold, so that fp32 and
fp64 decide alike), pad contents that move no block onto the online path and leave valid
rows bitwise unchanged, and blocks forced onto the online path that still match."""
import math

import numpy as np
import pytest
import torch

from helpers import compare, dev_bf16, gpu_tables_self, oracle_angles_self
from oracle.attention import attention
from oracle.fixed_m import FIXED_M_SPAN_LN, fixed_path_blocks, row_bounds
from video_dit_attention_gb300.inputs import AttnCase, make_qkv, sample_rows, wan480_case

pytestmark = pytest.mark.gpu


def _run(lib, case, q, k, v):
    tabs = gpu_tables_self(lib, case)
    n_online = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.dit_attn_fwd_ws_fixed_m(dev_bf16(q), dev_bf16(k), dev_bf16(v), case.q_valid,
                                           int(case.kv_valid), *tabs, n_online=n_online,
                                           softmax_scale=case.scale)
    torch.cuda.synchronize()
    assert lib.dit_device_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(n_online.item())


def _oracle_online_blocks(case, q, k):
    """Blocks the oracle sends to the online path, after checking that no block's largest
    2 m_i lies within 5 % of the threshold (where fp32 and fp64 could decide differently)."""
    m = row_bounds(q, k, case.q_valid, int(case.kv_valid), case.scale)
    B, Sq, H = m.shape
    mv = m[:, :case.q_valid]
    for c in range(0, case.q_valid, 32):
        top = 2.0 * np.max(mv[:, c:c + 32], axis=1)
        assert np.all((top < 0.95 * FIXED_M_SPAN_LN) | (top > 1.05 * FIXED_M_SPAN_LN)), "too close to the threshold"
    return int(np.sum(~fixed_path_blocks(m, case.q_valid)))


CASES = [
    AttnCase("fm-tiny", B=1, H=2, D=64, Sq=384, Skv=384, q_valid=300, kv_valid=300, rope="1d", seed=140),
    AttnCase("fm-ragged", B=2, H=3, D=128, Sq=640, Skv=768, q_valid=601, kv_valid=700, rope="1d",
             seed=141, k_pos_offset=40),
    AttnCase("fm-3d", B=1, H=4, D=128, Sq=512, Skv=512, q_valid=495, kv_valid=495, rope="3d",
             grid=(3, 5, 33), seed=142),
    AttnCase("fm-rounds", B=1, H=200, D=64, Sq=768, Skv=768, q_valid=300, kv_valid=711, rope="1d", seed=143),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_fixed_m_matches_oracle(lib, case):
    q, k, v = make_qkv(case)
    O, L, n_online = _run(lib, case, q, k, v)
    assert n_online == _oracle_online_blocks(case, q, k) == 0   # N(0,1) rows: every block fixed
    aq, ak = oracle_angles_self(case)
    if case.H > 8:
        rows, heads = sample_rows(case.q_valid, case.Sq, 16, seed=41), [0, case.H // 2, case.H - 1]
    else:
        rows, heads = None, None
    Or, Lr = attention(q, k, v, case.q_valid, case.kv_valid, case.scale, aq, ak, rows=rows, heads=heads)
    compare(O, L, Or, Lr, case.q_valid, rows=rows, heads=heads)


@pytest.mark.parametrize("blocks", ["all", "some"])
def test_blocks_forced_onto_the_online_path(lib, blocks):
    """q rows scaled by a power of two (exact in bf16) push their blocks past the threshold:
    those blocks, and only those, take the online path, and the results still match. The
    scale stays at 2 so that the scores stay in the range the absolute tolerances assume: the
    fp16 rounding of q~ grows with the scores (at 4 the LSE error reaches 1.9e-3, at 16 the
    nearly one-hot softmax gives O errors of 2e-2), on the online path as on the fixed one."""
    case = AttnCase("fm-online", B=2, H=3, D=128, Sq=512, Skv=640, q_valid=450, kv_valid=600, rope="1d", seed=144)
    q, k, v = make_qkv(case)
    if blocks == "all":
        q[:, :case.q_valid] *= 2.0
    else:
        q[0, 64:96, 1] *= 2.0           # one block of batch 0, head 1
        q[1, 300:301, 2] *= 2.0         # one row: its block of batch 1, head 2
    O, L, n_online = _run(lib, case, q, k, v)
    expect = _oracle_online_blocks(case, q, k)
    assert expect == (2 * 3 * math.ceil(case.q_valid / 32) if blocks == "all" else 2)
    assert n_online == expect
    aq, ak = oracle_angles_self(case)
    Or, Lr = attention(q, k, v, case.q_valid, case.kv_valid, case.scale, aq, ak)
    compare(O, L, Or, Lr, case.q_valid)


def test_pad_contents_move_no_block_and_no_valid_row(lib):
    """Huge and non-finite pad rows in q, k and v: no block leaves the fixed path and valid rows
    are bitwise those of zero pads."""
    case = AttnCase("fm-pads", B=1, H=4, D=128, Sq=512, Skv=512, q_valid=333, kv_valid=401, rope="1d", seed=145)
    q, k, v = make_qkv(case)
    q0, k0, v0 = q.copy(), k.copy(), v.copy()
    for a, n in ((q0, case.q_valid), (k0, case.kv_valid), (v0, case.kv_valid)):
        a[:, n:] = 0.0
    q1, k1, v1 = q.copy(), k.copy(), v.copy()
    q1[:, case.q_valid:] = 3.0e4
    k1[:, case.kv_valid:] = -3.0e4
    k1[:, case.kv_valid + 5] = np.inf
    v1[:, case.kv_valid:] = np.nan
    O0, L0, n0 = _run(lib, case, q0, k0, v0)
    O1, L1, n1 = _run(lib, case, q1, k1, v1)
    assert n0 == n1 == 0
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)
    aq, ak = oracle_angles_self(case)
    Or, Lr = attention(q0, k0, v0, case.q_valid, case.kv_valid, case.scale, aq, ak)
    compare(O1, L1, Or, Lr, case.q_valid)


def test_fixed_m_against_the_online_workspace_path(lib):
    """Same inputs through dit_attn_fwd_ws (online softmax everywhere): the two differ only
    by where P is rounded, well inside the oracle tolerances."""
    case = AttnCase("fm-vs-ws", B=1, H=2, D=128, Sq=640, Skv=640, q_valid=600, kv_valid=611, rope="1d", seed=146)
    q, k, v = make_qkv(case)
    O1, L1, _ = _run(lib, case, q, k, v)
    tabs = gpu_tables_self(lib, case)
    out, lse = lib.dit_attn_fwd_ws(dev_bf16(q), dev_bf16(k), dev_bf16(v), case.q_valid, int(case.kv_valid),
                                   *tabs, softmax_scale=case.scale)
    torch.cuda.synchronize()
    O2, L2 = out.float().cpu().numpy(), lse.cpu().numpy()
    n = case.q_valid
    assert np.max(np.abs(O1[:, :n] - O2[:, :n])) <= 1e-2
    assert np.max(np.abs(L1[:, :n] - L2[:, :n])) <= 5e-4
    assert np.array_equal(O1[:, n:], O2[:, n:]) and np.array_equal(L1[:, n:], L2[:, n:])


def test_fixed_m_wan480_sampled(lib):
    case = wan480_case()
    q, k, v = make_qkv(case)
    O, L, n_online = _run(lib, case, q, k, v)
    assert n_online == 0
    rows = sample_rows(case.q_valid, case.Sq, 24, seed=43)
    heads = [3, 27]
    aq, ak = oracle_angles_self(case)
    Or, Lr = attention(q, k, v, case.q_valid, case.kv_valid, case.scale, aq, ak, rows=rows, heads=heads)
    compare(O, L, Or, Lr, case.q_valid, rows=rows, heads=heads)
    assert np.all(O[:, case.q_valid:] == 0) and np.all(L[:, case.q_valid:] == -np.inf)


@pytest.mark.parametrize("qv,kv", [(1, 1), (129, 1), (1, 300), (200, 127), (128, 129)])
def test_fixed_m_ragged_and_degenerate_lengths(lib, qv, kv):
    case = AttnCase(f"fm-edge-{qv}-{kv}", B=1, H=2, D=64, Sq=256, Skv=384, q_valid=qv, kv_valid=kv,
                    rope="1d", seed=170 + qv + kv)
    q, k, v = make_qkv(case)
    O, L, n_online = _run(lib, case, q, k, v)
    assert n_online == 0
    aq, ak = oracle_angles_self(case)
    Or, Lr = attention(q, k, v, case.q_valid, case.kv_valid, case.scale, aq, ak)
    compare(O, L, Or, Lr, case.q_valid)

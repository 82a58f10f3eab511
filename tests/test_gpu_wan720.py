"""GPU parity of the Wan 720p 81-frame self-attention at full size (maxdiffusion PR #491:
the 75,600 latent tokens of the 720p/81f Wan 2.2 runs, padded to whole 128-row tiles).

B1 H40 D128, grid 21 x 45 x 80 = 75,600 tokens padded to 75,648 (591 tiles), 3-D split-halves
RoPE (44/42/42, theta 10000), pad keys masked. The call is dit_attn_fwd_ws, the path the
benchmark times: k rotated once into the fp16 workspace (775 MB), each CTA walking about 78
work items of 591 key tiles each.

Checked against the fp64 oracle on sampled rows of four heads: the first rows, both sides of
the first tile boundary, both sides of the last valid tile boundary, rows inside the last
(ragged) tile, the last valid row, and random rows. On the device, every pad row of every
head must be exactly O = 0, LSE = -inf, and every valid LSE finite.
"""
import numpy as np
import pytest
import torch

from helpers import compare, dev_bf16, gpu_tables_self, oracle_self
from video_dit_attention_gb300.inputs import make_qkv, sample_rows, wan720_case

pytestmark = pytest.mark.gpu


def test_wan720_full_size_sampled_rows(lib):
    case = wan720_case()
    q, k, v = make_qkv(case)
    tabs = gpu_tables_self(lib, case)
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    out, lse = lib.dit_attn_fwd_ws(qd, kd, vd, case.q_valid, case.kv_valid, *tabs)
    torch.cuda.synchronize()
    del qd, kd, vd
    assert lib.dit_device_status() == 0

    n = case.q_valid
    # every pad row of every head is exact, every valid LSE finite (checked on the device)
    assert bool(torch.all(out[:, n:] == 0).item()), "pad rows of O must be exactly 0"
    assert bool(torch.all(lse[:, n:] == float("-inf")).item()), "pad rows of LSE must be -inf"
    assert bool(torch.all(torch.isfinite(lse[:, :n])).item()), "non-finite LSE on a valid row"
    assert bool(torch.all(torch.isfinite(out[:, :n].float())).item()), "non-finite O on a valid row"

    last_tile = (n // 128) * 128          # 75,520: the last, ragged tile holds 80 valid rows
    extra = [last_tile + 1, last_tile + 40, n - 2, last_tile - 2]
    rows = np.unique(np.concatenate([sample_rows(n, case.Sq, 24, seed=29), extra]))
    heads = [0, 13, 26, 39]
    ridx = torch.from_numpy(rows).cuda()
    O = out.index_select(1, ridx).float().cpu().numpy()
    L = lse.index_select(1, ridx).cpu().numpy()
    Or, Lr = oracle_self(case, q, k, v, rows=rows, heads=heads)
    # `compare` indexes rows of the full arrays: hand it the gathered rows as positions 0..n-1
    # with the matching pad/valid split.
    pos = np.arange(len(rows))
    n_valid_sampled = int(np.sum(rows < n))
    assert np.all(rows[:n_valid_sampled] < n) and np.all(rows[n_valid_sampled:] >= n)
    assert {0, 127, 128, last_tile - 1, last_tile, n - 1}.issubset(set(rows.tolist()))
    assert len(rows) >= 24
    compare(O[:, :, heads], L[:, :, heads], Or, Lr, n_valid_sampled, rows=pos, heads=np.arange(len(heads)))

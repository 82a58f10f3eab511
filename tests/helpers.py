"""Shared helpers for the GPU parity tests: build the same seeded inputs for both sides,
run the CUDA path through the binding, run the fp64 oracle, and compare.

Tolerances are the ones fixed for this path: max-abs 2e-2 on O and 1e-3 on the LSE
(bf16 inputs, bf16-rounded rotated q/k and P, fp32 accumulation), and exact values on pad
rows (O = 0, LSE = -inf).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle.attention import attention
from oracle.rope import pad_angles, rope_angles_1d, rope_angles_3d

O_TOL = 2e-2
LSE_TOL = 1e-3


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    """fp32 array of bf16-exact values -> bf16 CUDA tensor (exact)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def oracle_angles_self(case):
    """(angles_q, angles_k) for the oracle, or (None, None)."""
    if case.rope is None:
        return None, None
    if case.rope == "1d":
        aq = pad_angles(rope_angles_1d(np.arange(case.q_valid) + case.q_pos_offset, case.D, case.theta), case.Sq)
        ak = pad_angles(rope_angles_1d(np.arange(int(case.kv_valid)) + case.k_pos_offset, case.D, case.theta), case.Skv)
        return aq, ak
    T, Hh, W = case.grid
    a = rope_angles_3d(T, Hh, W, case.D, case.axis_dims, case.theta)
    return pad_angles(a, case.Sq), pad_angles(a, case.Skv)


def gpu_tables_self(lib, case):
    """Device (cos_q, sin_q, cos_k, sin_k) built by the library's host table builders."""
    if case.rope is None:
        return None, None, None, None
    if case.rope == "1d":
        cq, sq = lib.dit_rope_table_1d(case.Sq, case.q_valid, case.D, case.theta, case.q_pos_offset)
        ck, sk = lib.dit_rope_table_1d(case.Skv, int(case.kv_valid), case.D, case.theta, case.k_pos_offset)
    else:
        cq, sq = lib.dit_rope_table_3d(case.Sq, case.grid, case.D, case.axis_dims, case.theta)
        ck, sk = lib.dit_rope_table_3d(case.Skv, case.grid, case.D, case.axis_dims, case.theta)
    return tuple(torch.from_numpy(t).cuda() for t in (cq, sq, ck, sk))


def run_self(lib, case, q, k, v):
    """CUDA path for a self-attention case; returns (O fp32 numpy, LSE numpy)."""
    tabs = gpu_tables_self(lib, case)
    out, lse = lib.dit_attn_fwd(dev_bf16(q), dev_bf16(k), dev_bf16(v), case.q_valid,
                                int(case.kv_valid), *tabs, softmax_scale=case.scale)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def compare(O_gpu, L_gpu, O_ref, L_ref, q_valid, rows=None, heads=None):
    """Asserts parity on valid rows and exactness on pad rows. O_gpu/L_gpu are full
    [B, Sq, H, (D)] arrays; O_ref/L_ref are the oracle's values on `rows` x `heads`."""
    Sq = O_gpu.shape[1]
    rows = np.arange(Sq) if rows is None else np.asarray(rows)
    heads = np.arange(O_gpu.shape[2]) if heads is None else np.asarray(heads)
    Og = O_gpu[:, rows][:, :, heads]
    Lg = L_gpu[:, rows][:, :, heads]
    valid = rows < q_valid
    # pad rows: exact
    assert np.all(Og[:, ~valid] == 0.0), "pad rows of O must be exactly 0"
    assert np.all(Lg[:, ~valid] == -np.inf), "pad rows of LSE must be -inf"
    ov, lv = Og[:, valid], Lg[:, valid]
    orf, lrf = O_ref[:, valid], L_ref[:, valid]
    assert np.all(np.isfinite(ov)), "non-finite O on a valid row"
    fin = np.isfinite(lrf)
    assert np.array_equal(np.isfinite(lv), fin), "LSE finiteness differs from the oracle"
    o_err = float(np.max(np.abs(ov - orf))) if ov.size else 0.0
    l_err = float(np.max(np.abs(lv[fin] - lrf[fin]))) if fin.any() else 0.0
    assert o_err <= O_TOL, f"O max-abs error {o_err} > {O_TOL}"
    assert l_err <= LSE_TOL, f"LSE max-abs error {l_err} > {LSE_TOL}"
    return o_err, l_err


def oracle_self(case, q, k, v, rows=None, heads=None):
    aq, ak = oracle_angles_self(case)
    return attention(q, k, v, case.q_valid, case.kv_valid, case.scale, aq, ak, rows=rows, heads=heads)

"""dit_attn_fwd_ws_static, whose scratch is the library's fixed device array, against
dit_attn_fwd_ws with a workspace the caller allocates, on calls issued back to back.

The file name sorts last so that it also runs after every other GPU test in one session."""
import dataclasses

import numpy as np
import pytest
import torch

from helpers import LSE_TOL, O_TOL, dev_bf16, gpu_tables_self
from video_dit_attention_gb300.inputs import AttnCase, make_qkv, tiny_case, wan480_case

pytestmark = pytest.mark.gpu


def _inputs(lib, case):
    q, k, v = make_qkv(case)
    return (dev_bf16(q), dev_bf16(k), dev_bf16(v)), gpu_tables_self(lib, case)


def _existing(lib, case, qkv, tabs):
    return lib.dit_attn_fwd_ws(*qkv, case.q_valid, int(case.kv_valid), *tabs, softmax_scale=case.scale)


def _static(lib, case, qkv, tabs):
    return lib.dit_attn_fwd_ws_static(*qkv, case.q_valid, int(case.kv_valid), *tabs,
                                      softmax_scale=case.scale)


def _assert_close(got, ref, q_valid):
    (og, lg), (orf, lrf) = got, ref
    og, orf = og.float().cpu(), orf.float().cpu()
    lg, lrf = lg.cpu(), lrf.cpu()
    assert torch.equal(torch.isfinite(lg), torch.isfinite(lrf))
    fin = torch.isfinite(lrf)
    assert torch.max(torch.abs(og - orf)).item() <= O_TOL
    if fin.any():
        assert torch.max(torch.abs(lg[fin] - lrf[fin])).item() <= LSE_TOL
    assert torch.all(og[:, q_valid:] == 0) and torch.all(lg[:, q_valid:] == -np.inf)


def test_static_scratch_two_problems_in_a_row(lib):
    """A small 1-D RoPE problem (D 64) and the Wan 480p problem (D 128), issued one after
    the other on the same stream with no synchronisation between them."""
    a, b = tiny_case(), wan480_case()
    ia, ib = _inputs(lib, a), _inputs(lib, b)
    ra, rb = _existing(lib, a, *ia), _existing(lib, b, *ib)
    torch.cuda.synchronize()
    sa = _static(lib, a, *ia)
    sb = _static(lib, b, *ib)
    torch.cuda.synchronize()
    _assert_close(sa, ra, a.q_valid)
    _assert_close(sb, rb, b.q_valid)
    assert lib.dit_device_status() == 0


def test_static_scratch_same_shape_twice(lib):
    """Two calls of one shape with different inputs: nothing of the first call's scratch
    (rotated k copy, barrier word) leaks into the second."""
    c1 = AttnCase("ws-static", B=2, H=3, D=128, Sq=640, Skv=768, q_valid=601, kv_valid=700,
                  rope="1d", seed=90)
    c2 = dataclasses.replace(c1, seed=91)
    i1, i2 = _inputs(lib, c1), _inputs(lib, c2)
    s1 = _static(lib, c1, *i1)
    s2 = _static(lib, c2, *i2)
    torch.cuda.synchronize()
    r1, r2 = _existing(lib, c1, *i1), _existing(lib, c2, *i2)
    torch.cuda.synchronize()
    _assert_close(s1, r1, c1.q_valid)
    _assert_close(s2, r2, c2.q_valid)
    assert lib.dit_device_status() == 0


def test_static_scratch_rejects_problems_beyond_its_size(lib):
    B, S, H, D = 1, 9856, 40, 128            # 96.25 MiB of rotated keys > 96 MiB
    assert lib.dit_attn_workspace_bytes(B, S, S, H, D) > lib.DIT_ATTN_STATIC_SCRATCH_BYTES
    x = torch.zeros((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    t = torch.zeros((S, D // 2), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError, match="more than the library's fixed"):
        lib.dit_attn_fwd_ws_static(x, x, x, S, S, t, t, t, t)
    out = torch.empty_like(x)
    lse = torch.empty((B, S, H), dtype=torch.float32, device="cuda")
    p = lambda z: z.data_ptr()
    st = lib._lib.dit_attn_fwd_ws_static(p(x), p(x), p(x), B, S, S, H, D, S, S, p(t), p(t), p(t), p(t),
                                         0.125, p(out), p(lse), None)
    assert st == lib.DIT_ERR_UNSUPPORTED

"""A bounded wait that runs out, on the GPU, without faulting or hanging it.

Every wait in the attention kernels (self-attention and short-KV cross-attention: mbarrier,
named barrier, grid counter) gives up after a time limit: it records a bit in the device
status word, raises the CTA's abort flag so the other roles fall through, waits (again with
a limit) for its own copies and MMAs in flight, frees tensor memory and returns. These tests
exercise that path through the test-only library libdit_attn_testhooks.so (the product
sources compiled with DIT_TEST_HOOKS), whose wait limit a test can shorten and whose K/V
producers can be told to count one load (or one fill) without issuing it, a flag that
nothing else sets. Nothing faults or traps: the kernel gives up and
exits, and the next call on the same device computes the right result.
"""
import ctypes
import os
import time

import numpy as np
import pytest
import torch

from helpers import compare, dev_bf16
from oracle.attention import attention
from video_dit_attention_gb300.inputs import AttnCase, make_qkv

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
TEST_LIB = os.path.join(os.path.dirname(HERE), "video_dit_attention_gb300", "libdit_attn_testhooks.so")

TIMEOUT_BITS = 0x01 | 0x02 | 0x04 | 0x08 | 0x20   # load, MMA, softmax, aux, grid
DRAIN_BIT = 0x10


@pytest.fixture(scope="module")
def tlib(lib):
    if not os.path.exists(TEST_LIB):
        pytest.fail(f"{TEST_LIB} is missing: build() links it beside the product library")
    from video_dit_attention_gb300 import dit_attn
    t = ctypes.CDLL(TEST_LIB)
    for name, (args, res) in dit_attn._SIGNATURES.items():
        fn = getattr(t, name)
        fn.argtypes, fn.restype = args, res
    t.dit_test_set_wait_hooks.argtypes = [ctypes.c_ulonglong, ctypes.c_int]
    t.dit_test_set_wait_hooks.restype = ctypes.c_int
    yield t
    t.dit_test_set_wait_hooks(2_000_000_000, -1)


def _status(t):
    out = ctypes.c_uint(0)
    assert t.dit_device_status(ctypes.byref(out), 1) == 0
    return int(out.value)


def _plain_call(t, case, qd, kd, vd, out, lse):
    """dit_attn_fwd without RoPE through the given library."""
    return t.dit_attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), case.B, case.Sq, case.Skv, case.H,
                          case.D, case.q_valid, case.kv_valid, None, None, None, None, case.scale,
                          out.data_ptr(), lse.data_ptr(), None)


@pytest.mark.parametrize("skip_load", [0, 2])
def test_wait_runs_out_and_kernel_recovers(lib, tlib, skip_load):
    """One CTA, one item of one query tile and three key tiles. The producer skips load 0
    (K_0: the first S product waits) or load 2 (V_0: the first P.V waits). The call returns
    well within a second, the status word holds timeout bits only (no drain failure), it
    clears, and the next call through the same library, and one through the product
    library, match the oracle."""
    case = AttnCase("stall", B=1, H=1, D=128, Sq=128, Skv=384, q_valid=100, kv_valid=300, seed=97)
    q, k, v = make_qkv(case)
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    out = torch.empty_like(qd)
    lse = torch.empty((case.B, case.Sq, case.H), dtype=torch.float32, device="cuda")
    assert _status(tlib) == 0
    assert tlib.dit_test_set_wait_hooks(50_000_000, skip_load) == 0   # 50 ms, one load skipped
    t0 = time.perf_counter()
    assert _plain_call(tlib, case, qd, kd, vd, out, lse) == 0
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    st = _status(tlib)
    assert st != 0 and (st & ~TIMEOUT_BITS) == 0, f"status {st:#x}"
    assert not (st & DRAIN_BIT)
    assert wall < 2.0, f"the stalled call took {wall:.2f} s"
    assert _status(tlib) == 0   # cleared by the read above

    assert tlib.dit_test_set_wait_hooks(2_000_000_000, -1) == 0
    Or, Lr = attention(q, k, v, case.q_valid, case.kv_valid, case.scale)
    assert _plain_call(tlib, case, qd, kd, vd, out, lse) == 0
    torch.cuda.synchronize()
    assert _status(tlib) == 0
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), Or, Lr, case.q_valid)
    O2, L2 = lib.dit_attn_fwd(qd, kd, vd, case.q_valid, case.kv_valid)
    torch.cuda.synchronize()
    assert lib.dit_device_status() == 0
    assert torch.equal(O2, out) and torch.equal(L2, lse)


def _cross_call(t, case, qd, kd, vd, kv, out, lse):
    """dit_cross_attn_shortkv through the given library."""
    return t.dit_cross_attn_shortkv(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), case.B, case.Sq, case.Skv,
                                    case.H, case.D, case.q_valid, kv.data_ptr(), case.scale, out.data_ptr(),
                                    lse.data_ptr(), None)


@pytest.mark.parametrize("skip_fill", [0, 1])
def test_cross_wait_runs_out_and_kernel_recovers(lib, tlib, skip_fill):
    """Short-KV cross-attention, four CTAs of one query tile each over 300 text keys (so a tile
    reads two fills: key tiles 0-1, then key tile 2). Each CTA's fill warp counts fill
    `skip_fill` without issuing it: with 0 the first S product's wait runs out; with 1 the
    tile's first two products complete and the third one's wait runs out, with the softmax
    warps, the P.V issuer and the Q loader waiting at their next steps. The call returns well
    within a second with timeout bits only (no drain failure), the bits clear, and the next
    calls, through this library and through the product library, match the oracle."""
    case = AttnCase("xstall", B=1, H=2, D=128, Sq=256, Skv=512, q_valid=200, kv_valid=[300], seed=98)
    q, k, v = make_qkv(case)
    qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    kv = torch.tensor(case.kv_valid, dtype=torch.int32, device="cuda")
    out = torch.empty_like(qd)
    lse = torch.empty((case.B, case.Sq, case.H), dtype=torch.float32, device="cuda")
    assert _status(tlib) == 0
    assert tlib.dit_test_set_wait_hooks(50_000_000, skip_fill) == 0   # 50 ms, one fill skipped
    t0 = time.perf_counter()
    assert _cross_call(tlib, case, qd, kd, vd, kv, out, lse) == 0
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    st = _status(tlib)
    assert st != 0 and (st & ~TIMEOUT_BITS) == 0, f"status {st:#x}"
    assert not (st & DRAIN_BIT)
    assert wall < 2.0, f"the stalled call took {wall:.2f} s"
    assert _status(tlib) == 0

    assert tlib.dit_test_set_wait_hooks(2_000_000_000, -1) == 0
    Or, Lr = attention(q, k, v, case.q_valid, case.kv_valid, case.scale)
    assert _cross_call(tlib, case, qd, kd, vd, kv, out, lse) == 0
    torch.cuda.synchronize()
    assert _status(tlib) == 0
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), Or, Lr, case.q_valid)
    O2, L2 = lib.dit_cross_attn_shortkv(qd, kd, vd, case.q_valid, kv)
    torch.cuda.synchronize()
    assert lib.dit_device_status() == 0
    assert torch.equal(O2, out) and torch.equal(L2, lse)

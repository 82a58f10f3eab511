"""The C-ABI library without a GPU: it loads, exports every function include/dit_attn.h
declares, its host-side table builders agree with the oracle's angles, and invalid
arguments return the documented status before any CUDA call is made."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle.rope import pad_angles, rope_angles_1d, rope_angles_3d

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dit_attn.h")
LIB = os.path.join(ROOT, "video_dit_attention_gb300", "libdit_attn.so")


@pytest.fixture(scope="module")
def clib():
    if not os.path.exists(LIB):
        from video_dit_attention_gb300.build import build
        build()
    return ctypes.CDLL(LIB)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dit_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_hot_path_calls():
    names = declared_functions()
    for n in ("dit_rope_split_halves", "dit_attn_fwd", "dit_cross_attn_shortkv", "dit_attn_lse_merge"):
        assert n in names


def test_library_exports_every_declared_symbol(clib):
    for name in declared_functions():
        assert hasattr(clib, name), f"{name} declared in dit_attn.h but not exported"


def test_binding_defines_every_declared_symbol():
    import ast
    src = open(os.path.join(ROOT, "video_dit_attention_gb300", "dit_attn.py")).read()
    defined = {n.name for n in ast.parse(src).body if isinstance(n, ast.FunctionDef)}
    missing = [n for n in declared_functions() if n not in defined and n != "dit_last_cuda_error"]
    assert not missing, missing


def _tables(clib, fn, *args, S_pad, half):
    cos = np.empty((S_pad, half), dtype=np.float32)
    sin = np.empty((S_pad, half), dtype=np.float32)
    fp = ctypes.POINTER(ctypes.c_float)
    st = fn(cos.ctypes.data_as(fp), sin.ctypes.data_as(fp), *args)
    return st, cos, sin


def test_rope_table_1d_matches_oracle_angles(clib):
    fn = clib.dit_rope_table_1d
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_double, ctypes.c_int]
    st, c, s = _tables(clib, fn, 300, 290, 64, 10000.0, 37799 - 290, S_pad=300, half=32)
    assert st == 0
    ang = pad_angles(rope_angles_1d(np.arange(290) + 37799 - 290, 64), 300)
    assert np.max(np.abs(c - np.cos(ang))) < 1e-7 and np.max(np.abs(s - np.sin(ang))) < 1e-7
    assert np.all(c[290:] == 1.0) and np.all(s[290:] == 0.0)


def test_rope_table_3d_matches_oracle_angles(clib):
    fn = clib.dit_rope_table_3d
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 8 + [ctypes.c_double]
    st, c, s = _tables(clib, fn, 4736, 3, 30, 52, 128, 44, 42, 42, 10000.0, S_pad=4736, half=64)
    assert st == 0
    ang = pad_angles(rope_angles_3d(3, 30, 52), 4736)
    assert np.max(np.abs(c - np.cos(ang))) < 1e-7 and np.max(np.abs(s - np.sin(ang))) < 1e-7
    # bad channel split
    st2, _, _ = _tables(clib, fn, 4736, 3, 30, 52, 128, 44, 42, 40, 10000.0, S_pad=4736, half=64)
    assert st2 == -2
    st3, _, _ = _tables(clib, fn, 100, 3, 30, 52, 128, 44, 42, 42, 10000.0, S_pad=100, half=64)
    assert st3 == -1


def _attn(clib):
    fn = clib.dit_attn_fwd
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 7 + [ctypes.c_void_p] * 4 + \
                  [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def test_attention_argument_validation_before_any_cuda_call(clib):
    fn = _attn(clib)
    P = 0x10000   # never dereferenced: every case below fails validation first
    base = dict(q=P, k=P, v=P, B=1, Sq=256, Skv=256, H=2, D=128, qv=256, kv=256,
                cq=None, sq=None, ck=None, sk=None, scale=0.088, out=P, lse=P, stream=None)

    def call(**over):
        a = dict(base, **over)
        return fn(a["q"], a["k"], a["v"], a["B"], a["Sq"], a["Skv"], a["H"], a["D"], a["qv"], a["kv"],
                  a["cq"], a["sq"], a["ck"], a["sk"], a["scale"], a["out"], a["lse"], a["stream"])

    assert call(q=None) == -1
    assert call(B=0) == -1
    assert call(qv=257) == -1
    assert call(kv=-1) == -1
    assert call(scale=0.0) == -1
    assert call(scale=float("nan")) == -1
    assert call(cq=P) == -1                 # some tables but not all four
    assert call(D=96) == -2
    assert call(Sq=200, qv=200) == -2
    assert call(Skv=300) == -2
    assert call(q=P + 8) == -3
    assert call(lse=P + 2) == -3


def test_cross_and_merge_validation(clib):
    cross = clib.dit_cross_attn_shortkv
    cross.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 6 + [ctypes.c_void_p, ctypes.c_float,
                                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    P = 0x10000
    assert cross(P, P, P, 2, 256, 640, 2, 128, 256, P, 0.1, P, P, None) == -2     # Skv > 512
    assert cross(P, P, P, 2, 256, 512, 2, 128, 256, None, 0.1, P, P, None) == -1  # no lengths
    merge = clib.dit_attn_lse_merge
    merge.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 5 + [ctypes.c_void_p] * 3
    assert merge(P, P, 0, 1, 8, 2, 128, P, P, None) == -1
    assert merge(P, P, 65, 1, 8, 2, 128, P, P, None) == -1
    assert merge(P, P, 2, 1, 8, 2, 32, P, P, None) == -2
    assert merge(P + 4, P, 2, 1, 8, 2, 128, P, P, None) == -3
    rope = clib.dit_rope_split_halves
    rope.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    assert rope(P, P, P, P, 1, 8, 2, 80, None) == -2
    assert rope(P, P, P + 4, P, 1, 8, 2, 64, None) == -3


def test_status_strings(clib):
    clib.dit_status_string.restype = ctypes.c_char_p
    for code in (0, -1, -2, -3, -4, -5):
        assert clib.dit_status_string(code).startswith(b"DIT_")


def test_static_scratch_size_agrees_between_header_and_binding():
    h = re.search(r"#define DIT_ATTN_STATIC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", open(HEADER).read())
    src = open(os.path.join(ROOT, "video_dit_attention_gb300", "dit_attn.py")).read()
    b = re.search(r"^DIT_ATTN_STATIC_SCRATCH_BYTES = (\d+) << (\d+)$", src, re.M)
    assert h and b and (int(h[1]) << int(h[2])) == (int(b[1]) << int(b[2])) == 96 << 20


def test_static_scratch_entry_rejects_oversized_problems_before_any_cuda_call(clib):
    fn = clib.dit_attn_fwd_ws_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 7 + [ctypes.c_void_p] * 4 + \
        [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    ws = clib.dit_attn_workspace_bytes
    ws.restype = ctypes.c_size_t
    assert ws(1, 9856, 9856, 40, 128) > 96 << 20 >= ws(1, 9728, 9728, 40, 128) >= ws(1, 4736, 4736, 40, 128)
    assert fn(None, None, None, 1, 9856, 9856, 40, 128, 9856, 9856, None, None, None, None,
              0.125, None, None, None) == -2            # DIT_ERR_UNSUPPORTED: needs 96.25 MiB
    assert fn(None, None, None, 0, 128, 128, 1, 128, 1, 1, None, None, None, None,
              0.125, None, None, None) == -1            # DIT_ERR_INVALID_ARG
    assert fn(None, None, None, 1, 128, 128, 1, 96, 1, 1, None, None, None, None,
              0.125, None, None, None) == -2            # head dim not supported


def test_fixed_m_entry_validation_before_any_cuda_call(clib):
    wsb = clib.dit_attn_fixed_m_workspace_bytes
    wsb.restype = ctypes.c_size_t
    base = clib.dit_attn_workspace_bytes
    base.restype = ctypes.c_size_t
    # the ws layout, then the key-norm maxima [B*H] u32 and q row norms [B, Sq, H] fp32, 256-aligned
    r256 = lambda n: (n + 255) // 256 * 256
    assert wsb(1, 4736, 4736, 40, 128) == base(1, 4736, 4736, 40, 128) + r256(40 * 4) + r256(4736 * 40 * 4)
    assert wsb(2, 384, 512, 3, 64) == base(2, 384, 512, 3, 64) + r256(2 * 3 * 4) + r256(2 * 384 * 3 * 4)
    assert wsb(0, 128, 128, 1, 128) == 0 and wsb(1, 128, 128, 1, 96) == 0
    fn = clib.dit_attn_fwd_ws_fixed_m
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 7 + [ctypes.c_void_p] * 4 + \
        [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
         ctypes.c_void_p, ctypes.c_void_p]
    P = 0x10000   # never dereferenced: every case below fails validation first
    need = wsb(1, 256, 256, 2, 128)

    def call(B=1, H=2, wsz=need, ws=P, cos=P, n_online=None, kv=256):
        return fn(P, P, P, B, 256, 256, H, 128, 256, kv, cos, P, P, P, 0.088, P, P, ws, wsz, n_online, None)

    assert call(cos=None) == -1                 # all four tables are required
    assert call(ws=None) == -1
    assert call(wsz=need - 1) == -1             # workspace too small
    assert call(kv=257) == -1
    assert call(B=1, H=24577, wsz=wsb(1, 256, 256, 24577, 128)) == -2   # B * H above 24576
    assert call(n_online=P + 2) == -3           # misaligned counter
    assert call(ws=P + 128) == -3               # workspace not 256-byte aligned


def test_fp8_entry_validation_before_any_cuda_call(clib):
    wsb = clib.dit_attn_fp8_workspace_bytes
    wsb.restype = ctypes.c_size_t
    r256 = lambda n: (n + 255) // 256 * 256
    B, Sq, Skv, H, D = 1, 4736, 4736, 40, 128
    ntq, ntk = Sq // 128, Skv // 128
    # e4m3 q~, k~, v^T, then tile maxima (q, k, v), q scales per tile, k and v scales per head
    expect = (r256(B * Sq * H * D) + r256(B * Skv * H * D) + r256(B * H * D * Skv) + r256(B * H * ntq * 4)
              + 2 * r256(B * H * ntk * 4) + r256(B * H * ntq * 4) + 2 * r256(B * H * 4))
    assert wsb(B, Sq, Skv, H, D) == expect
    assert wsb(1, 128, 128, 1, 64) == 0 and wsb(0, 128, 128, 1, 128) == 0
    fn = clib.dit_attn_fwd_fp8
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 7 + [ctypes.c_void_p] * 4 + \
        [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    P = 0x10000   # never dereferenced: every case below fails validation first
    need = wsb(1, 256, 256, 2, 128)

    def call(D=128, wsz=need, ws=P, tabs=(P, P, P, P), kv=256):
        return fn(P, P, P, 1, 256, 256, 2, D, 256, kv, *tabs, 0.088, P, P, ws, wsz, None)

    assert call(D=64, wsz=10 ** 9) == -2        # built for D = 128 only
    assert call(ws=None) == -1
    assert call(wsz=need - 1) == -1
    assert call(tabs=(P, None, P, P)) == -1     # some tables but not all four
    assert call(kv=257) == -1
    assert call(ws=P + 64) == -3                # workspace not 256-byte aligned
    assert call(tabs=(P + 4, P, P, P)) == -3    # tables must be 16-byte aligned
    assert call(tabs=(P, P, P + 8, P)) == -3


def test_status_bits_agree_between_header_binding_and_kernels():
    """The status-word bits the header documents are the ones the kernels set and the
    binding names."""
    text = open(HEADER).read()
    hdr = {m.group(1): int(m.group(2), 16) for m in re.finditer(r"#define (DIT_STATUS_\w+) 0x([0-9a-fA-F]+)u", text)}
    ptx = open(os.path.join(ROOT, "video_dit_attention_gb300", "csrc", "ptx.cuh")).read()
    kern = {m.group(1): 1 << int(m.group(2)) for m in re.finditer(r"(kStatus\w+) = 1u << (\d+)", ptx)}
    pairs = {"DIT_STATUS_TIMEOUT_LOAD": "kStatusTimeoutLoad", "DIT_STATUS_TIMEOUT_MMA": "kStatusTimeoutMma",
             "DIT_STATUS_TIMEOUT_SOFTMAX": "kStatusTimeoutSoftmax", "DIT_STATUS_TIMEOUT_AUX": "kStatusTimeoutRope",
             "DIT_STATUS_TIMEOUT_DRAIN": "kStatusTimeoutDrain", "DIT_STATUS_TIMEOUT_GRID": "kStatusTimeoutGrid",
             "DIT_STATUS_BAD_KV_LENGTH": "kStatusBadKvLength"}
    assert set(hdr) == set(pairs) and set(kern) == set(pairs.values())
    for h, k in pairs.items():
        assert hdr[h] == kern[k], h
    import ast
    src = open(os.path.join(ROOT, "video_dit_attention_gb300", "dit_attn.py")).read()
    consts = {t.id: n.value.value for n in ast.parse(src).body if isinstance(n, ast.Assign)
              for t in n.targets if isinstance(t, ast.Name) and t.id.startswith("DIT_STATUS_")}
    assert consts == hdr


def test_test_hook_library_is_separate_from_the_product():
    """The test-only library exports the hook (and the product calls); the product library
    does not contain it."""
    test_lib = os.path.join(ROOT, "video_dit_attention_gb300", "libdit_attn_testhooks.so")
    if not os.path.exists(test_lib):
        from video_dit_attention_gb300.build import build
        build()
    t = ctypes.CDLL(test_lib)
    assert hasattr(t, "dit_test_set_wait_hooks")
    for name in declared_functions():
        assert hasattr(t, name), name
    p = ctypes.CDLL(LIB)
    assert not hasattr(p, "dit_test_set_wait_hooks")
    hdr = open(os.path.join(ROOT, "include", "dit_attn_test_hooks.h")).read()
    assert "int dit_test_set_wait_hooks(unsigned long long wait_limit_ns, int skip_load);" in hdr


def test_sharded_workspace_size_and_argument_checks(clib):
    """The chunk plan (and so the workspace size) depends only on the arguments; invalid
    shard descriptions give 0 / the documented statuses before any CUDA call."""
    f = clib.dit_attn_sharded_workspace_bytes
    f.restype = ctypes.c_size_t
    ia = lambda v: (ctypes.c_int * len(v))(*v)
    pad, val = [9472, 9472, 9472, 9472], [9472, 9472, 9472, 9384]
    n = f(1, 1024, 32, 128, 4, ia(pad), ia(val))
    rot = sum(1 * p * 32 * 128 * 2 for p in pad)
    # the plan cuts the 4 shards into 8 chunks of 37 tiles (128 items each: ~6 per SM)
    chunks = 8
    assert n == rot + 256 + chunks * 1024 * 32 * 128 * 2 + chunks * 1024 * 32 * 4
    assert f(1, 1024, 32, 128, 4, ia(pad), ia(val)) == n
    assert f(1, 1024, 32, 96, 4, ia(pad), ia(val)) == 0          # D not supported
    assert f(1, 1024, 32, 128, 0, ia(pad), ia(val)) == 0         # no shard
    assert f(1, 1024, 32, 128, 1, ia([100]), ia([50])) == 0      # padded length not whole tiles
    assert f(1, 1024, 32, 128, 1, ia([128]), ia([129])) == 0     # valid > padded
    assert f(1, 1000, 32, 128, 1, ia([128]), ia([100])) == 0     # Sq not whole tiles
    assert f(1, 1024, 32, 128, 17, ia([128] * 17), ia([1] * 17)) == 0   # more than 16 non-empty shards
    assert f(1, 1024, 32, 128, 2, ia([0, 128]), ia([0, 100])) > 0        # an empty shard may have no rows
    assert f(1, 1024, 32, 128, 1, ia([0]), ia([0])) > 0                  # no key at all: one empty chunk
    g = clib.dit_attn_fwd_sharded
    g.restype = ctypes.c_int
    vp = ctypes.c_void_p
    fake = vp(256)
    ptrs = (vp * 1)(fake)
    args = [fake, 1, 256, 2, 128, 200, 1, ptrs, ptrs, ia([256]), ia([200]), fake, fake, ptrs, ptrs,
            ctypes.c_float(0.088), fake, fake, fake, ctypes.c_size_t(1 << 30), None]
    a = list(args); a[0] = None
    assert g(*a) == -1                       # null q
    a = list(args); a[15] = ctypes.c_float(0.0)
    assert g(*a) == -1                       # bad scale
    a = list(args); a[19] = ctypes.c_size_t(16)
    assert g(*a) == -1                       # workspace too small
    a = list(args); a[4] = 96
    assert g(*a) == -2                       # D
    a = list(args); a[18] = vp(256 + 8)
    assert g(*a) == -3                       # workspace not 256-byte aligned

"""Python binding of libdit_attn.so: one function per C-ABI entry point, same names.

This layer only marshals arguments: it checks tensor placement, dtype, layout and shapes,
allocates outputs with torch (device memory only), passes raw pointers and the current CUDA
stream, and raises ``DitError`` on a non-zero status. At the end, attn_self, attn_cross,
attn_sharded, merge and rope take unpadded tensors and compose those calls (pad, cached RoPE
tables, attention, unpad). Every step of the computation runs in
the library's CUDA kernels; there is no fallback. Importing this module raises ImportError
if the library has not been built (``video_dit_attention_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

from .padding import TILE, plan_token_padding

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdit_attn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python video_dit_attention_gb300/build.py` "
                      "(nvcc, sm_103a). There is no CPU fallback.")
_lib = ctypes.CDLL(LIB_PATH)

_vp, _i, _f, _d, _ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_longlong
_fp = ctypes.POINTER(ctypes.c_float)

_SIGNATURES = {
    "dit_status_string": ([_i], ctypes.c_char_p),
    "dit_last_cuda_error": ([], _i),
    "dit_device_status": ([ctypes.POINTER(ctypes.c_uint), _i], _i),
    "dit_rope_table_1d": ([_fp, _fp, _i, _i, _i, _d, _i], _i),
    "dit_rope_table_3d": ([_fp, _fp, _i, _i, _i, _i, _i, _i, _i, _i, _d], _i),
    "dit_rope_split_halves": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp], _i),
    "dit_attn_fwd": ([_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _vp, _vp, _vp], _i),
    "dit_cross_attn_shortkv": ([_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _f, _vp, _vp, _vp], _i),
    "dit_attn_lse_merge": ([_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp], _i),
    "dit_pad_tokens": ([_vp, _vp, _i, _i, _i, _ll, _vp], _i),
    "dit_unpad_tokens": ([_vp, _vp, _i, _i, _i, _ll, _vp], _i),
    "dit_exp2_fma_eval": ([_vp, _vp, _ll, _vp], _i),
    "dit_attn_workspace_bytes": ([_i, _i, _i, _i, _i], ctypes.c_size_t),
    "dit_attn_fwd_ws": ([_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _vp, _vp,
                         _vp, ctypes.c_size_t, _vp], _i),
    "dit_attn_fwd_ws_static": ([_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _vp,
                                _vp, _vp], _i),
    "dit_attn_fwd_ws_qknorm": ([_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _f, _vp, _vp, _vp, _vp,
                                _f, _vp, _vp, _vp, ctypes.c_size_t, _vp], _i),
    "dit_qk_rmsnorm_rope": ([_vp, _vp, _vp, _f, _vp, _vp, _i, _i, _i, _i, _vp], _i),
    "dit_attn_fixed_m_workspace_bytes": ([_i, _i, _i, _i, _i], ctypes.c_size_t),
    "dit_attn_fp8_workspace_bytes": ([_i, _i, _i, _i, _i], ctypes.c_size_t),
    "dit_attn_fwd_fp8": ([_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _vp, _vp,
                          _vp, ctypes.c_size_t, _vp], _i),
    "dit_attn_fwd_ws_fixed_m": ([_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _vp,
                                 _vp, _vp, ctypes.c_size_t, _vp, _vp], _i),
    "dit_attn_sharded_workspace_bytes": ([_i, _i, _i, _i, _i, _vp, _vp], ctypes.c_size_t),
    "dit_attn_fwd_sharded": ([_vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f, _vp, _vp,
                              _vp, ctypes.c_size_t, _vp], _i),
}
for _name, (_args, _res) in _SIGNATURES.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res

DIT_OK, DIT_ERR_INVALID_ARG, DIT_ERR_UNSUPPORTED, DIT_ERR_ALIGNMENT, DIT_ERR_CUDA, DIT_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5


class DitError(ValueError):
    """A library call returned a non-zero status."""

    def __init__(self, name, status):
        msg = _lib.dit_status_string(status).decode()
        if status == DIT_ERR_CUDA:
            msg += f" (cudaError {_lib.dit_last_cuda_error()})"
        super().__init__(f"{name}: {msg}")
        self.status = status


def _check(name, status):
    if status != DIT_OK:
        raise DitError(name, status)


def _stream_handle(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def dit_status_string(status: int) -> str:
    return _lib.dit_status_string(status).decode()


# Bits of the device status word (include/dit_attn.h).
DIT_STATUS_TIMEOUT_LOAD = 0x01
DIT_STATUS_TIMEOUT_MMA = 0x02
DIT_STATUS_TIMEOUT_SOFTMAX = 0x04
DIT_STATUS_TIMEOUT_AUX = 0x08
DIT_STATUS_TIMEOUT_DRAIN = 0x10
DIT_STATUS_TIMEOUT_GRID = 0x20
DIT_STATUS_BAD_KV_LENGTH = 0x40


def dit_device_status(clear: bool = True) -> int:
    """Status word of the current device: bits of kernels that gave up on a bounded wait
    (DIT_STATUS_TIMEOUT_*) and of cross-attention calls given a key length out of range
    (DIT_STATUS_BAD_KV_LENGTH)."""
    out = ctypes.c_uint(0)
    _check("dit_device_status", _lib.dit_device_status(ctypes.byref(out), 1 if clear else 0))
    return int(out.value)


# ----------------------------------------------------------------------------- RoPE tables
def dit_rope_table_1d(S_pad: int, L: int, D: int, theta: float = 10000.0, pos_offset: int = 0):
    """Host cos/sin tables [S_pad, D/2] fp32 (numpy) for positions pos_offset .. pos_offset+L-1;
    rows >= L are the identity rotation."""
    cos = np.empty((S_pad, D // 2), dtype=np.float32)
    sin = np.empty((S_pad, D // 2), dtype=np.float32)
    _check("dit_rope_table_1d", _lib.dit_rope_table_1d(
        cos.ctypes.data_as(_fp), sin.ctypes.data_as(_fp), S_pad, L, D, float(theta), pos_offset))
    return cos, sin


def dit_rope_table_3d(S_pad: int, grid, D: int = 128, axis_dims=(44, 42, 42), theta: float = 10000.0):
    """Host cos/sin tables [S_pad, D/2] fp32 (numpy) for a T x Hh x W token grid (row-major);
    rows >= T*Hh*W are the identity rotation."""
    T, Hh, W = grid
    cos = np.empty((S_pad, D // 2), dtype=np.float32)
    sin = np.empty((S_pad, D // 2), dtype=np.float32)
    _check("dit_rope_table_3d", _lib.dit_rope_table_3d(
        cos.ctypes.data_as(_fp), sin.ctypes.data_as(_fp), S_pad, T, Hh, W, D,
        axis_dims[0], axis_dims[1], axis_dims[2], float(theta)))
    return cos, sin


# ----------------------------------------------------------------------------- device calls
def dit_rope_split_halves(x, cos, sin, out=None, stream=None):
    """y = split-halves RoPE of x [B, S, H, D] bf16 with device tables [S, D/2] fp32.
    out may be x itself (in place)."""
    _need(x, "x", torch.bfloat16, 4)
    B, S, H, D = x.shape
    _need(cos, "cos", torch.float32, 2)
    _need(sin, "sin", torch.float32, 2)
    if tuple(cos.shape) != (S, D // 2) or tuple(sin.shape) != (S, D // 2):
        raise ValueError(f"tables must be [{S}, {D // 2}]")
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", torch.bfloat16, 4)
    if out.shape != x.shape:
        raise ValueError("out must have x's shape")
    _check("dit_rope_split_halves", _lib.dit_rope_split_halves(
        _ptr(x), _ptr(out), _ptr(cos), _ptr(sin), B, S, H, D, _stream_handle(stream)))
    return out


def _attn_outputs(q, out, lse):
    B, Sq, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Sq, H), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    if out.shape != q.shape or tuple(lse.shape) != (B, Sq, H):
        raise ValueError("out must be [B, Sq, H, D] and lse [B, Sq, H]")
    return out, lse


def dit_attn_fwd(q, k, v, q_valid_len: int, kv_valid_len: int, cos_q=None, sin_q=None,
                 cos_k=None, sin_k=None, softmax_scale=None, out=None, lse=None, stream=None):
    """Masked attention over padded BSHD bf16 tensors, RoPE fused when tables are given.
    Returns (out [B, Sq, H, D] bf16, lse [B, Sq, H] fp32, natural log)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    if tuple(k.shape) != (B, Skv, H, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Skv, H, D] matching q")
    tables = (cos_q, sin_q, cos_k, sin_k)
    if any(t is not None for t in tables):
        if any(t is None for t in tables):
            raise ValueError("give all four RoPE tables or none")
        for t, n, rows in ((cos_q, "cos_q", Sq), (sin_q, "sin_q", Sq), (cos_k, "cos_k", Skv), (sin_k, "sin_k", Skv)):
            _need(t, n, torch.float32, 2)
            if tuple(t.shape) != (rows, D // 2):
                raise ValueError(f"{n} must be [{rows}, {D // 2}]")
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    out, lse = _attn_outputs(q, out, lse)
    _check("dit_attn_fwd", _lib.dit_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, H, D, int(q_valid_len), int(kv_valid_len),
        _ptr(cos_q), _ptr(sin_q), _ptr(cos_k), _ptr(sin_k), scale, _ptr(out), _ptr(lse),
        _stream_handle(stream)))
    return out, lse


def dit_attn_workspace_bytes(B: int, Sq: int, Skv: int, H: int, D: int) -> int:
    """Bytes of workspace dit_attn_fwd_ws needs (rotated fp16 q and k, and a barrier word)."""
    return int(_lib.dit_attn_workspace_bytes(B, Sq, Skv, H, D))


def dit_attn_fwd_ws(q, k, v, q_valid_len: int, kv_valid_len: int, cos_q, sin_q, cos_k, sin_k,
                    workspace=None, softmax_scale=None, out=None, lse=None, stream=None):
    """dit_attn_fwd with RoPE that rotates each q/k row once into `workspace` (a uint8 CUDA
    tensor of at least dit_attn_workspace_bytes(...) bytes; allocated here if None)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    if tuple(k.shape) != (B, Skv, H, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Skv, H, D] matching q")
    for t, n, rows in ((cos_q, "cos_q", Sq), (sin_q, "sin_q", Sq), (cos_k, "cos_k", Skv), (sin_k, "sin_k", Skv)):
        _need(t, n, torch.float32, 2)
        if tuple(t.shape) != (rows, D // 2):
            raise ValueError(f"{n} must be [{rows}, {D // 2}]")
    need = dit_attn_workspace_bytes(B, Sq, Skv, H, D)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    out, lse = _attn_outputs(q, out, lse)
    _check("dit_attn_fwd_ws", _lib.dit_attn_fwd_ws(
        _ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, H, D, int(q_valid_len), int(kv_valid_len),
        _ptr(cos_q), _ptr(sin_q), _ptr(cos_k), _ptr(sin_k), scale, _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel(), _stream_handle(stream)))
    return out, lse


def dit_attn_fwd_ws_qknorm(q, k, v, q_valid_len: int, kv_valid_len: int, norm_q, norm_k, cos_q, sin_q,
                           cos_k, sin_k, eps: float = 1e-6, workspace=None, softmax_scale=None, out=None,
                           lse=None, stream=None):
    """dit_attn_fwd_ws with a per-head RMSNorm of q and k (weights norm_q, norm_k: fp32 CUDA
    tensors [D]) ahead of the rotation."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    if tuple(k.shape) != (B, Skv, H, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Skv, H, D] matching q")
    for t, n in ((norm_q, "norm_q"), (norm_k, "norm_k")):
        _need(t, n, torch.float32, 1)
        if t.shape[0] != D:
            raise ValueError(f"{n} must be [{D}]")
    for t, n, rows in ((cos_q, "cos_q", Sq), (sin_q, "sin_q", Sq), (cos_k, "cos_k", Skv), (sin_k, "sin_k", Skv)):
        _need(t, n, torch.float32, 2)
        if tuple(t.shape) != (rows, D // 2):
            raise ValueError(f"{n} must be [{rows}, {D // 2}]")
    need = dit_attn_workspace_bytes(B, Sq, Skv, H, D)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    out, lse = _attn_outputs(q, out, lse)
    _check("dit_attn_fwd_ws_qknorm", _lib.dit_attn_fwd_ws_qknorm(
        _ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, H, D, int(q_valid_len), int(kv_valid_len),
        _ptr(norm_q), _ptr(norm_k), float(eps), _ptr(cos_q), _ptr(sin_q), _ptr(cos_k), _ptr(sin_k),
        scale, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream_handle(stream)))
    return out, lse


def dit_attn_fixed_m_workspace_bytes(B: int, Sq: int, Skv: int, H: int, D: int) -> int:
    """Bytes of device workspace dit_attn_fwd_ws_fixed_m needs (0 for an invalid shape)."""
    return int(_lib.dit_attn_fixed_m_workspace_bytes(B, Sq, Skv, H, D))


def dit_attn_fwd_ws_fixed_m(q, k, v, q_valid_len: int, kv_valid_len: int, cos_q, sin_q, cos_k, sin_k,
                            workspace=None, n_online=None, softmax_scale=None, out=None, lse=None,
                            stream=None):
    """dit_attn_fwd_ws with the fixed-m softmax: 32-row query blocks whose norm bound allows it
    skip the running maximum. n_online: None or an int32/uint32-sized CUDA tensor [1] to which
    the call adds the number of blocks that took the online path (the caller zeroes it)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    if tuple(k.shape) != (B, Skv, H, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Skv, H, D] matching q")
    for t, n, rows in ((cos_q, "cos_q", Sq), (sin_q, "sin_q", Sq), (cos_k, "cos_k", Skv), (sin_k, "sin_k", Skv)):
        _need(t, n, torch.float32, 2)
        if tuple(t.shape) != (rows, D // 2):
            raise ValueError(f"{n} must be [{rows}, {D // 2}]")
    need = dit_attn_fixed_m_workspace_bytes(B, Sq, Skv, H, D)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    if n_online is not None:
        _need(n_online, "n_online", torch.int32, 1)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    out, lse = _attn_outputs(q, out, lse)
    _check("dit_attn_fwd_ws_fixed_m", _lib.dit_attn_fwd_ws_fixed_m(
        _ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, H, D, int(q_valid_len), int(kv_valid_len),
        _ptr(cos_q), _ptr(sin_q), _ptr(cos_k), _ptr(sin_k), scale, _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel(), _ptr(n_online), _stream_handle(stream)))
    return out, lse


def dit_attn_fp8_workspace_bytes(B: int, Sq: int, Skv: int, H: int, D: int) -> int:
    """Bytes of device workspace dit_attn_fwd_fp8 needs (0 for an invalid shape or D != 128)."""
    return int(_lib.dit_attn_fp8_workspace_bytes(B, Sq, Skv, H, D))


def dit_attn_fwd_fp8(q, k, v, q_valid_len: int, kv_valid_len: int, cos_q=None, sin_q=None, cos_k=None,
                     sin_k=None, workspace=None, softmax_scale=None, out=None, lse=None, stream=None):
    """FP8 (e4m3) attention (D = 128): q~ quantised per 128-row tile, k~ and v per head, P as
    e4m3(112 p) (the running maximum lags by at most 2 in log2 units); tables as in
    dit_attn_fwd (all four, or none for no RoPE)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    if tuple(k.shape) != (B, Skv, H, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Skv, H, D] matching q")
    tabs = (cos_q, sin_q, cos_k, sin_k)
    if any(t is not None for t in tabs):
        for t, n, rows in zip(tabs, ("cos_q", "sin_q", "cos_k", "sin_k"), (Sq, Sq, Skv, Skv)):
            _need(t, n, torch.float32, 2)
            if tuple(t.shape) != (rows, D // 2):
                raise ValueError(f"{n} must be [{rows}, {D // 2}]")
    need = dit_attn_fp8_workspace_bytes(B, Sq, Skv, H, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", torch.uint8, 1)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    out, lse = _attn_outputs(q, out, lse)
    _check("dit_attn_fwd_fp8", _lib.dit_attn_fwd_fp8(
        _ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, H, D, int(q_valid_len), int(kv_valid_len),
        *(_ptr(t) for t in tabs), scale, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _stream_handle(stream)))
    return out, lse


def dit_qk_rmsnorm_rope(x, w, cos, sin, eps: float = 1e-6, out=None, stream=None):
    """y = split-halves RoPE of the per-head RMSNorm of x [B, S, H, D] bf16 (weights w: fp32
    [D]; tables [S, D/2] fp32). out may be x itself (in place)."""
    _need(x, "x", torch.bfloat16, 4)
    B, S, H, D = x.shape
    _need(w, "w", torch.float32, 1)
    if w.shape[0] != D:
        raise ValueError(f"w must be [{D}]")
    _need(cos, "cos", torch.float32, 2)
    _need(sin, "sin", torch.float32, 2)
    if tuple(cos.shape) != (S, D // 2) or tuple(sin.shape) != (S, D // 2):
        raise ValueError(f"tables must be [{S}, {D // 2}]")
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", torch.bfloat16, 4)
    if out.shape != x.shape:
        raise ValueError("out must have x's shape")
    _check("dit_qk_rmsnorm_rope", _lib.dit_qk_rmsnorm_rope(
        _ptr(x), _ptr(out), _ptr(w), float(eps), _ptr(cos), _ptr(sin), B, S, H, D, _stream_handle(stream)))
    return out


# Size of the library's fixed device scratch array used by dit_attn_fwd_ws_static.
DIT_ATTN_STATIC_SCRATCH_BYTES = 96 << 20


def dit_attn_fwd_ws_static(q, k, v, q_valid_len: int, kv_valid_len: int, cos_q, sin_q, cos_k, sin_k,
                           softmax_scale=None, out=None, lse=None, stream=None):
    """dit_attn_fwd_ws with the workspace taken from the library's fixed 96 MiB device array,
    so the C call allocates nothing. Calls in flight at the same time on one device share
    that array and must not overlap; the first call on a device does a one-time set-up."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    if tuple(k.shape) != (B, Skv, H, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Skv, H, D] matching q")
    for t, n, rows in ((cos_q, "cos_q", Sq), (sin_q, "sin_q", Sq), (cos_k, "cos_k", Skv), (sin_k, "sin_k", Skv)):
        _need(t, n, torch.float32, 2)
        if tuple(t.shape) != (rows, D // 2):
            raise ValueError(f"{n} must be [{rows}, {D // 2}]")
    need = dit_attn_workspace_bytes(B, Sq, Skv, H, D)
    if need > DIT_ATTN_STATIC_SCRATCH_BYTES:
        raise ValueError(f"dit_attn_fwd_ws_static: this problem needs {need} bytes of scratch, more than "
                         f"the library's fixed {DIT_ATTN_STATIC_SCRATCH_BYTES} bytes; "
                         f"use dit_attn_fwd_ws with a caller workspace")
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    out, lse = _attn_outputs(q, out, lse)
    _check("dit_attn_fwd_ws_static", _lib.dit_attn_fwd_ws_static(
        _ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, H, D, int(q_valid_len), int(kv_valid_len),
        _ptr(cos_q), _ptr(sin_q), _ptr(cos_k), _ptr(sin_k), scale, _ptr(out), _ptr(lse),
        _stream_handle(stream)))
    return out, lse


def dit_cross_attn_shortkv(q, k, v, q_valid_len: int, kv_valid_len_dev, softmax_scale=None,
                           out=None, lse=None, stream=None):
    """Short-KV cross-attention; kv_valid_len_dev: int32 CUDA tensor [B] of valid key counts."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    _need(kv_valid_len_dev, "kv_valid_len_dev", torch.int32, 1)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    if tuple(k.shape) != (B, Skv, H, D) or v.shape != k.shape or kv_valid_len_dev.shape[0] != B:
        raise ValueError("k, v must be [B, Skv, H, D] and kv_valid_len_dev [B]")
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    out, lse = _attn_outputs(q, out, lse)
    _check("dit_cross_attn_shortkv", _lib.dit_cross_attn_shortkv(
        _ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, H, D, int(q_valid_len), _ptr(kv_valid_len_dev),
        scale, _ptr(out), _ptr(lse), _stream_handle(stream)))
    return out, lse


def _int_array(vals):
    return (ctypes.c_int * len(vals))(*[int(x) for x in vals])


def _ptr_array(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def dit_attn_sharded_workspace_bytes(B: int, Sq: int, H: int, D: int, shard_padded, shard_valid) -> int:
    n = len(shard_padded)
    return int(_lib.dit_attn_sharded_workspace_bytes(B, Sq, H, D, n, _int_array(shard_padded),
                                                     _int_array(shard_valid)))


def dit_attn_fwd_sharded(q, shards, q_valid_len: int, cos_q, sin_q, softmax_scale=None, workspace=None,
                         out=None, lse=None, stream=None):
    """Attention of padded q [B, Sq, H, D] over key shards in one call: shards is a sequence of
    (k_s, v_s, valid_s, cos_k_s, sin_k_s) with k_s, v_s [B, S_s, H, D] bf16 (S_s a multiple of
    128) and the shard's tables [S_s, D/2] fp32 at its global key positions."""
    _need(q, "q", torch.bfloat16, 4)
    B, Sq, H, D = q.shape
    ks, vs, valid, ck, sk = [], [], [], [], []
    for i, (k, v, n, c, sn) in enumerate(shards):
        _need(k, f"k[{i}]", torch.bfloat16, 4)
        _need(v, f"v[{i}]", torch.bfloat16, 4)
        _need(c, f"cos_k[{i}]", torch.float32, 2)
        _need(sn, f"sin_k[{i}]", torch.float32, 2)
        if tuple(k.shape) != (B, k.shape[1], H, D) or v.shape != k.shape:
            raise ValueError(f"shard {i}: k and v must be [B, S_s, H, D] matching q")
        ks.append(k); vs.append(v); valid.append(int(n)); ck.append(c); sk.append(sn)
    padded = [k.shape[1] for k in ks]
    _need(cos_q, "cos_q", torch.float32, 2)
    _need(sin_q, "sin_q", torch.float32, 2)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    need = dit_attn_sharded_workspace_bytes(B, Sq, H, D, padded, valid)
    if need == 0:
        raise DitError("dit_attn_sharded_workspace_bytes", -2)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    out, lse = _attn_outputs(q, out, lse)
    _check("dit_attn_fwd_sharded", _lib.dit_attn_fwd_sharded(
        _ptr(q), B, Sq, H, D, int(q_valid_len), len(ks), _ptr_array(ks), _ptr_array(vs), _int_array(padded),
        _int_array(valid), _ptr(cos_q), _ptr(sin_q), _ptr_array(ck), _ptr_array(sk), scale, _ptr(out), _ptr(lse),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()), _stream_handle(stream)))
    return out, lse


def dit_attn_lse_merge(partial_o, partial_lse, out=None, lse=None, stream=None):
    """Merges n partials: partial_o [n, B, S, H, D] bf16, partial_lse [n, B, S, H] fp32."""
    _need(partial_o, "partial_o", torch.bfloat16, 5)
    _need(partial_lse, "partial_lse", torch.float32, 4)
    n, B, S, H, D = partial_o.shape
    if tuple(partial_lse.shape) != (n, B, S, H):
        raise ValueError("partial_lse must be [n, B, S, H]")
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=partial_o.device)
    if lse is None:
        lse = torch.empty((B, S, H), dtype=torch.float32, device=partial_o.device)
    _need(out, "out", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    _check("dit_attn_lse_merge", _lib.dit_attn_lse_merge(
        _ptr(partial_o), _ptr(partial_lse), n, B, S, H, D, _ptr(out), _ptr(lse), _stream_handle(stream)))
    return out, lse


def dit_pad_tokens(x, S_pad: int, out=None, stream=None):
    """Copies x [B, L, ...] into the first L rows of a [B, S_pad, ...] buffer (pad rows untouched)."""
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    B, L = x.shape[:2]
    if out is None:
        out = torch.empty((B, S_pad) + tuple(x.shape[2:]), dtype=x.dtype, device=x.device)
    if not out.is_contiguous() or out.dtype != x.dtype or tuple(out.shape) != (B, S_pad) + tuple(x.shape[2:]):
        raise ValueError("out must be a contiguous [B, S_pad, ...] tensor of x's dtype")
    row_bytes = x[0, 0].numel() * x.element_size() if L > 0 else out[0, 0].numel() * out.element_size()
    _check("dit_pad_tokens", _lib.dit_pad_tokens(_ptr(x), _ptr(out), B, L, S_pad, row_bytes,
                                                 _stream_handle(stream)))
    return out


def dit_unpad_tokens(x_pad, L: int, out=None, stream=None):
    """Copies the first L rows of x_pad [B, S_pad, ...] into a [B, L, ...] tensor."""
    if not x_pad.is_cuda or not x_pad.is_contiguous():
        raise ValueError("x_pad must be a contiguous CUDA tensor")
    B, S_pad = x_pad.shape[:2]
    if out is None:
        out = torch.empty((B, L) + tuple(x_pad.shape[2:]), dtype=x_pad.dtype, device=x_pad.device)
    if not out.is_contiguous() or out.dtype != x_pad.dtype or tuple(out.shape) != (B, L) + tuple(x_pad.shape[2:]):
        raise ValueError("out must be a contiguous [B, L, ...] tensor of x_pad's dtype")
    row_bytes = x_pad[0, 0].numel() * x_pad.element_size()
    _check("dit_unpad_tokens", _lib.dit_unpad_tokens(_ptr(x_pad), _ptr(out), B, L, S_pad, row_bytes,
                                                     _stream_handle(stream)))
    return out


def dit_exp2_fma_eval(x, out=None, stream=None):
    """Diagnostic: the softmax's FMA-pipe 2^x applied to a float32 CUDA tensor."""
    _need(x, "x", torch.float32)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", torch.float32)
    _check("dit_exp2_fma_eval", _lib.dit_exp2_fma_eval(_ptr(x), _ptr(out), x.numel(), _stream_handle(stream)))
    return out


# ----------------------------------------------------------------------------- unpadded layer
# What a model calls: unpadded [B, L, H, D] bf16 tensors in, unpadded O [B, L, H, D] bf16 and
# LSE [B, L, H] fp32 (natural log) out. Each call pads to whole 128-row tiles on the device
# (dit_pad_tokens; pad rows keep whatever the buffer held, since no kernel reads them), takes
# its RoPE tables from a per-geometry cache (built once by the host table functions and kept
# on the device, as the pages build them once per forward and share them across blocks),
# calls one attention entry point and cuts the pad (dit_unpad_tokens). Sequences already a
# whole number of tiles go in and out without copies.
_MODES = ("exact", "fixed_m", "fp8")
_TABLE_CACHE: dict = {}
_TABLE_CACHE_MAX = 64


def _tiles(n: int) -> int:
    """Padded length of n rows: whole tiles, at least one (a 0-row key set still needs a
    buffer; its valid length 0 gives O = 0 and LSE = -inf)."""
    return max(TILE, plan_token_padding(n))


def rope_tables(S_pad: int, D: int, rope, device, L: int = None, pos_offset: int = 0,
                theta: float = 10000.0, axis_dims=(44, 42, 42)):
    """Device (cos, sin) [S_pad, D/2] fp32 tables, cached per geometry and device.

    rope = "1d": positions pos_offset .. pos_offset + L - 1 on rows 0 .. L - 1.
    rope = (T, Hh, W): the 3-D latent grid (rows 0 .. T*Hh*W - 1, t slowest).
    Rows past the valid ones are the identity rotation."""
    dev = torch.device(device)
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if rope == "1d":
        if L is None:
            raise ValueError("rope_tables: a 1-D table needs L")
        key = ("1d", S_pad, D, int(L), int(pos_offset), float(theta), str(dev))
    else:
        grid = tuple(int(x) for x in rope)
        key = ("3d", S_pad, D, grid, tuple(int(x) for x in axis_dims), float(theta), str(dev))
    hit = _TABLE_CACHE.get(key)
    if hit is not None:
        return hit
    if rope == "1d":
        c, s = dit_rope_table_1d(S_pad, int(L), D, theta, int(pos_offset))
    else:
        c, s = dit_rope_table_3d(S_pad, key[3], D, axis_dims, theta)
    if len(_TABLE_CACHE) >= _TABLE_CACHE_MAX:
        _TABLE_CACHE.clear()
    hit = (torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev))
    _TABLE_CACHE[key] = hit
    return hit


def _pad(x, S_pad, stream):
    if x.shape[1] == S_pad:
        return x
    if x.shape[1] == 0:       # nothing to copy (and an empty tensor has no data pointer)
        return torch.empty((x.shape[0], S_pad) + tuple(x.shape[2:]), dtype=x.dtype, device=x.device)
    return dit_pad_tokens(x, S_pad, stream=stream)


def _unpad(x, L, stream):
    return x if x.shape[1] == L else dit_unpad_tokens(x, L, stream=stream)


def _check_grid(rope, Lq, Lk):
    if rope is None or rope == "1d":
        return
    try:
        grid = tuple(int(x) for x in rope)
    except TypeError:
        raise ValueError(f'rope must be None, "1d" or a (T, Hh, W) grid, got {rope!r}') from None
    if len(grid) != 3 or min(grid) < 1:
        raise ValueError(f"a 3-D RoPE grid is (T, Hh, W) with positive sizes, got {rope!r}")
    if Lq != Lk or grid[0] * grid[1] * grid[2] != Lq:
        raise ValueError(f"a 3-D grid {grid} needs Lq = Lk = T*Hh*W (got Lq={Lq}, Lk={Lk})")


def attn_self(q, k, v, rope=None, *, mode: str = "exact", norm_q=None, norm_k=None, eps: float = 1e-6,
              q_pos_offset: int = 0, k_pos_offset: int = 0, theta: float = 10000.0, axis_dims=(44, 42, 42),
              softmax_scale=None, stream=None):
    """Attention of unpadded q [B, Lq, H, D] over unpadded k, v [B, Lk, H, D] (bf16, CUDA).

    rope: None; "1d" (query i at position q_pos_offset + i, key j at k_pos_offset + j); or a
    (T, Hh, W) latent grid for 3-D RoPE (Lq = Lk = T*Hh*W).
    mode: "exact" (dit_attn_fwd_ws with RoPE, dit_attn_fwd without), "fixed_m"
    (dit_attn_fwd_ws_fixed_m, needs RoPE) or "fp8" (dit_attn_fwd_fp8, D = 128).
    norm_q, norm_k: fp32 CUDA [D] weights of a per-head RMSNorm of q and k ahead of the
    rotation (dit_attn_fwd_ws_qknorm: exact mode, with RoPE).
    Returns (out [B, Lq, H, D] bf16, lse [B, Lq, H] fp32)."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, L, H, D]")
    B, Lq, H, D = q.shape
    Lk = k.shape[1]
    if tuple(k.shape) != (B, Lk, H, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Lk, H, D] matching q")
    if mode not in _MODES:
        raise ValueError(f"mode must be one of {_MODES}, got {mode!r}")
    normed = norm_q is not None or norm_k is not None
    if normed and (norm_q is None or norm_k is None):
        raise ValueError("give both norm_q and norm_k, or neither")
    if normed and (rope is None or mode != "exact"):
        raise ValueError("the fused q/k RMSNorm runs in the exact mode with RoPE")
    if mode == "fixed_m" and rope is None:
        raise ValueError("the fixed-m mode runs with RoPE")
    _check_grid(rope, Lq, Lk)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    if Lq == 0:
        return (torch.empty((B, 0, H, D), dtype=torch.bfloat16, device=q.device),
                torch.empty((B, 0, H), dtype=torch.float32, device=q.device))
    Sq, Skv = _tiles(Lq), _tiles(Lk)
    qp, kp, vp = _pad(q, Sq, stream), _pad(k, Skv, stream), _pad(v, Skv, stream)
    if rope is None:
        tabs = ()
    elif rope == "1d":
        tabs = rope_tables(Sq, D, "1d", q.device, L=Lq, pos_offset=q_pos_offset, theta=theta) + \
               rope_tables(Skv, D, "1d", q.device, L=Lk, pos_offset=k_pos_offset, theta=theta)
    else:
        t3 = rope_tables(Sq, D, rope, q.device, theta=theta, axis_dims=axis_dims)
        tabs = t3 + t3
    kw = dict(softmax_scale=softmax_scale, stream=stream)
    if mode == "fp8":
        op, lp = dit_attn_fwd_fp8(qp, kp, vp, Lq, Lk, *tabs, **kw)
    elif mode == "fixed_m":
        op, lp = dit_attn_fwd_ws_fixed_m(qp, kp, vp, Lq, Lk, *tabs, **kw)
    elif normed:
        op, lp = dit_attn_fwd_ws_qknorm(qp, kp, vp, Lq, Lk, norm_q, norm_k, *tabs, eps=eps, **kw)
    elif tabs:
        op, lp = dit_attn_fwd_ws(qp, kp, vp, Lq, Lk, *tabs, **kw)
    else:
        op, lp = dit_attn_fwd(qp, kp, vp, Lq, Lk, **kw)
    return _unpad(op, Lq, stream), _unpad(lp, Lq, stream)


def attn_cross(q, k, v, kv_valid_len, *, softmax_scale=None, stream=None):
    """Short-KV cross-attention of unpadded q [B, Lq, H, D] against k, v [B, Lk, H, D]
    (bf16, CUDA, Lk <= 512): batch b attends to its first kv_valid_len[b] keys
    (a sequence of B host integers in [0, Lk]). No RoPE.
    Returns (out [B, Lq, H, D] bf16, lse [B, Lq, H] fp32)."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, L, H, D]")
    B, Lq, H, D = q.shape
    Lk = k.shape[1]
    if tuple(k.shape) != (B, Lk, H, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Lk, H, D] matching q")
    if Lk > 512:
        raise ValueError(f"the short-KV path takes at most 512 keys, got {Lk}")
    lens = [int(x) for x in kv_valid_len]
    if len(lens) != B or min(lens) < 0 or max(lens) > Lk:
        raise ValueError(f"kv_valid_len must hold B={B} integers in [0, {Lk}], got {lens}")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    if Lq == 0:
        return (torch.empty((B, 0, H, D), dtype=torch.bfloat16, device=q.device),
                torch.empty((B, 0, H), dtype=torch.float32, device=q.device))
    Sq, Skv = _tiles(Lq), _tiles(Lk)
    qp, kp, vp = _pad(q, Sq, stream), _pad(k, Skv, stream), _pad(v, Skv, stream)
    kv_dev = torch.tensor(lens, dtype=torch.int32).to(q.device)
    op, lp = dit_cross_attn_shortkv(qp, kp, vp, Lq, kv_dev, softmax_scale=softmax_scale, stream=stream)
    return _unpad(op, Lq, stream), _unpad(lp, Lq, stream)


def attn_sharded(q, shards, rope="1d", *, q_pos_offset: int = 0, theta: float = 10000.0,
                 softmax_scale=None, stream=None):
    """Attention of unpadded q [B, Lq, H, D] over keys held in shards [(k_0, v_0), (k_1, v_1),
    ...] (each [B, L_s, H, D] bf16, CUDA, in global key order). With rope = "1d" every key
    keeps its global position (shard s starts after the keys of shards 0 .. s-1) and query i
    sits at q_pos_offset + i: one dit_attn_fwd_sharded call (all shards in one launch, then
    the LSE merge). rope = None runs one partial per shard without RoPE, then the merge.
    Returns (out [B, Lq, H, D] bf16, lse [B, Lq, H] fp32)."""
    if rope not in (None, "1d"):
        raise ValueError('attn_sharded takes rope = "1d" or None')
    if not 1 <= len(shards) <= 64:
        raise ValueError(f"between 1 and 64 shards, got {len(shards)}")
    if q.dim() != 4:
        raise ValueError("q must be [B, L, H, D]")
    B, Lq, H, D = q.shape
    for s, (ks, vs) in enumerate(shards):
        if ks.dim() != 4 or tuple(ks.shape) != (B, ks.shape[1], H, D) or vs.shape != ks.shape:
            raise ValueError(f"shard {s}: k and v must be [B, L_s, H, D] matching q")
    _need(q, "q", torch.bfloat16, 4)
    for s, (ks, vs) in enumerate(shards):
        _need(ks, f"k[{s}]", torch.bfloat16, 4)
        _need(vs, f"v[{s}]", torch.bfloat16, 4)
    if Lq == 0:
        return (torch.empty((B, 0, H, D), dtype=torch.bfloat16, device=q.device),
                torch.empty((B, 0, H), dtype=torch.float32, device=q.device))
    n, Sq = len(shards), _tiles(Lq)
    qp = _pad(q, Sq, stream)
    if rope:
        tq = rope_tables(Sq, D, "1d", q.device, L=Lq, pos_offset=q_pos_offset, theta=theta)
        entries, offset = [], 0
        for ks, vs in shards:
            Ls = ks.shape[1]
            Ss = _tiles(Ls)
            kp, vp = _pad(ks, Ss, stream), _pad(vs, Ss, stream)
            tk = rope_tables(Ss, D, "1d", q.device, L=Ls, pos_offset=offset, theta=theta)
            entries.append((kp, vp, Ls, *tk))
            offset += Ls
        op, lp = dit_attn_fwd_sharded(qp, entries, Lq, *tq, softmax_scale=softmax_scale, stream=stream)
        return _unpad(op, Lq, stream), _unpad(lp, Lq, stream)
    po = torch.empty((n, B, Sq, H, D), dtype=torch.bfloat16, device=q.device)
    pl = torch.empty((n, B, Sq, H), dtype=torch.float32, device=q.device)
    for s, (ks, vs) in enumerate(shards):
        Ls = ks.shape[1]
        Ss = _tiles(Ls)
        kp, vp = _pad(ks, Ss, stream), _pad(vs, Ss, stream)
        dit_attn_fwd(qp, kp, vp, Lq, Ls, softmax_scale=softmax_scale, out=po[s], lse=pl[s], stream=stream)
    op, lp = dit_attn_lse_merge(po, pl, stream=stream)
    return _unpad(op, Lq, stream), _unpad(lp, Lq, stream)


def merge(partial_o, partial_lse, stream=None):
    """LSE merge of n partials, given stacked ([n, B, S, H, D] bf16, [n, B, S, H] fp32) or as
    sequences of n [B, S, H, D] / [B, S, H] tensors. Returns (out, lse)."""
    if isinstance(partial_o, (list, tuple)):
        partial_o = torch.stack(list(partial_o))
    if isinstance(partial_lse, (list, tuple)):
        partial_lse = torch.stack(list(partial_lse))
    return dit_attn_lse_merge(partial_o.contiguous(), partial_lse.contiguous(), stream=stream)


def rope(x, rope, *, pos_offset: int = 0, norm=None, eps: float = 1e-6, theta: float = 10000.0,
         axis_dims=(44, 42, 42), out=None, stream=None):
    """Split-halves RoPE of unpadded x [B, L, H, D] bf16 (CUDA): rope = "1d" (row i at
    position pos_offset + i) or a (T, Hh, W) grid (L = T*Hh*W). With norm (fp32 CUDA [D]
    weights) a per-head RMSNorm comes first (dit_qk_rmsnorm_rope). out may be x."""
    if x.dim() != 4:
        raise ValueError("x must be [B, L, H, D]")
    B, L, H, D = x.shape
    if rope is None:
        raise ValueError('rope must be "1d" or a (T, Hh, W) grid')
    _check_grid(rope, L, L)
    _need(x, "x", torch.bfloat16, 4)
    if L == 0:
        return x if out is None else out
    if rope == "1d":
        c, s = rope_tables(L, D, "1d", x.device, L=L, pos_offset=pos_offset, theta=theta)
    else:
        c, s = rope_tables(L, D, rope, x.device, theta=theta, axis_dims=axis_dims)
    if norm is not None:
        return dit_qk_rmsnorm_rope(x, norm, c, s, eps=eps, out=out, stream=stream)
    return dit_rope_split_halves(x, c, s, out=out, stream=stream)

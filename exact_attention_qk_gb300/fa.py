"""Thin Python binding of libfa.so (ctypes). Argument marshalling only.

Every function here has the name of the C entry point it calls (include/fa.h).
Tensors are torch CUDA tensors; PyTorch allocates device memory and supplies
the stream, the library computes. There is no fallback: if libfa.so is missing
or fails to load, importing this module raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_ALIGNMENT = 3
FA_ERR_WORKSPACE = 4
FA_ERR_LAUNCH = 5
FA_ERR_DEVICE_TIMEOUT = 6
FA_ERR_CUDA = 7


class FaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: status {code} ({fa_status_string(code)})")
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")

_lib = ctypes.CDLL(LIB_PATH)


class FwdArgs(ctypes.Structure):
    """Mirror of `fa_fwd_args` in include/fa.h (same field order and types)."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("q_batch_stride", ctypes.c_int64), ("q_row_stride", ctypes.c_int64), ("q_head_stride", ctypes.c_int64),
        ("k_batch_stride", ctypes.c_int64), ("k_row_stride", ctypes.c_int64), ("k_head_stride", ctypes.c_int64),
        ("v_batch_stride", ctypes.c_int64), ("v_row_stride", ctypes.c_int64), ("v_head_stride", ctypes.c_int64),
        ("o_batch_stride", ctypes.c_int64), ("o_row_stride", ctypes.c_int64), ("o_head_stride", ctypes.c_int64),
        ("batch", ctypes.c_int32), ("seqlen_q", ctypes.c_int32), ("seqlen_k", ctypes.c_int32),
        ("num_heads_q", ctypes.c_int32), ("num_heads_kv", ctypes.c_int32),
        ("head_dim_qk", ctypes.c_int32), ("head_dim_v", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p), ("seqused_k", ctypes.c_void_p),
        ("total_q", ctypes.c_int32), ("total_k", ctypes.c_int32),
        ("max_seqlen_q", ctypes.c_int32), ("max_seqlen_k", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("causal", ctypes.c_int32), ("window_left", ctypes.c_int32), ("window_right", ctypes.c_int32),
        ("num_splits", ctypes.c_int32),
        ("kv_format", ctypes.c_int32), ("k_descale", ctypes.c_void_p), ("v_descale", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("max_pages_per_seq", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
    ]


# K/V element formats (fa.h FA_KV_*)
KV_FORMATS = {"bf16": 0, "e4m3": 1, "e5m2": 2}


def _kv_format_of(k: torch.Tensor, kv_format) -> int:
    if kv_format is not None:
        return KV_FORMATS[kv_format] if isinstance(kv_format, str) else int(kv_format)
    if hasattr(torch, "float8_e4m3fn") and k.dtype == torch.float8_e4m3fn:
        return KV_FORMATS["e4m3"]
    if hasattr(torch, "float8_e5m2") and k.dtype == torch.float8_e5m2:
        return KV_FORMATS["e5m2"]
    if k.dtype == torch.uint8:
        raise ValueError("uint8 K/V need kv_format='e4m3' or 'e5m2'")
    return KV_FORMATS["bf16"]


_P = ctypes.POINTER(FwdArgs)
_vp = ctypes.c_void_p
_lib.fa_fwd.argtypes = [_P, _vp, ctypes.c_size_t, _vp]
_lib.fa_fwd.restype = ctypes.c_int
_lib.fa_fwd_splitkv.argtypes = [_P, ctypes.c_int, _vp, _vp, _vp, ctypes.c_size_t, _vp]
_lib.fa_fwd_splitkv.restype = ctypes.c_int
_lib.fa_combine.argtypes = [_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                            _vp, ctypes.c_int, _vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _vp, _vp]
_lib.fa_combine.restype = ctypes.c_int
_lib.fa_workspace_size.argtypes = [_P]
_lib.fa_workspace_size.restype = ctypes.c_size_t
_lib.fa_num_splits.argtypes = [_P, ctypes.c_int]
_lib.fa_num_splits.restype = ctypes.c_int
_lib.fa_split_len.argtypes = [_P, ctypes.c_int]
_lib.fa_split_len.restype = ctypes.c_int
_lib.fa_get_status.argtypes = [_vp]
_lib.fa_get_status.restype = ctypes.c_int
_lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
_lib.fa_set_wait_timeout_ns.restype = None
_lib.fa_status_string.argtypes = [ctypes.c_int]
_lib.fa_status_string.restype = ctypes.c_char_p
_lib.fa_fwd_decode_noalloc.argtypes = [_P, _vp]
_lib.fa_fwd_decode_noalloc.restype = ctypes.c_int
_lib.fa_bwd.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
_lib.fa_bwd.restype = ctypes.c_int
_lib.fa_bwd_two_streams.argtypes = [_P, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp]
_lib.fa_bwd_two_streams.restype = ctypes.c_int
_lib.fa_bwd_workspace_size.argtypes = [_P]
_lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
_lib.fa_abi_version.argtypes = []
_lib.fa_abi_version.restype = ctypes.c_int


def lib() -> ctypes.CDLL:
    return _lib


def fa_status_string(code: int) -> str:
    return _lib.fa_status_string(int(code)).decode()


def fa_abi_version() -> int:
    return _lib.fa_abi_version()


def fa_set_wait_timeout_ns(ns: int) -> None:
    _lib.fa_set_wait_timeout_ns(int(ns))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_args(q, k, v, out=None, lse=None, *, softmax_scale=None, causal=False, window_left=-1,
              window_right=-1, cu_seqlens_q=None, cu_seqlens_k=None, seqused_k=None, max_seqlen_q=None,
              max_seqlen_k=None, num_splits=0, kv_format=None, k_descale=None, v_descale=None,
              page_table=None) -> FwdArgs:
    """Fill fa_fwd_args from tensors (q/out bf16, last dim contiguous).

    k / v: bf16, or one-byte fp8 codes (uint8 with kv_format 'e4m3' / 'e5m2', or
    torch's float8 dtypes) with fp32 k_descale / v_descale of shape
    (batch, num_heads_kv). With page_table (int32 (batch, max_pages_per_seq)),
    k and v are page pools (num_pages, page_size, num_heads_kv, head_dim).
    """
    a = FwdArgs()
    a.q, a.k, a.v, a.out, a.lse = _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse)
    varlen = cu_seqlens_q is not None
    if varlen:
        a.q_row_stride, a.q_head_stride = q.stride(0), q.stride(1)
        a.k_row_stride, a.k_head_stride = k.stride(0), k.stride(1)
        a.v_row_stride, a.v_head_stride = v.stride(0), v.stride(1)
        if out is not None:
            a.o_row_stride, a.o_head_stride = out.stride(0), out.stride(1)
        a.batch = cu_seqlens_q.numel() - 1
        a.total_q, a.total_k = q.shape[0], k.shape[0]
        a.max_seqlen_q = int(max_seqlen_q)
        a.max_seqlen_k = int(max_seqlen_k)
        a.num_heads_q, a.num_heads_kv = q.shape[1], k.shape[1]
    else:
        a.q_batch_stride, a.q_row_stride, a.q_head_stride = q.stride(0), q.stride(1), q.stride(2)
        a.k_batch_stride, a.k_row_stride, a.k_head_stride = k.stride(0), k.stride(1), k.stride(2)
        a.v_batch_stride, a.v_row_stride, a.v_head_stride = v.stride(0), v.stride(1), v.stride(2)
        if out is not None:
            a.o_batch_stride, a.o_row_stride, a.o_head_stride = out.stride(0), out.stride(1), out.stride(2)
        a.batch, a.seqlen_q, a.seqlen_k = q.shape[0], q.shape[1], k.shape[1]
        a.num_heads_q, a.num_heads_kv = q.shape[2], k.shape[2]
        if page_table is not None:
            a.seqlen_k = page_table.shape[1] * k.shape[1]
    a.head_dim_qk, a.head_dim_v = q.shape[-1], v.shape[-1]
    a.cu_seqlens_q, a.cu_seqlens_k, a.seqused_k = _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(seqused_k)
    a.softmax_scale = 0.0 if softmax_scale is None else float(softmax_scale)
    a.causal = 1 if causal else 0
    a.window_left, a.window_right = int(window_left), int(window_right)
    a.num_splits = int(num_splits)
    if page_table is not None:
        a.page_table = _ptr(page_table)
        a.max_pages_per_seq = page_table.shape[1]
        a.num_pages, a.page_size = k.shape[0], k.shape[1]
    a.kv_format = _kv_format_of(k, kv_format)
    a.k_descale, a.v_descale = _ptr(k_descale), _ptr(v_descale)
    return a


def _check(code: int, where: str) -> None:
    if code != FA_OK:
        raise FaError(code, where)


def fa_workspace_size(args: FwdArgs) -> int:
    return int(_lib.fa_workspace_size(ctypes.byref(args)))


def fa_num_splits(args: FwdArgs, num_sms: int = 0) -> int:
    return int(_lib.fa_num_splits(ctypes.byref(args), int(num_sms)))


def fa_split_len(args: FwdArgs, num_splits: int) -> int:
    return int(_lib.fa_split_len(ctypes.byref(args), int(num_splits)))


def fa_get_status(stream=None) -> int:
    return int(_lib.fa_get_status(_vp(_stream_handle(stream))))


def fa_fwd(q, k, v, out=None, lse=None, *, workspace=None, stream=None, return_lse=True, **kw
           ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """O (and LSE) of the exact attention forward. kw: see make_args."""
    varlen = kw.get("cu_seqlens_q") is not None
    hq, dv = q.shape[-2], v.shape[-1]
    if out is None:
        out = torch.empty(q.shape[:-1] + (dv,), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        shape = (hq, q.shape[0]) if varlen else (q.shape[0], hq, q.shape[1])
        lse = torch.empty(shape, dtype=torch.float32, device=q.device)
    args = make_args(q, k, v, out, lse, **kw)
    need = fa_workspace_size(args)
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _ptr(workspace) if need > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if (need > 0) else 0
    _check(_lib.fa_fwd(ctypes.byref(args), ws_ptr, ws_bytes, _vp(_stream_handle(stream))), "fa_fwd")
    return out, lse


def fa_fwd_splitkv(q, k, v, num_splits: int, out_partial=None, lse_partial=None, *, stream=None, **kw):
    """fp32 split partials (num_splits, ...). kw: see make_args."""
    varlen = kw.get("cu_seqlens_q") is not None
    hq, dv = q.shape[-2], v.shape[-1]
    rows_shape = (q.shape[0],) if varlen else (q.shape[0], q.shape[1])
    if out_partial is None:
        out_partial = torch.empty((num_splits,) + rows_shape + (hq, dv), dtype=torch.float32, device=q.device)
    if lse_partial is None:
        shape = (num_splits, hq, q.shape[0]) if varlen else (num_splits, q.shape[0], hq, q.shape[1])
        lse_partial = torch.empty(shape, dtype=torch.float32, device=q.device)
    args = make_args(q, k, v, **kw)
    _check(_lib.fa_fwd_splitkv(ctypes.byref(args), int(num_splits), _ptr(out_partial), _ptr(lse_partial),
                               None, 0, _vp(_stream_handle(stream))), "fa_fwd_splitkv")
    return out_partial, lse_partial


def fa_combine(out_partial, lse_partial, out=None, lse=None, *, cu_seqlens_q=None, stream=None):
    """Merge (num_splits, ...) fp32 partials into bf16 O and fp32 LSE."""
    ns = out_partial.shape[0]
    dv, hq = out_partial.shape[-1], out_partial.shape[-2]
    varlen = cu_seqlens_q is not None
    if varlen:
        total_q, batch, seqlen_q = out_partial.shape[1], cu_seqlens_q.numel() - 1, 0
    else:
        total_q, batch, seqlen_q = 0, out_partial.shape[1], out_partial.shape[2]
    if out is None:
        out = torch.empty(out_partial.shape[1:], dtype=torch.bfloat16, device=out_partial.device)
    if lse is None:
        lse = torch.empty(lse_partial.shape[1:], dtype=torch.float32, device=out_partial.device)
    if varlen:
        obs, ors, ohs = 0, out.stride(0), out.stride(1)
    else:
        obs, ors, ohs = out.stride(0), out.stride(1), out.stride(2)
    _check(_lib.fa_combine(_ptr(out_partial), _ptr(lse_partial), ns, batch, seqlen_q, hq, dv,
                           _ptr(cu_seqlens_q), total_q, _ptr(out), obs, ors, ohs, _ptr(lse),
                           _vp(_stream_handle(stream))), "fa_combine")
    return out, lse


def fa_bwd_workspace_size(args: FwdArgs) -> int:
    return int(_lib.fa_bwd_workspace_size(ctypes.byref(args)))


_SIDE = {}


def side_stream_objects(device) -> tuple:
    """A high-priority torch stream and two events per device, made once and
    reused by fa_bwd(concurrent=True): PyTorch owns them, not the library."""
    idx = torch.device(device).index
    if idx is None:
        idx = torch.cuda.current_device()
    if idx not in _SIDE:
        with torch.cuda.device(idx):
            side = torch.cuda.Stream(priority=-1)
            fork, join = torch.cuda.Event(), torch.cuda.Event()
            fork.record(side)       # torch creates the CUDA event at its first record
            join.record(side)
            _SIDE[idx] = (side, fork, join)
    return _SIDE[idx]


def fa_bwd(q, k, v, out, lse, dout, dq=None, dk=None, dv=None, *, workspace=None, stream=None,
           concurrent=True, **kw):
    """dQ, dK, dV of the forward (q, k, v) -> (out, lse), given dO.

    Batched or packed varlen layout (pass the forward's cu_seqlens_q/k and
    max_seqlen_q/k). out and lse are the forward's results; dout has out's
    shape and strides; dq / dk / dv (allocated when None) take q's / k's / v's.
    kw: the forward's mask, scale and varlen keywords (see make_args).
    concurrent: run dK/dV on a second (torch-owned, high-priority) stream
    alongside dQ (fa_bwd_two_streams); otherwise every kernel on `stream`.
    Deterministic: the same inputs give the same bits.
    """
    if dq is None:
        dq = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    if dk is None:
        dk = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
    if dv is None:
        dv = torch.empty_strided(v.shape, v.stride(), dtype=v.dtype, device=v.device)
    for name, a, b in (("dout", dout, out), ("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if a.shape != b.shape or a.stride() != b.stride():
            raise ValueError(f"{name} must have the shape and strides of its forward tensor")
    args = make_args(q, k, v, out, lse, **kw)
    need = fa_bwd_workspace_size(args)
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _ptr(workspace) if need > 0 else None
    ws_bytes = workspace.numel() * workspace.element_size() if need > 0 else 0
    if concurrent:
        side, fork, join = side_stream_objects(q.device)
        _check(_lib.fa_bwd_two_streams(ctypes.byref(args), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), ws_ptr,
                                       ws_bytes, _vp(_stream_handle(stream)), _vp(side.cuda_stream),
                                       _vp(fork.cuda_event), _vp(join.cuda_event)), "fa_bwd_two_streams")
    else:
        _check(_lib.fa_bwd(ctypes.byref(args), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), ws_ptr, ws_bytes,
                           _vp(_stream_handle(stream))), "fa_bwd")
    return dq, dk, dv


def default_scale(head_dim_qk: int) -> float:
    return 1.0 / math.sqrt(head_dim_qk)


NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def fa_fwd_decode_noalloc(q, k, v, out, lse=None, *, stream=None, **kw):
    """Split-KV decode + combine with the library's fixed scratch (no workspace).

    For callers that cannot allocate device memory at the call: `out` (and
    `lse`, if wanted) must already exist. See fa.h for the limits and the
    sharing rules of the scratch array.
    """
    args = make_args(q, k, v, out, lse, **kw)
    _check(_lib.fa_fwd_decode_noalloc(ctypes.byref(args), _vp(_stream_handle(stream))), "fa_fwd_decode_noalloc")
    return out, lse

"""GB300-native fused attention with an in-kernel relative-position bias (T5 buckets, ALiBi),
padding-free varlen packing, forward and backward.

This module is a thin ctypes binding over libfatattn.so (C ABI in include/fat_attn.h): it only
marshals torch tensors into pointers and sizes. Every step of the computation runs in the CUDA
kernels of the library; there is no other implementation to fall back to, and a missing or
unloadable library raises immediately.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "FatAttnError", "load", "fat_attn_fwd", "fat_attn_fwd_workspace_size", "fat_attn_bwd",
    "fat_attn_bwd_workspace_size",
    "fat_attn_get_device_error", "fat_attn_strerror", "fat_attn_bucket_thresholds",
    "fat_attn_debug_buckets", "fat_attn_debug_set_watchdog", "fat_attn_bwd_stages",
    "fat_attn_bwd_noalloc", "fat_xattn_fwd", "fat_xattn_bwd", "fat_xattn_bwd_workspace_size",
    "fat_xattn_splitkv_num_splits", "fat_rope_apply", "fat_rmsnorm_fwd", "fat_rmsnorm_bwd",
    "fat_cross_entropy", "FAT_DEVERR_TIMEOUT_FWD", "FAT_DEVERR_TIMEOUT_BWD", "FAT_DEVERR_INDEX",
    "FAT_DEVERR_SEQLENS", "LIB_PATH",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfatattn.so")

FAT_DEVERR_TIMEOUT_FWD = 1
FAT_DEVERR_TIMEOUT_BWD = 2
FAT_DEVERR_SEQLENS = 4
FAT_DEVERR_INDEX = 8


class FatAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = ""
        if code == -4:
            detail = "; " + load().fat_attn_last_error_message().decode()
        super().__init__(f"{where} failed: {code} ({fat_attn_strerror(code)}{detail})")


class _Shape(ctypes.Structure):
    _fields_ = [("total_tokens", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("max_seqlen", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("stream", ctypes.c_void_p)]


class _XShape(ctypes.Structure):
    _fields_ = [("total_q", ctypes.c_int32), ("total_k", ctypes.c_int32),
                ("num_seqs", ctypes.c_int32), ("max_seqlen_q", ctypes.c_int32),
                ("max_seqlen_k", ctypes.c_int32), ("num_heads_q", ctypes.c_int32),
                ("num_heads_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("stream", ctypes.c_void_p)]


_lib = None


def load(path: Optional[str] = None):
    """Load libfatattn.so (built by __graft_entry__.build()). Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FileNotFoundError(
            f"{p} not found: build the CUDA library first (python -c 'import __graft_entry__ as g; "
            f"g.build()')")
    lib = ctypes.CDLL(p)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    S = ctypes.POINTER(_Shape)
    lib.fat_attn_fwd.argtypes = [S, vp, vp, vp, vp, i32, i32, i32, vp, vp, i32, f32, vp, vp]
    lib.fat_attn_fwd.restype = i32
    lib.fat_attn_fwd_ws.argtypes = [S, vp, vp, vp, vp, i32, i32, i32, vp, vp, i32, f32, vp, vp,
                                    vp, ctypes.c_size_t]
    lib.fat_attn_fwd_ws.restype = i32
    lib.fat_attn_fwd_workspace_size.argtypes = [S]
    lib.fat_attn_fwd_workspace_size.restype = ctypes.c_size_t
    lib.fat_attn_bwd_workspace_size.argtypes = [S]
    lib.fat_attn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fat_attn_bwd.argtypes = [S, vp, vp, vp, vp, i32, i32, i32, vp, vp, i32, f32, vp, vp, vp,
                                 vp, ctypes.c_size_t, vp, vp, vp, vp]
    lib.fat_attn_bwd.restype = i32
    lib.fat_attn_bwd_preprocess.argtypes = [S, vp, vp, vp, ctypes.c_size_t, vp, i32]
    lib.fat_attn_bwd_preprocess.restype = i32
    lib.fat_attn_bwd_main.argtypes = [S, vp, vp, vp, vp, i32, i32, i32, vp, vp, i32, f32, vp, vp,
                                      vp, ctypes.c_size_t, vp, vp, vp]
    lib.fat_attn_bwd_main.restype = i32
    lib.fat_attn_bwd_finalize.argtypes = [S, vp, ctypes.c_size_t, f32, vp]
    lib.fat_attn_bwd_finalize.restype = i32
    lib.fat_attn_bwd_noalloc.argtypes = [S, vp, vp, vp, vp, i32, i32, i32, vp, vp, i32, f32, vp,
                                         vp, vp, vp, vp, vp, vp]
    lib.fat_attn_bwd_noalloc.restype = i32
    X = ctypes.POINTER(_XShape)
    lib.fat_xattn_fwd.argtypes = [X, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, i32, f32, vp, vp]
    lib.fat_xattn_fwd.restype = i32
    lib.fat_xattn_splitkv_num_splits.argtypes = [X]
    lib.fat_xattn_splitkv_num_splits.restype = i32
    lib.fat_xattn_splitkv_workspace_size.argtypes = [X, i32]
    lib.fat_xattn_splitkv_workspace_size.restype = ctypes.c_size_t
    lib.fat_xattn_fwd_splitkv.argtypes = [X, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, i32, f32,
                                          i32, vp, ctypes.c_size_t, vp, vp]
    lib.fat_xattn_fwd_splitkv.restype = i32
    lib.fat_xattn_bwd_workspace_size.argtypes = [X]
    lib.fat_xattn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fat_xattn_bwd.argtypes = [X, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, i32, f32, vp, vp,
                                  vp, vp, ctypes.c_size_t, vp, vp, vp, vp]
    lib.fat_xattn_bwd.restype = i32
    ll = ctypes.c_longlong
    lib.fat_rmsnorm_fwd.argtypes = [ll, i32, vp, vp, f32, vp, vp, vp]
    lib.fat_rmsnorm_fwd.restype = i32
    lib.fat_rmsnorm_bwd.argtypes = [ll, i32, vp, vp, vp, vp, vp, vp, vp]
    lib.fat_rmsnorm_bwd.restype = i32
    lib.fat_cross_entropy.argtypes = [ll, i32, vp, vp, f32, f32, vp, vp, vp, vp]
    lib.fat_cross_entropy.restype = i32
    lib.fat_rope_apply.argtypes = [S, vp, vp, vp, ctypes.c_double, i32]
    lib.fat_rope_apply.restype = i32
    lib.fat_attn_get_device_error.argtypes = [vp, ctypes.POINTER(i32)]
    lib.fat_attn_get_device_error.restype = i32
    lib.fat_attn_strerror.argtypes = [i32]
    lib.fat_attn_strerror.restype = ctypes.c_char_p
    lib.fat_attn_last_error_message.argtypes = []
    lib.fat_attn_last_error_message.restype = ctypes.c_char_p
    lib.fat_attn_bucket_thresholds.argtypes = [i32, i32, i32, ctypes.POINTER(ctypes.c_int32),
                                               ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.fat_attn_bucket_thresholds.restype = i32
    lib.fat_attn_debug_buckets.argtypes = [ctypes.c_longlong, i32, i32, i32, i32, vp, vp]
    lib.fat_attn_debug_buckets.restype = i32
    lib.fat_attn_debug_set_watchdog.argtypes = [ctypes.c_longlong, i32]
    lib.fat_attn_debug_set_watchdog.restype = None
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream, device) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _on(device):
    """Context that makes `device` the current CUDA device for the duration of a library call:
    the library launches on, and looks up its per-GPU state for, the current device."""
    import torch
    return torch.cuda.device(device)


def _shape(total_tokens, num_seqs, max_seqlen, num_heads, head_dim, stream_ptr) -> _Shape:
    return _Shape(int(total_tokens), int(num_seqs), int(max_seqlen), int(num_heads),
                  int(head_dim), stream_ptr)


def _check_tensor(name, t, dtype, ndim=None):
    import torch
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")


def fat_attn_fwd(q, k, v, cu_seqlens, max_seqlen: int, bias_table=None, num_buckets: int = 0,
                 max_distance: int = 0, bidirectional: bool = True, alibi_slopes=None,
                 causal: bool = False, softmax_scale: float = 1.0, out=None, lse=None,
                 workspace=None, stream=None):
    """Forward pass. q, k, v: bf16 [T, H, d] (CUDA, contiguous); cu_seqlens: int32 [n+1] (CUDA).
    workspace: device bytes for a split last wave (fat_attn_fwd_workspace_size); None allocates
    what the shape uses, False runs without one. Returns (out bf16 [T, H, d], lse fp32 [H, T])."""
    import torch
    lib = load()
    T, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _check_tensor(name, t, torch.bfloat16, 3)
    _check_tensor("cu_seqlens", cu_seqlens, torch.int32, 1)
    _check_tensor("bias_table", bias_table, torch.float32)
    _check_tensor("alibi_slopes", alibi_slopes, torch.float32)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    sh = _shape(T, cu_seqlens.numel() - 1, max_seqlen, H, d, _stream_ptr(stream, q.device))
    args = (ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(bias_table), int(num_buckets),
            int(max_distance), int(bool(bidirectional)), _ptr(alibi_slopes), _ptr(cu_seqlens),
            int(bool(causal)), float(softmax_scale), _ptr(out), _ptr(lse))
    if workspace is None and not causal:
        need = int(lib.fat_attn_fwd_workspace_size(ctypes.byref(sh)))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    with _on(q.device):
        if workspace is None or workspace is False:
            rc = lib.fat_attn_fwd(*args)
        else:
            rc = lib.fat_attn_fwd_ws(*args, _ptr(workspace),
                                     int(workspace.numel() * workspace.element_size()))
    if rc != 0:
        raise FatAttnError(rc, "fat_attn_fwd")
    return out, lse


def fat_attn_fwd_workspace_size(total_tokens: int, num_seqs: int, max_seqlen: int,
                                num_heads: int, head_dim: int) -> int:
    """Device bytes that let the forward split its last wave for this shape (0: none)."""
    sh = _shape(total_tokens, num_seqs, max_seqlen, num_heads, head_dim, None)
    return int(load().fat_attn_fwd_workspace_size(ctypes.byref(sh)))


def fat_attn_bwd_workspace_size(total_tokens: int, num_heads: int, head_dim: int,
                                num_seqs: int = 1, max_seqlen: int = 1) -> int:
    """Backward workspace bytes. With the defaults: the minimum every backward call accepts (dQ
    accumulator and D); with the problem's num_seqs and max_seqlen: the size for its fastest
    schedule (adds the rows of a split last wave when the shape has one)."""
    lib = load()
    sh = _shape(total_tokens, num_seqs, max_seqlen, num_heads, head_dim, None)
    return int(lib.fat_attn_bwd_workspace_size(ctypes.byref(sh)))


def fat_attn_bwd(q, k, v, cu_seqlens, max_seqlen: int, out, lse, dout, bias_table=None,
                 num_buckets: int = 0, max_distance: int = 0, bidirectional: bool = True,
                 alibi_slopes=None, causal: bool = False, softmax_scale: float = 1.0,
                 want_dbias: bool = True, workspace=None, dq=None, dk=None, dv=None,
                 dbias_table=None, stream=None):
    """Backward pass of sum(out * dout). Returns (dq, dk, dv, dbias_table or None)."""
    import torch
    lib = load()
    T, H, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        _check_tensor(name, t, torch.bfloat16, 3)
    _check_tensor("lse", lse, torch.float32, 2)
    _check_tensor("cu_seqlens", cu_seqlens, torch.int32, 1)
    _check_tensor("bias_table", bias_table, torch.float32)
    _check_tensor("alibi_slopes", alibi_slopes, torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dbias_table is None and want_dbias and bias_table is not None:
        dbias_table = torch.empty_like(bias_table)
    sh = _shape(T, cu_seqlens.numel() - 1, max_seqlen, H, d, _stream_ptr(stream, q.device))
    need = int(lib.fat_attn_bwd_workspace_size(ctypes.byref(sh)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    with _on(q.device):
        rc = lib.fat_attn_bwd(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(bias_table),
                              int(num_buckets), int(max_distance), int(bool(bidirectional)),
                              _ptr(alibi_slopes), _ptr(cu_seqlens), int(bool(causal)),
                              float(softmax_scale), _ptr(out), _ptr(lse), _ptr(dout),
                              _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                              _ptr(dq), _ptr(dk), _ptr(dv),
                              _ptr(dbias_table))
    if rc != 0:
        raise FatAttnError(rc, "fat_attn_bwd")
    return dq, dk, dv, dbias_table


def fat_attn_bwd_stages(q, k, v, cu_seqlens, max_seqlen: int, out, lse, dout, workspace, dq, dk,
                        dv, dbias_table=None, bias_table=None, num_buckets: int = 0,
                        max_distance: int = 0, bidirectional: bool = True, alibi_slopes=None,
                        causal: bool = False, softmax_scale: float = 1.0, stream=None,
                        between=None):
    """The backward as its three C-ABI stages (preprocess, main, finalize) with every buffer
    supplied by the caller. `between(i)` (optional) is called after enqueueing stage i, e.g. to
    record CUDA events around the main kernel."""
    lib = load()
    T, H, d = q.shape
    sh = _shape(T, cu_seqlens.numel() - 1, max_seqlen, H, d, _stream_ptr(stream, q.device))
    nbytes = int(workspace.numel() * workspace.element_size())
    if between is not None:
        between(-1)
    with _on(q.device):
        rc = lib.fat_attn_bwd_preprocess(ctypes.byref(sh), _ptr(out), _ptr(dout), _ptr(workspace),
                                         nbytes, _ptr(dbias_table), int(num_buckets))
    if rc != 0:
        raise FatAttnError(rc, "fat_attn_bwd_preprocess")
    if between is not None:
        between(0)
    with _on(q.device):
        rc = lib.fat_attn_bwd_main(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(bias_table),
                                   int(num_buckets), int(max_distance), int(bool(bidirectional)),
                                   _ptr(alibi_slopes), _ptr(cu_seqlens), int(bool(causal)),
                                   float(softmax_scale), _ptr(lse), _ptr(dout), _ptr(workspace),
                                   nbytes, _ptr(dk), _ptr(dv), _ptr(dbias_table))
    if rc != 0:
        raise FatAttnError(rc, "fat_attn_bwd_main")
    if between is not None:
        between(1)
    with _on(q.device):
        rc = lib.fat_attn_bwd_finalize(ctypes.byref(sh), _ptr(workspace), nbytes,
                                       float(softmax_scale), _ptr(dq))
    if rc != 0:
        raise FatAttnError(rc, "fat_attn_bwd_finalize")
    if between is not None:
        between(2)
    return dq, dk, dv, dbias_table


def fat_attn_bwd_noalloc(q, k, v, cu_seqlens, max_seqlen: int, out, lse, dout, dq, dk, dv,
                         dbias_table=None, bias_table=None, num_buckets: int = 0,
                         max_distance: int = 0, bidirectional: bool = True, alibi_slopes=None,
                         causal: bool = False, softmax_scale: float = 1.0, stream=None):
    """The backward with the library's built-in scratch instead of a workspace, for callers that
    cannot allocate device memory (see fat_attn_bwd_noalloc in include/fat_attn.h). All output
    buffers are supplied by the caller; nothing is allocated here."""
    lib = load()
    T, H, d = q.shape
    sh = _shape(T, cu_seqlens.numel() - 1, max_seqlen, H, d, _stream_ptr(stream, q.device))
    with _on(q.device):
        rc = lib.fat_attn_bwd_noalloc(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(bias_table),
                                      int(num_buckets), int(max_distance), int(bool(bidirectional)),
                                      _ptr(alibi_slopes), _ptr(cu_seqlens), int(bool(causal)),
                                      float(softmax_scale), _ptr(out), _ptr(lse), _ptr(dout),
                                      _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias_table))
    if rc != 0:
        raise FatAttnError(rc, "fat_attn_bwd_noalloc")
    return dq, dk, dv, dbias_table


def _xshape(q, k, cu_seqlens_q, max_seqlen_q, max_seqlen_k, stream) -> _XShape:
    Tq, Hq, d = q.shape
    Tk, Hkv, _ = k.shape
    return _XShape(int(Tq), int(Tk), int(cu_seqlens_q.numel() - 1), int(max_seqlen_q),
                   int(max_seqlen_k), int(Hq), int(Hkv), int(d), _stream_ptr(stream, q.device))


def fat_xattn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                  bias_table=None, num_buckets: int = 0, max_distance: int = 0,
                  bidirectional: bool = True, alibi_slopes=None, causal: bool = False,
                  softmax_scale: float = 1.0, out=None, lse=None, num_splits: int = 1,
                  workspace=None, stream=None):
    """Forward with its own query and key lengths per document (cross-attention, decode over a
    key cache) and grouped-query heads. q: bf16 [Tq, Hq, d]; k, v: bf16 [Tk, Hkv, d];
    cu_seqlens_q / cu_seqlens_k: int32 [n + 1]. num_splits > 1 splits every document's keys
    into that many ranges (merged by a second grid); 0 lets the library choose.
    Returns (out bf16 [Tq, Hq, d], lse fp32 [Hq, Tq])."""
    import torch
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _check_tensor(name, t, torch.bfloat16, 3)
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        _check_tensor(name, t, torch.int32, 1)
    _check_tensor("bias_table", bias_table, torch.float32)
    _check_tensor("alibi_slopes", alibi_slopes, torch.float32)
    Tq, Hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    sh = _xshape(q, k, cu_seqlens_q, max_seqlen_q, max_seqlen_k, stream)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(bias_table), int(num_buckets), int(max_distance),
            int(bool(bidirectional)), _ptr(alibi_slopes), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
            int(bool(causal)), float(softmax_scale))
    with _on(q.device):
        if num_splits == 0:
            num_splits = int(lib.fat_xattn_splitkv_num_splits(ctypes.byref(sh)))
        if num_splits == 1:
            rc = lib.fat_xattn_fwd(ctypes.byref(sh), *args, _ptr(out), _ptr(lse))
        else:
            need = int(lib.fat_xattn_splitkv_workspace_size(ctypes.byref(sh), int(num_splits)))
            if workspace is None:
                workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
            rc = lib.fat_xattn_fwd_splitkv(ctypes.byref(sh), *args, int(num_splits),
                                           _ptr(workspace),
                                           int(workspace.numel() * workspace.element_size()),
                                           _ptr(out), _ptr(lse))
    if rc != 0:
        raise FatAttnError(rc, "fat_xattn_fwd")
    return out, lse


def fat_xattn_splitkv_num_splits(q, k, cu_seqlens_q, max_seqlen_q: int, max_seqlen_k: int) -> int:
    """The number of key splits the library suggests for this problem."""
    sh = _xshape(q, k, cu_seqlens_q, max_seqlen_q, max_seqlen_k, None)
    return int(load().fat_xattn_splitkv_num_splits(ctypes.byref(sh)))


def fat_xattn_bwd_workspace_size(total_q: int, total_k: int, num_heads_q: int,
                                 num_heads_kv: int, head_dim: int) -> int:
    sh = _XShape(int(total_q), int(total_k), 1, 1, 1, int(num_heads_q), int(num_heads_kv),
                 int(head_dim), None)
    return int(load().fat_xattn_bwd_workspace_size(ctypes.byref(sh)))


def fat_xattn_bwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                  out, lse, dout, bias_table=None, num_buckets: int = 0, max_distance: int = 0,
                  bidirectional: bool = True, alibi_slopes=None, causal: bool = False,
                  softmax_scale: float = 1.0, want_dbias: bool = True, workspace=None, dq=None,
                  dk=None, dv=None, dbias_table=None, stream=None):
    """Backward of sum(out * dout) for fat_xattn_fwd. Returns (dq, dk, dv, dbias or None)."""
    import torch
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        _check_tensor(name, t, torch.bfloat16, 3)
    _check_tensor("lse", lse, torch.float32, 2)
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        _check_tensor(name, t, torch.int32, 1)
    _check_tensor("bias_table", bias_table, torch.float32)
    _check_tensor("alibi_slopes", alibi_slopes, torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dbias_table is None and want_dbias and bias_table is not None:
        dbias_table = torch.empty_like(bias_table)
    sh = _xshape(q, k, cu_seqlens_q, max_seqlen_q, max_seqlen_k, stream)
    need = int(lib.fat_xattn_bwd_workspace_size(ctypes.byref(sh)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    with _on(q.device):
        rc = lib.fat_xattn_bwd(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(bias_table),
                               int(num_buckets), int(max_distance), int(bool(bidirectional)),
                               _ptr(alibi_slopes), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                               int(bool(causal)), float(softmax_scale), _ptr(out), _ptr(lse),
                               _ptr(dout), _ptr(workspace),
                               int(workspace.numel() * workspace.element_size()), _ptr(dq),
                               _ptr(dk), _ptr(dv), _ptr(dbias_table))
    if rc != 0:
        raise FatAttnError(rc, "fat_xattn_bwd")
    return dq, dk, dv, dbias_table


def fat_rope_apply(x, cu_seqlens, max_seqlen: int, base: float = 10000.0, inverse: bool = False,
                   out=None, stream=None):
    """Rotary position embedding of bf16 [T, H, d] rows, positions local to each document
    (inverse=True turns a gradient back). out may be x itself (in place). Returns out."""
    import torch
    lib = load()
    _check_tensor("x", x, torch.bfloat16, 3)
    _check_tensor("out", out, torch.bfloat16, 3)
    _check_tensor("cu_seqlens", cu_seqlens, torch.int32, 1)
    if out is None:
        out = torch.empty_like(x)
    T, H, d = x.shape
    sh = _shape(T, cu_seqlens.numel() - 1, max_seqlen, H, d, _stream_ptr(stream, x.device))
    with _on(x.device):
        rc = lib.fat_rope_apply(ctypes.byref(sh), _ptr(x), _ptr(out), _ptr(cu_seqlens),
                                float(base), int(bool(inverse)))
    if rc != 0:
        raise FatAttnError(rc, "fat_rope_apply")
    return out


def fat_rmsnorm_fwd(x, weight, eps: float = 1e-6, y=None, rstd=None, stream=None):
    """RMSNorm of the rows of x (bf16 [..., dim], contiguous) with an fp32 weight [dim].
    Returns (y bf16 like x, rstd fp32 [rows])."""
    import torch
    lib = load()
    _check_tensor("x", x, torch.bfloat16)
    _check_tensor("weight", weight, torch.float32, 1)
    dim = x.shape[-1]
    rows = x.numel() // dim if dim else 0
    y = torch.empty_like(x) if y is None else y
    rstd = torch.empty(rows, dtype=torch.float32, device=x.device) if rstd is None else rstd
    with _on(x.device):
        rc = lib.fat_rmsnorm_fwd(rows, int(dim), _ptr(x), _ptr(weight), float(eps), _ptr(y),
                                 _ptr(rstd), _stream_ptr(stream, x.device))
    if rc != 0:
        raise FatAttnError(rc, "fat_rmsnorm_fwd")
    return y, rstd


def fat_rmsnorm_bwd(x, weight, rstd, dy, dx=None, dweight=None, stream=None):
    """Gradients of sum(y * dy) for fat_rmsnorm_fwd: (dx bf16 like x, dweight fp32 [dim])."""
    import torch
    lib = load()
    for name, t in (("x", x), ("dy", dy), ("dx", dx)):
        _check_tensor(name, t, torch.bfloat16)
    _check_tensor("weight", weight, torch.float32, 1)
    _check_tensor("rstd", rstd, torch.float32, 1)
    dim = x.shape[-1]
    rows = x.numel() // dim if dim else 0
    dx = torch.empty_like(x) if dx is None else dx
    dweight = torch.empty_like(weight) if dweight is None else dweight
    with _on(x.device):
        rc = lib.fat_rmsnorm_bwd(rows, int(dim), _ptr(x), _ptr(weight), _ptr(rstd), _ptr(dy),
                                 _ptr(dx), _ptr(dweight), _stream_ptr(stream, x.device))
    if rc != 0:
        raise FatAttnError(rc, "fat_rmsnorm_bwd")
    return dx, dweight


def fat_cross_entropy(logits, target, z_loss: float = 0.0, grad_scale: float = 1.0,
                      want_grad: bool = True, loss=None, lse=None, dlogits=None, stream=None):
    """Cross-entropy with a z-loss term per row of logits (bf16 [rows, vocab]) against int32
    targets [rows] (negative = ignored); with want_grad the gradient of grad_scale * sum(loss)
    comes from the same pass. Returns (loss fp32 [rows], lse fp32 [rows], dlogits or None)."""
    import torch
    lib = load()
    _check_tensor("logits", logits, torch.bfloat16, 2)
    _check_tensor("target", target, torch.int32, 1)
    rows, vocab = logits.shape
    loss = torch.empty(rows, dtype=torch.float32, device=logits.device) if loss is None else loss
    lse = torch.empty(rows, dtype=torch.float32, device=logits.device) if lse is None else lse
    if want_grad and dlogits is None:
        dlogits = torch.empty_like(logits)
    with _on(logits.device):
        rc = lib.fat_cross_entropy(int(rows), int(vocab), _ptr(logits), _ptr(target),
                                   float(z_loss), float(grad_scale), _ptr(loss), _ptr(lse),
                                   _ptr(dlogits) if want_grad else None,
                                   _stream_ptr(stream, logits.device))
    if rc != 0:
        raise FatAttnError(rc, "fat_cross_entropy")
    return loss, lse, (dlogits if want_grad else None)


def fat_attn_get_device_error(stream=None, device=None) -> int:
    """Synchronise, read and clear the device error word; returns its bits (0 = no error)."""
    lib = load()
    bits = ctypes.c_int(0)
    rc = lib.fat_attn_get_device_error(_stream_ptr(stream, device), ctypes.byref(bits))
    if rc not in (0, -6):
        raise FatAttnError(rc, "fat_attn_get_device_error")
    return int(bits.value)


def fat_attn_strerror(code: int) -> str:
    return load().fat_attn_strerror(int(code)).decode()


def fat_attn_bucket_thresholds(num_buckets: int, max_distance: int, bidirectional: bool):
    """Host-side thresholds the kernels compare distances with: (thresholds list, saturation)."""
    lib = load()
    arr = (ctypes.c_int32 * 64)()
    cnt, sat = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib.fat_attn_bucket_thresholds(int(num_buckets), int(max_distance),
                                        int(bool(bidirectional)), arr, ctypes.byref(cnt),
                                        ctypes.byref(sat))
    if rc != 0:
        raise FatAttnError(rc, "fat_attn_bucket_thresholds")
    return list(arr[: cnt.value]), int(sat.value)


def fat_attn_debug_buckets(delta_lo: int, n: int, num_buckets: int, max_distance: int,
                           bidirectional: bool, out=None, stream=None, device="cuda"):
    """Device-side T5 bucket ids for delta_lo .. delta_lo+n-1 (int32 CUDA tensor)."""
    import torch
    lib = load()
    if out is None:
        out = torch.empty(n, dtype=torch.int32, device=device)
    with _on(out.device):
        rc = lib.fat_attn_debug_buckets(int(delta_lo), int(n), int(num_buckets), int(max_distance),
                                        int(bool(bidirectional)), _ptr(out),
                                        _stream_ptr(stream, out.device))
    if rc != 0:
        raise FatAttnError(rc, "fat_attn_debug_buckets")
    return out


def fat_attn_debug_set_watchdog(timeout_ns: int = 0, flags: int = 0) -> None:
    load().fat_attn_debug_set_watchdog(int(timeout_ns), int(flags))

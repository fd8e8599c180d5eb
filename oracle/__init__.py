"""fp64 CPU oracle for attention with an in-kernel relative-position bias.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` are the only callers. The product library never imports this package, and this
package never imports the product library.

The arithmetic lives in ``oracle.c`` (self-attention with the relative-position bias) and
``oracle_xattn.c`` (own query and key lengths per document, grouped-query heads, bottom-right
causal alignment), plain C, fp64, OpenMP; this module compiles them with gcc and marshals numpy
arrays through ctypes. The rotary embedding (``rope_*``) is numpy fp64 around the plain oracle;
RMSNorm and the cross-entropy with z-loss (the report's other fused kernels) are numpy fp64 in
``oracle.norm_ce``.
Inputs may be the exact bf16 bit patterns the GPU path receives (numpy ``uint16``), fp32 or fp64
arrays; all are widened exactly to fp64 here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "oracle_xattn.c")]
_HDRS = [os.path.join(_HERE, "oracle.h"), os.path.join(_HERE, "oracle_xattn.h")]
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c and oracle_xattn.c into liboracle.so next to them (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(f) for f in _SRCS + _HDRS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           *_SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [
        ("total_tokens", ctypes.c_int),
        ("num_seqs", ctypes.c_int),
        ("num_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("cu_seqlens", ctypes.c_void_p),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("bias_table", ctypes.c_void_p),
        ("num_buckets", ctypes.c_int),
        ("max_distance", ctypes.c_int),
        ("bidirectional", ctypes.c_int),
        ("alibi_slopes", ctypes.c_void_p),
        ("causal", ctypes.c_int),
        ("softmax_scale", ctypes.c_double),
        ("d_from_bf16_out", ctypes.c_int),
    ]


class _XProblem(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int),
        ("total_q", ctypes.c_int),
        ("total_k", ctypes.c_int),
        ("num_heads_q", ctypes.c_int),
        ("num_heads_kv", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("cu_seqlens_q", ctypes.c_void_p),
        ("cu_seqlens_k", ctypes.c_void_p),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("bias_table", ctypes.c_void_p),
        ("num_buckets", ctypes.c_int),
        ("max_distance", ctypes.c_int),
        ("bidirectional", ctypes.c_int),
        ("alibi_slopes", ctypes.c_void_p),
        ("causal", ctypes.c_int),
        ("softmax_scale", ctypes.c_double),
    ]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER(_Problem)
        vp = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_t5_bucket.argtypes = [ctypes.c_longlong, i, i, i]
        lib.oracle_t5_bucket.restype = i
        lib.oracle_alibi_bias.argtypes = [ctypes.c_longlong, ctypes.c_double]
        lib.oracle_alibi_bias.restype = ctypes.c_double
        lib.oracle_attn_fwd.argtypes = [P, vp, vp]
        lib.oracle_attn_bwd.argtypes = [P, vp, vp, vp, vp, vp]
        lib.oracle_attn_fwd_rows.argtypes = [P, i, i, vp, i, vp, vp]
        lib.oracle_attn_bwd_rows.argtypes = [P, vp, i, i, vp, i, vp, i, vp, vp, vp, vp]
        XP = ctypes.POINTER(_XProblem)
        lib.oracle_xattn_fwd.argtypes = [XP, vp, vp]
        lib.oracle_xattn_bwd.argtypes = [XP, vp, vp, vp, vp, vp]
        for f in ("oracle_attn_fwd", "oracle_attn_bwd", "oracle_attn_fwd_rows",
                  "oracle_attn_bwd_rows", "oracle_num_threads", "oracle_xattn_fwd",
                  "oracle_xattn_bwd"):
            getattr(lib, f).restype = i
        _lib = lib
    return _lib


def widen(a) -> np.ndarray:
    """Exact fp64 copy of a uint16 array of bf16 bit patterns, or of an fp32/fp64 array."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.ascontiguousarray(a, dtype=np.float64)


@dataclass
class Problem:
    """One packed varlen attention problem, host side.

    q, k, v: [T, H, d] as bf16 bit patterns (uint16) or floats; cu_seqlens: int32 [n+1];
    table: [nb, H] floats or None; slopes: [H] floats or None. Stored widened to fp64.
    """
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    cu_seqlens: np.ndarray
    table: Optional[np.ndarray] = None
    num_buckets: int = 0
    max_distance: int = 0
    bidirectional: bool = True
    slopes: Optional[np.ndarray] = None
    causal: bool = False
    scale: float = 1.0
    d_from_bf16_out: bool = False  # backward row statistic from the bf16-rounded output

    def __post_init__(self):
        self.q, self.k, self.v = widen(self.q), widen(self.k), widen(self.v)
        self.cu_seqlens = np.ascontiguousarray(self.cu_seqlens, dtype=np.int32)
        if self.table is not None:
            self.table = widen(self.table)
        if self.slopes is not None:
            self.slopes = widen(self.slopes)

    @property
    def shape(self):
        return self.q.shape

    def _c(self) -> _Problem:
        T, H, d = self.q.shape
        p = _Problem()
        p.total_tokens, p.num_seqs, p.num_heads, p.head_dim = T, len(self.cu_seqlens) - 1, H, d
        p.cu_seqlens = self.cu_seqlens.ctypes.data
        p.q, p.k, p.v = self.q.ctypes.data, self.k.ctypes.data, self.v.ctypes.data
        p.bias_table = self.table.ctypes.data if self.table is not None else None
        p.num_buckets, p.max_distance = int(self.num_buckets), int(self.max_distance)
        p.bidirectional = int(bool(self.bidirectional))
        p.alibi_slopes = self.slopes.ctypes.data if self.slopes is not None else None
        p.causal = int(bool(self.causal))
        p.softmax_scale = float(self.scale)
        p.d_from_bf16_out = int(bool(self.d_from_bf16_out))
        return p


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def t5_bucket(delta: int, num_buckets: int, max_distance: int, bidirectional: bool) -> int:
    return int(_load().oracle_t5_bucket(int(delta), int(num_buckets), int(max_distance),
                                        int(bool(bidirectional))))


def alibi_bias(delta: int, slope: float) -> float:
    return float(_load().oracle_alibi_bias(int(delta), float(slope)))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def attn_fwd(pb: Problem):
    """Full forward. Returns (out fp64 [T,H,d], lse fp64 [H,T])."""
    T, H, d = pb.shape
    out = np.zeros((T, H, d), np.float64)
    lse = np.full((H, T), np.nan, np.float64)
    c = pb._c()
    _check(_load().oracle_attn_fwd(ctypes.byref(c), out.ctypes.data, lse.ctypes.data), "fwd")
    return out, lse


def attn_bwd(pb: Problem, dout: np.ndarray):
    """Full backward of sum(out*dout). Returns (dq, dk, dv, dtable-or-None), fp64."""
    T, H, d = pb.shape
    dout = widen(dout)
    dq = np.zeros((T, H, d), np.float64)
    dk = np.zeros_like(dq)
    dv = np.zeros_like(dq)
    dtab = np.zeros((pb.num_buckets, H), np.float64) if pb.table is not None else None
    c = pb._c()
    _check(_load().oracle_attn_bwd(ctypes.byref(c), dout.ctypes.data, dq.ctypes.data,
                                   dk.ctypes.data, dv.ctypes.data,
                                   dtab.ctypes.data if dtab is not None else None), "bwd")
    return dq, dk, dv, dtab


def attn_fwd_rows(pb: Problem, doc: int, head: int, rows: Sequence[int]):
    """out and lse for query rows (document-local positions) of one (doc, head)."""
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    d = pb.shape[2]
    out = np.zeros((len(rows), d), np.float64)
    lse = np.zeros(len(rows), np.float64)
    c = pb._c()
    _check(_load().oracle_attn_fwd_rows(ctypes.byref(c), int(doc), int(head), rows.ctypes.data,
                                        len(rows), out.ctypes.data, lse.ctypes.data), "fwd_rows")
    return out, lse


def attn_bwd_rows(pb: Problem, dout: np.ndarray, doc: int, head: int, qrows: Sequence[int],
                  krows: Sequence[int], want_dtable: bool = False):
    """dq for query rows, dk/dv for key rows of one (doc, head) (document-local positions), and
    optionally this (doc, head)'s contribution to the bucket gradient [nb]."""
    dout = widen(dout)
    qrows = np.ascontiguousarray(qrows, dtype=np.int32)
    krows = np.ascontiguousarray(krows, dtype=np.int32)
    d = pb.shape[2]
    dq = np.zeros((len(qrows), d), np.float64)
    dk = np.zeros((len(krows), d), np.float64)
    dv = np.zeros((len(krows), d), np.float64)
    dcol = np.zeros(pb.num_buckets, np.float64) if (want_dtable and pb.table is not None) else None
    c = pb._c()
    _check(_load().oracle_attn_bwd_rows(
        ctypes.byref(c), dout.ctypes.data, int(doc), int(head), qrows.ctypes.data, len(qrows),
        krows.ctypes.data, len(krows), dq.ctypes.data, dk.ctypes.data, dv.ctypes.data,
        dcol.ctypes.data if dcol is not None else None), "bwd_rows")
    return dq, dk, dv, dcol


# ---- generalised problem: own query and key lengths, grouped-query heads, bottom-right causal ----
@dataclass
class XProblem:
    """Per document a query sequence and a key/value sequence of their own lengths.

    q: [total_q, Hq, d]; k, v: [total_k, Hkv, d] (Hq a multiple of Hkv; query head h reads
    key/value head h // (Hq // Hkv)); cu_seqlens_q / cu_seqlens_k: int32 [n + 1]. Causal masking
    is aligned at the bottom right (query p of a document sees keys r <= p + Lk - Lq), and the
    relative position of the bias is r - (p + Lk - Lq). Stored widened to fp64.
    """
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    cu_seqlens_q: np.ndarray
    cu_seqlens_k: np.ndarray
    table: Optional[np.ndarray] = None
    num_buckets: int = 0
    max_distance: int = 0
    bidirectional: bool = True
    slopes: Optional[np.ndarray] = None
    causal: bool = False
    scale: float = 1.0

    def __post_init__(self):
        self.q, self.k, self.v = widen(self.q), widen(self.k), widen(self.v)
        self.cu_seqlens_q = np.ascontiguousarray(self.cu_seqlens_q, dtype=np.int32)
        self.cu_seqlens_k = np.ascontiguousarray(self.cu_seqlens_k, dtype=np.int32)
        if self.table is not None:
            self.table = widen(self.table)
        if self.slopes is not None:
            self.slopes = widen(self.slopes)

    def _c(self) -> _XProblem:
        p = _XProblem()
        p.num_seqs = len(self.cu_seqlens_q) - 1
        p.total_q, p.num_heads_q, p.head_dim = self.q.shape
        p.total_k, p.num_heads_kv = self.k.shape[0], self.k.shape[1]
        p.cu_seqlens_q = self.cu_seqlens_q.ctypes.data
        p.cu_seqlens_k = self.cu_seqlens_k.ctypes.data
        p.q, p.k, p.v = self.q.ctypes.data, self.k.ctypes.data, self.v.ctypes.data
        p.bias_table = self.table.ctypes.data if self.table is not None else None
        p.num_buckets, p.max_distance = int(self.num_buckets), int(self.max_distance)
        p.bidirectional = int(bool(self.bidirectional))
        p.alibi_slopes = self.slopes.ctypes.data if self.slopes is not None else None
        p.causal = int(bool(self.causal))
        p.softmax_scale = float(self.scale)
        return p


def xattn_fwd(pb: XProblem):
    """Returns (out fp64 [total_q, Hq, d], lse fp64 [Hq, total_q])."""
    if len(pb.cu_seqlens_k) != len(pb.cu_seqlens_q) or pb.k.shape != pb.v.shape:
        raise ValueError("oracle xattn_fwd: mismatched problem")
    Tq, Hq, d = pb.q.shape
    out = np.zeros((Tq, Hq, d))
    lse = np.zeros((Hq, Tq))
    c = pb._c()
    _check(_load().oracle_xattn_fwd(ctypes.byref(c), out.ctypes.data, lse.ctypes.data),
           "xattn_fwd")
    return out, lse


def xattn_bwd(pb: XProblem, dout: np.ndarray):
    """Gradients of sum(out * dout): (dq, dk, dv, dtable or None)."""
    if len(pb.cu_seqlens_k) != len(pb.cu_seqlens_q) or pb.k.shape != pb.v.shape:
        raise ValueError("oracle xattn_bwd: mismatched problem")
    dout = widen(dout)
    if dout.shape != pb.q.shape:
        raise ValueError("oracle xattn_bwd: dout shape")
    dq = np.zeros(pb.q.shape)
    dk = np.zeros(pb.k.shape)
    dv = np.zeros(pb.v.shape)
    dt = np.zeros((pb.num_buckets, pb.q.shape[1])) if pb.table is not None else None
    c = pb._c()
    _check(_load().oracle_xattn_bwd(ctypes.byref(c), dout.ctypes.data, dq.ctypes.data,
                                    dk.ctypes.data, dv.ctypes.data,
                                    dt.ctypes.data if dt is not None else None), "xattn_bwd")
    return dq, dk, dv, dt


# ---- rotary position embedding (RoPE), applied to Q and K before plain attention ----
def rope_rotate_at(x, positions, base: float = 10000.0, inverse: bool = False) -> np.ndarray:
    """Rotary position embedding of RoFormer, the RoPE the FAT5 report lists among the
    positional encodings its kernels accept (positional-encoding note of the "Noyau CUDA"
    section). Channel pair (2i, 2i+1) of a row at position m is turned by the angle
    m * base^(-2i/d); inverse=True turns it back (the transpose, used for gradients).
    x: [T, H, d] (d even); positions: [T]. fp64 throughout."""
    x = widen(x)
    T, H, d = x.shape
    if d % 2:
        raise ValueError("rotary embedding needs an even head_dim")
    pos = np.asarray(positions, dtype=np.float64).reshape(T)
    theta = base ** (-np.arange(0, d, 2, dtype=np.float64) / d)  # [d/2]
    ang = pos[:, None] * theta[None, :]  # [T, d/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    if inverse:
        s = -s
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def doc_positions(cu_seqlens) -> np.ndarray:
    """Position of every packed token within its document (restarting at 0 per document)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    pos = np.zeros(int(cu[-1]), dtype=np.int64)
    for i in range(len(cu) - 1):
        pos[cu[i]:cu[i + 1]] = np.arange(cu[i + 1] - cu[i])
    return pos


def rope_attn_fwd(pb: Problem, base: float = 10000.0):
    """Attention with RoPE on Q and K (positions local to each document) and the problem's own
    bias/mask settings: the plain oracle on the rotated inputs. Returns (out, lse)."""
    pos = doc_positions(pb.cu_seqlens)
    rot = _replace_qk(pb, rope_rotate_at(pb.q, pos, base), rope_rotate_at(pb.k, pos, base))
    return attn_fwd(rot)


def rope_attn_bwd(pb: Problem, dout: np.ndarray, base: float = 10000.0):
    """Gradients of sum(out * dout) with respect to the unrotated q, k, v (and the table): the
    rotation is orthogonal, so dq and dk are the rotated-space gradients turned back."""
    pos = doc_positions(pb.cu_seqlens)
    rot = _replace_qk(pb, rope_rotate_at(pb.q, pos, base), rope_rotate_at(pb.k, pos, base))
    dq_r, dk_r, dv, dt = attn_bwd(rot, dout)
    return (rope_rotate_at(dq_r, pos, base, inverse=True),
            rope_rotate_at(dk_r, pos, base, inverse=True), dv, dt)


def _replace_qk(pb: Problem, q, k) -> Problem:
    return Problem(q, k, pb.v, pb.cu_seqlens, table=pb.table, num_buckets=pb.num_buckets,
                   max_distance=pb.max_distance, bidirectional=pb.bidirectional,
                   slopes=pb.slopes, causal=pb.causal, scale=pb.scale,
                   d_from_bf16_out=pb.d_from_bf16_out)

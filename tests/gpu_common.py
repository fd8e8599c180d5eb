"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI, build the
matching oracle problem from the same seeded inputs, and compare."""
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
# per-bucket tolerance (causal T5, unscaled logits; oracle against oracle). So the small cases
# compare the table gradient with the oracle in its bf16-output mode (D from the bf16-rounded
# output, the quantity this backward is defined on).
U_D = 2.0 ** -8
ATOL = 2e-2
RTOL = 1e-2
LSE_ATOL = 1e-3
DBIAS_REL = 1e-2


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


def assert_close(name, got, ref, atol=ATOL, rtol=RTOL, slack=0.0):
    err = np.abs(got - ref)
    lim = atol + rtol * np.abs(ref) + slack
    bad = err > lim
    if bad.any():
        idx = np.unravel_index(np.argmax(err - lim), err.shape)
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {err.size} elements out of tolerance; worst at {idx}: "
            f"got {got[idx]!r} ref {ref[idx]!r} (max abs err {err.max():.3e})")
    return float(err.max())


def assert_dbias(got, ref):
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    assert rel <= DBIAS_REL, f"dbias norm-wise relative error {rel:.3e}"
    per = np.abs(got - ref)
    lim = 1e-2 * np.abs(ref).max() + 1e-3
    assert (per <= lim).all(), f"dbias per-bucket error {per.max():.3e} > {lim:.3e}"
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

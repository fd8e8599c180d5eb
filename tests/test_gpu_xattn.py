"""GPU parity of the generalised problem: own query and key lengths per document
(cross-attention, queries over a longer key cache, decode steps), grouped-query heads and
bottom-right causal alignment, forward and backward through the C ABI, against the fp64
cross-attention oracle on the same seeded inputs; the split-key forward against the oracle and
against the unsplit forward."""
import numpy as np
import pytest
import torch

import attention_relative_position_gb300 as fa
import oracle
from attention_relative_position_gb300 import workloads as wl
from gpu_common import LSE_ATOL, U_D, U_OP, _bias, assert_dbias, check, grad_tol

pytestmark = pytest.mark.gpu

XW = wl.XWorkload
CASES = [
    # T5 decoder cross-attention: no bias, queries over the encoder output, empty documents on
    # either side (no keys: out 0, lse -inf)
    XW("xattn_cross_nobias_d64", (100, 257, 1, 0, 64, 130), (300, 40, 129, 50, 0, 700), 4, 4,
       64, 0.7, seed=61),
    # decoder self-attention over a longer cache: causal bottom-right, unidirectional T5 bias,
    # grouped heads
    XW("xattn_cache_causal_t5_gqa_d64", (50, 128, 200, 1), (300, 128, 513, 257), 8, 2, 64, 0.5,
       (32, 128, False), causal=True, seed=62),
    # more queries than keys, causal: the first Lq - Lk rows see no key
    XW("xattn_causal_fewer_keys_alibi_d128", (300, 40), (100, 170), 4, 1, 128, 1.0, None, True,
       True, 128 ** -0.5, seed=63),
    # bidirectional T5 + ALiBi with grouped heads, non-causal, d 128
    XW("xattn_t5_alibi_gqa_d128", (129, 77), (200, 333), 4, 2, 128, 0.6, (32, 128, True), True,
       False, 0.3, seed=64),
    # equal documents, grouped heads, no causal mask: the backward's key-tile CTAs are split
    # along the query tiles, their dK, dV added into the grouped-head accumulators
    XW("xattn_equal_docs_split_bwd_gqa_d128", (300,) * 3, (520,) * 3, 4, 2, 128, 0.6,
       (32, 128, True), True, False, 0.3, seed=71),
]


def _args(w):
    t5 = w.t5 or (0, 0, True)
    return dict(num_buckets=t5[0], max_distance=t5[1], bidirectional=t5[2], causal=w.causal,
                softmax_scale=w.scale)


def _xproblem(w, x, **over):
    t5 = w.t5 or (0, 0, True)
    d = dict(q=wl.bf16_bits(x["q"]), k=wl.bf16_bits(x["k"]), v=wl.bf16_bits(x["v"]),
             cu_seqlens_q=x["cu_seqlens_q"].cpu().numpy(),
             cu_seqlens_k=x["cu_seqlens_k"].cpu().numpy(),
             table=x["table"].cpu().numpy() if x["table"] is not None else None,
             num_buckets=t5[0], max_distance=t5[1], bidirectional=t5[2],
             slopes=x["slopes"].cpu().numpy() if x["slopes"] is not None else None,
             causal=w.causal, scale=w.scale)
    d.update(over)
    return oracle.XProblem(**d)


def _gpu(w, x, num_splits=1, bwd=True):
    kw = _args(w)
    out, lse = fa.fat_xattn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"],
                                w.max_seqlen_q, w.max_seqlen_k, bias_table=x["table"],
                                alibi_slopes=x["slopes"], num_splits=num_splits, **kw)
    res = dict(out=out, lse=lse)
    if bwd:
        dq, dk, dv, dt = fa.fat_xattn_bwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                                          x["cu_seqlens_k"], w.max_seqlen_q, w.max_seqlen_k, out,
                                          lse, x["dout"], bias_table=x["table"],
                                          alibi_slopes=x["slopes"], **kw)
        res.update(dq=dq, dk=dk, dv=dv, dbias=dt)
    torch.cuda.synchronize()
    assert fa.fat_attn_get_device_error() == 0
    return {k: (v.float().cpu().numpy() if v is not None else None) for k, v in res.items()}


def _xbounds(pb, dout64, ro, rl):
    """bf16-operand bounds (see gpu_common) of the generalised problem: dq per query head, dk and
    dv summed over the query heads that share a key/value head."""
    bq, bk, bv = np.zeros_like(pb.q), np.zeros_like(pb.k), np.zeros_like(pb.v)
    Hq, Hkv = pb.q.shape[1], pb.k.shape[1]
    cq, ck = pb.cu_seqlens_q, pb.cu_seqlens_k
    for doc in range(len(cq) - 1):
        sq, lq = int(cq[doc]), int(cq[doc + 1] - cq[doc])
        sk, lk = int(ck[doc]), int(ck[doc + 1] - ck[doc])
        if lq == 0 or lk == 0:
            continue
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            Q, K, V = pb.q[sq:sq + lq, h], pb.k[sk:sk + lk, hk], pb.v[sk:sk + lk, hk]
            dO = dout64[sq:sq + lq, h]
            b, delta = _bias(pb, h, np.arange(lq), np.arange(lk), shift=lk - lq)
            x = pb.scale * Q @ K.T + b
            if pb.causal:
                x = np.where(delta > 0, -np.inf, x)
            lse = rl[h, sq:sq + lq][:, None]
            ok = np.isfinite(lse)
            P = np.where(ok, np.exp(x - np.where(ok, lse, 0.0)), 0.0)
            D = (dO * ro[sq:sq + lq, h]).sum(-1)
            dS = P * (dO @ V.T - D[:, None])
            bq[sq:sq + lq, h] = U_OP * pb.scale * np.abs(dS) @ np.abs(K)
            bk[sk:sk + lk, hk] += U_OP * pb.scale * np.abs(dS).T @ np.abs(Q)
            bv[sk:sk + lk, hk] += U_OP * P.T @ np.abs(dO)
    return dict(dq=bq, dk=bk, dv=bv)


def _check_grads(case, res, pb, w, dout, ro, rl):
    rq, rk, rv, rt = oracle.xattn_bwd(pb, dout)
    # D = rowsum(dout * out) is formed from the bf16 output; its propagated effect on dq and dk
    # (see gpu_common): |d dq| <= scale |delta| sum_k P |K|, |d dk| <= scale sum_q P |delta| |Q|
    b1 = U_D * np.abs(dout * ro).sum(-1)
    pk, _ = oracle.xattn_fwd(oracle.XProblem(pb.q, pb.k, np.abs(pb.k), pb.cu_seqlens_q,
                                             pb.cu_seqlens_k, table=pb.table,
                                             num_buckets=pb.num_buckets,
                                             max_distance=pb.max_distance,
                                             bidirectional=pb.bidirectional, slopes=pb.slopes,
                                             causal=pb.causal, scale=pb.scale))
    _, _, dkw, _ = oracle.xattn_bwd(pb, b1[..., None] * np.abs(pb.q))
    ob = _xbounds(pb, dout, ro, rl)
    check(case, "dv", res["dv"], rv, grad_tol(rv, ob["dv"]), mode="exact+op")
    check(case, "dq", res["dq"], rq, grad_tol(rq, w.scale * b1[..., None] * pk + ob["dq"]),
          mode="exact+D+op")
    check(case, "dk", res["dk"], rk, grad_tol(rk, w.scale * dkw + ob["dk"]), mode="exact+D+op")
    if rt is not None:
        assert_dbias(res["dbias"], rt, case, mode="exact", per_bucket=False)


def _check_fwd(case, res, ro, rl):
    check(case, "out", res["out"], ro, grad_tol(ro))
    finite = np.isfinite(rl)
    # rows that see no key: lse -inf on both sides, out exactly 0
    assert np.array_equal(np.isfinite(res["lse"]), finite), case
    assert (res["out"][~finite.T] == 0).all(), case
    check(case, "lse", res["lse"][finite], rl[finite], LSE_ATOL)


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_xattn_forward_and_backward(w):
    x = wl.make_xinputs(w, device="cuda")
    res = _gpu(w, x)
    pb = _xproblem(w, x)
    ro, rl = oracle.xattn_fwd(pb)
    _check_fwd(w.name, res, ro, rl)
    dout = oracle.widen(wl.bf16_bits(x["dout"]))
    _check_grads(w.name, res, pb, w, dout, ro, rl)


def test_xattn_equals_self_attention_when_lengths_match():
    """Lq = Lk per document and one key/value head per query head: the generalised calls give
    bit-identical results to the self-attention calls."""
    w = wl.Workload("xattn_vs_self", (300, 129, 77), 2, 64, 0.5, (32, 128, False), False, True,
                    1.0, seed=65)
    x = wl.make_inputs(w, device="cuda")
    kw = dict(bias_table=x["table"], num_buckets=32, max_distance=128, bidirectional=False,
              causal=True, softmax_scale=1.0)
    o1, l1 = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, **kw)
    o2, l2 = fa.fat_xattn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens"],
                              w.max_seqlen, w.max_seqlen, **kw)
    g1 = fa.fat_attn_bwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, o1, l1,
                         x["dout"], **kw)
    g2 = fa.fat_xattn_bwd(x["q"], x["k"], x["v"], x["cu_seqlens"], x["cu_seqlens"],
                          w.max_seqlen, w.max_seqlen, o2, l2, x["dout"], **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1[:3], g2[:3]):
        assert torch.equal(a, b)
    torch.testing.assert_close(g1[3], g2[3], rtol=1e-5, atol=1e-5)  # atomic order only


DECODE = [
    # one new query per document over its key cache (T5 decoder, causal, unidirectional bias)
    XW("decode_t5_causal_d64", (1,) * 12, tuple(int(x) for x in
       np.random.default_rng(66).integers(200, 3000, 12)), 8, 8, 64, 0.5, (32, 128, False),
       causal=True, seed=66),
    # grouped heads, d 128, ALiBi, a few queries per document (chunked decode)
    XW("decode_gqa_alibi_d128", (1, 4, 2, 1), (4000, 1500, 129, 7), 8, 2, 128, 1.0, None, True,
       True, 128 ** -0.5, seed=67),
    # the few-row kernel's row tiles: 8 rows (one query x 8 heads of a group; two queries x 4
    # heads), 4 rows (4 heads over one key/value head), with a document without keys, a
    # document with more queries than keys (its first query sees nothing under the causal
    # mask) and empty key ranges when the split count exceeds the key tiles
    XW("decode_gqa8_t5bidir_d128", (1,) * 6, (3000, 0, 1, 513, 4096, 77), 16, 2, 128, 0.5,
       (32, 128, True), False, False, 128 ** -0.5, seed=68),
    XW("decode_chunk2_gqa4_t5_alibi_causal_d64", (2, 1, 2, 0, 2), (700, 1, 2049, 30, 1), 8, 2,
       64, 0.5, (32, 64, False), True, True, 0.125, seed=69),
    XW("decode_mqa_causal_d128", (1, 1, 1), (5000, 2500, 640), 4, 1, 128, 1.0, None, False,
       True, 128 ** -0.5, seed=70),
    # query chunks of up to 64 rows with grouped heads at d 64: too many rows for the few-row
    # kernel, so the tiled forward with one Q tile per CTA takes the key splits
    XW("chunk64_gqa2_t5_causal_splitkv_d64", (20, 3, 64), (900, 2000, 700), 4, 2, 64, 0.5,
       (32, 128, False), causal=True, seed=72),
]


@pytest.mark.parametrize("w", DECODE, ids=[w.name for w in DECODE])
def test_decode_split_kv(w):
    x = wl.make_xinputs(w, device="cuda")
    pb = _xproblem(w, x)
    ro, rl = oracle.xattn_fwd(pb)
    whole = _gpu(w, x, num_splits=1, bwd=False)
    _check_fwd(w.name + " (unsplit)", whole, ro, rl)
    auto = fa.fat_xattn_splitkv_num_splits(x["q"], x["k"], x["cu_seqlens_q"], w.max_seqlen_q,
                                           w.max_seqlen_k)
    assert auto > 1  # few rows, long keys: the library splits
    for ns in sorted({2, 3, auto, 64}):
        res = _gpu(w, x, num_splits=ns, bwd=False)
        _check_fwd(f"{w.name} ({ns} splits)", res, ro, rl)
        # the merge reproduces the unsplit result up to the bf16 rounding of out
        assert np.abs(res["out"] - whole["out"]).max() <= 2 ** -7 * max(1.0, np.abs(ro).max())
        fin = np.isfinite(whole["lse"])  # rows without keys: -inf on both sides
        assert np.array_equal(np.isfinite(res["lse"]), fin)
        assert np.abs(res["lse"][fin] - whole["lse"][fin]).max() <= 1e-4
    # and the backward of a decode step (one query over the cache) against the oracle
    res = _gpu(w, x, num_splits=0, bwd=True)
    dout = oracle.widen(wl.bf16_bits(x["dout"]))
    _check_grads(w.name, res, pb, w, dout, ro, rl)

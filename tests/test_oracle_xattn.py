"""Pins for the generalised fp64 oracle (own query and key lengths per document, grouped-query
heads, bottom-right causal alignment; no GPU).

The generalised oracle is tied to things other than itself: the already pinned self-attention
oracle (to which it must reduce when Lq = Lk and every query head has its own key/value head),
the same oracle with key/value heads repeated (grouped-query heads), torch SDPA and autograd in
fp64 with an explicit mask built from the independent exact bucket function, and central finite
differences. A slip in the alignment shift, the head grouping, the group sums of dK/dV or the
sign of the relative position fails at least one of them.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_buckets import exact_bucket


def _xproblem(lq, lk, hq, hkv, d, seed, t5=None, alibi=False, causal=False, scale=0.7):
    rng = np.random.default_rng(seed)
    tq, tk = sum(lq), sum(lk)
    q = rng.standard_normal((tq, hq, d))
    k = rng.standard_normal((tk, hkv, d))
    v = rng.standard_normal((tk, hkv, d))
    table = rng.standard_normal((t5[0], hq)) * 0.5 if t5 else None
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / hq) for h in range(hq)]) if alibi else None
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    kw = dict(num_buckets=t5[0], max_distance=t5[1], bidirectional=t5[2]) if t5 else {}
    return oracle.XProblem(q, k, v, cq, ck, table=table, slopes=slopes, causal=causal,
                           scale=scale, **kw)


def _self_problem(xp):
    """The same problem in the self-attention oracle's form (needs Lq = Lk and Hq = Hkv)."""
    return oracle.Problem(xp.q, xp.k, xp.v, xp.cu_seqlens_q, table=xp.table,
                          num_buckets=xp.num_buckets, max_distance=xp.max_distance,
                          bidirectional=xp.bidirectional, slopes=xp.slopes, causal=xp.causal,
                          scale=xp.scale)


def _torch_loss(xp, dout, q, k, v, table):
    """sum(out * dout) through torch SDPA (fp64) with an explicit additive mask per document and
    head; the relative position is r - (p + Lk - Lq), bucketed by the exact integer form."""
    hq, hkv = xp.q.shape[1], xp.k.shape[1]
    grp = hq // hkv
    loss = torch.zeros((), dtype=torch.float64)
    for i in range(len(xp.cu_seqlens_q) - 1):
        sq, eq = int(xp.cu_seqlens_q[i]), int(xp.cu_seqlens_q[i + 1])
        sk, ek = int(xp.cu_seqlens_k[i]), int(xp.cu_seqlens_k[i + 1])
        lq, lk = eq - sq, ek - sk
        if lq == 0 or lk == 0:
            continue
        rel = torch.arange(lk)[None, :] - (torch.arange(lq)[:, None] + (lk - lq))
        for h in range(hq):
            mask = torch.zeros((lq, lk), dtype=torch.float64)
            if table is not None:
                bidx = torch.tensor([[exact_bucket(int(r), xp.num_buckets, xp.max_distance,
                                                   xp.bidirectional) for r in row] for row in rel])
                mask = mask + table[:, h][bidx]
            if xp.slopes is not None:
                mask = mask - float(xp.slopes[h]) * rel.abs().double()
            if xp.causal:
                mask = mask.masked_fill(rel > 0, float("-inf"))
            o = torch.nn.functional.scaled_dot_product_attention(
                q[sq:eq, h][None], k[sk:ek, h // grp][None], v[sk:ek, h // grp][None],
                attn_mask=mask, scale=xp.scale)
            loss = loss + (o[0] * torch.from_numpy(dout[sq:eq, h])).sum()
    return loss


@pytest.mark.parametrize("t5,alibi,causal", [((8, 16, True), False, False),
                                             ((16, 24, False), True, True),
                                             (None, True, False)])
def test_reduces_to_self_attention_oracle(t5, alibi, causal):
    xp = _xproblem([9, 1, 14], [9, 1, 14], 2, 2, 5, seed=50, t5=t5, alibi=alibi, causal=causal)
    sp = _self_problem(xp)
    o1, l1 = oracle.xattn_fwd(xp)
    o0, l0 = oracle.attn_fwd(sp)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-13)
    dout = np.random.default_rng(51).standard_normal(xp.q.shape)
    g1 = oracle.xattn_bwd(xp, dout)
    g0 = oracle.attn_bwd(sp, dout)
    for a, b in zip(g1, g0):
        if a is None:
            assert b is None
            continue
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_grouped_heads_equal_repeated_key_value_heads():
    xp = _xproblem([11, 6], [11, 6], 6, 2, 4, seed=52, t5=(8, 16, True), alibi=True, causal=True)
    grp = 3
    rep = oracle.Problem(xp.q, np.repeat(xp.k, grp, axis=1), np.repeat(xp.v, grp, axis=1),
                         xp.cu_seqlens_q, table=xp.table, num_buckets=xp.num_buckets,
                         max_distance=xp.max_distance, bidirectional=xp.bidirectional,
                         slopes=xp.slopes, causal=True, scale=xp.scale)
    o1, l1 = oracle.xattn_fwd(xp)
    o0, l0 = oracle.attn_fwd(rep)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-13)
    dout = np.random.default_rng(53).standard_normal(xp.q.shape)
    dq1, dk1, dv1, dt1 = oracle.xattn_bwd(xp, dout)
    dq0, dk0, dv0, dt0 = oracle.attn_bwd(rep, dout)
    np.testing.assert_allclose(dq1, dq0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dt1, dt0, rtol=0, atol=1e-12)
    # a key/value head's gradient is the sum over the query heads that read it
    T, _, d = xp.k.shape
    np.testing.assert_allclose(dk1, dk0.reshape(T, 2, grp, d).sum(axis=2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv1, dv0.reshape(T, 2, grp, d).sum(axis=2), rtol=0, atol=1e-12)


@pytest.mark.parametrize("t5,alibi,causal", [(None, False, False), (None, False, True),
                                             ((8, 16, True), True, False),
                                             ((16, 24, False), False, True)])
def test_cross_lengths_match_torch_sdpa_and_autograd(t5, alibi, causal):
    # documents with fewer queries than keys (decoder over an encoder output, or new tokens over
    # a longer key cache); Lq <= Lk keeps every causal row non-empty for the SDPA comparison
    xp = _xproblem([3, 7, 1], [10, 7, 5], 4, 2, 6, seed=54, t5=t5, alibi=alibi, causal=causal,
                   scale=0.9)
    dout = np.random.default_rng(55).standard_normal(xp.q.shape)
    out, _ = oracle.xattn_fwd(xp)
    dq, dk, dv, dt = oracle.xattn_bwd(xp, dout)
    q = torch.from_numpy(xp.q.copy()).requires_grad_()
    k = torch.from_numpy(xp.k.copy()).requires_grad_()
    v = torch.from_numpy(xp.v.copy()).requires_grad_()
    table = torch.from_numpy(xp.table.copy()).requires_grad_() if xp.table is not None else None
    loss = _torch_loss(xp, dout, q, k, v, table)
    assert abs(float(loss.detach()) - float((out * dout).sum())) < 1e-10
    loss.backward()
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=1e-9, atol=1e-11)
    if dt is not None:
        np.testing.assert_allclose(dt, table.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_alignment_is_bottom_right():
    # one document, 2 queries over 6 keys, causal: query 0 sits at key position 4, query 1 at 5
    xp = _xproblem([2], [6], 1, 1, 3, seed=56, causal=True)
    out, _ = oracle.xattn_fwd(xp)
    xp_cut = oracle.XProblem(xp.q, xp.k[:5], xp.v[:5], xp.cu_seqlens_q, np.array([0, 5]),
                             causal=False, scale=xp.scale)
    o_cut, _ = oracle.xattn_fwd(xp_cut)  # query 0 sees keys 0..4 only
    np.testing.assert_allclose(out[0], o_cut[0], rtol=0, atol=1e-14)
    xp_all = oracle.XProblem(xp.q, xp.k, xp.v, xp.cu_seqlens_q, xp.cu_seqlens_k, causal=False,
                             scale=xp.scale)
    o_all, _ = oracle.xattn_fwd(xp_all)  # the last query sees every key
    np.testing.assert_allclose(out[1], o_all[1], rtol=0, atol=1e-14)


def test_rows_without_keys():
    # causal with more queries than keys: the first Lq - Lk queries see no key at all
    xp = _xproblem([5, 2], [3, 0], 2, 1, 4, seed=57, causal=True)
    out, lse = oracle.xattn_fwd(xp)
    assert np.all(np.isneginf(lse[:, [0, 1, 5, 6]]))
    assert np.all(np.isfinite(lse[:, 2:5]))
    np.testing.assert_array_equal(out[[0, 1, 5, 6]], 0.0)
    dout = np.random.default_rng(58).standard_normal(xp.q.shape)
    dq, dk, dv, _ = oracle.xattn_bwd(xp, dout)
    np.testing.assert_array_equal(dq[[0, 1, 5, 6]], 0.0)
    # the remaining rows of document 0 are plain causal self-attention over its 3 keys
    sub = oracle.XProblem(xp.q[2:5], xp.k, xp.v, np.array([0, 3]), np.array([0, 3]),
                          causal=True, scale=xp.scale)
    o_sub, _ = oracle.xattn_fwd(sub)
    np.testing.assert_allclose(out[2:5], o_sub, rtol=0, atol=1e-14)
    _, dk_sub, dv_sub, _ = oracle.xattn_bwd(sub, dout[2:5])
    np.testing.assert_allclose(dk, dk_sub, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dv_sub, rtol=0, atol=1e-13)


def test_finite_differences():
    xp = _xproblem([4, 3], [6, 3], 4, 2, 3, seed=59, t5=(8, 12, True), alibi=True, causal=True,
                   scale=0.8)
    dout = np.random.default_rng(60).standard_normal(xp.q.shape)
    dq, dk, dv, dt = oracle.xattn_bwd(xp, dout)
    eps = 1e-6

    def loss():
        return float((oracle.xattn_fwd(xp)[0] * dout).sum())

    def fd(arr, idx):
        old = arr[idx]
        arr[idx] = old + eps
        lp = loss()
        arr[idx] = old - eps
        lm = loss()
        arr[idx] = old
        return (lp - lm) / (2 * eps)

    for name, arr, grad, picks in (
            ("q", xp.q, dq, [(0, 0, 0), (3, 2, 1), (6, 3, 2)]),
            ("k", xp.k, dk, [(0, 0, 0), (5, 1, 2), (8, 0, 1)]),
            ("v", xp.v, dv, [(1, 1, 0), (4, 0, 2), (7, 1, 1)])):
        for idx in picks:
            want = fd(arr, idx)
            assert abs(grad[idx] - want) <= 1e-6 * max(1.0, abs(want)), (name, idx)
    for b in range(8):
        for h in range(4):
            want = fd(xp.table, (b, h))
            assert abs(dt[b, h] - want) <= 1e-6 * max(1.0, abs(want)), ("table", b, h)


def test_argument_errors():
    xp = _xproblem([3], [4], 3, 2, 4, seed=61)  # 3 query heads cannot share 2 key/value heads
    with pytest.raises(ValueError):
        oracle.xattn_fwd(xp)
    xp = _xproblem([3], [4], 2, 1, 4, seed=62)
    xp.cu_seqlens_k = np.array([0, 3], dtype=np.int32)  # does not end at total_k
    with pytest.raises(ValueError):
        oracle.xattn_fwd(xp)


@pytest.mark.parametrize("t5,alibi", [((32, 128, False), False), (None, True)])
def test_decode_row_equals_last_row_of_self_attention(t5, alibi):
    # decode step: one new query over the whole key cache of its document (causal decoder with
    # T5 or ALiBi bias) equals the last row of causal self-attention over the full sequence
    L = [40, 17]
    full = _xproblem(L, L, 2, 2, 8, seed=63, t5=t5, alibi=alibi, causal=True)
    o_full, l_full = oracle.xattn_fwd(full)
    last = np.cumsum(L) - 1
    dec = oracle.XProblem(full.q[last], full.k, full.v, np.array([0, 1, 2]), full.cu_seqlens_k,
                          table=full.table, num_buckets=full.num_buckets,
                          max_distance=full.max_distance, bidirectional=full.bidirectional,
                          slopes=full.slopes, causal=True, scale=full.scale)
    o_dec, l_dec = oracle.xattn_fwd(dec)
    np.testing.assert_allclose(o_dec, o_full[last], rtol=0, atol=1e-14)
    np.testing.assert_allclose(l_dec, l_full[:, last], rtol=0, atol=1e-14)

"""Pins for the fp64 CPU oracle (no GPU).

The pages fix no numeric examples, so each pin comes from mathematics the oracle must obey:
closed forms of the T5 bucket thresholds, the ALiBi form, uniform attention, softmax row sums,
shift invariance, a library routine (torch SDPA in fp64 with an explicit additive mask, built
here from an independent exact bucket implementation), causality, packing independence,
finite differences and gradient invariants. Each is chosen so that a plausible slip in the
oracle (dropped scale, wrong sign of the relative position, transposed operand, wrong bucket
rounding, missing mask) fails at least one of them.
"""
import math
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from attention_relative_position_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "t5_buckets.txt")


from exact_buckets import exact_bucket, exact_thresholds  # noqa: E402


BUCKET_CASES = [(32, 128, True), (32, 128, False), (64, 1024, True), (64, 1024, False),
                (32, 64, True), (128, 4096, True), (8, 16, True), (8, 16, False), (16, 20, False)]


@pytest.mark.parametrize("nb,md,bidir", BUCKET_CASES)
def test_bucket_matches_exact_threshold_form(nb, md, bidir):
    for delta in range(-20000, 20001):
        if abs(delta) > 3000 and delta % 37:
            continue  # dense near the origin, sparse beyond (saturated there)
        assert oracle.t5_bucket(delta, nb, md, bidir) == exact_bucket(delta, nb, md, bidir), delta


def test_bucket_golden_hand_derived():
    n = 0
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            nb, md, bidir, delta, want = map(int, line.split())
            assert oracle.t5_bucket(delta, nb, md, bool(bidir)) == want, line
            n += 1
    assert n >= 50


@pytest.mark.parametrize("nb,md,bidir", BUCKET_CASES)
def test_bucket_structure(nb, md, bidir):
    nbh = nb // 2 if bidir else nb
    prev = -1
    for n in range(0, 5000):
        b_neg = oracle.t5_bucket(-n, nb, md, bidir)
        assert 0 <= b_neg < nbh
        assert b_neg >= prev  # monotone in distance
        prev = b_neg
        if n < nbh // 2:
            assert b_neg == n  # exact region
    assert oracle.t5_bucket(-10 ** 7, nb, md, bidir) == nbh - 1  # saturation
    if bidir:
        assert oracle.t5_bucket(1, nb, md, bidir) == nbh + 1
        assert oracle.t5_bucket(10 ** 7, nb, md, bidir) == nb - 1
    else:
        for dl in (0, 1, 5, 10 ** 6):
            assert oracle.t5_bucket(dl, nb, md, bidir) == 0


def test_alibi_closed_form():
    for dl in (-300, -1, 0, 1, 17, 8191):
        assert oracle.alibi_bias(dl, 0.25) == -0.25 * abs(dl)
    s = workloads.alibi_slopes(16)
    assert s[0] == np.float32(2 ** -0.5)
    assert s[15] == np.float32(2 ** -8)
    assert np.all(np.diff(s) < 0)
    s8 = workloads.alibi_slopes(8)
    np.testing.assert_allclose(s8, [2.0 ** -(h + 1) for h in range(8)], rtol=0)


# --------------------------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------------------------
def _rand_problem(seqlens, H, d, seed, t5=None, alibi=False, causal=False, scale=0.7,
                  table_scale=0.5):
    rng = np.random.default_rng(seed)
    T = sum(seqlens)
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    table = rng.standard_normal((t5[0], H)) * table_scale if t5 else None
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)]) if alibi else None
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    kw = dict(num_buckets=t5[0], max_distance=t5[1], bidirectional=t5[2]) if t5 else {}
    return oracle.Problem(q, k, v, cu, table=table, slopes=slopes, causal=causal, scale=scale,
                          **kw)


def _bias_matrix(pb: oracle.Problem, L: int, h: int) -> np.ndarray:
    """Independent construction of the additive bias for one document and head."""
    B = np.zeros((L, L))
    for p in range(L):
        for r in range(L):
            b = 0.0
            if pb.table is not None:
                b += pb.table[exact_bucket(r - p, pb.num_buckets, pb.max_distance,
                                           pb.bidirectional), h]
            if pb.slopes is not None:
                b += -pb.slopes[h] * abs(r - p)
            B[p, r] = b
    return B


def _sdpa_reference(pb: oracle.Problem):
    """torch SDPA (CPU, fp64) per document with the bias as an explicit float mask."""
    T, H, d = pb.shape
    out = np.zeros((T, H, d))
    cu = pb.cu_seqlens
    for i in range(len(cu) - 1):
        s, e = int(cu[i]), int(cu[i + 1])
        L = e - s
        if L == 0:
            continue
        for h in range(H):
            q = torch.from_numpy(pb.q[s:e, h]).unsqueeze(0)
            k = torch.from_numpy(pb.k[s:e, h]).unsqueeze(0)
            v = torch.from_numpy(pb.v[s:e, h]).unsqueeze(0)
            mask = torch.from_numpy(_bias_matrix(pb, L, h))
            if pb.causal:
                mask = mask.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool), 1),
                                        float("-inf"))
            o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                                 scale=pb.scale)
            out[s:e, h] = o[0].numpy()
    return out


# --------------------------------------------------------------------------------------------
# forward pins
# --------------------------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_uniform_attention_when_q_zero_and_bias_constant(causal):
    pb = _rand_problem([7, 13], 2, 8, seed=1, t5=(8, 16, True), causal=causal)
    pb.q[:] = 0.0
    c = 0.375
    pb.table[:] = c
    out, lse = oracle.attn_fwd(pb)
    for i in range(2):
        s, e = pb.cu_seqlens[i], pb.cu_seqlens[i + 1]
        for p in range(e - s):
            n_allowed = (p + 1) if causal else (e - s)
            want = pb.v[s:s + n_allowed].mean(axis=0)
            np.testing.assert_allclose(out[s + p], want, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse[:, s + p], math.log(n_allowed) + c, rtol=1e-13)


def test_rows_of_p_sum_to_one():
    pb = _rand_problem([5, 11, 1], 3, 8, seed=2, t5=(16, 32, False), alibi=True, causal=True)
    pb.v[:] = 1.0
    out, _ = oracle.attn_fwd(pb)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-13)


def test_constant_table_shift_moves_only_lse():
    pb = _rand_problem([9, 6], 2, 8, seed=3, t5=(8, 16, True))
    out0, lse0 = oracle.attn_fwd(pb)
    pb.table += 1.25
    out1, lse1 = oracle.attn_fwd(pb)
    np.testing.assert_allclose(out1, out0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse1, lse0 + 1.25, rtol=0, atol=1e-12)


@pytest.mark.parametrize("cfg", [
    dict(t5=None, alibi=False, causal=False),
    dict(t5=None, alibi=False, causal=True),
    dict(t5=(8, 16, True), alibi=False, causal=False),
    dict(t5=(16, 24, False), alibi=False, causal=True),
    dict(t5=None, alibi=True, causal=False),
    dict(t5=(8, 16, True), alibi=True, causal=True),
])
def test_forward_matches_torch_sdpa_fp64(cfg):
    pb = _rand_problem([12, 1, 20, 0, 5], 2, 8, seed=4, scale=0.6, **cfg)
    out, lse = oracle.attn_fwd(pb)
    ref = _sdpa_reference(pb)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_relative_position_sign_convention():
    """A large bias on bucket(+1) only (bidirectional) makes each query copy the next key's
    value: delta = key - query, positive to the right."""
    L = 10
    pb = _rand_problem([L], 1, 4, seed=5, t5=(8, 16, True))
    pb.q[:] = 0.0
    pb.table[:] = 0.0
    pb.table[exact_bucket(+1, 8, 16, True), 0] = 60.0
    out, _ = oracle.attn_fwd(pb)
    for p in range(L - 1):
        np.testing.assert_allclose(out[p, 0], pb.v[p + 1, 0], atol=1e-12)


def test_scale_applies_to_qk_only():
    pb = _rand_problem([9], 1, 8, seed=6, t5=(8, 16, True), scale=1.0)
    out1, lse1 = oracle.attn_fwd(pb)
    pb.scale = 0.5
    pb.q *= 2.0
    out2, lse2 = oracle.attn_fwd(pb)
    np.testing.assert_allclose(out2, out1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse2, lse1, rtol=1e-12, atol=1e-12)


def test_causal_ignores_future():
    pb = _rand_problem([16], 2, 8, seed=7, t5=(16, 32, False), causal=True)
    out0, lse0 = oracle.attn_fwd(pb)
    pb.k[10:] += 3.0
    pb.v[10:] -= 2.0
    out1, lse1 = oracle.attn_fwd(pb)
    np.testing.assert_array_equal(out1[:10], out0[:10])
    np.testing.assert_array_equal(lse1[:, :10], lse0[:, :10])
    assert not np.allclose(out1[10:], out0[10:])


def test_packed_equals_separate_documents():
    lens = [6, 0, 11, 3]
    pb = _rand_problem(lens, 2, 8, seed=8, t5=(8, 16, True), alibi=True)
    out, lse = oracle.attn_fwd(pb)
    cu = pb.cu_seqlens
    for i, L in enumerate(lens):
        if L == 0:
            continue
        s, e = cu[i], cu[i + 1]
        single = oracle.Problem(pb.q[s:e], pb.k[s:e], pb.v[s:e], np.array([0, L], np.int32),
                                table=pb.table, num_buckets=8, max_distance=16,
                                bidirectional=True, slopes=pb.slopes, scale=pb.scale)
        o1, l1 = oracle.attn_fwd(single)
        np.testing.assert_array_equal(out[s:e], o1)
        np.testing.assert_array_equal(lse[:, s:e], l1)


def test_rows_api_matches_full():
    pb = _rand_problem([30, 45], 3, 8, seed=9, t5=(16, 40, True), alibi=True, causal=True)
    out, lse = oracle.attn_fwd(pb)
    rng = np.random.default_rng(0)
    dout = rng.standard_normal(pb.shape)
    dq, dk, dv, dtab = oracle.attn_bwd(pb, dout)
    for doc in (0, 1):
        s = pb.cu_seqlens[doc]
        L = pb.cu_seqlens[doc + 1] - s
        rows = [0, 3, L - 1, L // 2]
        for h in range(3):
            o, l = oracle.attn_fwd_rows(pb, doc, h, rows)
            np.testing.assert_allclose(o, out[s + np.array(rows), h], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(l, lse[h, s + np.array(rows)], rtol=1e-13)
            gq, gk, gv, gcol = oracle.attn_bwd_rows(pb, dout, doc, h, rows, rows[::-1],
                                                    want_dtable=True)
            np.testing.assert_allclose(gq, dq[s + np.array(rows), h], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(gk, dk[s + np.array(rows[::-1]), h], rtol=1e-10,
                                       atol=1e-12)
            np.testing.assert_allclose(gv, dv[s + np.array(rows[::-1]), h], rtol=1e-10,
                                       atol=1e-12)
    # single-head, single-document bucket gradients add up to the full table gradient
    tot = np.zeros_like(dtab)
    for doc in (0, 1):
        for h in range(3):
            _, _, _, gcol = oracle.attn_bwd_rows(pb, dout, doc, h, [0], [0], want_dtable=True)
            tot[:, h] += gcol
    np.testing.assert_allclose(tot, dtab, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------------------------
# backward pins
# --------------------------------------------------------------------------------------------
def _loss(pb, dout):
    out, _ = oracle.attn_fwd(pb)
    return float(np.sum(out * dout))


@pytest.mark.parametrize("bidir,causal,alibi", [(True, False, False), (False, True, False),
                                                (True, True, True), (False, False, True)])
def test_backward_finite_differences(bidir, causal, alibi):
    pb = _rand_problem([9, 4], 2, 5, seed=10, t5=(8, 16, bidir), alibi=alibi, causal=causal,
                       scale=0.8)
    rng = np.random.default_rng(11)
    dout = rng.standard_normal(pb.shape)
    dq, dk, dv, dtab = oracle.attn_bwd(pb, dout)
    eps = 1e-6

    def fd(arr, idx):
        old = arr[idx]
        arr[idx] = old + eps
        lp = _loss(pb, dout)
        arr[idx] = old - eps
        lm = _loss(pb, dout)
        arr[idx] = old
        return (lp - lm) / (2 * eps)

    picks = [(0, 0, 0), (3, 1, 4), (8, 0, 2), (10, 1, 1), (12, 1, 3)]
    for name, arr, grad in (("q", pb.q, dq), ("k", pb.k, dk), ("v", pb.v, dv)):
        for idx in picks:
            want = fd(arr, idx)
            assert abs(grad[idx] - want) <= 1e-6 * max(1.0, abs(want)), (name, idx)
    for b in range(8):
        for h in range(2):
            want = fd(pb.table, (b, h))
            assert abs(dtab[b, h] - want) <= 1e-6 * max(1.0, abs(want)), ("table", b, h)


def test_backward_invariants():
    pb = _rand_problem([17, 1, 33], 3, 8, seed=12, t5=(16, 40, True), causal=True)
    rng = np.random.default_rng(13)
    dout = rng.standard_normal(pb.shape)
    dq, dk, dv, dtab = oracle.attn_bwd(pb, dout)
    # every row of dS sums to zero, so each head's bucket gradients sum to zero
    np.testing.assert_allclose(dtab.sum(axis=0), 0.0, atol=1e-11)
    # every row of P sums to one, so per document the dV rows add up to the dO rows
    cu = pb.cu_seqlens
    for i in range(3):
        s, e = cu[i], cu[i + 1]
        np.testing.assert_allclose(dv[s:e].sum(axis=0), dout[s:e].sum(axis=0), atol=1e-11)
    # shift invariance: dQ and dK have no component from a constant added to all logits, so the
    # gradient of the table along the all-ones direction (per head) is zero -- same as above


@pytest.mark.parametrize("cfg", [dict(t5=(8, 16, True), alibi=False, causal=False),
                                 dict(t5=(16, 24, False), alibi=True, causal=True)])
def test_backward_matches_torch_autograd(cfg):
    pb = _rand_problem([10, 3, 14], 2, 6, seed=14, scale=0.9, **cfg)
    rng = np.random.default_rng(15)
    dout = rng.standard_normal(pb.shape)
    dq, dk, dv, dtab = oracle.attn_bwd(pb, dout)
    q = torch.from_numpy(pb.q).requires_grad_()
    k = torch.from_numpy(pb.k).requires_grad_()
    v = torch.from_numpy(pb.v).requires_grad_()
    table = torch.from_numpy(pb.table).requires_grad_()
    slopes = torch.from_numpy(pb.slopes) if pb.slopes is not None else None
    loss = 0.0
    cu = pb.cu_seqlens
    for i in range(len(cu) - 1):
        s, e = int(cu[i]), int(cu[i + 1])
        L = e - s
        pos = torch.arange(L)
        rel = pos[None, :] - pos[:, None]
        bidx = torch.tensor([[exact_bucket(int(r), pb.num_buckets, pb.max_distance,
                                           pb.bidirectional) for r in row] for row in rel])
        for h in range(pb.shape[1]):
            mask = table[:, h][bidx]
            if slopes is not None:
                mask = mask - slopes[h] * rel.abs().double()
            if pb.causal:
                mask = mask.masked_fill(rel > 0, float("-inf"))
            o = torch.nn.functional.scaled_dot_product_attention(
                q[s:e, h][None], k[s:e, h][None], v[s:e, h][None], attn_mask=mask, scale=pb.scale)
            loss = loss + (o[0] * torch.from_numpy(dout[s:e, h])).sum()
    loss.backward()
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dtab, table.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_oracle_argument_errors():
    pb = _rand_problem([4], 1, 4, seed=16, t5=(7, 16, True))
    with pytest.raises(ValueError):
        oracle.attn_fwd(pb)  # odd bucket count with bidirectional buckets
    pb = _rand_problem([4], 1, 4, seed=16, t5=(8, 2, True))
    with pytest.raises(ValueError):
        oracle.attn_fwd(pb)  # max_distance inside the exact region


@pytest.mark.parametrize("causal,alibi", [(False, False), (True, True)])
def test_backward_with_bf16_output_statistic_identity(causal, alibi):
    """With D formed from the bf16-rounded output, the gradients differ from the exact ones by
    terms linear in delta = D_exact - D_rounded: dq by scale*delta*(P K), dk by
    scale*sum_q P delta Q, the table gradient by sum of P*delta per bucket; dv is unchanged."""
    pb = _rand_problem([11, 6], 2, 5, seed=40, t5=(8, 16, not causal), alibi=alibi,
                       causal=causal, scale=0.9)
    rng = np.random.default_rng(41)
    dout = rng.standard_normal(pb.shape)
    out, _ = oracle.attn_fwd(pb)
    dq0, dk0, dv0, dt0 = oracle.attn_bwd(pb, dout)
    pb.d_from_bf16_out = True
    dq1, dk1, dv1, dt1 = oracle.attn_bwd(pb, dout)
    pb.d_from_bf16_out = False
    out_b = torch.from_numpy(out).to(torch.bfloat16).double().numpy()
    delta = (dout * out).sum(-1) - (dout * out_b).sum(-1)  # [T, H]
    assert np.abs(delta).max() > 0
    np.testing.assert_array_equal(dv1, dv0)
    pk = oracle.Problem(pb.q, pb.k, pb.k, pb.cu_seqlens, table=pb.table,
                        num_buckets=pb.num_buckets, max_distance=pb.max_distance,
                        bidirectional=pb.bidirectional, slopes=pb.slopes, causal=causal,
                        scale=pb.scale)
    PK, _ = oracle.attn_fwd(pk)
    np.testing.assert_allclose(dq1 - dq0, pb.scale * delta[..., None] * PK, atol=1e-12)
    _, _, dv_w, _ = oracle.attn_bwd(pb, delta[..., None] * pb.q)
    np.testing.assert_allclose(dk1 - dk0, pb.scale * dv_w, atol=1e-12)
    want = np.zeros_like(dt0)
    cu = pb.cu_seqlens
    for i in range(len(cu) - 1):
        s, e = cu[i], cu[i + 1]
        L = e - s
        for h in range(pb.shape[1]):
            B = _bias_matrix(pb, L, h)
            S = pb.scale * pb.q[s:e, h] @ pb.k[s:e, h].T + B
            if causal:
                S = np.where(np.triu(np.ones((L, L), bool), 1), -np.inf, S)
            P = np.exp(S - S.max(1, keepdims=True))
            P /= P.sum(1, keepdims=True)
            for p in range(L):
                for r in range(L):
                    b = exact_bucket(r - p, pb.num_buckets, pb.max_distance, pb.bidirectional)
                    want[b, h] += P[p, r] * delta[s + p, h]
    np.testing.assert_allclose(dt1 - dt0, want, atol=1e-12)


@pytest.mark.parametrize("nb,md,bidir", BUCKET_CASES)
def test_vectorised_exact_bucket_matches_scalar_form(nb, md, bidir):
    from exact_buckets import exact_bucket_array
    deltas = np.arange(-3000, 3001)
    want = np.array([exact_bucket(int(x), nb, md, bidir) for x in deltas])
    np.testing.assert_array_equal(exact_bucket_array(deltas, nb, md, bidir), want)

"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on identical seeded
bf16 inputs. Small cases are compared element by element over every output; the full-size
benchmark workloads, run in the benchmark's launch configuration, are compared on sampled rows
the oracle computes one by one, plus invariants that hold at any size."""
import numpy as np
import pytest
import torch

import attention_relative_position_gb300 as fa
import oracle
from attention_relative_position_gb300 import workloads as wl
from gpu_common import (LSE_ATOL, assert_dbias, check, compare_grads, compare_grads_exact_d,
                        grad_bounds_full, grad_bounds_rows, grad_tol, operand_bounds,
                        operand_bounds_full, oracle_problem, run_gpu, run_gpu_bwd_exact_d)

pytestmark = pytest.mark.gpu

W = wl.Workload
SMALL = [
    wl.WORKLOADS[0],
    W("t5enc_varlen_ragged_d64", (200, 77, 1, 0, 384), 2, 64, 1.0, (32, 128, True), False, False,
      0.5, seed=11),
    W("t5dec_causal_varlen_d64", (130, 16, 1, 257, 2047), 3, 64, 1.0, (32, 128, False), False,
      True, 0.7, seed=12),
    W("alibi_causal_d128", (300, 129), 2, 128, 1.0, None, True, True, 128 ** -0.5, seed=13),
    W("t5_alibi_bidir_d128", (513,), 2, 128, 1.0, (32, 128, True), True, False, 0.3, seed=14),
    W("plain_d64", (128, 256), 2, 64, 1.0, None, False, False, 0.125, seed=15),
    W("plain_causal_d128", (257, 3), 2, 128, 1.0, None, False, True, 0.1, seed=16),
    W("t5enc_long_buckets_d64", (1000,), 1, 64, 0.5, (64, 1024, True), False, False, 1.0,
      seed=17),
    W("t5enc_long_buckets_d128", (900, 33), 1, 128, 0.5, (64, 1024, True), False, False, 0.5,
      seed=18),
    W("alibi_bidir_d64", (260,), 4, 64, 1.0, None, True, False, 0.125, seed=19),
    W("t5dec_alibi_causal_d64", (700, 45), 2, 64, 1.0, (32, 128, False), True, True, 0.25,
      seed=20),
    # many short documents: the persistent backward gives CTAs several items, switching heads,
    # skipping key tiles past short documents and an empty one
    W("t5enc_many_docs_d64", (300,) * 12 + (64,) * 6 + (0, 129), 4, 64, 1.0, (32, 128, True),
      False, False, 0.5, seed=22),
    W("t5dec_many_docs_causal_d64", (200,) * 16 + (1,) * 4 + (383,), 3, 64, 1.0,
      (32, 128, False), False, True, 0.5, seed=23),
    # documents of different lengths past the persistent backward's longest-first limits, so
    # that it falls back to the round-robin order: more (key tile, document) groups than the
    # sort takes, and (20000 items on one CTA per SM) more rounds per CTA than its list holds
    W("t5enc_many_tiny_docs_d64", tuple([1, 2, 17, 5, 30, 9, 3, 16] * 1100), 1, 64, 1.0,
      (32, 128, True), False, False, 0.3, seed=41),
    W("t5dec_many_short_docs_heads_d64", tuple([20, 3, 33, 9] * 625), 8, 64, 1.0,
      (32, 128, False), False, True, 0.3, seed=42),
    # bucket layouts with large lookup tables: at head_dim 128 the backward drops to two Q/dO
    # stages (4265 entries), at head_dim 64 the table nearly fills the backward's shared memory
    # (3031 of at most 3083 entries)
    W("t5_bidir_big_table_d128", (700, 300), 2, 128, 1.0, (32, 4096, True), False, False, 0.3,
      seed=43),
    W("t5_bidir_big_table_d64", (900, 200), 2, 64, 1.0, (32, 2600, True), False, False, 0.3,
      seed=44),
    # documents of at most 8 tokens: the forward takes the few-row kernel (rows = the
    # document's queries), the backward the tiled kernels
    W("tiny_docs_t5_alibi_causal_d64", (1, 3, 8, 2, 5, 0, 7, 8, 4), 4, 64, 1.0,
      (32, 128, False), True, True, 0.5, seed=24),
    W("tiny_docs_t5_bidir_d128", (6, 1, 8, 8, 3), 2, 128, 1.0, (32, 128, True), False, False,
      0.3, seed=25),
    # documents of equal length, no causal mask, grids of less than a wave: the forward's CTAs
    # are split along the keys (partial rows merged), the backward's along the query tiles (dK,
    # dV summed in fp32)
    W("t5enc_equal_docs_split_d128", (520,) * 3, 4, 128, 1.0, (32, 128, True), False, False,
      0.3, seed=26),
]


def _full_compare(w, x, res, case=None, gpu_fwd=None):
    """Every output of a small case against the oracle: the forward, the public backward (D
    from the bf16 output, with its propagated bound), and the same backward kernels run on the
    oracle's exact D (no slack). gpu_fwd: the forward's (out, lse) tensors on the device."""
    case = case or w.name
    pb = oracle_problem(w, x)
    ro, rl = oracle.attn_fwd(pb)
    check(case, "out", res["out"], ro, grad_tol(ro))
    check(case, "lse", res["lse"], rl, LSE_ATOL)
    dout = oracle.widen(wl.bf16_bits(x["dout"]))
    rq, rk, rv, rt = oracle.attn_bwd(pb, dout)
    dq_slack, dk_slack = grad_bounds_full(pb, dout, ro)
    exact = dict(dq=rq, dk=rk, dv=rv)
    ob = operand_bounds_full(pb, dout, ro, rl)
    compare_grads(case, res, exact, dq_slack, dk_slack, ob)
    if rt is not None:
        # held norm-wise to the backward defined on the stored bf16 output (D formed from it);
        # per-bucket error and the distance to the exact calculus are logged beside it
        bt = oracle.attn_bwd(oracle_problem(w, x, d_from_bf16_out=True), dout)[3]
        assert_dbias(res["dbias"], bt, case, mode="bf16-out", per_bucket=False)
        assert_dbias(res["dbias"], rt, case, mode="exact", enforce=False)
    if gpu_fwd is not None:
        d_exact = np.einsum("thc,thc->ht", dout, ro)  # D = rowsum(dout * out), exact
        ex = run_gpu_bwd_exact_d(w, x, gpu_fwd[0], gpu_fwd[1], d_exact)
        compare_grads_exact_d(case, ex, exact, ob)
        if rt is not None:
            assert_dbias(ex["dbias"], rt, case, mode="exact-D run")


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_cases_full(w):
    x = wl.make_inputs(w, device="cuda")
    res = run_gpu(w, x, keep_fwd=True)
    _full_compare(w, x, res, gpu_fwd=res.pop("fwd_tensors"))


def test_zero_table_equals_plain_attention():
    w = W("zero_table", (333,), 2, 64, 1.0, (32, 128, True), False, False, 0.125, seed=21)
    x = wl.make_inputs(w, device="cuda")
    x["table"].zero_()
    res = run_gpu(w, x)
    plain = w.with_(t5=None)
    xp = dict(x, table=None)
    res_p = run_gpu(plain, xp)
    np.testing.assert_array_equal(res["out"], res_p["out"])
    np.testing.assert_array_equal(res["lse"], res_p["lse"])
    _full_compare(w, x, res)


def test_max_seqlen_larger_than_needed():
    w = W("oversized_grid", (150, 40), 2, 64, 1.0, (32, 128, True), False, True, 0.5, seed=22)
    x = wl.make_inputs(w, device="cuda")
    res = run_gpu(w, x, max_seqlen=1000)
    _full_compare(w, x, res)


def test_repeat_calls_are_deterministic_except_dbias():
    w = SMALL[1]
    x = wl.make_inputs(w, device="cuda")
    a = run_gpu(w, x)
    b = run_gpu(w, x)
    for k in ("out", "lse", "dk", "dv"):
        np.testing.assert_array_equal(a[k], b[k])


def _sample_rows(L, n, rng):
    rows = {0, L - 1, L // 2, min(127, L - 1), min(128, L - 1)}
    rows |= set(int(r) for r in rng.integers(0, L, size=n))
    return sorted(rows)


@pytest.mark.parametrize("idx", [1, 2, 3, 4], ids=[wl.WORKLOADS[i].name for i in (1, 2, 3, 4)])
def test_full_size_workloads_sampled(idx):
    w = wl.WORKLOADS[idx]
    x = wl.make_inputs(w, device="cuda")
    res = run_gpu(w, x, keep_fwd=True)
    pb = oracle_problem(w, x)
    pb16 = oracle_problem(w, x, d_from_bf16_out=True)
    d_exact = np.full((w.num_heads, w.total_tokens), np.nan)  # NaN: keep the GPU's own D
    checks = []
    dout = wl.bf16_bits(x["dout"])
    dout64 = oracle.widen(dout)
    rng = np.random.default_rng(100 + idx)
    cu = x["cu_seqlens"].cpu().numpy()
    lens = np.diff(cu)
    docs = sorted({int(np.argmax(lens)), int(rng.integers(0, len(lens)))})
    heads = sorted({0, w.num_heads - 1})
    for doc in docs:
        s, L = int(cu[doc]), int(lens[doc])
        rows0 = _sample_rows(L, 6, rng)
        for h in heads:
            rows = rows0
            if L > 4096 and h > 0:
                # the last head of a long document: the first 2048 queries (the forward's split
                # last wave when the documents are equal and not causal) and the last 2048 keys
                # (the backward's)
                rows = sorted({int(v) for v in rng.integers(0, 2048, 3)} |
                              {int(v) for v in rng.integers(L - 2048, L, 3)})
            case = f"{w.name}[doc {doc}, head {h}]"
            r = s + np.array(rows)
            o, l = oracle.attn_fwd_rows(pb, doc, h, rows)
            check(case, "out", res["out"][r, h], o, grad_tol(o))
            check(case, "lse", res["lse"][h, r], l, LSE_ATOL)
            want_col = len(lens) == 1
            gq, gk, gv, gcol = oracle.attn_bwd_rows(pb, dout, doc, h, rows, rows,
                                                    want_dtable=want_col)
            sq, sk = grad_bounds_rows(pb, dout64, doc, h, rows, rows)
            got = dict(dq=res["dq"][r, h], dk=res["dk"][r, h], dv=res["dv"][r, h])
            exact = dict(dq=gq, dk=gk, dv=gv)
            o_all, l_all = oracle.attn_fwd_rows(pb, doc, h, list(range(L)))
            ob = operand_bounds(pb, dout64, doc, h, rows, rows, o_all, l_all)
            compare_grads(case, got, exact, sq, sk, ob)
            if gcol is not None:
                bcol = oracle.attn_bwd_rows(pb16, dout, doc, h, [0], [0], want_dtable=True)[3]
                assert_dbias(res["dbias"][:, h], bcol, case, mode="bf16-out", per_bucket=False)
                assert_dbias(res["dbias"][:, h], gcol, case, mode="exact", enforce=False)
            # the exact row statistic of this (document, head), for the exact-D run below
            d_exact[h, s:s + L] = (dout64[s:s + L, h] * o_all).sum(-1)
            checks.append((case, r, h, exact, gcol, ob))
    ex = run_gpu_bwd_exact_d(w, x, res["fwd_tensors"][0], res["fwd_tensors"][1], d_exact)
    for case, r, h, exact, gcol, ob in checks:
        got = dict(dq=ex["dq"][r, h], dk=ex["dk"][r, h], dv=ex["dv"][r, h])
        compare_grads_exact_d(case, got, exact, ob)
        if gcol is not None:
            assert_dbias(ex["dbias"][:, h], gcol, case, mode="exact-D run")
    # invariants at full size
    dvs = res["dv"].astype(np.float64)
    dos = x["dout"].float().cpu().numpy().astype(np.float64)
    for i in range(len(lens)):
        s, e = int(cu[i]), int(cu[i + 1])
        got = dvs[s:e].sum(axis=0)
        want = dos[s:e].sum(axis=0)
        # each row of P sums to one, so the dV rows of a document add up to its dO rows
        assert (np.abs(got - want) <= 1e-2 * np.abs(dvs[s:e]).sum(axis=0) + 1e-2).all(), i
    if res["dbias"] is not None:
        col_sum = res["dbias"].sum(axis=0)
        scale = np.abs(res["dbias"]).sum(axis=0) + 1e-6
        assert (np.abs(col_sum) <= 1e-2 * scale + 1e-3).all(), col_sum


def _table_gradient_over_documents(w, heads):
    """The packed batch's table gradient, column by column, is the sum of every document's
    contribution, each computed by the oracle from whole documents: the public path against the
    bf16-output oracle (norm-wise), the exact-D run against the exact oracle (norm-wise and per
    bucket)."""
    x = wl.make_inputs(w, device="cuda")
    res = run_gpu(w, x, keep_fwd=True)
    dout = wl.bf16_bits(x["dout"])
    dout64 = oracle.widen(dout)
    pb = oracle_problem(w, x)
    pb16 = oracle_problem(w, x, d_from_bf16_out=True)
    cu = x["cu_seqlens"].cpu().numpy()
    ndoc = len(cu) - 1
    d_exact = np.full((w.num_heads, w.total_tokens), np.nan)
    want = {}
    for h in heads:
        tot = np.zeros(w.t5[0])
        tot16 = np.zeros(w.t5[0])
        for doc in range(ndoc):
            s, L = int(cu[doc]), int(cu[doc + 1] - cu[doc])
            if L == 0:
                continue
            tot += oracle.attn_bwd_rows(pb, dout, doc, h, [0], [0], want_dtable=True)[3]
            tot16 += oracle.attn_bwd_rows(pb16, dout, doc, h, [0], [0], want_dtable=True)[3]
            o_all, _ = oracle.attn_fwd_rows(pb, doc, h, list(range(L)))
            d_exact[h, s:s + L] = (dout64[s:s + L, h] * o_all).sum(-1)
        case = f"{w.name}[all {ndoc} documents, head {h}]"
        assert_dbias(res["dbias"][:, h], tot16, case, mode="bf16-out", per_bucket=False)
        assert_dbias(res["dbias"][:, h], tot, case, mode="exact", enforce=False)
        want[h] = (case, tot)
    ex = run_gpu_bwd_exact_d(w, x, res["fwd_tensors"][0], res["fwd_tensors"][1], d_exact)
    for h, (case, tot) in want.items():
        assert_dbias(ex["dbias"][:, h], tot, case, mode="exact-D run")


def test_multi_doc_table_gradient_sums_over_documents():
    _table_gradient_over_documents(wl.WORKLOADS[1], heads=[3])


def test_varlen_causal_table_gradient_full_size():
    """The 46-document causal T5 decoder workload: its whole table gradient for two heads."""
    w = wl.WORKLOADS[2]
    _table_gradient_over_documents(w, heads=[0, w.num_heads - 1])


def test_split_last_wave_matches_whole_ctas():
    """The long T5 encoder workload (one 16K document, 12 heads, d 64: 768 forward CTAs and 1536
    backward key-tile CTAs on 152 SMs) with its last waves split, against the same problem run
    without the split (forward without a workspace; backward as its stage calls, which do not
    split), on every row: they agree up to the rounding of the merges."""
    w = wl.WORKLOADS[4]
    x = wl.make_inputs(w, device="cuda")
    kw = dict(bias_table=x["table"], num_buckets=w.t5[0], max_distance=w.t5[1],
              bidirectional=w.t5[2], causal=w.causal, softmax_scale=w.scale)
    T, H, d = x["q"].shape
    assert fa.fat_attn_fwd_workspace_size(T, 1, w.max_seqlen, H, d) > 0
    o1, l1 = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen,
                             workspace=False, **kw)
    o2, l2 = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, **kw)
    torch.cuda.synchronize()
    a, b = o1.float(), o2.float()
    # out: each key range's P is rounded to bf16 against its own running max before P V, so the
    # two schedules differ by bf16 roundings of P (relative 2^-9 each) besides the final rounding
    # of out: held to the parity regime's absolute bound (both are within it of the exact
    # result); a wrong row, head or range would differ by the size of out itself
    diff = (a - b).abs()
    assert (diff <= 2e-2 + 2 ** -8 * a.abs()).all(), float(diff.max())
    assert (l1 - l2).abs().max().item() <= 1e-5 * max(1.0, l1.abs().max().item())
    full = fa.fat_attn_bwd_workspace_size(T, H, d, 1, w.max_seqlen)
    assert full > fa.fat_attn_bwd_workspace_size(T, H, d)
    g1 = fa.fat_attn_bwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, o1, l1,
                         x["dout"], **kw)
    ws = torch.empty(full, dtype=torch.uint8, device="cuda")
    g2 = fa.fat_attn_bwd_stages(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, o1, l1,
                                x["dout"], ws, torch.empty_like(x["q"]), torch.empty_like(x["q"]),
                                torch.empty_like(x["q"]), dbias_table=torch.empty_like(x["table"]),
                                **kw)
    torch.cuda.synchronize()
    assert fa.fat_attn_get_device_error() == 0
    for name, u, v in zip(("dq", "dk", "dv"), g1[:3], g2[:3]):
        u, v = u.float(), v.float()
        # fp32 sums in another order, then one bf16 rounding
        err = (u - v).abs() - 2 ** -8 * v.abs()
        assert (err <= 1e-3 * v.abs().max()).all(), (name, err.max().item())
    torch.testing.assert_close(g1[3], g2[3], rtol=1e-4, atol=1e-3)


def test_split_schedules_fall_back_without_room():
    """Equal documents without a causal mask, grids of less than a wave: a forward workspace
    smaller than fat_attn_fwd_workspace_size runs the one-launch schedule (bit-identical to no
    workspace), and a backward given only the minimum workspace does not split either (dK, dV
    bit-identical to the stage calls, which never split)."""
    w = wl.Workload("equal_docs_fallback_d128", (520,) * 3, 4, 128, 1.0, (32, 128, True), False,
                    False, 0.3, seed=27)
    x = wl.make_inputs(w, device="cuda")
    kw = dict(bias_table=x["table"], num_buckets=32, max_distance=128, bidirectional=True,
              causal=False, softmax_scale=w.scale)
    T, H, d = x["q"].shape
    need = fa.fat_attn_fwd_workspace_size(T, 3, w.max_seqlen, H, d)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    o1, l1 = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen,
                             workspace=False, **kw)
    o2, l2 = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen,
                             workspace=small, **kw)
    o3, l3 = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert ((o1.float() - o3.float()).abs() <= 2e-2 + 2 ** -8 * o1.float().abs()).all()
    minimum = fa.fat_attn_bwd_workspace_size(T, H, d)
    assert fa.fat_attn_bwd_workspace_size(T, H, d, 3, w.max_seqlen) > minimum
    ws = torch.empty(minimum, dtype=torch.uint8, device="cuda")
    g1 = fa.fat_attn_bwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, o1, l1, x["dout"],
                         workspace=ws, **kw)
    g2 = fa.fat_attn_bwd_stages(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, o1, l1,
                                x["dout"], torch.empty_like(ws), torch.empty_like(x["q"]),
                                torch.empty_like(x["q"]), torch.empty_like(x["q"]),
                                dbias_table=torch.empty_like(x["table"]), **kw)
    torch.cuda.synchronize()
    assert fa.fat_attn_get_device_error() == 0
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    torch.testing.assert_close(g1[0].float(), g2[0].float(), rtol=2 ** -7, atol=1e-3)

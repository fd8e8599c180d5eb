"""GPU: the persistent one-tile forward (head_dim 64, documents of at most 2048 rows) against the
grid of one-tile CTAs that runs when there are fewer blocks (the same arithmetic per row, so the
results are bit-identical; both paths forced through the debug flags)
and, on a varlen causal T5 case walked longest-first, against the fp64 oracle. The cases cover
both work orders (sorted for documents of different lengths, round-robin for equal ones or when
the sort's limits are exceeded), head changes between items, rows without keys, grouped heads
and every bias form."""
import numpy as np
import pytest
import torch

import attention_relative_position_gb300 as fa
import oracle
from attention_relative_position_gb300 import workloads as wl
from gpu_common import ATOL, check, oracle_problem

pytestmark = pytest.mark.gpu

W = wl.Workload
SELF_CASES = [
    # documents of different lengths, causal, unidirectional T5: the longest-first order
    W("pers_varlen_causal_t5", tuple(wl.lognormal_lengths(6000, 5.8, 0.8, 16, 2048, seed=81)),
      6, 64, 1.0, (32, 128, False), False, True, 1.0, seed=81),
    # equal documents, bidirectional T5 + ALiBi, no mask: the round-robin order
    W("pers_equal_t5_alibi", (640,) * 6, 4, 64, 0.5, (32, 128, True), True, False, 0.4, seed=82),
    # one document, ALiBi causal, ragged last block
    W("pers_one_doc_alibi_causal", (1999,), 8, 64, 1.0, None, True, True, 0.125, seed=83),
    # many tiny documents, no bias: more groups than the sort takes (round-robin order)
    W("pers_many_tiny_nobias", tuple([1, 2, 17, 5, 30, 9, 3, 16] * 1100), 1, 64, 1.0, None,
      False, False, 0.3, seed=84),
    # many short documents and heads: more rounds per CTA than the sorted list holds
    W("pers_many_short_heads", tuple([40, 3, 70, 21] * 625), 16, 64, 1.0, (32, 128, True),
      False, True, 0.3, seed=85),
]
X = wl.XWorkload
X_CASES = [
    # more queries than keys, causal: the first rows see no key (items without key tiles)
    X("pers_x_fewer_keys_causal_gqa", (300, 200, 1000), (100, 250, 64), 8, 2, 64, 1.0,
      (32, 128, False), False, True, 0.5, seed=86),
    # cross-attention without bias, empty documents on either side
    X("pers_x_cross_empty", (100, 0, 257, 700), (300, 40, 0, 129), 4, 4, 64, 0.7, seed=87),
]


def _self_fwd(w, x, flags):
    t5 = w.t5 or (0, 0, True)
    fa.fat_attn_debug_set_watchdog(0, flags)
    try:
        out, lse = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen,
                                   bias_table=x["table"], num_buckets=t5[0],
                                   max_distance=t5[1], bidirectional=t5[2],
                                   alibi_slopes=x["slopes"], causal=w.causal,
                                   softmax_scale=w.scale)
        torch.cuda.synchronize()
    finally:
        fa.fat_attn_debug_set_watchdog(0, 0)
    assert fa.fat_attn_get_device_error() == 0
    return out, lse


def _x_fwd(w, x, flags):
    t5 = w.t5 or (0, 0, True)
    fa.fat_attn_debug_set_watchdog(0, flags)
    try:
        out, lse = fa.fat_xattn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"],
                                    w.max_seqlen_q, w.max_seqlen_k, bias_table=x["table"],
                                    num_buckets=t5[0], max_distance=t5[1],
                                    bidirectional=t5[2], alibi_slopes=x["slopes"],
                                    causal=w.causal, softmax_scale=w.scale)
        torch.cuda.synchronize()
    finally:
        fa.fat_attn_debug_set_watchdog(0, 0)
    assert fa.fat_attn_get_device_error() == 0
    return out, lse


def _same(a, b):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def _same_lse(a, b):
    fa_, fb_ = torch.isfinite(a), torch.isfinite(b)
    assert torch.equal(fa_, fb_)
    assert torch.equal(a[fa_], b[fb_])
    assert torch.equal(a[~fa_], b[~fb_])  # -inf rows (no key) on both sides


@pytest.mark.parametrize("w", SELF_CASES, ids=lambda w: w.name)
def test_persistent_forward_matches_one_tile_grid(w):
    x = wl.make_inputs(w, device="cuda", with_dout=False)
    out_p, lse_p = _self_fwd(w, x, 8)  # persistent CTAs
    out_g, lse_g = _self_fwd(w, x, 4)  # the grid of one-tile CTAs
    _same(out_p, out_g)
    _same_lse(lse_p, lse_g)


@pytest.mark.parametrize("w", X_CASES, ids=lambda w: w.name)
def test_persistent_xattn_forward_matches_one_tile_grid(w):
    x = wl.make_xinputs(w, device="cuda")
    out_p, lse_p = _x_fwd(w, x, 8)
    out_g, lse_g = _x_fwd(w, x, 4)
    _same(out_p, out_g)
    _same_lse(lse_p, lse_g)


def test_persistent_forward_against_oracle():
    # a smaller varlen causal T5 case than the ones above, walked longest-first
    w = W("pers_oracle_varlen", (700, 33, 129, 1, 256, 400, 64), 3, 64, 1.0, (32, 128, False),
          False, True, 1.0, seed=88)
    x = wl.make_inputs(w, device="cuda", with_dout=False)
    out, lse = _self_fwd(w, x, 8)
    ro, rl = oracle.attn_fwd(oracle_problem(w, x))
    check(w.name, "out", out.float().cpu().numpy(), ro, ATOL)
    got = lse.float().cpu().numpy()
    assert np.max(np.abs(got - rl)) <= 1e-3


def test_persistent_forward_watchdog():
    # the producer issues no copies: every consumer wait runs out, the kernel records the
    # forward timeout and exits; the context stays usable
    w = W("pers_watchdog", (300, 40, 129), 2, 64, 1.0, (32, 128, True), False, False, 0.5,
          seed=89)
    x = wl.make_inputs(w, device="cuda", with_dout=False)
    assert fa.fat_attn_get_device_error() == 0
    fa.fat_attn_debug_set_watchdog(50_000_000, 1 | 8)
    try:
        fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen,
                        bias_table=x["table"], num_buckets=32, max_distance=128,
                        bidirectional=True, softmax_scale=w.scale)
        torch.cuda.synchronize()
        bits = fa.fat_attn_get_device_error()
    finally:
        fa.fat_attn_debug_set_watchdog(0, 0)
    assert bits == fa.FAT_DEVERR_TIMEOUT_FWD
    out, lse = _self_fwd(w, x, 8)
    ro, rl = oracle.attn_fwd(oracle_problem(w, x))
    check(w.name, "out", out.float().cpu().numpy(), ro, ATOL)

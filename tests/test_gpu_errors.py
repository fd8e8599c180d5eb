"""GPU checks of the device-side bucket mapping and of failure handling without faulting the GPU:
the watchdog makes a pipeline wait run out (the producer issues nothing), the kernel records a
status bit and exits, and the context stays usable; corrupt cu_seqlens are reported, not read
out of bounds."""
import numpy as np
import pytest
import torch

import attention_relative_position_gb300 as fa
import oracle
from attention_relative_position_gb300 import workloads as wl
from exact_buckets import exact_bucket_array
from gpu_common import ATOL, check, oracle_problem, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nb,md,bidir", [(32, 128, True), (32, 128, False), (64, 1024, True),
                                         (64, 1024, False), (128, 4096, True), (8, 16, False)])
def test_device_bucket_ids_bit_exact(nb, md, bidir):
    """Every one of the 131 073 deltas in [-65536, 65536]: the device's bucket id equals the
    exact integer-root threshold form."""
    lo, n = -65536, 131073
    got = fa.fat_attn_debug_buckets(lo, n, nb, md, bidir).cpu().numpy().astype(np.int64)
    want = exact_bucket_array(np.arange(lo, lo + n), nb, md, bidir)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(lo + int(i), int(got[i]), int(want[i])) for i in bad[:10]]
    # and the oracle agrees on a stride plus the whole near region
    for i in np.concatenate([np.arange(0, n, 509), np.arange(65536 - 300, 65536 + 301)]):
        assert oracle.t5_bucket(lo + int(i), nb, md, bidir) == want[i]


def test_watchdog_timeout_sets_status_and_context_survives():
    w = wl.Workload("watchdog", (300,), 2, 64, 1.0, (32, 128, True), False, False, 0.5, seed=31)
    x = wl.make_inputs(w, device="cuda")
    assert fa.fat_attn_get_device_error() == 0
    try:
        fa.fat_attn_debug_set_watchdog(50_000_000, 1)  # 50 ms, producer issues no copies
        fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen,
                        bias_table=x["table"], num_buckets=32, max_distance=128,
                        bidirectional=True, softmax_scale=w.scale)
        torch.cuda.synchronize()
        bits = fa.fat_attn_get_device_error()
    finally:
        fa.fat_attn_debug_set_watchdog(0, 0)
    assert bits == fa.FAT_DEVERR_TIMEOUT_FWD
    assert fa.fat_attn_get_device_error() == 0  # cleared by the read
    # the context is still usable and results are right
    res = run_gpu(w, x, with_bwd=False)
    ro, rl = oracle.attn_fwd(oracle_problem(w, x))
    check("watchdog_recovered", "out", res["out"], ro, ATOL)


def test_backward_watchdog_timeout():
    w = wl.Workload("watchdog_bwd", (200,), 1, 128, 1.0, None, True, True, 0.1, seed=32)
    x = wl.make_inputs(w, device="cuda")
    out, lse = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen,
                               alibi_slopes=x["slopes"], causal=True, softmax_scale=w.scale)
    try:
        fa.fat_attn_debug_set_watchdog(50_000_000, 2)
        fa.fat_attn_bwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, out, lse,
                        x["dout"], alibi_slopes=x["slopes"], causal=True, softmax_scale=w.scale)
        torch.cuda.synchronize()
        bits = fa.fat_attn_get_device_error()
    finally:
        fa.fat_attn_debug_set_watchdog(0, 0)
    assert bits == fa.FAT_DEVERR_TIMEOUT_BWD


def test_corrupt_cu_seqlens_reported():
    w = wl.Workload("bad_cu", (100, 50), 2, 64, 1.0, None, False, False, 0.5, seed=33)
    x = wl.make_inputs(w, device="cuda")
    cu = torch.tensor([0, 400, 150], dtype=torch.int32, device="cuda")  # 400 > total tokens
    fa.fat_attn_fwd(x["q"], x["k"], x["v"], cu, 256, softmax_scale=0.5)
    torch.cuda.synchronize()
    assert fa.fat_attn_get_device_error() & fa.FAT_DEVERR_SEQLENS


def test_document_longer_than_max_seqlen_reported():
    """max_seqlen sizes the grids; a document longer than it is reported by the forward and by
    both backward launch shapes (status bit, no fault)."""
    for d, H in ((64, 2), (128, 1)):
        w = wl.Workload(f"long_doc_d{d}", (100, 700), H, d, 1.0, (32, 128, True), False, False,
                        0.5, seed=34)
        x = wl.make_inputs(w, device="cuda")
        kw = dict(bias_table=x["table"], num_buckets=32, max_distance=128, bidirectional=True,
                  softmax_scale=w.scale)
        out, lse = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], 300, **kw)
        torch.cuda.synchronize()
        assert fa.fat_attn_get_device_error() & fa.FAT_DEVERR_SEQLENS
        fa.fat_attn_bwd(x["q"], x["k"], x["v"], x["cu_seqlens"], 300, out, lse, x["dout"], **kw)
        torch.cuda.synchronize()
        assert fa.fat_attn_get_device_error() & fa.FAT_DEVERR_SEQLENS
        # the same call with a correct bound reports nothing
        run_gpu(w, x)

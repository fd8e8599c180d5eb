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
from gpu_common import assert_close, oracle_problem, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nb,md,bidir", [(32, 128, True), (32, 128, False), (64, 1024, True),
                                         (64, 1024, False), (128, 4096, True), (8, 16, False)])
def test_device_bucket_ids_bit_exact(nb, md, bidir):
    lo, n = -65536, 131073
    got = fa.fat_attn_debug_buckets(lo, n, nb, md, bidir).cpu().numpy()
    # every distinct value is checked near the origin, a stride beyond
    idx = np.concatenate([np.arange(0, n, 97), np.arange(65536 - 5000, 65536 + 5001)])
    for i in np.unique(idx):
        assert got[i] == oracle.t5_bucket(lo + int(i), nb, md, bidir), lo + int(i)


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
    assert_close("out", res["out"], ro)


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

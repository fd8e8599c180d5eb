"""The allocation-free backward (fat_attn_bwd_noalloc): for callers that cannot allocate device
memory it runs the backward on a scratch array the library keeps on each GPU. Its results must
match the ordinary entry point (fat_attn_bwd with a caller workspace) on two calls in a row, the
second call reusing the scratch the first one left behind. This file sorts last so that a run
that stops at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import attention_relative_position_gb300 as fa
from attention_relative_position_gb300 import workloads as wl
from gpu_common import ATOL, RTOL, t5_args

CASES = [
    wl.Workload("noalloc_t5enc_varlen_d64", (300, 77, 1, 512), 2, 64, 1.0, (32, 128, True),
                False, False, 0.5, seed=51),
    wl.Workload("noalloc_alibi_causal_d128", (257, 130), 2, 128, 1.0, None, True, True,
                128 ** -0.5, seed=52),
    wl.Workload("noalloc_t5dec_causal_d64", (129, 640), 3, 64, 1.0, (32, 128, False), False,
                True, 0.7, seed=53),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_noalloc_matches_workspace_backward(w):
    x = wl.make_inputs(w, device="cuda")
    a = t5_args(w)
    kw = dict(bias_table=x["table"], alibi_slopes=x["slopes"], causal=w.causal,
              softmax_scale=w.scale, num_buckets=a["num_buckets"],
              max_distance=a["max_distance"], bidirectional=a["bidirectional"])
    out, lse = fa.fat_attn_fwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, **kw)
    ref = fa.fat_attn_bwd(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, out, lse,
                          x["dout"], **kw)
    torch.cuda.synchronize()
    ref = [t.float().cpu().numpy() if t is not None else None for t in ref]
    for call in range(2):
        dq, dk, dv = (torch.full_like(x["q"], float("nan")) for _ in range(3))
        dtab = torch.full_like(x["table"], float("nan")) if x["table"] is not None else None
        fa.fat_attn_bwd_noalloc(x["q"], x["k"], x["v"], x["cu_seqlens"], w.max_seqlen, out, lse,
                                x["dout"], dq, dk, dv, dbias_table=dtab, **kw)
        torch.cuda.synchronize()
        assert fa.fat_attn_get_device_error() == 0
        got = [t.float().cpu().numpy() if t is not None else None for t in (dq, dk, dv, dtab)]
        for name, g, r in zip(("dq", "dk", "dv", "dbias"), got, ref):
            if r is None:
                assert g is None
                continue
            assert np.isfinite(g).all(), (call, name)
            err = np.abs(g - r)
            assert (err <= ATOL + RTOL * np.abs(r)).all(), (call, name, float(err.max()))


def test_noalloc_rejects_problems_beyond_the_scratch():
    lib = fa.load()
    T, H, d = 1 << 20, 8, 64  # needs far more than the built-in scratch
    sh = fa._Shape(T, 1, T, H, d, None)
    assert lib.fat_attn_bwd_workspace_size(ctypes.byref(sh)) > (32 << 20)
    fake = 1 << 20
    rc = lib.fat_attn_bwd_noalloc(ctypes.byref(sh), fake, fake, fake, None, 0, 0, 1, None, fake,
                                  0, 1.0, fake, fake, fake, fake, fake, fake, None)
    assert rc == -5
    assert b"scratch" in lib.fat_attn_last_error_message()

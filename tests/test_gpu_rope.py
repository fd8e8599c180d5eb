"""GPU parity of the rotary position embedding (RoPE): the rotation kernel against the oracle's
RoFormer rotation (rounded to bf16 the same way), and RoPE attention end to end (rotate Q and K,
attention forward and backward on the rotated tensors, dQ and dK turned back) against the
oracle's RoPE attention."""
import numpy as np
import pytest
import torch

import attention_relative_position_gb300 as fa
import oracle
from attention_relative_position_gb300 import workloads as wl
from gpu_common import (LSE_ATOL, check, grad_bounds_full, grad_tol, operand_bounds_full,
                        run_gpu)

pytestmark = pytest.mark.gpu


def _bf16(a):
    """fp64 -> the bf16 value (round to nearest even), as fp64."""
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("d,base", [(64, 10000.0), (128, 10000.0), (64, 500.0)])
def test_rotation_matches_oracle(d, base):
    w = wl.Workload(f"rope_rot_d{d}", (1, 300, 16384 - 301), 3, d, 1.0, seed=81)
    x = wl.make_inputs(w, device="cuda")
    cu = x["cu_seqlens"]
    pos = oracle.doc_positions(cu.cpu().numpy())
    for name in ("q", "k"):
        got = fa.fat_rope_apply(x[name], cu, w.max_seqlen, base=base).double().cpu().numpy()
        want = _bf16(oracle.rope_rotate_at(wl.bf16_bits(x[name]), pos, base))
        diff = np.abs(got - want)
        # the same bf16 value nearly everywhere; never more than one bf16 ulp apart
        ulp = 2 * np.exp2(np.floor(np.log2(np.maximum(np.abs(want), 2.0 ** -126))) - 8)
        assert (diff <= ulp + 1e-30).all(), float((diff / ulp).max())
        assert (diff == 0).mean() > 0.999, (diff == 0).mean()
        check(w.name, name + "_rot", got, want, 2 * ulp, mode="bf16(oracle)")
        # position 0 of every document is left as it is
        zero = np.asarray(cu.cpu().numpy()[:-1])
        np.testing.assert_array_equal(got[zero], oracle.widen(wl.bf16_bits(x[name]))[zero])
    # inverse turns back, in place
    y = fa.fat_rope_apply(x["q"], cu, w.max_seqlen, base=base)
    fa.fat_rope_apply(y, cu, w.max_seqlen, base=base, inverse=True, out=y)
    back = y.double().cpu().numpy()
    assert np.abs(back - oracle.widen(wl.bf16_bits(x["q"]))).max() <= 2 ** -6 * 4
    torch.cuda.synchronize()
    assert fa.fat_attn_get_device_error() == 0


CASES = [
    wl.Workload("rope_causal_varlen_d64", (300, 129, 1, 700), 2, 64, 1.0, None, False, True,
                0.125, seed=82),
    wl.Workload("rope_bidir_d128", (513, 77), 2, 128, 1.0, None, False, False, 128 ** -0.5,
                seed=83),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_rope_attention_end_to_end(w):
    base = 10000.0
    x = wl.make_inputs(w, device="cuda")
    cu = x["cu_seqlens"]
    qr = fa.fat_rope_apply(x["q"], cu, w.max_seqlen, base=base)
    kr = fa.fat_rope_apply(x["k"], cu, w.max_seqlen, base=base)
    xr = dict(x, q=qr, k=kr)
    res = run_gpu(w, xr)
    dq = fa.fat_rope_apply(torch.from_numpy(res["dq"]).to(torch.bfloat16).cuda(), cu, w.max_seqlen,
                           base=base, inverse=True).double().cpu().numpy()
    dk = fa.fat_rope_apply(torch.from_numpy(res["dk"]).to(torch.bfloat16).cuda(), cu, w.max_seqlen,
                           base=base, inverse=True).double().cpu().numpy()
    pb = oracle.Problem(wl.bf16_bits(x["q"]), wl.bf16_bits(x["k"]), wl.bf16_bits(x["v"]),
                        cu.cpu().numpy(), causal=w.causal, scale=w.scale)
    ro, rl = oracle.rope_attn_fwd(pb, base)
    check(w.name, "out", res["out"], ro, grad_tol(ro))
    check(w.name, "lse", res["lse"], rl, LSE_ATOL)
    dout = oracle.widen(wl.bf16_bits(x["dout"]))
    rq, rk, rv, _ = oracle.rope_attn_bwd(pb, dout, base)
    # bounds on the rotated problem the kernels ran (bf16 operands, D from the bf16 output;
    # see gpu_common), plus the bf16 rounding of the rotated gradients before they turn back
    pos = oracle.doc_positions(cu.cpu().numpy())
    prot = oracle.Problem(_bf16(oracle.rope_rotate_at(pb.q, pos, base)),
                          _bf16(oracle.rope_rotate_at(pb.k, pos, base)), pb.v, pb.cu_seqlens,
                          causal=w.causal, scale=w.scale)
    ro2, rl2 = oracle.attn_fwd(prot)
    sq, sk = grad_bounds_full(prot, dout, ro2)
    ob = operand_bounds_full(prot, dout, ro2, rl2)
    rq2, rk2, _, _ = oracle.attn_bwd(prot, dout)
    rnd_q = 2 ** -8 * np.abs(rq2).max(-1, keepdims=True)  # one bf16 rounding, any channel
    rnd_k = 2 ** -8 * np.abs(rk2).max(-1, keepdims=True)
    check(w.name, "dv", res["dv"], rv, grad_tol(rv, ob["dv"]), mode="exact+op")
    check(w.name, "dq", dq, rq, grad_tol(rq, sq + ob["dq"] + rnd_q), mode="exact+D+op")
    check(w.name, "dk", dk, rk, grad_tol(rk, sk + ob["dk"] + rnd_k), mode="exact+D+op")

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
        xin = oracle.widen(wl.bf16_bits(x[name]))
        exact = oracle.rope_rotate_at(xin, pos, base)
        want = _bf16(exact)
        diff = np.abs(got - want)
        # fp32 rotation: error ~1e-7 of the pair's norm (where the rotated value cancels to near
        # zero that is many of its own ulps), then one bf16 rounding: within one bf16 ulp of the
        # exact rotation plus that fp32 error, and the same bf16 value nearly everywhere
        norm = np.sqrt(xin[..., 0::2] ** 2 + xin[..., 1::2] ** 2).repeat(2, axis=-1)
        ulp = 2 * np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 2.0 ** -126))) - 8)
        check(w.name, name + "_rot", got, exact, ulp + 1e-6 * norm, mode="exact rotation")
        assert (diff == 0).mean() > 0.99, (diff == 0).mean()
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
    # The attention kernels take bf16 inputs, so the rotated Q and K are stored in bf16: the
    # expected values are the oracle's attention on its own rotation rounded to bf16 (the
    # rotation itself is checked above), with the oracle's unrounded RoPE attention logged.
    pos = oracle.doc_positions(cu.cpu().numpy())
    prot = oracle.Problem(_bf16(oracle.rope_rotate_at(pb.q, pos, base)),
                          _bf16(oracle.rope_rotate_at(pb.k, pos, base)), pb.v, pb.cu_seqlens,
                          causal=w.causal, scale=w.scale)
    ro2, rl2 = oracle.attn_fwd(prot)
    check(w.name, "out", res["out"], ro2, grad_tol(ro2), mode="bf16 rotation")
    check(w.name, "lse", res["lse"], rl2, LSE_ATOL, mode="bf16 rotation")
    ro, rl = oracle.rope_attn_fwd(pb, base)
    check(w.name, "out", res["out"], ro, grad_tol(ro), mode="exact rotation", enforce=False)
    check(w.name, "lse", res["lse"], rl, LSE_ATOL, mode="exact rotation", enforce=False)
    dout = oracle.widen(wl.bf16_bits(x["dout"]))
    # gradients of the unrotated inputs: the rotated problem's, turned back in fp64; bounds of
    # the bf16 operands and of D from the bf16 output (see gpu_common), plus the bf16 rounding
    # of the rotated gradients before they turn back
    rq2, rk2, rv2, _ = oracle.attn_bwd(prot, dout)
    rq = oracle.rope_rotate_at(rq2, pos, base, inverse=True)
    rk = oracle.rope_rotate_at(rk2, pos, base, inverse=True)
    sq, sk = grad_bounds_full(prot, dout, ro2)
    ob = operand_bounds_full(prot, dout, ro2, rl2)
    rnd_q = 2 ** -8 * np.abs(rq2).max(-1, keepdims=True)  # one bf16 rounding, any channel
    rnd_k = 2 ** -8 * np.abs(rk2).max(-1, keepdims=True)
    check(w.name, "dv", res["dv"], rv2, grad_tol(rv2, ob["dv"]), mode="exact+op")
    check(w.name, "dq", dq, rq, grad_tol(rq, sq + ob["dq"] + rnd_q), mode="exact+D+op")
    check(w.name, "dk", dk, rk, grad_tol(rk, sk + ob["dk"] + rnd_k), mode="exact+D+op")
    eq, ek, ev, _ = oracle.rope_attn_bwd(pb, dout, base)  # the unrounded definition, logged
    check(w.name, "dq", dq, eq, grad_tol(eq, sq + ob["dq"] + rnd_q), mode="exact rotation",
          enforce=False)

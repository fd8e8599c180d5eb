"""GPU parity of RMSNorm and of the cross-entropy with z-loss against their fp64 oracle on the
same seeded bf16 inputs."""
import numpy as np
import pytest
import torch

import attention_relative_position_gb300 as fa
from attention_relative_position_gb300 import workloads as wl
from gpu_common import check, grad_tol
from oracle import norm_ce as nc

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,dim", [(1000, 256), (3001, 768), (4096, 1024), (517, 2048),
                                      (1, 512)])
def test_rmsnorm_forward_backward(rows, dim):
    x, w, dy = wl.make_norm_inputs(rows, dim, seed=90 + dim, device="cuda")
    eps = 1e-6
    y, rstd = fa.fat_rmsnorm_fwd(x, w, eps)
    dx, dw = fa.fat_rmsnorm_bwd(x, w, rstd, dy)
    torch.cuda.synchronize()
    case = f"rmsnorm_{rows}x{dim}"
    ry, rr = nc.rmsnorm_fwd(wl.bf16_bits(x), w.cpu().numpy(), eps)
    rdx, rdw = nc.rmsnorm_bwd(wl.bf16_bits(x), w.cpu().numpy(), wl.bf16_bits(dy), eps)
    check(case, "y", y.double().cpu().numpy(), ry, grad_tol(ry))
    check(case, "rstd", rstd.double().cpu().numpy(), rr, 1e-5 * np.abs(rr))
    check(case, "dx", dx.double().cpu().numpy(), rdx, grad_tol(rdx))
    # dw sums rows of fp32 products: relative to the sum of the terms' magnitudes
    xs, dys = x.double().cpu().numpy(), dy.double().cpu().numpy()
    terms = np.abs(dys * xs * rr[:, None]).sum(0)
    check(case, "dw", dw.double().cpu().numpy(), rdw, 1e-5 * terms + 1e-6)


@pytest.mark.parametrize("rows,vocab,z_loss", [(256, 32768, 1e-4), (1000, 1000, 0.0),
                                               (64, 50000, 1e-3), (3, 8, 0.5)])
def test_cross_entropy(rows, vocab, z_loss):
    z, t = wl.make_ce_inputs(rows, vocab, seed=95 + rows, device="cuda")
    valid = int((t >= 0).sum())
    scale = 1.0 / max(valid, 1)
    loss, lse, dz = fa.fat_cross_entropy(z, t, z_loss=z_loss, grad_scale=scale)
    torch.cuda.synchronize()
    assert fa.fat_attn_get_device_error() == 0
    case = f"ce_{rows}x{vocab}"
    tn = t.cpu().numpy()
    rl, rlse = nc.cross_entropy_fwd(wl.bf16_bits(z), tn, z_loss)
    rdz = nc.cross_entropy_bwd(wl.bf16_bits(z), tn, z_loss, scale)
    check(case, "lse", lse.double().cpu().numpy(), rlse, 2e-5 * np.maximum(1, np.abs(rlse)))
    check(case, "loss", loss.double().cpu().numpy(), rl, 2e-5 * np.maximum(1, np.abs(rlse)))
    assert (loss.cpu().numpy()[tn < 0] == 0).all()
    # one bf16 ulp of each gradient element (the fp32 value may land on either side of a
    # rounding midpoint: up to 2^-7 |ref|), plus the fp32 exponentials and sum
    check(case, "dlogits", dz.double().cpu().numpy(), rdz, 2 ** -7 * np.abs(rdz) + 1e-6 * scale)
    assert (dz.float().cpu().numpy()[tn < 0] == 0).all()
    # forward only: the same loss without a gradient buffer
    loss2, _, none = fa.fat_cross_entropy(z, t, z_loss=z_loss, want_grad=False)
    assert none is None
    torch.testing.assert_close(loss2, loss, rtol=0, atol=0)


def test_cross_entropy_target_out_of_range_reported():
    z, t = wl.make_ce_inputs(4, 64, seed=99, device="cuda")
    t[1] = 64
    loss, _, _ = fa.fat_cross_entropy(z, t)
    torch.cuda.synchronize()
    assert fa.fat_attn_get_device_error() & fa.FAT_DEVERR_INDEX
    assert loss[1].item() == 0.0

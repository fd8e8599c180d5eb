"""Pins for the RMSNorm and cross-entropy (+ z-loss) oracle (no GPU).

Closed forms (a constant row, uniform logits, a dominant logit), invariances (scale invariance of
RMSNorm without eps, the gradient rows' sums), library routines in fp64 (torch's rms_norm and
cross_entropy, logsumexp, autograd through them) and central finite differences. Each is chosen so
that a plausible slip (a mean where a sum belongs, a dropped eps or weight, the z-loss factor 2, a
wrong sign on the target term, ignored rows leaking) fails at least one of them.
"""
import numpy as np
import pytest
import torch

from oracle import norm_ce as nc


def _rng(seed):
    return np.random.default_rng(seed)


# ---- RMSNorm -------------------------------------------------------------------------------
def test_rmsnorm_constant_row_closed_form():
    # x = c * ones: mean of squares c^2, so y = w * c / sqrt(c^2 + eps)
    D, c, eps = 16, -1.5, 1e-6
    w = np.linspace(0.5, 2.0, D)
    y, rstd = nc.rmsnorm_fwd(np.full((1, D), c), w, eps)
    np.testing.assert_allclose(rstd[0], 1.0 / np.sqrt(c * c + eps), rtol=1e-15)
    np.testing.assert_allclose(y[0], w * c / np.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_scale_invariance_and_unit_rms():
    x = _rng(1).standard_normal((5, 64))
    w = np.ones(64)
    y1, _ = nc.rmsnorm_fwd(x, w, 0.0)
    y2, _ = nc.rmsnorm_fwd(37.0 * x, w, 0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-13)
    np.testing.assert_allclose((y1 ** 2).mean(-1), 1.0, rtol=1e-13)


def test_rmsnorm_matches_torch():
    x = _rng(2).standard_normal((7, 96))
    w = _rng(3).standard_normal(96)
    y, _ = nc.rmsnorm_fwd(x, w, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), 1e-6)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_rmsnorm_backward_matches_autograd():
    x = _rng(4).standard_normal((6, 40))
    w = _rng(5).standard_normal(40)
    dy = _rng(6).standard_normal((6, 40))
    dx, dw = nc.rmsnorm_bwd(x, w, dy, 1e-5)
    xt = torch.from_numpy(x).requires_grad_(True)
    wt = torch.from_numpy(w).requires_grad_(True)
    y = torch.nn.functional.rms_norm(xt, (40,), wt, 1e-5)
    (y * torch.from_numpy(dy)).sum().backward()
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_rmsnorm_backward_finite_differences():
    rng = _rng(7)
    x, w, dy = rng.standard_normal((3, 8)), rng.standard_normal(8), rng.standard_normal((3, 8))
    eps, h = 1e-3, 1e-6
    dx, dw = nc.rmsnorm_bwd(x, w, dy, eps)

    def f(xx, ww):
        return (nc.rmsnorm_fwd(xx, ww, eps)[0] * dy).sum()

    for (i, j) in [(0, 0), (1, 5), (2, 7)]:
        e = np.zeros_like(x)
        e[i, j] = h
        assert abs((f(x + e, w) - f(x - e, w)) / (2 * h) - dx[i, j]) < 1e-7
    for j in (0, 3, 7):
        e = np.zeros_like(w)
        e[j] = h
        assert abs((f(x, w + e) - f(x, w - e)) / (2 * h) - dw[j]) < 1e-7


# ---- cross-entropy with z-loss ------------------------------------------------------------------
def test_ce_uniform_logits_closed_form():
    V, zc = 1000, 1e-4
    z = np.full((2, V), 3.0)
    loss, lse = nc.cross_entropy_fwd(z, [5, 999], zc)
    want_lse = 3.0 + np.log(V)
    np.testing.assert_allclose(lse, want_lse, rtol=1e-14)
    np.testing.assert_allclose(loss, np.log(V) + zc * want_lse ** 2, rtol=1e-13)


def test_ce_dominant_logit():
    z = np.zeros((1, 50))
    z[0, 7] = 60.0
    loss, lse = nc.cross_entropy_fwd(z, [7], 0.0)
    assert abs(lse[0] - 60.0) <= 49 * np.exp(-60.0) * 1.01
    assert loss[0] < 1e-24
    loss2, _ = nc.cross_entropy_fwd(z, [3], 0.0)  # the wrong class costs the whole margin
    np.testing.assert_allclose(loss2[0], 60.0, rtol=1e-14)


def test_ce_matches_torch_and_ignores_negative_targets():
    rng = _rng(8)
    z = rng.standard_normal((9, 300)) * 3
    t = rng.integers(0, 300, 9)
    t[[2, 6]] = -100
    zc = 2e-4
    loss, lse = nc.cross_entropy_fwd(z, t, zc)
    zt = torch.from_numpy(z)
    ref = torch.nn.functional.cross_entropy(zt, torch.from_numpy(t), ignore_index=-100,
                                            reduction="none")
    ref = ref + zc * torch.logsumexp(zt, -1) ** 2 * (torch.from_numpy(t) >= 0)
    np.testing.assert_allclose(loss, ref.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, torch.logsumexp(zt, -1).numpy(), rtol=1e-14)
    assert loss[2] == 0.0 and loss[6] == 0.0


def test_ce_backward_matches_autograd_and_row_sums():
    rng = _rng(9)
    z = rng.standard_normal((6, 77)) * 2
    t = rng.integers(0, 77, 6)
    t[4] = -1
    zc, scale = 3e-3, 0.25
    dz = nc.cross_entropy_bwd(z, t, zc, scale)
    zt = torch.from_numpy(z).requires_grad_(True)
    lse = torch.logsumexp(zt, -1)
    valid = torch.from_numpy(t >= 0)
    tt = torch.from_numpy(np.where(t >= 0, t, 0))
    loss = (lse - zt.gather(1, tt[:, None])[:, 0] + zc * lse * lse) * valid
    (scale * loss.sum()).backward()
    np.testing.assert_allclose(dz, zt.grad.numpy(), rtol=1e-11, atol=1e-13)
    # each valid row sums to scale * 2 zc lse (the softmax sums to one), ignored rows to zero
    _, lse_np = nc.cross_entropy_fwd(z, t, zc)
    np.testing.assert_allclose(dz.sum(-1), np.where(t >= 0, scale * 2 * zc * lse_np, 0.0),
                               atol=1e-13)


def test_ce_backward_finite_differences():
    rng = _rng(10)
    z = rng.standard_normal((2, 9))
    t = np.array([4, 0])
    zc, h = 0.05, 1e-6
    dz = nc.cross_entropy_bwd(z, t, zc, 1.0)
    for (i, j) in [(0, 4), (0, 1), (1, 0), (1, 8)]:
        e = np.zeros_like(z)
        e[i, j] = h
        num = (nc.cross_entropy_fwd(z + e, t, zc)[0].sum() -
               nc.cross_entropy_fwd(z - e, t, zc)[0].sum()) / (2 * h)
        assert abs(num - dz[i, j]) < 1e-8

"""fp64 CPU oracle for the two other fused kernels of the FAT5 report: RMSNorm and the
cross-entropy loss with a z-loss term ("Noyau Triton" section, whose benchmarks are in "Torch vs
Triton"). TEST INFRASTRUCTURE ONLY, with the same callers as the rest of the oracle package.

The pages name the kernels and report their speed and memory, but print no formula; the
readings (each the plainest one, stated where it is used):

RMSNorm (the T5 layer norm the report's encoder-decoder uses; Zhang and Sennrich's RMSNorm):
    r = 1 / sqrt(mean_j x_j^2 + eps),   y = w * x * r      (no mean subtraction, no bias)
    backward of sum(y * dy):  with xh = x * r,
        dx = r * (w * dy - xh * mean_j(w_j dy_j xh_j)),   dw = sum over rows of dy * xh.

Cross-entropy with z-loss (the PaLM auxiliary loss that keeps the log-partition near 0):
    lse = log sum_v exp(z_v),   loss = lse - z_target + zc * lse^2
    (rows whose target is negative are ignored: loss 0, gradient 0)
    gradient of scale * loss:  dz_v = scale * (softmax_v * (1 + 2 zc lse) - [v == target]).

All arithmetic is fp64 on fp64 copies of the inputs (bf16 inputs widened exactly), one row at a
time, with numpy array operations as the only library primitives.
"""
from __future__ import annotations

import numpy as np

from . import widen


def rmsnorm_fwd(x, w, eps: float):
    """x: [N, D] (bf16 bits or floats), w: [D]. Returns (y [N, D], rstd [N]), fp64."""
    x = widen(x)
    w = widen(w)
    ms = (x * x).mean(axis=-1)          # mean of squares per row
    rstd = 1.0 / np.sqrt(ms + eps)
    y = w[None, :] * x * rstd[:, None]
    return y, rstd


def rmsnorm_bwd(x, w, dy, eps: float):
    """Gradients of sum(y * dy) for rmsnorm_fwd: (dx [N, D], dw [D]), fp64."""
    x = widen(x)
    w = widen(w)
    dy = widen(dy)
    _, rstd = rmsnorm_fwd(x, w, eps)
    xh = x * rstd[:, None]
    g = w[None, :] * dy
    c = (g * xh).mean(axis=-1)         # mean_j(w_j dy_j xh_j) per row
    dx = rstd[:, None] * (g - xh * c[:, None])
    dw = (dy * xh).sum(axis=0)
    return dx, dw


def cross_entropy_fwd(z, target, z_loss: float):
    """z: [N, V] logits (bf16 bits or floats); target: [N] ints (negative = ignored).
    Returns (loss [N], lse [N]) in fp64; ignored rows have loss 0 (their lse is still given)."""
    z = widen(z)
    target = np.asarray(target, dtype=np.int64)
    m = z.max(axis=-1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(axis=-1))
    valid = target >= 0
    zt = np.where(valid, z[np.arange(len(z)), np.where(valid, target, 0)], 0.0)
    loss = np.where(valid, lse - zt + z_loss * lse * lse, 0.0)
    return loss, lse


def cross_entropy_bwd(z, target, z_loss: float, scale: float):
    """Gradient of scale * sum(loss) with respect to the logits: dz [N, V] fp64."""
    z = widen(z)
    target = np.asarray(target, dtype=np.int64)
    _, lse = cross_entropy_fwd(z, target, z_loss)
    p = np.exp(z - lse[:, None])
    dz = p * (1.0 + 2.0 * z_loss * lse)[:, None]
    valid = target >= 0
    rows = np.nonzero(valid)[0]
    dz[rows, target[rows]] -= 1.0
    dz[~valid] = 0.0
    return scale * dz

"""Pins for the rotary-position-embedding oracle (no GPU).

RoPE is tied to properties that characterise it rather than to its formula: each channel pair
keeps its norm; a query-key score depends on the two positions only through their difference;
attention is therefore unchanged when every position of a document moves by the same amount;
at position 0 nothing turns; and the gradients match central finite differences and torch
autograd through an independent complex-number implementation.
"""
import numpy as np
import pytest
import torch

import oracle


def _x(T, H, d, seed):
    return np.random.default_rng(seed).standard_normal((T, H, d))


def test_pairs_keep_their_norm():
    x = _x(37, 3, 16, 70)
    y = oracle.rope_rotate_at(x, np.arange(37) * 7 + 3)
    n0 = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n1 = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-13, atol=1e-13)


def test_position_zero_is_the_identity_and_inverse_turns_back():
    x = _x(5, 2, 8, 71)
    np.testing.assert_array_equal(oracle.rope_rotate_at(x, np.zeros(5)), x)
    pos = np.array([0, 1, 10, 100, 1000])
    back = oracle.rope_rotate_at(oracle.rope_rotate_at(x, pos), pos, inverse=True)
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-12)


def test_first_pair_turns_by_the_position_in_radians():
    # theta_0 = base^0 = 1 for any base and head_dim: the unit vector (1, 0) at position m
    # lands on (cos m, sin m)
    x = np.zeros((4, 1, 6))
    x[:, 0, 0] = 1.0
    m = np.array([0.0, 1.0, 2.5, 40.0])
    y = oracle.rope_rotate_at(x, m, base=500.0)
    np.testing.assert_allclose(y[:, 0, 0], np.cos(m), atol=1e-15)
    np.testing.assert_allclose(y[:, 0, 1], np.sin(m), atol=1e-15)


def test_frequency_ladder_hand_values():
    """The frequency of pair i is base^(-2i/d), pinned by values worked out by hand:
    d = 4, base = 100 gives theta_1 = 100^(-1/2) = 0.1, so pair 1 at position 10 turns by one
    radian; d = 8, base = 10^4 gives theta_i = 10^(-i) (1, 0.1, 0.01, 0.001), so pair i at
    position 10^i turns by one radian. A ladder over d/2 instead of d, or starting at i = 1,
    moves every one of these."""
    x = np.zeros((1, 1, 4))
    x[0, 0, 2] = 1.0
    y = oracle.rope_rotate_at(x, [10], base=100.0)
    np.testing.assert_allclose(y[0, 0], [0.0, 0.0, np.cos(1.0), np.sin(1.0)], atol=1e-14)
    for i in range(4):
        x = np.zeros((1, 1, 8))
        x[0, 0, 2 * i] = 1.0
        y = oracle.rope_rotate_at(x, [10 ** i], base=1e4)
        want = np.zeros(8)
        want[2 * i], want[2 * i + 1] = np.cos(1.0), np.sin(1.0)
        np.testing.assert_allclose(y[0, 0], want, atol=1e-12)
    # a second pair at the same time: pair 1 of d = 8 at position 5 turns by 0.5 radian
    x = np.zeros((1, 1, 8))
    x[0, 0, 3] = 1.0  # the odd channel of pair 1: (0, 1) turns to (-sin, cos)
    y = oracle.rope_rotate_at(x, [5], base=1e4)
    np.testing.assert_allclose(y[0, 0, 2:4], [-np.sin(0.5), np.cos(0.5)], atol=1e-14)


def test_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(72)
    q = rng.standard_normal((1, 1, 32))
    k = rng.standard_normal((1, 1, 32))

    def score(m, n):
        return float((oracle.rope_rotate_at(q, [m]) * oracle.rope_rotate_at(k, [n])).sum())

    for m, n in [(0, 0), (5, 2), (2, 5), (100, 37)]:
        for t in (1, 17, 1000):
            assert abs(score(m + t, n + t) - score(m, n)) < 1e-11
    # and it does depend on the difference
    assert abs(score(5, 2) - score(2, 5)) > 1e-3


def test_attention_unchanged_by_a_common_position_shift():
    pb = oracle.Problem(_x(40, 2, 8, 73), _x(40, 2, 8, 74), _x(40, 2, 8, 75),
                        np.array([0, 25, 40]), causal=True, scale=0.4)
    out0, lse0 = oracle.rope_attn_fwd(pb)
    pos = oracle.doc_positions(pb.cu_seqlens) + 123
    shifted = oracle.Problem(oracle.rope_rotate_at(pb.q, pos), oracle.rope_rotate_at(pb.k, pos),
                             pb.v, pb.cu_seqlens, causal=True, scale=0.4)
    out1, lse1 = oracle.attn_fwd(shifted)
    np.testing.assert_allclose(out1, out0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse1, lse0, rtol=0, atol=1e-12)


def test_single_token_documents_equal_plain_attention():
    pb = oracle.Problem(_x(6, 2, 8, 76), _x(6, 2, 8, 77), _x(6, 2, 8, 78),
                        np.arange(7), scale=0.3)
    o_r, l_r = oracle.rope_attn_fwd(pb)
    o_p, l_p = oracle.attn_fwd(pb)
    np.testing.assert_array_equal(o_r, o_p)
    np.testing.assert_array_equal(l_r, l_p)


def test_backward_finite_differences():
    pb = oracle.Problem(_x(9, 2, 6, 79), _x(9, 2, 6, 80), _x(9, 2, 6, 81), np.array([0, 6, 9]),
                        causal=True, scale=0.7)
    dout = np.random.default_rng(82).standard_normal(pb.shape)
    dq, dk, dv, _ = oracle.rope_attn_bwd(pb, dout)
    eps = 1e-6

    def loss():
        return float((oracle.rope_attn_fwd(pb)[0] * dout).sum())

    for name, arr, grad in (("q", pb.q, dq), ("k", pb.k, dk), ("v", pb.v, dv)):
        for idx in [(0, 0, 0), (3, 1, 5), (5, 0, 2), (7, 1, 3), (8, 0, 4)]:
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss()
            arr[idx] = old - eps
            lm = loss()
            arr[idx] = old
            want = (lp - lm) / (2 * eps)
            assert abs(grad[idx] - want) <= 1e-6 * max(1.0, abs(want)), (name, idx)


def test_matches_torch_autograd_through_complex_rotation():
    T, H, d, base = 13, 2, 8, 10000.0
    pb = oracle.Problem(_x(T, H, d, 83), _x(T, H, d, 84), _x(T, H, d, 85),
                        np.array([0, 8, 13]), causal=False, scale=0.5)
    dout = np.random.default_rng(86).standard_normal(pb.shape)
    out, _ = oracle.rope_attn_fwd(pb, base)
    dq, dk, dv, _ = oracle.rope_attn_bwd(pb, dout, base)
    q = torch.from_numpy(pb.q.copy()).requires_grad_()
    k = torch.from_numpy(pb.k.copy()).requires_grad_()
    v = torch.from_numpy(pb.v.copy()).requires_grad_()
    pos = torch.from_numpy(oracle.doc_positions(pb.cu_seqlens).astype(np.float64))
    freq = base ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    turn = torch.polar(torch.ones(T, d // 2, dtype=torch.float64), pos[:, None] * freq[None])

    def rot(x):  # channel pairs as complex numbers, multiplied by e^(i m theta)
        z = torch.view_as_complex(x.reshape(T, H, d // 2, 2).contiguous())
        return torch.view_as_real(z * turn[:, None, :]).reshape(T, H, d)

    qr, kr = rot(q), rot(k)
    loss = torch.zeros((), dtype=torch.float64)
    got = np.zeros_like(out)
    for i in range(2):
        s, e = int(pb.cu_seqlens[i]), int(pb.cu_seqlens[i + 1])
        for h in range(H):
            o = torch.nn.functional.scaled_dot_product_attention(
                qr[s:e, h][None], kr[s:e, h][None], v[s:e, h][None], scale=pb.scale)[0]
            got[s:e, h] = o.detach().numpy()
            loss = loss + (o * torch.from_numpy(dout[s:e, h])).sum()
    np.testing.assert_allclose(out, got, rtol=1e-10, atol=1e-12)
    loss.backward()
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_odd_head_dim_rejected():
    with pytest.raises(ValueError):
        oracle.rope_rotate_at(np.zeros((2, 1, 5)), [0, 1])

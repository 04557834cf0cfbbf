"""Pins of the oracle's QKV-post (norms + RoPE) (CPU only).

Pinned against: the rotation written as a complex multiplication (torch
complex128, a different formula for the same map), closed forms (RMS of a
normalised vector, position 0 is the identity, pair norms are preserved),
the relative-position property that makes RoPE useful (a query-key dot
product depends only on the distance of the positions), and the scale
invariance of RMS normalisation.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64)


def test_rope_equals_complex_rotation():
    Hq, Hkv, d, T = 4, 2, 16, 7
    x = _rand((T, Hq + 2 * Hkv, d), 0)
    pos = torch.tensor([0, 1, 5, 100, 4095, 32767, 12345])
    theta = 10000.0
    q, k, v = oracle.qkv_post(x, pos, Hq, Hkv, rope_theta=theta)
    half = d // 2
    freqs = theta ** (-torch.arange(half, dtype=torch.float64) * 2 / d)
    rot = torch.polar(torch.ones(T, half, dtype=torch.float64), pos[:, None].double() * freqs)
    def ref(a):
        z = torch.complex(a[..., :half], a[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1).numpy()
    assert np.abs(q - ref(x[:, :Hq])).max() < 1e-12
    assert np.abs(k - ref(x[:, Hq:Hq + Hkv])).max() < 1e-12
    assert np.array_equal(v, x[:, Hq + Hkv:].numpy())


def test_position_zero_and_no_theta_are_identity():
    x = _rand((3, 6, 8), 1)
    q, k, v = oracle.qkv_post(x, torch.zeros(3, dtype=torch.long), 2, 2, rope_theta=1e6)
    assert np.abs(q - x[:, :2].numpy()).max() < 1e-15
    q2, _, _ = oracle.qkv_post(x, torch.tensor([5, 6, 7]), 2, 2, rope_theta=0.0)
    assert np.array_equal(q2, x[:, :2].numpy())


def test_rope_preserves_pair_norms():
    x = _rand((5, 3, 32), 2)
    q, _, _ = oracle.qkv_post(x, torch.tensor([3, 9, 27, 81, 243]), 1, 1, rope_theta=500000.0)
    a = x[:, :1].numpy()
    n_in = a[..., :16] ** 2 + a[..., 16:] ** 2
    n_out = q[..., :16] ** 2 + q[..., 16:] ** 2
    assert np.abs(n_in - n_out).max() < 1e-12


def test_rope_dot_product_depends_on_distance_only():
    d = 16
    base = _rand((1, 2, d), 3)
    x = base.repeat(4, 1, 1)
    pos_q = torch.tensor([10, 110, 1010, 5])
    pos_k = pos_q - 7
    q, _, _ = oracle.qkv_post(x, pos_q, 1, 0, rope_theta=10000.0)
    xk = torch.stack([base[0, 1:2]] * 4)  # the key vector as a query head
    kk, _, _ = oracle.qkv_post(torch.cat([xk, xk], dim=1), pos_k, 1, 0, rope_theta=10000.0)
    dots = (q[:, 0] * kk[:, 0]).sum(-1)
    assert np.abs(dots - dots[0]).max() < 1e-10


def test_rms_norm_closed_forms():
    x = _rand((4, 3, 64), 4) * 3.0
    w = torch.ones(64, dtype=torch.float64)
    q, k, _ = oracle.qkv_post(x, torch.zeros(4, dtype=torch.long), 2, 0, q_norm_w=w, eps=0.0)
    assert np.abs(np.sqrt((q ** 2).mean(-1)) - 1.0).max() < 1e-12
    q5, _, _ = oracle.qkv_post(x * 5.0, torch.zeros(4, dtype=torch.long), 2, 0, q_norm_w=w, eps=0.0)
    assert np.abs(q5 - q).max() < 1e-12
    w2 = torch.linspace(0.5, 2.0, 64, dtype=torch.float64)
    q2, _, _ = oracle.qkv_post(x, torch.zeros(4, dtype=torch.long), 2, 0, q_norm_w=w2, eps=0.0)
    assert np.abs(q2 - q * w2.numpy()).max() < 1e-12


def test_norm_before_rotation():
    """The norm acts on the head vector before the rotation: rotating first
    and normalising with a non-uniform weight gives a different result."""
    x = _rand((2, 2, 8), 5)
    w = torch.tensor([1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0, 8.0], dtype=torch.float64)
    pos = torch.tensor([3, 11])
    q, _, _ = oracle.qkv_post(x, pos, 1, 0, q_norm_w=w, eps=0.0, rope_theta=100.0)
    nq = (x[:, :1] * w / torch.sqrt((x[:, :1] ** 2).mean(-1, keepdim=True))).numpy()
    r, _, _ = oracle.qkv_post(torch.from_numpy(nq), pos, 1, 0, rope_theta=100.0)
    assert np.abs(q - r).max() < 1e-12


def test_rms_norm_epsilon_closed_forms():
    """The epsilon of the RMS norm sits inside the square root, added to the
    mean of the squares (not scaled by d, not outside the root).  A constant
    head vector x = c with weight 1 normalises to c / sqrt(c^2 + eps); with
    c = 1e-3 and eps = 1e-6 the two terms are equal, so any other placement
    of eps moves the result far from 1/sqrt(2)."""
    d = 64
    c, eps = 1e-3, 1e-6
    x = torch.full((3, 2, d), c, dtype=torch.float64)
    w = torch.ones(d, dtype=torch.float64)
    q, k, _ = oracle.qkv_post(x, torch.zeros(3, dtype=torch.long), 1, 0, q_norm_w=w, eps=eps)
    want = c / math.sqrt(c * c + eps)
    assert abs(want - 1.0 / math.sqrt(2.0)) < 1e-12
    assert np.abs(q - want).max() < 1e-12
    # the slips a reader could make all give other numbers
    assert abs(c / (math.sqrt(c * c) + eps) - want) > 1e-3          # eps outside the root
    assert abs(c / math.sqrt(c * c + d * eps) - want) > 1e-2        # eps scaled by d
    assert abs(c / math.sqrt(c * c + eps / d) - want) > 1e-2        # eps divided by d
    # eps dominating: x tiny against sqrt(eps) gives x / sqrt(eps) to first order
    x2 = torch.full((1, 1, d), 1e-9, dtype=torch.float64)
    q2, _, _ = oracle.qkv_post(x2, torch.zeros(1, dtype=torch.long), 1, 0, q_norm_w=w, eps=1e-2)
    assert np.abs(q2 - 1e-9 / math.sqrt(1e-18 + 1e-2)).max() < 1e-20
    # the key heads use their own weight, with the same epsilon
    xk = torch.cat([x, x], dim=1)
    _, k2, _ = oracle.qkv_post(xk, torch.zeros(3, dtype=torch.long), 1, 1, k_norm_w=2.0 * w,
                               eps=eps)
    assert np.abs(k2 - 2.0 * want).max() < 1e-12


def test_rms_norm_epsilon_non_uniform_weight_and_vector():
    """Non-uniform x and w with eps of the same size as mean(x^2): the output
    is w_i x_i / sqrt(mean(x^2) + eps), checked against sums written out in
    plain Python for a 4-element head."""
    xs = [3e-3, -1e-3, 2e-3, 0.0]
    ws = [0.5, 1.5, -2.0, 4.0]
    eps = 4e-6
    ms = sum(v * v for v in xs) / 4.0          # 3.5e-6, same order as eps
    x = torch.tensor([[xs]], dtype=torch.float64)
    w = torch.tensor(ws, dtype=torch.float64)
    q, _, _ = oracle.qkv_post(x, torch.zeros(1, dtype=torch.long), 1, 0, q_norm_w=w, eps=eps)
    want = [wi * xi / math.sqrt(ms + eps) for xi, wi in zip(xs, ws)]
    assert np.abs(q[0, 0] - np.array(want)).max() < 1e-15
    # and eps = 0 would have given a result about 1.46x larger
    assert abs(want[0] / (ws[0] * xs[0] / math.sqrt(ms)) - math.sqrt(ms / (ms + eps))) < 1e-12

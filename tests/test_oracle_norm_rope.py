"""Pins of the oracle's Q/K RMSNorm + RoPE (the pages name the steps, not the
formulas; the reading is RMSNorm over the head dimension and the RoFormer
rotation of consecutive pairs).  Pinned by closed forms (unit mean square,
scale invariance, quarter-turn), invariants (pair norms, the relative-position
property of rotary products), torch's rms_norm as a library special case, and
a complex-number restatement of the rotation."""
import numpy as np
import pytest
import torch

import oracle


def _x(shape, seed=0):
    return np.random.default_rng(seed).standard_normal(shape) * 3.0


def test_rms_norm_closed_forms():
    x = _x((5, 7, 64))
    y = oracle.rms_norm(x, None, 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-12)
    np.testing.assert_allclose(oracle.rms_norm(4.5 * x, None, 0.0), y, rtol=1e-12)   # scale invariance
    w = np.linspace(0.5, 2.0, 64)
    np.testing.assert_allclose(oracle.rms_norm(x, w, 0.0), y * w, rtol=1e-12)
    # eps matters for tiny rows: a zero row stays zero, a constant row c -> c / sqrt(c^2 + eps)
    z = oracle.rms_norm(np.full((1, 64), 1e-3), None, 1e-6)
    np.testing.assert_allclose(z, 1e-3 / np.sqrt(1e-6 + 1e-6), rtol=1e-12)
    assert np.all(oracle.rms_norm(np.zeros((2, 64)), None, 1e-6) == 0)


def test_rms_norm_matches_torch():
    x = _x((3, 11, 128), 1)
    w = np.random.default_rng(2).uniform(0.5, 1.5, 128)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (128,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rms_norm(x, w, 1e-6), ref, rtol=1e-12, atol=1e-14)


def test_rope_is_a_rotation():
    y = _x((6, 4, 128), 3)
    theta = np.random.default_rng(4).uniform(-np.pi, np.pi, (6, 1, 64))
    r = oracle.rope_pairs(y, np.cos(theta), np.sin(theta))
    np.testing.assert_allclose(r[..., 0::2] ** 2 + r[..., 1::2] ** 2, y[..., 0::2] ** 2 + y[..., 1::2] ** 2,
                               rtol=1e-12)
    # identity and a quarter turn
    assert np.array_equal(oracle.rope_pairs(y, np.ones((6, 1, 64)), np.zeros((6, 1, 64))), y)
    q = oracle.rope_pairs(y, np.zeros((6, 1, 64)), np.ones((6, 1, 64)))
    assert np.array_equal(q[..., 0::2], -y[..., 1::2]) and np.array_equal(q[..., 1::2], y[..., 0::2])
    # the complex-number form: pair (a, b) is a + ib multiplied by e^{i theta}
    z = (y[..., 0::2] + 1j * y[..., 1::2]) * np.exp(1j * theta)
    np.testing.assert_allclose(r[..., 0::2], z.real, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r[..., 1::2], z.imag, rtol=1e-12, atol=1e-12)


def test_rope_relative_position_property():
    """With angles theta_i * n, <R(n) q, R(m) k> depends on n - m only."""
    D = 64
    freq = 10000.0 ** (-np.arange(D // 2) / (D // 2))
    ang = np.arange(40)[:, None] * freq[None, :]
    q, k = _x((D,), 5), _x((D,), 6)
    Rq = oracle.rope_pairs(np.broadcast_to(q, (40, D)), np.cos(ang), np.sin(ang))
    Rk = oracle.rope_pairs(np.broadcast_to(k, (40, D)), np.cos(ang), np.sin(ang))
    for shift in (0, 3, 17):
        dots = [Rq[n] @ Rk[n - shift] for n in range(shift, 40)]
        np.testing.assert_allclose(dots, dots[0], rtol=1e-9, atol=1e-9)


def test_fused_layout_applies_q_k_only_and_moves_heads():
    rng = np.random.default_rng(7)
    B, N, H, D = 2, 9, 3, 16
    x = torch.from_numpy(rng.standard_normal((B, N, 3, H, D)) * 2).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    wq, wk = rng.uniform(0.5, 1.5, D), rng.uniform(0.5, 1.5, D)
    ang = rng.uniform(-3, 3, (N, D // 2))
    q, k, v = oracle.qkv_norm_rope_to_head_major(bits, wq, wk, 1e-6, np.cos(ang), np.sin(ang))
    xf = x.to(torch.float64).numpy()
    assert np.array_equal(v, np.transpose(xf[:, :, 2], (0, 2, 1, 3)))            # v untouched
    b, n, h = 1, 4, 2
    yq = oracle.rms_norm(xf[b, n, 0, h], wq, 1e-6)
    c, s = np.cos(ang[n]), np.sin(ang[n])
    np.testing.assert_allclose(q[b, h, n, 0::2], yq[0::2] * c - yq[1::2] * s, rtol=1e-12)
    # no weights, no tables: pure split
    q0, k0, _ = oracle.qkv_norm_rope_to_head_major(bits, None, None, 1e-6, None, None)
    assert np.array_equal(k0, np.transpose(xf[:, :, 1], (0, 2, 1, 3)))

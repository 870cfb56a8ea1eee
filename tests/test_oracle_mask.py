"""Pins of the oracle's general (B, T, T) mask and the padding rule of "8 卡怎么
分 token", "构造 padding mask" (pad key columns masked, pad query rows attend
every valid key): special cases that reduce to the key-only mask or to no mask,
torch's fp64 SDPA with a boolean mask, and the empty-row convention."""
import numpy as np
import torch

import oracle
from dit_long_sequence_gb300 import workloads as wl


def _bits(t):
    return wl.bf16_bits(t.contiguous())


def _case(B=2, N=50, H=2, D=32, seed=3):
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed=seed)
    return q, k, v, _bits(q), _bits(k), _bits(v)


def test_all_true_mask_is_no_mask():
    q, k, v, qb, kb, vb = _case()
    allow = np.ones((2, 50, 50), dtype=bool)
    O1, L1 = oracle.attn(qb, kb, vb, allow=allow)
    O0, L0 = oracle.attn(qb, kb, vb)
    assert np.array_equal(O1, O0) and np.array_equal(L1, L0)


def test_prefix_mask_is_the_key_only_mask():
    q, k, v, qb, kb, vb = _case()
    allow = np.zeros((2, 50, 50), dtype=bool)
    allow[:, :, :31] = True
    O1, L1 = oracle.attn(qb, kb, vb, allow=allow)
    O0, L0 = oracle.attn(qb, kb, vb, key_valid_len=31)
    assert np.array_equal(O1, O0) and np.array_equal(L1, L0)


def test_random_mask_matches_sdpa_and_empty_rows_are_zero():
    q, k, v, qb, kb, vb = _case(seed=8)
    g = torch.Generator().manual_seed(1)
    allow = torch.rand((2, 50, 50), generator=g) < 0.3
    allow[0, 7, :] = False                       # an empty row
    O, L = oracle.attn(qb, kb, vb, allow=allow.numpy(), scale=0.3)
    qt, kt, vt = (x.to(torch.float64).permute(0, 2, 1, 3) for x in (q, k, v))
    am = allow[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=am, scale=0.3)
    ref = ref.permute(0, 2, 1, 3).numpy()
    lref = torch.logsumexp((0.3 * torch.einsum("bhid,bhjd->bhij", qt, kt)).masked_fill(~am, -np.inf), -1).numpy()
    rows = allow.any(-1).numpy()
    np.testing.assert_allclose(O[rows], ref[rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(L.transpose(0, 2, 1)[rows], lref.transpose(0, 2, 1)[rows], rtol=0, atol=1e-12)
    assert np.all(O[0, 7] == 0) and np.all(np.isneginf(L[0, :, 7]))


def test_padding_rule():
    T, Tp = 37, 48
    g = np.random.default_rng(2)
    m = g.random((2, T, T)) < 0.5
    e = oracle.expand_mask(m, Tp)
    assert e.shape == (2, Tp, Tp)
    assert np.array_equal(e[:, :T, :T], m)
    assert not e[:, :, T:].any()                 # pad keys never attended
    assert e[:, T:, :T].all()                    # pad queries see every valid key
    # pad query rows then equal the key-only-mask result over the T valid keys
    q, k, v, qb, kb, vb = _case(N=Tp, seed=4)
    O1, L1 = oracle.attn(qb, kb, vb, allow=e)
    O0, L0 = oracle.attn(qb, kb, vb, key_valid_len=T)
    assert np.array_equal(O1[:, T:], O0[:, T:]) and np.array_equal(L1[:, :, T:], L0[:, :, T:])

"""Pins of the fp64 CPU oracle against things other than itself.

Each test ties the oracle to the mathematics or to an independent library
routine: brute force on tiny inputs, torch's fp64 scaled-dot-product attention
and scipy's logsumexp (library special cases), closed forms, and the
invariants the pages fix (softmax rows sum to one, constant V, key
permutation, masked pad keys have no effect, chunked (O, LSE) merge equals one
global pass).  A plausible slip in the oracle -- a dropped scale, a missing
max term in the LSE, a transposed operand, an off-by-one mask, a wrong stride
-- fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from dit_long_sequence_gb300 import workloads as wl


def _bits(t):
    return wl.bf16_bits(t.contiguous())


def _vals(t):
    return t.to(torch.float64).numpy()


def _inputs(B, N, H, D, seed, Nkv=None):
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed, device="cpu", Nkv=Nkv)
    return q, k, v


def _from_values(arr):
    """bf16 tensor holding exactly the given (bf16-representable) values."""
    t = torch.tensor(np.asarray(arr, dtype=np.float64), dtype=torch.float64)
    tb = t.to(torch.bfloat16)
    assert torch.equal(tb.to(torch.float64), t), "fixture values must be exact in bf16"
    return tb


# ---------------------------------------------------------------- brute force

def _brute(q, k, v, scale, kvl):
    """Scalar Python with math.fsum: [B,N,H,D] float64 arrays."""
    B, Nq, H, D = q.shape
    O = np.zeros((B, Nq, H, D))
    L = np.zeros((B, H, Nq))
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                s = [scale * math.fsum(q[b, i, h, d] * k[b, j, h, d] for d in range(D))
                     for j in range(kvl)]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                l = math.fsum(e)
                for d in range(D):
                    O[b, i, h, d] = math.fsum(e[j] * v[b, j, h, d] for j in range(kvl)) / l
                L[b, h, i] = m + math.log(l)
    return O, L


@pytest.mark.parametrize("B,N,Nkv,H,D,kvl,scale", [
    (1, 7, 7, 1, 4, 7, 0.5),
    (2, 9, 12, 3, 8, 12, 0.35),
    (1, 12, 12, 2, 8, 5, 0.9),     # key mask, not a multiple of anything
    (2, 5, 16, 2, 4, 1, 0.7),      # one valid key
])
def test_brute_force_tiny(B, N, Nkv, H, D, kvl, scale):
    q, k, v = _inputs(B, N, H, D, seed=11 + N, Nkv=Nkv)
    O, L = oracle.attn(_bits(q), _bits(k), _bits(v), key_valid_len=kvl, scale=scale)
    Ob, Lb = _brute(_vals(q), _vals(k), _vals(v), scale, kvl)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)


# ------------------------------------------------------ library special cases

@pytest.mark.parametrize("B,N,Nkv,H,D,kvl", [
    (1, 64, 64, 2, 64, None),
    (2, 33, 97, 3, 128, None),      # cross lengths, ragged
    (1, 50, 80, 2, 64, 61),         # key mask
])
def test_matches_torch_sdpa_fp64(B, N, Nkv, H, D, kvl):
    q, k, v = _inputs(B, N, H, D, seed=5, Nkv=Nkv)
    scale = 1.0 / math.sqrt(D)
    O, L = oracle.attn(_bits(q), _bits(k), _bits(v), key_valid_len=kvl, scale=scale)
    qt, kt, vt = (x.to(torch.float64).permute(0, 2, 1, 3) for x in (q, k, v))  # [B,H,N,D]
    mask = None
    n_valid = Nkv if kvl is None else kvl
    if kvl is not None:
        mask = torch.zeros(1, Nkv, dtype=torch.bool)
        mask[:, :kvl] = True
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(O, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    s = scale * torch.einsum("bhid,bhjd->bhij", qt, kt[:, :, :n_valid])
    np.testing.assert_allclose(L, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, scipy.special.logsumexp(s.numpy(), axis=-1), rtol=0, atol=1e-12)


# ------------------------------------------------------------- closed forms

def test_closed_form_weights_one_two_four():
    # scale = ln 2 and scores 0, ln2, 2 ln2 give weights 1:2:4, l = 7 (times 2^-2 after
    # the max shift), so O = (v0 + 2 v1 + 4 v2) / 7 and LSE = ln 7.
    q = _from_values([[[[1.0, 0.0]]]])                            # [1,1,1,2]
    k = _from_values([[[[0.0, 0.0]], [[1.0, 0.0]], [[2.0, 0.0]]]])  # [1,3,1,2]
    v = _from_values([[[[7.0, 0.0]], [[0.0, 7.0]], [[7.0, 7.0]]]])
    O, L = oracle.attn(_bits(q), _bits(k), _bits(v), scale=math.log(2.0))
    np.testing.assert_allclose(O[0, 0, 0], [5.0, 6.0], rtol=0, atol=1e-14)
    assert abs(L[0, 0, 0] - math.log(7.0)) < 1e-14
    # masking the last key leaves weights 1:2 -> O = (v0 + 2 v1)/3, LSE = ln 3
    O, L = oracle.attn(_bits(q), _bits(k), _bits(v), scale=math.log(2.0), key_valid_len=2)
    np.testing.assert_allclose(O[0, 0, 0], [7.0 / 3.0, 14.0 / 3.0], rtol=0, atol=1e-14)
    assert abs(L[0, 0, 0] - math.log(3.0)) < 1e-14


def test_closed_form_two_keys_sigmoid():
    # D = 1, two keys: w0 = sigmoid(s0 - s1); O = w0 v0 + (1 - w0) v1;
    # LSE = s0 + ln(1 + exp(s1 - s0)).
    q = _from_values([[[[2.0]]]])
    k = _from_values([[[[1.0]], [[-1.0]]]])
    v = _from_values([[[[3.0]], [[-1.0]]]])
    scale = 0.5
    O, L = oracle.attn(_bits(q), _bits(k), _bits(v), scale=scale)
    s0, s1 = 1.0, -1.0
    w0 = 1.0 / (1.0 + math.exp(-(s0 - s1)))
    assert abs(O[0, 0, 0, 0] - (3.0 * w0 - 1.0 * (1.0 - w0))) < 1e-14
    assert abs(L[0, 0, 0] - (s0 + math.log1p(math.exp(s1 - s0)))) < 1e-14


def test_closed_form_zero_query_is_mean():
    # q = 0: every score is 0, weights are uniform over the valid keys.
    B, N, H, D, kvl = 1, 40, 2, 64, 29
    _, k, v = _inputs(B, N, H, D, seed=3)
    q = torch.zeros(B, N, H, D, dtype=torch.bfloat16)
    O, L = oracle.attn(_bits(q), _bits(k), _bits(v), key_valid_len=kvl)
    mean = _vals(v)[:, :kvl].mean(axis=1)                        # [B,H,D]
    np.testing.assert_allclose(O, np.broadcast_to(mean[:, None], O.shape), rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, math.log(kvl), rtol=0, atol=1e-12)


def test_closed_form_single_valid_key():
    B, N, H, D = 2, 16, 2, 64
    q, k, v = _inputs(B, N, H, D, seed=4)
    O, L = oracle.attn(_bits(q), _bits(k), _bits(v), key_valid_len=1)
    vv, qq, kk = _vals(v), _vals(q), _vals(k)
    np.testing.assert_array_equal(O, np.broadcast_to(vv[:, :1], O.shape))
    s0 = np.einsum("bihd,bhd->bhi", qq, kk[:, 0]) / 8.0
    np.testing.assert_allclose(L, s0, rtol=0, atol=1e-12)


def test_closed_form_dominant_key():
    # A huge scale turns softmax into argmax: O -> the value row of the best key.
    B, N, H, D = 1, 24, 2, 64
    q, k, v = _inputs(B, N, H, D, seed=6)
    O, L = oracle.attn(_bits(q), _bits(k), _bits(v), scale=1e4)
    s = np.einsum("bihd,bjhd->bhij", _vals(q), _vals(k))
    best = s.argmax(axis=-1)                                      # [B,H,N]
    vv = _vals(v)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(O[b, :, h], vv[b, best[b, h], h], rtol=0, atol=1e-9)
            np.testing.assert_allclose(L[b, h], 1e4 * s[b, h].max(axis=-1), rtol=1e-13)


def test_statistical_lse_sanity():
    # N(0,1) inputs: scale*q.k is about N(0,1), so LSE is about ln N + 1/2 (a smoke check).
    B, N, H, D = 1, 4096, 1, 128
    q, k, v = _inputs(B, N, H, D, seed=8)
    rows = np.arange(0, N, 64, dtype=np.int32)[None, None]
    _, L = oracle.attn(_bits(q), _bits(k), _bits(v), rows=rows)
    assert abs(L.mean() - (math.log(N) + 0.5)) < 0.15


# --------------------------------------------------------------- invariants

def test_softmax_rows_sum_to_one():
    B, N, H, D = 1, 96, 2, 64
    q, k, v = _inputs(B, N, H, D, seed=9)
    scale = 0.125
    _, L = oracle.attn(_bits(q), _bits(k), _bits(v), scale=scale)
    s = scale * np.einsum("bihd,bjhd->bhij", _vals(q), _vals(k))
    total = np.exp(s - L[..., None]).sum(axis=-1)
    np.testing.assert_allclose(total, 1.0, rtol=0, atol=1e-12)


def test_constant_v_gives_constant_output():
    B, N, H, D = 1, 70, 2, 64
    q, k, _ = _inputs(B, N, H, D, seed=10)
    c = torch.linspace(-3, 3, D, dtype=torch.float64).to(torch.bfloat16)
    v = c.expand(B, N, H, D).contiguous()
    O, _ = oracle.attn(_bits(q), _bits(k), _bits(v), key_valid_len=53)
    np.testing.assert_allclose(O, np.broadcast_to(c.to(torch.float64).numpy(), O.shape),
                               rtol=0, atol=1e-12)


def test_key_permutation_invariance():
    B, N, H, D = 1, 80, 2, 64
    q, k, v = _inputs(B, N, H, D, seed=12)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(1))
    O1, L1 = oracle.attn(_bits(q), _bits(k), _bits(v))
    O2, L2 = oracle.attn(_bits(q), _bits(k[:, perm]), _bits(v[:, perm]))
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-13)


def test_masked_pad_keys_have_no_effect():
    B, N, H, D, kvl = 1, 64, 2, 64, 41
    q, k, v = _inputs(B, N, H, D, seed=13)
    O1, L1 = oracle.attn(_bits(q), _bits(k), _bits(v), key_valid_len=kvl)
    k2, v2 = k.clone(), v.clone()
    k2[:, kvl:] = 1e4
    v2[:, kvl:] = float("nan")
    O2, L2 = oracle.attn(_bits(q), _bits(k2), _bits(v2), key_valid_len=kvl)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)
    # and the mask is not a no-op: dropping it changes the result
    O3, _ = oracle.attn(_bits(q), _bits(k), _bits(v))
    assert np.abs(O3 - O1).max() > 1e-3


def test_zero_valid_keys_convention():
    B, N, H, D = 1, 8, 2, 64
    q, k, v = _inputs(B, N, H, D, seed=14)
    O, L = oracle.attn(_bits(q), _bits(k), _bits(v), key_valid_len=0)
    assert (O == 0).all() and np.isneginf(L).all()


def test_fused_strided_views_equal_contiguous():
    B, N, H, D = 2, 48, 3, 64
    q, k, v, buf = wl.make_qkv(B, N, H, D, seed=15, fused=True)
    assert q.stride(1) == 3 * H * D and not q.is_contiguous()
    bits = wl.bf16_bits(buf)
    qv, kv, vv = bits[:, :, 0], bits[:, :, 1], bits[:, :, 2]
    O1, L1 = oracle.attn(qv, kv, vv)
    O2, L2 = oracle.attn(_bits(q), _bits(k), _bits(v))
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_row_sampling_matches_full():
    B, N, H, D = 1, 200, 2, 64
    q, k, v = _inputs(B, N, H, D, seed=16)
    Of, Lf = oracle.attn(_bits(q), _bits(k), _bits(v))
    rows = wl.sample_rows(B, H, N, 17, seed=16, must=(100,))
    Os, Ls = oracle.attn(_bits(q), _bits(k), _bits(v), rows=rows)
    for b in range(B):
        for h in range(H):
            np.testing.assert_array_equal(Os[b, h], Of[b, rows[b, h], h])
            np.testing.assert_array_equal(Ls[b, h], Lf[b, h, rows[b, h]])


# -------------------------------------------------------------------- merge

def _chunked(q, k, v, bounds, scale=None):
    parts_o, parts_l = [], []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        o, l = oracle.attn(_bits(q), _bits(k[:, lo:hi]), _bits(v[:, lo:hi]), scale=scale)
        parts_o.append(o)
        parts_l.append(l)
    return np.stack(parts_o), np.stack(parts_l)


@pytest.mark.parametrize("bounds", [[0, 96], [0, 50, 96], [0, 10, 11, 40, 77, 96], list(range(0, 97, 32))])
def test_chunked_merge_equals_single_pass(bounds):
    B, N, H, D = 1, 96, 2, 64
    q, k, v = _inputs(B, N, H, D, seed=17)
    Of, Lf = oracle.attn(_bits(q), _bits(k), _bits(v))
    po, pl = _chunked(q, k, v, bounds)
    Om, Lm = oracle.lse_merge(po, pl)
    np.testing.assert_allclose(Om, Of, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lm, Lf, rtol=0, atol=1e-12)
    Os, Ls = oracle.lse_merge_streaming(po, pl)
    np.testing.assert_allclose(Os, Of, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Ls, Lf, rtol=0, atol=1e-12)


def test_merge_empty_chunk_is_identity_and_order_free():
    B, N, H, D = 1, 64, 2, 64
    q, k, v = _inputs(B, N, H, D, seed=18)
    po, pl = _chunked(q, k, v, [0, 20, 64])
    empty_o = np.full_like(po[:1], np.nan)
    empty_l = np.full_like(pl[:1], -np.inf)
    Om, Lm = oracle.lse_merge(po, pl)
    Oe, Le = oracle.lse_merge(np.concatenate([empty_o, po]), np.concatenate([empty_l, pl]))
    np.testing.assert_array_equal(Oe, Om)
    np.testing.assert_array_equal(Le, Lm)
    Or, Lr = oracle.lse_merge(po[::-1], pl[::-1])
    np.testing.assert_allclose(Or, Om, rtol=0, atol=1e-14)
    np.testing.assert_allclose(Lr, Lm, rtol=0, atol=1e-14)
    Os, Ls = oracle.lse_merge_streaming(np.concatenate([empty_o, po]), np.concatenate([empty_l, pl]))
    np.testing.assert_allclose(Os, Om, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Ls, Lm, rtol=0, atol=1e-12)
    # every chunk empty -> O = 0, LSE = -inf
    Oz, Lz = oracle.lse_merge(np.concatenate([empty_o, empty_o]), np.concatenate([empty_l, empty_l]))
    assert (Oz == 0).all() and np.isneginf(Lz).all()


def test_merge_closed_form_two_chunks():
    # two chunks with L = ln 1 and ln 3 -> weights 1/4, 3/4 and LSE = ln 4
    o = np.array([[[[[1.0, 0.0]]]], [[[[0.0, 1.0]]]]])        # [2,1,1,1,2]
    l = np.array([[[[0.0]]], [[[math.log(3.0)]]]])            # [2,1,1,1]
    O, L = oracle.lse_merge(o, l)
    np.testing.assert_allclose(O[0, 0, 0], [0.25, 0.75], rtol=0, atol=1e-15)
    assert abs(L[0, 0, 0] - math.log(4.0)) < 1e-15


# ------------------------------------------------------------------- layout

def test_layout_index_identity():
    B, N, H, D = 2, 5, 3, 8
    # every element holds a unique code of its own (b, n, t, h, d) position
    codes = np.arange(B * N * 3 * H * D, dtype=np.uint16).reshape(B, N, 3, H, D)
    outs = oracle.qkv_to_head_major(codes)
    for t in range(3):
        assert outs[t].shape == (B, H, N, D) and outs[t].flags["C_CONTIGUOUS"]
        for b in range(B):
            for h in range(H):
                for n in range(N):
                    for d in range(D):
                        want = (((b * N + n) * 3 + t) * H + h) * D + d
                        assert outs[t][b, h, n, d] == want

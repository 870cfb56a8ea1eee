"""Pins of the oracle's FP8 E4M3 codec, scaled QKV cast and FP8 attention.

The codec is pinned by the format's fixed points (every code decodes to its
defining value and encodes back), hand-worked ties and saturation, and by
torch's float8_e4m3fn conversion as a library special case; the FP8 attention
reduces exactly to the bf16 attention oracle (every E4M3 value is a bf16 value)
and to torch's fp64 SDPA on the decoded values.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def test_every_code_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    nan = np.isnan(vals)
    assert nan.sum() == 2 and set(codes[nan]) == {0x7F, 0xFF}
    back = oracle.e4m3_encode(vals[~nan])
    assert np.array_equal(back, codes[~nan])
    assert vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6
    assert vals[0x38] == 1.0 and vals[0xB8] == -1.0


@pytest.mark.parametrize("x,code", [
    (1.0625, 0x38),                  # halfway 1.0 / 1.125 -> even mantissa (1.0)
    (1.1875, 0x3A),                  # halfway 1.125 / 1.25 -> even (1.25)
    (2.0 ** -10, 0x00),              # half the smallest subnormal -> 0 (even)
    (3 * 2.0 ** -10, 0x02),          # halfway 2^-9 / 2^-8 -> even (2^-8)
    (15 * 2.0 ** -10, 0x08),         # rounds up into the smallest normal
    (460.0, 0x7E), (1e9, 0x7E), (-1e9, 0xFE), (float("inf"), 0x7E),   # saturation
    (-0.0, 0x80), (0.0, 0x00),
])
def test_hand_worked_rounding_and_saturation(x, code):
    assert int(oracle.e4m3_encode(np.array([x]))[0]) == code


def test_matches_torch_float8_in_range():
    g = torch.Generator().manual_seed(0)
    x = torch.cat([torch.randn(20000, generator=g, dtype=torch.float64) * s for s in (1e-3, 0.1, 1.0, 30.0)])
    x = x.clamp(-448.0, 448.0)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x.numpy())
    assert np.array_equal(got, ref)


def test_cast_of_stacked_buffer_uses_per_tensor_scales():
    g = torch.Generator().manual_seed(1)
    buf = (torch.randn(2, 5, 3, 2, 8, generator=g) * 4).to(torch.bfloat16)
    bits = buf.view(torch.int16).numpy().view(np.uint16)
    scales = (0.5, 2.0, 16.0)
    out = oracle.qkv_cast_fp8(bits, scales)
    x = buf.to(torch.float64).numpy()
    for t in range(3):
        assert np.array_equal(out[:, :, t], oracle.e4m3_encode(x[:, :, t] * scales[t]))


def test_e4m3_values_are_exact_bf16():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    bits = oracle.e4m3_to_bf16_bits(codes)
    back = oracle.bf16_bits_to_f64(bits)
    assert np.array_equal(back, oracle.e4m3_decode(codes))


def test_fp8_attention_matches_sdpa_on_decoded_values():
    g = torch.Generator().manual_seed(2)
    B, N, H, D = 1, 40, 2, 16
    q8, k8, v8 = (oracle.e4m3_encode((torch.randn(B, N, H, D, generator=g, dtype=torch.float64) * 3).numpy())
                  for _ in range(3))
    dq, dk, dv, scale = 0.25, 0.5, 2.0, 1.0 / math.sqrt(D)
    O, L = oracle.attn_fp8(q8, k8, v8, scale=scale, descale_q=dq, descale_k=dk, descale_v=dv, key_valid_len=31)
    Q, K, V = (torch.from_numpy(oracle.e4m3_decode(a)).permute(0, 2, 1, 3) for a in (q8, k8, v8))
    Q, K, V = Q * dq, K * dk, V * dv
    mask = torch.zeros(1, N, dtype=torch.bool)
    mask[:, :31] = True
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(O, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    s = scale * torch.einsum("bhid,bhjd->bhij", Q, K[:, :, :31])
    np.testing.assert_allclose(L, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)

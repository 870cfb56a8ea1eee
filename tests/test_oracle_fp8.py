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


# The cast forms x * s in fp32 (one fp32 rounding), then rounds that to E4M3.
# Each case below puts the exact product x * s on one side of an E4M3 rounding
# tie and its fp32 rounding exactly on the tie, so a cast that multiplies in
# fp64 (or skips the fp32 step) lands on the other neighbour.  x = 3 is exact in
# bf16; s is an fp32 value given by its hex form.  Worked by hand:
#   s = 0x1.6aaaacp-2 (17/48 rounded up):  3s = 17/16 + 2^-24.  In fp32 that is
#     halfway between 17/16 and 17/16 + 2^-23 and goes to the even one, 17/16;
#     17/16 is halfway between 1 and 9/8 in E4M3 and goes to the even mantissa,
#     1 (0x38).  From the exact product the E4M3 rounding gives 9/8 (0x39).
#   s = 0x1.955554p-2:  3s = 19/16 - 2^-24 -> fp32 19/16 (even) -> E4M3 tie
#     between 9/8 (odd mantissa) and 5/4 -> 5/4 (0x3A); exact: 9/8 (0x39).
#   s = 0x1.aaaaacp-10: 3s = 5 * 2^-10 + 2^-33 -> fp32 5 * 2^-10 -> subnormal
#     tie between 2 * 2^-9 and 3 * 2^-9 -> 2 * 2^-9 (0x02); exact: 0x03.
#   x = -3 with the first s: the same magnitude, sign bit set (0xB8 / 0xB9).
FP32_STEP_CASES = [
    # (x, s as hex, code after the fp32 product, code from the exact product)
    (3.0, "0x1.6aaaacp-2", 0x38, 0x39),
    (3.0, "0x1.955554p-2", 0x3A, 0x39),
    (3.0, "0x1.aaaaacp-10", 0x02, 0x03),
    (-3.0, "0x1.6aaaacp-2", 0xB8, 0xB9),
]


def _cast_one(mod, x, s, slot):
    """Cast a [1, 1, 3, 1, 16] stacked buffer whose tensor `slot` holds x with
    scale s (the other two tensors hold 1.0 with scale 1)."""
    buf = torch.ones((1, 1, 3, 1, 16), dtype=torch.bfloat16)
    buf[:, :, slot] = x
    scales = [1.0, 1.0, 1.0]
    scales[slot] = s
    out = mod.qkv_cast_fp8(buf.view(torch.int16).numpy().view(np.uint16), scales)
    return out


@pytest.mark.parametrize("x,s_hex,code,exact_code", FP32_STEP_CASES)
def test_cast_rounds_the_product_in_fp32_first(x, s_hex, code, exact_code):
    s = float.fromhex(s_hex)
    assert float(np.float32(s)) == s                      # s is an fp32 value
    # preconditions of the hand-worked case (pure fp64 / fp32 arithmetic)
    p32 = float(np.float32(x) * np.float32(s))
    assert p32 != x * s                                   # the fp32 product rounded
    assert int(oracle.e4m3_encode(np.array([x * s]))[0]) == exact_code
    for slot in range(3):
        out = _cast_one(oracle, x, s, slot)
        assert np.all(out[:, :, slot] == code), (slot, out[:, :, slot])
        others = [t for t in range(3) if t != slot]
        assert np.all(out[:, :, others] == 0x38)          # 1.0 with scale 1


# ---- planted slips in the numpy part of the oracle (the FP8 cast) ----------
# Each mutant is a copy of oracle/__init__.py with one plausible slip, loaded
# from a temporary directory; the cast pins above must reject every one.
CAST_MUTANTS = {
    "product_in_fp64": ("out[:, n0:n0 + step] = e4m3_encode((x * sc).astype(np.float64))",
                        "out[:, n0:n0 + step] = e4m3_encode(x.astype(np.float64) * sc.astype(np.float64))"),
    "no_fp32_step": ("x = bf16_bits_to_f64(bits[:, n0:n0 + step]).astype(np.float32)",
                     "x = bf16_bits_to_f64(bits[:, n0:n0 + step])"),
    "scale_after_rounding": ("out[:, n0:n0 + step] = e4m3_encode((x * sc).astype(np.float64))",
                             "out[:, n0:n0 + step] = e4m3_encode(e4m3_decode(e4m3_encode(x)) * sc)"),
    "scales_rotated": ("sc = np.asarray(scales, dtype=np.float32).reshape(1, 1, 3, 1, 1)",
                       "sc = np.roll(np.asarray(scales, dtype=np.float32), 1).reshape(1, 1, 3, 1, 1)"),
}


def _cast_pin_failures(mod):
    failures = []
    for x, s_hex, code, _ in FP32_STEP_CASES:
        s = float.fromhex(s_hex)
        for slot in range(3):
            try:
                out = _cast_one(mod, x, s, slot)
            except Exception:
                return ["raised"]
            if not (np.all(out[:, :, slot] == code) and np.all(out[:, :, [t for t in range(3) if t != slot]] == 0x38)):
                failures.append((x, s_hex, slot))
    return failures


def _load_mutant(tmp_path, old, new):
    import importlib.util
    src = open(oracle.__file__, encoding="utf-8").read()
    assert src.count(old) == 1, "mutation anchor not found"
    d = tmp_path / "oracle_mutant"
    d.mkdir()
    (d / "__init__.py").write_text(src.replace(old, new), encoding="utf-8")
    spec = importlib.util.spec_from_file_location("oracle_mutant", str(d / "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_real_cast_passes_the_cast_pins():
    assert _cast_pin_failures(oracle) == []


@pytest.mark.parametrize("name", sorted(CAST_MUTANTS))
def test_cast_mutant_is_caught(name, tmp_path):
    mod = _load_mutant(tmp_path, *CAST_MUTANTS[name])
    assert _cast_pin_failures(mod), f"cast mutant {name} slipped through every pin"

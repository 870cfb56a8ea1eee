"""Seeded shape fuzzing of the attention entry points against the oracle:
random batch, rows, keys, heads, head dim, key-valid length, padded or fused
strides and output dtype (tiny extremes included), each compared element-wise
with the parity gates of tests/parity.py."""
import numpy as np
import pytest
import torch

import oracle
from dit_long_sequence_gb300 import workloads as wl

from parity import compare, compare_fp8, host_bits, host_u8

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def dl():
    import dit_long_sequence_gb300 as m
    return m


def _views(B, Nq, Nkv, H, D, layout, seed):
    """q, k, v bf16 views: separate tensors with padded head rows, or strided
    views of one fused [B, N, 3, H, D] buffer (Nq = Nkv then)."""
    if layout == "fused":
        q, k, v, _ = wl.make_qkv(B, Nq, H, D, seed=seed, device=DEV, fused=True)
        return q, k, v
    pad = 8 * (seed % 3)
    g = wl.generator(DEV, seed)
    q = torch.randn((B, Nq, H, D + pad), generator=g, device=DEV).to(torch.bfloat16)[..., :D]
    k = torch.randn((B, Nkv, H, D + pad), generator=g, device=DEV).to(torch.bfloat16)[..., :D]
    v = torch.randn((B, Nkv, H, D), generator=g, device=DEV).to(torch.bfloat16)
    return q, k, v


CASES = []
_rng = np.random.default_rng(2026)
for i in range(24):
    D = int(_rng.choice([64, 128]))
    layout = "fused" if i % 4 == 0 else "separate"
    Nq = int(_rng.choice([1, 2, 127, 128, 129, 255, 256, 257, 700, 1500]))
    Nkv = Nq if layout == "fused" else int(_rng.choice([1, 3, 96, 128, 129, 640, 1111]))
    kvl = int(_rng.integers(0, Nkv + 1)) if i % 3 == 0 else Nkv
    CASES.append((i, int(_rng.integers(1, 3)), Nq, Nkv, int(_rng.integers(1, 4)), D, kvl, layout,
                  torch.bfloat16 if i % 5 == 0 else torch.float32))


@pytest.mark.parametrize("i,B,Nq,Nkv,H,D,kvl,layout,out_dtype", CASES)
def test_attention_fuzz(dl, i, B, Nq, Nkv, H, D, kvl, layout, out_dtype):
    q, k, v = _views(B, Nq, Nkv, H, D, layout, 500 + i)
    O, L = dl.attn_fwd(q, k, v, key_valid_len=kvl, out_dtype=out_dtype)
    torch.cuda.synchronize()
    Or, Lr = oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=kvl)
    compare(O.double().permute(0, 2, 1, 3).cpu().numpy(), L.double().cpu().numpy(), Or.transpose(0, 2, 1, 3), Lr)


@pytest.mark.parametrize("i", range(6))
def test_fp8_and_masked_fuzz(dl, i):
    rng = np.random.default_rng(77 + i)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 3))
    N = int(rng.choice([130, 257, 600, 1024]))
    kvl = int(rng.integers(1, N + 1))
    # FP8 on a stacked buffer
    qkv8 = wl.randn_e4m3((B, N, 3, H, 128), 900 + i, 64.0, DEV)
    q8, k8, v8 = dl.split_stacked_fp8(qkv8)
    d = 1.0 / 64
    O8, L8 = dl.attn_fwd_fp8(q8, k8, v8, (d, d, d), key_valid_len=kvl)
    # general mask on bf16 views, mask rows fewer than the queries
    D = int(rng.choice([64, 128]))
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed=950 + i, device=DEV)
    rows = int(rng.integers(0, N + 1))
    m = torch.rand((B, max(rows, 1), kvl), generator=torch.Generator().manual_seed(i)) < float(rng.uniform(0.02, 0.9))
    bits = wl.pack_mask_bits(m).to(DEV)
    Om, Lm = dl.attn_fwd_masked(q, k, v, bits, mask_rows=rows, key_valid_len=kvl)
    torch.cuda.synchronize()
    codes = host_u8(qkv8)
    Or8, Lr8 = oracle.attn_fp8(codes[:, :, 0], codes[:, :, 1], codes[:, :, 2], scale=128 ** -0.5, descale_q=d,
                               descale_k=d, descale_v=d, key_valid_len=kvl)
    vmax = float(oracle.e4m3_decode(np.array([int((codes[:, :, 2] & 0x7F).max())], dtype=np.uint8))[0]) * d
    compare_fp8(O8.double().permute(0, 2, 1, 3).cpu().numpy(), L8.double().cpu().numpy(), Or8.transpose(0, 2, 1, 3),
                Lr8, vmax)
    allow = np.ones((B, N, kvl), dtype=bool)
    allow[:, :rows] = m.numpy()[:, :rows]
    Orm, Lrm = oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=kvl, allow=allow)
    compare(Om.double().permute(0, 2, 1, 3).cpu().numpy(), Lm.double().cpu().numpy(), Orm.transpose(0, 2, 1, 3), Lrm)

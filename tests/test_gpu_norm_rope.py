"""GPU parity of dit_qkv_norm_rope_to_head_major against the oracle.

Tolerance from the arithmetic: the kernel computes in fp32 and rounds to bf16
once, so |out - ref| <= 2^-9 |ref| (the rounding) + a few fp32 ulps of the
pair's magnitude (rsqrt, the products of the rotation); gated at
2^-8 |ref| + 2^-16 * (largest |y| of the row).  Most elements must round to
the same bf16 as the fp64 value; V must be bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from dit_long_sequence_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def dl():
    import dit_long_sequence_gb300 as m
    return m


def _check(out, ref, row_axis=-1):
    got = out.to(torch.float64).cpu().numpy()
    scale = np.abs(ref).max(axis=row_axis, keepdims=True)
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -16 * scale
    assert (err <= bound).all(), (err.max(), np.argwhere(err > bound)[:5])
    rn = torch.from_numpy(ref).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.mean(got == rn) > 0.98, np.mean(got == rn)


@pytest.mark.parametrize("B,N,H,D,pad,grid", [(2, 37, 3, 64, 0, None), (1, 300, 2, 128, 24, (3, 10, 10)),
                                              (1, 129, 4, 128, 0, None), (2, 64, 1, 64, 8, (4, 4, 4))])
def test_matches_oracle(dl, B, N, H, D, pad, grid):
    g = wl.generator(DEV, 21 + N)
    full = torch.randn((B, N, 3 * H * D + pad), generator=g, device=DEV).mul_(3.0).to(torch.bfloat16)
    qkv = full[:, :, :3 * H * D].view(B, N, 3, H, D)
    wq = torch.rand((D,), generator=g, device=DEV) + 0.5
    wk = torch.rand((D,), generator=g, device=DEV) + 0.5
    if grid is None:
        ang = torch.rand((N, D // 2), generator=g, device=DEV, dtype=torch.float64) * 100.0
        cos, sin = ang.cos().float(), ang.sin().float()
    else:
        cos, sin = wl.rope_tables_3d(grid, D, device=DEV)
    q, k, v = dl.qkv_norm_rope_to_head_major(qkv, q_weight=wq, k_weight=wk, eps=1e-6, rope_cos=cos, rope_sin=sin)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.qkv_norm_rope_to_head_major(wl.host_bf16_bits(qkv), wq.cpu().numpy(), wk.cpu().numpy(),
                                                    1e-6, cos.cpu().numpy(), sin.cpu().numpy())
    _check(q, rq)
    _check(k, rk)
    assert np.array_equal(v.to(torch.float64).cpu().numpy(), rv)


def test_each_step_can_be_skipped(dl):
    B, N, H, D = 1, 70, 2, 128
    qkv = wl.randn_bf16((B, N, 3, H, D), 5, DEV)
    cos, sin = wl.rope_tables_3d((2, 5, 7), D, device=DEV)
    w = torch.ones((D,), device=DEV)
    bits = wl.host_bf16_bits(qkv)
    # nothing applied: the plain split, bit for bit
    outs = dl.qkv_norm_rope_to_head_major(qkv)
    plain = dl.qkv_to_head_major(qkv)
    torch.cuda.synchronize()
    for a, b in zip(outs, plain):
        assert torch.equal(a, b)
    # rotation only (q), norm only (k): compare each with the oracle
    q, k, _ = dl.qkv_norm_rope_to_head_major(qkv, k_weight=w, rope_cos=cos, rope_sin=sin)
    torch.cuda.synchronize()
    rq, rk, _ = oracle.qkv_norm_rope_to_head_major(bits, None, np.ones(D), 1e-6, cos.cpu().numpy(), sin.cpu().numpy())
    _check(q, rq)
    _check(k, rk)


def test_ltx_sized_sampled_rows(dl):
    """LTX-2-shaped buffer (24,576 tokens = a 16 x 32 x 48 latent grid, 32 heads)
    with 3-D rotary tables; sampled sequence rows of every head."""
    B, N, H, D = 1, 24576, 32, 128
    qkv = wl.randn_bf16((B, N, 3, H, D), 1, DEV)
    cos, sin = wl.rope_tables_3d((16, 32, 48), D, device=DEV)
    g = wl.generator(DEV, 9)
    wq = torch.rand((D,), generator=g, device=DEV) + 0.5
    wk = torch.rand((D,), generator=g, device=DEV) + 0.5
    q, k, v = dl.qkv_norm_rope_to_head_major(qkv, q_weight=wq, k_weight=wk, rope_cos=cos, rope_sin=sin)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(3).choice(N, 256, replace=False))
    rows[0], rows[-1] = 0, N - 1
    idx = torch.as_tensor(rows, device=DEV)
    sub = qkv[:, idx].contiguous()
    rq, rk, rv = oracle.qkv_norm_rope_to_head_major(wl.host_bf16_bits(sub), wq.cpu().numpy(), wk.cpu().numpy(),
                                                    1e-6, cos[idx].cpu().numpy(), sin[idx].cpu().numpy())
    _check(q[:, :, idx], rq)
    _check(k[:, :, idx], rk)
    assert np.array_equal(v[:, :, idx].to(torch.float64).cpu().numpy(), rv)

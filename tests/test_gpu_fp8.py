"""GPU parity of the FP8 path: the one-pass E4M3 cast of a stacked QKV buffer
(bit-exact against the oracle's codec) and FP8 attention on its output
(against the fp64 oracle on the same E4M3 codes, with the tolerance derived in
tests/parity.py from E4M3's rounding of the probabilities)."""
import numpy as np
import pytest
import torch

import oracle
from dit_long_sequence_gb300 import workloads as wl

from parity import compare_fp8, gather_rows, host_u8

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def dl():
    import dit_long_sequence_gb300 as m
    return m


def _bits(t):
    return wl.host_bf16_bits(t)


def _absmax(codes) -> float:
    """Largest |value| among E4M3 codes: the magnitude is monotonic in the low 7 bits."""
    return float(oracle.e4m3_decode(np.array([int((np.asarray(codes) & 0x7F).max())], dtype=np.uint8))[0])


@pytest.mark.parametrize("B,N,H,D,pad", [(2, 37, 3, 32, 0), (1, 300, 2, 128, 16), (3, 5, 1, 16, 48)])
def test_cast_is_bit_exact(dl, B, N, H, D, pad):
    # values spanning subnormals, the normal range and saturation after scaling
    g = wl.generator(DEV, 11 + N)
    mag = torch.exp2(torch.empty((B, N, 3, H, D), device=DEV).uniform_(-14, 11, generator=g))
    sign = torch.where(torch.rand((B, N, 3, H, D), device=DEV, generator=g) < 0.5, -1.0, 1.0)
    full = torch.zeros((B, N, 3 * H * D + pad), dtype=torch.bfloat16, device=DEV)
    full[:, :, :3 * H * D] = (mag * sign).to(torch.bfloat16).reshape(B, N, -1)
    qkv = full[:, :, :3 * H * D].view(B, N, 3, H, D)
    scales = (1.0, 0.37, 3.5)
    out = dl.qkv_cast_fp8(qkv, scales)
    torch.cuda.synchronize()
    ref = oracle.qkv_cast_fp8(_bits(qkv), scales)
    got = out.cpu().numpy()
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]
    # saturation and zeros really occur in this input
    assert (got & 0x7F == 0x7E).any() and (got & 0x7F == 0).any()


def test_cast_bit_exact_at_full_size_sampled_rows(dl):
    w = wl.WORKLOADS["ltx2_padded"]
    buf = wl.randn_bf16((w.B, w.N, 3, w.H, w.D), w.seed, DEV)
    scales = (64.0, 64.0, 48.0)
    out = dl.qkv_cast_fp8(buf, scales)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(5).choice(w.N, 384, replace=False))
    rows[0], rows[-1] = 0, w.N - 1
    idx = torch.as_tensor(rows, device=DEV)
    ref = oracle.qkv_cast_fp8(_bits(buf[:, idx].contiguous()), scales)
    assert np.array_equal(out[:, idx].cpu().numpy(), ref)


def _stacked_case(B, N, H, D, seed, ramp=0.0):
    g = wl.generator(DEV, seed)
    x = torch.randn((B, N, 3, H, D), device=DEV, generator=g)
    if ramp:
        # key magnitudes grow along the sequence: later key tiles raise the row max
        x[:, :, 1] *= (1.0 + ramp * torch.arange(N, device=DEV, dtype=torch.float32) / N)[None, :, None, None]
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("B,N,H,kvl,out_dtype", [
    (1, 300, 2, None, torch.float32),
    (2, 513, 3, 400, torch.float32),
    (1, 1000, 1, 1, torch.float32),
    (1, 128, 2, None, torch.bfloat16),
    (1, 777, 2, 129, torch.bfloat16),
    (1, 2048, 2, 2000, torch.float32),
])
def test_fp8_attention_on_cast_output(dl, B, N, H, kvl, out_dtype):
    D = 128
    buf = _stacked_case(B, N, H, D, seed=100 + N)
    amax = [float(buf[:, :, t].abs().max()) for t in range(3)]
    scales = tuple(448.0 / a for a in amax)
    desc = tuple(1.0 / s for s in scales)
    qkv8 = dl.qkv_cast_fp8(buf, scales)
    q8, k8, v8 = dl.split_stacked_fp8(qkv8)
    O, L = dl.attn_fwd_fp8(q8, k8, v8, desc, key_valid_len=kvl, out_dtype=out_dtype)
    torch.cuda.synchronize()
    # the oracle casts the same bf16 bits with its own codec
    codes = oracle.qkv_cast_fp8(_bits(buf), scales)
    assert np.array_equal(codes, qkv8.cpu().numpy())
    Oref, Lref = oracle.attn_fp8(codes[:, :, 0], codes[:, :, 1], codes[:, :, 2], scale=D ** -0.5,
                                 descale_q=desc[0], descale_k=desc[1], descale_v=desc[2], key_valid_len=kvl)
    vmax = _absmax(codes[:, :, 2]) * desc[2]
    compare_fp8(O.to(torch.float64).permute(0, 2, 1, 3).cpu().numpy(), L.double().cpu().numpy(),
                Oref.transpose(0, 2, 1, 3), Lref, vmax)


def test_fp8_rescale_paths(dl):
    """Scores that keep growing along the keys make the running max move by more
    than the stale margin in later tiles, exercising the O rescale."""
    B, N, H, D = 1, 1536, 2, 128
    buf = _stacked_case(B, N, H, D, seed=7, ramp=3.0)
    scales = tuple(448.0 / float(buf[:, :, t].abs().max()) for t in range(3))
    desc = tuple(1.0 / s for s in scales)
    qkv8 = dl.qkv_cast_fp8(buf, scales)
    q8, k8, v8 = dl.split_stacked_fp8(qkv8)
    sc = 4.0 * D ** -0.5   # sharper softmax: jumps of several units in log2
    O, L = dl.attn_fwd_fp8(q8, k8, v8, desc, scale=sc)
    torch.cuda.synchronize()
    codes = oracle.qkv_cast_fp8(_bits(buf), scales)
    Oref, Lref = oracle.attn_fp8(codes[:, :, 0], codes[:, :, 1], codes[:, :, 2], scale=sc, descale_q=desc[0],
                                 descale_k=desc[1], descale_v=desc[2])
    vmax = _absmax(codes[:, :, 2]) * desc[2]
    compare_fp8(O.double().permute(0, 2, 1, 3).cpu().numpy(), L.double().cpu().numpy(), Oref.transpose(0, 2, 1, 3),
                Lref, vmax)


def test_fp8_zero_valid_keys_and_strided_output(dl):
    B, N, H, D = 1, 300, 2, 128
    qkv8 = wl.randn_e4m3((B, N, 3, H, D), 3, 64.0, DEV)
    q8, k8, v8 = dl.split_stacked_fp8(qkv8)
    O, L = dl.attn_fwd_fp8(q8, k8, v8, (1 / 64, 1 / 64, 1 / 64), key_valid_len=0)
    torch.cuda.synchronize()
    assert torch.all(O == 0) and torch.all(torch.isneginf(L))
    # output written through strides into a wider buffer, bf16
    wide = torch.full((B, N, H, 2 * D), 7.0, dtype=torch.bfloat16, device=DEV)
    O2, L2 = dl.attn_fwd_fp8(q8, k8, v8, (1 / 64, 1 / 64, 1 / 64), out=wide[..., :D], key_valid_len=250)
    torch.cuda.synchronize()
    assert torch.all(wide[..., D:] == 7.0)
    Oref, Lref = oracle.attn_fp8(*(host_u8(t) for t in (q8, k8, v8)), scale=D ** -0.5, descale_q=1 / 64,
                                 descale_k=1 / 64, descale_v=1 / 64, key_valid_len=250)
    vmax = _absmax(host_u8(v8)) / 64
    compare_fp8(O2.double().permute(0, 2, 1, 3).cpu().numpy(), L2.double().cpu().numpy(),
                Oref.transpose(0, 2, 1, 3), Lref, vmax)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["ltx2_padded", "wan22_a14b"])
def test_fp8_attention_sampled_rows_full_size(dl, name):
    w = wl.WORKLOADS[name]
    qkv8 = wl.randn_e4m3((w.B, w.N, 3, w.H, w.D), w.seed, 64.0, DEV)
    q8, k8, v8 = dl.split_stacked_fp8(qkv8)
    d = 1.0 / 64
    # the benchmark's call: the last partial wave of work items split over key ranges
    O, L = dl.attn_fwd_fp8_ws(q8, k8, v8, (d, d, d), key_valid_len=w.key_valid_len)
    torch.cuda.synchronize()
    rows = wl.sample_rows(w.B, w.H, w.N, 12, w.seed, must=(w.kv_len - 1, w.kv_len))
    codes = qkv8.cpu().numpy()
    Oref, Lref = oracle.attn_fp8(codes[:, :, 0], codes[:, :, 1], codes[:, :, 2], scale=w.scale, descale_q=d,
                                 descale_k=d, descale_v=d, key_valid_len=w.key_valid_len, rows=rows)
    Os, Ls = gather_rows(O, L, rows)
    vmax = _absmax(codes[:, :, 2]) * d
    compare_fp8(Os, Ls, Oref, Lref, vmax)


@pytest.mark.parametrize("Nq,Nkv,kvl", [(300, 77, None), (513, 2048, 1999), (129, 129, 128)])
def test_fp8_cross_attention_on_separate_tensors(dl, Nq, Nkv, kvl):
    """Separate (non-stacked) E4M3 tensors, Nq != Nkv, padded row strides."""
    B, H, D = 2, 2, 128
    g = 60 + Nq
    q8 = wl.randn_e4m3((B, Nq, H, D + 16), g, 64.0, DEV)[..., :D]
    k8 = wl.randn_e4m3((B, Nkv, H, D), g + 1, 64.0, DEV)
    v8 = wl.randn_e4m3((B, Nkv, H, D), g + 2, 64.0, DEV)
    d = 1.0 / 64
    O, L = dl.attn_fwd_fp8(q8, k8, v8, (d, d, d), key_valid_len=kvl)
    torch.cuda.synchronize()
    Oref, Lref = oracle.attn_fp8(host_u8(q8), host_u8(k8), host_u8(v8), scale=D ** -0.5, descale_q=d,
                                 descale_k=d, descale_v=d, key_valid_len=kvl)
    vmax = _absmax(host_u8(v8)) * d
    compare_fp8(O.double().permute(0, 2, 1, 3).cpu().numpy(), L.double().cpu().numpy(),
                Oref.transpose(0, 2, 1, 3), Lref, vmax)


def test_fp8_attention_sinks_and_long_tails(dl):
    """Rows whose scores have four dominant keys (attention sinks) over thousands
    of small ones: each sink sits ~13 units above a typical key in log2 terms, so
    the sinks hold most of each row's mass (~70%) and the tail, at P ~2^-6 of the
    row max, the rest -- which E4M3 must carry within the derived tolerance (the
    mass split is asserted from the oracle's decoded inputs)."""
    B, N, H, D = 1, 4096, 2, 128
    g = wl.generator(DEV, 77)
    x = torch.randn((B, N, 3, H, D), device=DEV, generator=g)
    direction = torch.randn((D,), device=DEV, generator=g)
    direction = direction / direction.norm()
    x[:, :, 0] += 4.0 * direction                     # every query leans towards `direction`
    x[:, :, 1, :, :] -= (x[:, :, 1] @ direction)[..., None] * direction   # keys orthogonal to it ...
    x[:, 100:104, 1] += 24.0 * direction              # ... except four sinks
    buf = x.to(torch.bfloat16)
    scales = tuple(448.0 / float(buf[:, :, t].abs().max()) for t in range(3))
    desc = tuple(1.0 / sc for sc in scales)
    qkv8 = dl.qkv_cast_fp8(buf, scales)
    O, L = dl.attn_fwd_fp8(*dl.split_stacked_fp8(qkv8), desc)
    torch.cuda.synchronize()
    codes = oracle.qkv_cast_fp8(_bits(buf), scales)
    Oref, Lref = oracle.attn_fp8(codes[:, :, 0], codes[:, :, 1], codes[:, :, 2], scale=D ** -0.5,
                                 descale_q=desc[0], descale_k=desc[1], descale_v=desc[2])
    # the mass split this case is about: sinks hold most, the tail a large share
    qd = oracle.e4m3_decode(codes[0, :64, 0, 0]) * desc[0]
    kd = oracle.e4m3_decode(codes[0, :, 1, 0]) * desc[1]
    sc = (qd @ kd.T) * D ** -0.5
    w = np.exp(sc - sc.max(axis=1, keepdims=True))
    sink_share = w[:, 100:104].sum(1) / w.sum(1)
    assert 0.3 < np.median(sink_share) < 0.97, np.median(sink_share)
    vmax = _absmax(codes[:, :, 2]) * desc[2]
    compare_fp8(O.double().permute(0, 2, 1, 3).cpu().numpy(), L.double().cpu().numpy(), Oref.transpose(0, 2, 1, 3),
                Lref, vmax)

"""GPU parity of dit_attn_lse_merge and dit_qkv_to_head_major (through the C ABI).

Merge: seeded synthetic partials (including -inf chunks and all -inf rows)
against the oracle's fp64 merge; chunked attention + merge against the oracle's
single pass (the identity "merged partials equal one global pass"); and the
ring-style workload: keys in 9 chunks, 9 attention calls + one merge, against
the oracle on sampled rows and against the GPU single pass.
Layout: bit-exact against the oracle's index identity, strided inputs included.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from dit_long_sequence_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _dev():
    return torch.device("cuda:0")


def _dl():
    import dit_long_sequence_gb300 as dl
    return dl


def _partials(n, B, Nq, H, D, seed, empty_frac=0.1):
    g = wl.generator(_dev(), seed)
    o = torch.randn(n, B, Nq, H, D, generator=g, device=_dev())
    l = 3.0 * torch.randn(n, B, H, Nq, generator=g, device=_dev()) + 8.0
    drop = torch.rand(n, B, H, Nq, generator=g, device=_dev()) < empty_frac
    l[drop] = float("-inf")
    if Nq > 3:
        l[:, :, 0, 3] = float("-inf")   # one row with every chunk empty
    o[drop.permute(0, 1, 3, 2).unsqueeze(-1).expand_as(o)] = float("nan")   # never read
    return o, l


@pytest.mark.parametrize("n,B,Nq,H,D", [(1, 1, 100, 2, 128), (2, 2, 257, 3, 64), (3, 1, 300, 5, 128),
                                        (9, 1, 129, 4, 128)])
def test_merge_matches_oracle(n, B, Nq, H, D):
    o, l = _partials(n, B, Nq, H, D, seed=20 + n)
    O, L = _dl().lse_merge(o, l)
    Ob, Lb = _dl().lse_merge(o, l, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    Or, Lr = oracle.lse_merge(o.double().cpu().numpy(), l.double().cpu().numpy())
    Og, Lg = O.double().cpu().numpy(), L.double().cpu().numpy()
    assert np.array_equal(np.isneginf(Lg), np.isneginf(Lr))
    fin = np.isfinite(Lr)
    assert np.abs(Lg[fin] - Lr[fin]).max() <= 1e-5
    assert np.isfinite(Og).all()
    assert np.abs(Og - Or).max() <= 1e-5
    assert np.abs(Ob.double().cpu().numpy() - Or).max() <= 2e-2 * max(1.0, np.abs(Or).max())
    assert torch.equal(L, Lb)


@pytest.mark.parametrize("n,B,Nq,H,D", [(9, 1, 200, 4, 128), (3, 2, 130, 3, 64)])
def test_merge_interleaved_layout(n, B, Nq, H, D):
    # chunks interleaved per row: a [B, Nq, H, n, D] buffer seen as [n, B, Nq, H, D]
    o, l = _partials(n, B, Nq, H, D, seed=50 + n)
    buf = o.permute(1, 2, 3, 0, 4).contiguous()
    o_il = buf.permute(3, 0, 1, 2, 4)
    assert o_il.stride(3) == n * D and o_il.stride(0) == D
    O, L = _dl().lse_merge(o_il, l)
    O2, L2 = _dl().lse_merge(o, l)
    torch.cuda.synchronize()
    Or, Lr = oracle.lse_merge(o.double().cpu().numpy(), l.double().cpu().numpy())
    assert torch.equal(O, O2) and torch.equal(L, L2), "layouts disagree"
    assert np.abs(O.double().cpu().numpy() - Or).max() <= 1e-5


def test_chunked_attention_merge_equals_single_pass():
    B, N, H, D = 1, 900, 2, 128
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed=30, device=_dev())
    bounds = [0, 128, 300, 301, 640, 900]
    n = len(bounds) - 1
    o_parts = torch.empty(n, B, N, H, D, device=_dev())
    l_parts = torch.empty(n, B, H, N, device=_dev())
    for c in range(n):
        lo, hi = bounds[c], bounds[c + 1]
        _dl().attn_fwd(q, k[:, lo:hi], v[:, lo:hi], out=o_parts[c], lse=l_parts[c])
    O, L = _dl().lse_merge(o_parts, l_parts)
    O1, L1 = _dl().attn_fwd(q, k, v)
    torch.cuda.synchronize()
    Or, Lr = parity.oracle_full(q, k, v)
    parity.compare(O.double().cpu().numpy(), L.double().cpu().numpy(), Or, Lr, head_axes=(0, 2))
    assert (O - O1).abs().max().item() <= 2e-3
    assert (L - L1).abs().max().item() <= 1e-4


def test_ring9_workload_chunked_vs_oracle_and_single_pass():
    # the benchmark's ring-9 step: 9 chunk calls through dit_attn_fwd_ws (each
    # chunk's last partial wave of work items split over key ranges); the
    # attention writes each chunk's O straight into a per-row interleaved
    # [B, N, H, n, D] buffer through its output strides; the merge reads it back
    w = wl.WORKLOADS["ring9"]
    q, k, v, _ = wl.make_workload_inputs(w, device=_dev())
    n = w.kv_chunks
    cl = w.N // n
    o_buf = torch.empty(w.B, w.N, w.H, n, w.D, device=_dev())
    l_parts = torch.empty(n, w.B, w.H, w.N, device=_dev())
    for c in range(n):
        _dl().attn_fwd_ws(q, k[:, c * cl:(c + 1) * cl], v[:, c * cl:(c + 1) * cl], out=o_buf[:, :, :, c],
                          lse=l_parts[c])
    O, L = _dl().lse_merge(o_buf.permute(3, 0, 1, 2, 4), l_parts)
    del o_buf, l_parts
    O1, L1 = _dl().attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert (O - O1).abs().max().item() <= 2e-3
    assert (L - L1).abs().max().item() <= 1e-4
    rows = wl.sample_rows(w.B, w.H, w.N, 1024, seed=w.seed, must=[cl - 1, cl, w.N - 1])
    Og, Lg = parity.gather_rows(O, L, rows)
    Or, Lr = parity.oracle_rows(q, k, v, rows)
    parity.compare(Og, Lg, Or, Lr, head_axes=(0, 1))


@pytest.mark.parametrize("B,N,H,D,pad_n,pad_b", [(1, 5, 3, 8, 0, 0), (2, 37, 4, 64, 0, 0),
                                                 (2, 130, 16, 128, 24, 64), (1, 1, 1, 8, 0, 0)])
def test_layout_bit_exact(B, N, H, D, pad_n, pad_b):
    row = 3 * H * D + pad_n
    flat = torch.randint(-32768, 32767, (B * (N * row + pad_b),), dtype=torch.int32,
                         generator=wl.generator("cpu", 40 + N)).to(torch.int16)
    flat = flat.to(_dev())
    qkv = flat.view(torch.bfloat16).as_strided((B, N, 3, H, D), (N * row + pad_b, row, H * D, D, 1))
    outs = _dl().qkv_to_head_major(qkv)
    torch.cuda.synchronize()
    host = flat.cpu().numpy().view(np.uint16)
    ref_in = np.lib.stride_tricks.as_strided(host, shape=(B, N, 3, H, D),
                                             strides=tuple(2 * s for s in (N * row + pad_b, row, H * D, D, 1)))
    refs = oracle.qkv_to_head_major(ref_in)
    for t in range(3):
        got = outs[t].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, refs[t]), f"plane {t} differs"


def test_layout_cosmos_sized_bit_exact():
    w = wl.WORKLOADS["cosmos3_nano"]
    _, _, _, buf = wl.make_workload_inputs(w, device=_dev())
    outs = _dl().qkv_to_head_major(buf)
    torch.cuda.synchronize()
    refs = oracle.qkv_to_head_major(wl.host_bf16_bits(buf))
    for t in range(3):
        got = wl.host_bf16_bits(outs[t])
        assert np.array_equal(got, refs[t]), f"plane {t} differs"

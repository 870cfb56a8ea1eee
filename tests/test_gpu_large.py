"""Attention at a size whose output has more than 2^31 elements.

B = 1, N = 270,000 tokens (the last key tile ragged), H = 64, D = 128: O holds
2.21e9 fp32 elements, so every row past 262,144 sits beyond a 32-bit element
offset, and the grid's last partial wave is split over key ranges.  The bf16
call runs in the benchmark's launch configuration (the workspace form); the FP8
call runs on E4M3 inputs of the same shape.  Sampled rows (among them the last
ones and those on either side of the 2^31 boundary) of the first and the last
head are compared with the fp64 oracle against all keys.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from dit_long_sequence_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
N, H, D = 270_000, 64, 128
HEADS = [0, H - 1]


@pytest.fixture(scope="module")
def dl():
    import dit_long_sequence_gb300 as m
    return m


def _rows(seed):
    fixed = [0, 1, 131_071, 262_143, 262_144, 262_145, 266_000, N - 129, N - 128, N - 2, N - 1]
    extra = np.random.default_rng(seed).choice(N, 37, replace=False)
    r = np.unique(np.concatenate([fixed, extra]))
    return np.broadcast_to(r, (1, len(HEADS), len(r))).copy()


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_bf16_attention_beyond_32_bit_offsets(dl):
    q, k, v, _ = wl.make_qkv(1, N, H, D, seed=70, device=DEV)
    O, L = dl.attn_fwd_ws(q, k, v)
    torch.cuda.synchronize()
    assert O.numel() > 2 ** 31
    assert dl.attn_fwd_workspace_bytes(1, N, H, D, N) > 0     # the split is in the timed form too
    rows = _rows(70)
    qh, kh, vh = (t[:, :, HEADS].contiguous() for t in (q, k, v))
    Os, Ls = parity.gather_rows(O[:, :, HEADS], L[:, HEADS], rows)
    del q, k, v, O, L
    _free()
    Or, Lr = parity.oracle_rows(qh, kh, vh, rows)
    parity.compare(Os, Ls, Or, Lr)
    rc, info = dl.check_watchdog()
    assert rc == 0, info


def test_fp8_attention_beyond_32_bit_offsets(dl):
    qkv8 = wl.randn_e4m3((1, N, 3, H, D), 71, 64.0, DEV)
    q8, k8, v8 = dl.split_stacked_fp8(qkv8)
    d = 1.0 / 64
    O, L = dl.attn_fwd_fp8_ws(q8, k8, v8, (d, d, d))
    torch.cuda.synchronize()
    assert O.numel() > 2 ** 31
    rows = _rows(71)
    codes = qkv8[:, :, :, HEADS].cpu().numpy()          # [1, N, 3, 2, D]
    Os, Ls = parity.gather_rows(O[:, :, HEADS], L[:, HEADS], rows)
    del qkv8, q8, k8, v8, O, L
    _free()
    Oref, Lref = oracle.attn_fp8(codes[:, :, 0], codes[:, :, 1], codes[:, :, 2], scale=D ** -0.5, descale_q=d,
                                 descale_k=d, descale_v=d, rows=rows)
    vmax = float(oracle.e4m3_decode(np.array([int((codes[:, :, 2] & 0x7F).max())], dtype=np.uint8))[0]) * d
    parity.compare_fp8(Os, Ls, Oref, Lref, vmax)
    rc, info = dl.check_watchdog()
    assert rc == 0, info

"""Shared helpers for the GPU parity tests: run the oracle on the very bf16
bits the GPU saw, and compare with the stated tolerances.

Tolerances (O in fp32 against the fp64 oracle on identical bf16 inputs):
  O   max-abs <= 2e-2 and mean-abs <= 2e-3;   LSE max-abs <= 1e-3.
Stricter internal gate, because |O| is small at long N with N(0,1) inputs:
  relative L2 error of O per (b, h) <= 1e-2.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dit_long_sequence_gb300 import workloads as wl

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3
O_REL_L2 = 1e-2


def host_bits(t: torch.Tensor) -> np.ndarray:
    return wl.host_bf16_bits(t)


def oracle_full(q, k, v, key_valid_len=None, scale=None):
    return oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=key_valid_len, scale=scale)


def oracle_rows(q, k, v, rows, key_valid_len=None, scale=None):
    return oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=key_valid_len, scale=scale,
                       rows=rows)


def gather_rows(O: torch.Tensor, L: torch.Tensor, rows: np.ndarray):
    """GPU O [B,Nq,H,D], LSE [B,H,Nq] at rows [B,H,R] -> host O [B,H,R,D], LSE [B,H,R]."""
    B, H, R = rows.shape
    idx = torch.as_tensor(rows, device=O.device, dtype=torch.long)
    bi = torch.arange(B, device=O.device)[:, None, None]
    hi = torch.arange(H, device=O.device)[None, :, None]
    Os = O[bi, idx, hi].to(torch.float64).cpu().numpy()
    Ls = L[bi, hi, idx].to(torch.float64).cpu().numpy()
    return Os, Ls


def compare(O_gpu: np.ndarray, L_gpu: np.ndarray, O_ref: np.ndarray, L_ref: np.ndarray, head_axes=(0, 1),
            o_max=O_MAX_ABS, o_mean=O_MEAN_ABS, lse_max=LSE_MAX_ABS, rel_l2=O_REL_L2):
    """Element-wise gates; returns a dict of the measured errors."""
    dO = np.abs(O_gpu - O_ref)
    dL = np.abs(L_gpu - L_ref)
    finite = np.isfinite(L_ref)
    res = {
        "o_max_abs": float(dO.max()) if dO.size else 0.0,
        "o_mean_abs": float(dO.mean()) if dO.size else 0.0,
        "lse_max_abs": float(dL[finite].max()) if finite.any() else 0.0,
    }
    # -inf LSE must match exactly
    assert np.array_equal(np.isneginf(L_gpu), np.isneginf(L_ref)), "LSE -inf pattern differs"
    assert np.isfinite(O_gpu).all(), "non-finite O"
    assert res["o_max_abs"] <= o_max, res
    assert res["o_mean_abs"] <= o_mean, res
    assert res["lse_max_abs"] <= lse_max, res
    if rel_l2 is not None and O_ref.size:
        # per head: O is [B, ..., D] with the head axis given
        num = np.sqrt(((O_gpu - O_ref) ** 2).sum(axis=tuple(a for a in range(O_ref.ndim) if a not in head_axes)))
        den = np.sqrt((O_ref ** 2).sum(axis=tuple(a for a in range(O_ref.ndim) if a not in head_axes)))
        rel = float((num / np.maximum(den, 1e-30)).max())
        res["o_rel_l2"] = rel
        assert rel <= rel_l2, res
    return res

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
    finite = np.isfinite(L_ref)
    dL = np.where(finite, np.abs(np.where(finite, L_gpu, 0.0) - np.where(finite, L_ref, 0.0)), 0.0)
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


# ---------------------------------------------------------------- FP8 path
# The FP8 kernel rounds each probability P to E4M3 before the P.V product
# (relative rounding error |delta| <= 2^-4 for the normal range; P's row max
# is >= 2^7 so subnormal P are >= 2^-16 below it).  LSE and the divisor l come
# from the unrounded fp32 P, so against the fp64 oracle on the same E4M3 inputs
#   e = O - O_ref = sum_j w_j delta_j v_j,   w_j = P_j / sum_k P_k.
# Hard per-element bound: |e| <= 2^-4 * max_j |v_j| (plus 1e-3 for the fp32
# arithmetic).
# Statistical bounds: delta = u / m with u uniform in [-2^-4, 2^-4] (half the
# E4M3 spacing at mantissa m in [1, 2)), so its RMS is
#   sigma = 2^-4 * sqrt(E[1/m^2] / 3) <= 2^-4 / sqrt(3) ~= 0.036
# (m >= 1), and ~0.027 for the near log-uniform mantissas of exponentials.
# With delta zero-mean and independent of v,
#   E[e^2] = sigma^2 * E[sum_j w_j^2 v_j^2],
# and for v drawn independently of the keys' weights E[O_ref^2] has the same
# value, so RMS(e) ~= sigma * RMS(O_ref).  Gates:
#   * per-head relative L2 of O <= 0.04 (sigma ~0.027 with margin);
#   * mean |e| <= 2^-4 / sqrt(3) * RMS(O_ref) + 1e-5: mean |e| <= RMS(e), and
#     the worst-case sigma bounds RMS(e) (1e-5 covers the fp32 arithmetic).
# LSE comes from the unrounded fp32 P: the bf16 gate (1e-3) applies.
FP8_O_REL_L2 = 0.04
FP8_DELTA_RMS_MAX = 2.0 ** -4 / np.sqrt(3.0)


def fp8_o_mean_bound(O_ref: np.ndarray) -> float:
    """The FP8 mean-abs gate on O for this reference (see the derivation above)."""
    rms = float(np.sqrt(np.mean(np.square(O_ref)))) if O_ref.size else 0.0
    return FP8_DELTA_RMS_MAX * rms + 1e-5


def compare_fp8(O_gpu, L_gpu, O_ref, L_ref, v_absmax: float, head_axes=(0, 1)):
    return compare(O_gpu, L_gpu, O_ref, L_ref, head_axes=head_axes, o_max=2.0 ** -4 * v_absmax + 1e-3,
                   o_mean=fp8_o_mean_bound(O_ref), lse_max=LSE_MAX_ABS, rel_l2=FP8_O_REL_L2)


def host_u8(t: torch.Tensor) -> np.ndarray:
    """Host copy of a (possibly strided) uint8 device view, strides kept."""
    if t.device.type == "cpu":
        return t.numpy()
    n = t.untyped_storage().nbytes()
    base = torch.empty(0, dtype=torch.uint8, device=t.device).set_(t.untyped_storage(), 0, (n,), (1,))
    return base.cpu().as_strided(t.shape, t.stride(), t.storage_offset()).numpy()

"""The FP8 parity gates (tests/parity.py) against a model of the kernel's rounding.

The FP8 kernel rounds each probability P = 2^(x - m + 7) to E4M3 before the
P.V product and divides by the row sum of the unrounded P.  A plain torch model
of exactly that rounding (torch's own float8 conversion, exact row max) must
pass compare_fp8 against the oracle; the same model with P rounded to E5M2 (one
mantissa bit fewer, twice the spacing) must fail the mean-abs gate, and a 5%
error in the V descale must fail the gates too.  This checks that the derived
tolerances are neither vacuous nor too tight for the rounding they model.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import FP8_DELTA_RMS_MAX, compare_fp8, fp8_o_mean_bound


def _inputs(B=1, H=2, Nq=192, Nkv=3000, D=128, seed=11):
    g = torch.Generator().manual_seed(seed)
    mk = lambda n: (torch.randn(B, n, H, D, generator=g, dtype=torch.float32) * 64).clamp(-448, 448).to(
        torch.float8_e4m3fn)
    return mk(Nq), mk(Nkv), mk(Nkv)


def _model(q8, k8, v8, dq, dk, dv, scale, p_dtype, kvl):
    """O and LSE with P = 2^(x - m + 7) rounded to p_dtype, the divisor from
    the unrounded P; fp64 everywhere else."""
    Q, K, V = (t.to(torch.float64).permute(0, 2, 1, 3) for t in (q8, k8, v8))
    K, V = K[:, :, :kvl], V[:, :, :kvl]
    x = (scale * dq * dk * math.log2(math.e)) * torch.einsum("bhid,bhjd->bhij", Q, K)
    m = x.amax(-1, keepdim=True)
    P = torch.exp2(x - m + 7.0)
    Pr = P.to(p_dtype).to(torch.float64)
    l = P.sum(-1, keepdim=True)
    O = (Pr @ V) * dv / l
    L = (m.squeeze(-1) + torch.log2(l.squeeze(-1)) - 7.0) * math.log(2.0)
    return O.permute(0, 2, 1, 3).numpy(), L.numpy()


@pytest.fixture(scope="module")
def case():
    q8, k8, v8 = _inputs()
    dq = dk = dv = 1.0 / 64
    scale, kvl = 1.0 / math.sqrt(128), 2900
    u8 = lambda t: t.view(torch.uint8).numpy()
    Oref, Lref = oracle.attn_fp8(u8(q8), u8(k8), u8(v8), scale=scale, descale_q=dq, descale_k=dk, descale_v=dv,
                                 key_valid_len=kvl)
    vmax = float(v8.to(torch.float64)[:, :kvl].abs().max()) * dv
    return q8, k8, v8, dq, dk, dv, scale, kvl, Oref, Lref, vmax


def test_e4m3_rounding_model_passes_the_gates(case):
    q8, k8, v8, dq, dk, dv, scale, kvl, Oref, Lref, vmax = case
    O, L = _model(q8, k8, v8, dq, dk, dv, scale, torch.float8_e4m3fn, kvl)
    res = compare_fp8(O, L, Oref, Lref, vmax, head_axes=(0, 2))
    rms = float(np.sqrt(np.mean(Oref ** 2)))
    # the model's error sits near the expected ~0.8 * 0.027 * RMS(O), under the gate
    assert 0.01 * rms < res["o_mean_abs"] < 0.8 * FP8_DELTA_RMS_MAX * rms, res


def test_coarser_p_rounding_fails_the_mean_abs_gate(case):
    q8, k8, v8, dq, dk, dv, scale, kvl, Oref, Lref, vmax = case
    O, L = _model(q8, k8, v8, dq, dk, dv, scale, torch.float8_e5m2, kvl)
    assert float(np.abs(O - Oref).mean()) > fp8_o_mean_bound(Oref)
    with pytest.raises(AssertionError):
        compare_fp8(O, L, Oref, Lref, vmax, head_axes=(0, 2))


def test_wrong_v_descale_fails(case):
    q8, k8, v8, dq, dk, dv, scale, kvl, Oref, Lref, vmax = case
    O, L = _model(q8, k8, v8, dq, dk, dv * 1.05, scale, torch.float8_e4m3fn, kvl)
    with pytest.raises(AssertionError):
        compare_fp8(O, L, Oref, Lref, vmax, head_axes=(0, 2))

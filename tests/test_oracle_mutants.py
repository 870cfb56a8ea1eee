"""The oracle's pins catch planted mistakes.

Each case copies the C oracle's source, plants one plausible slip in the copy
(on the CPU, in a temporary directory), compiles it and runs a compact pin
suite -- brute force, torch's fp64 SDPA, closed forms, the mask and fused-view
checks -- against the mutant.  The real oracle passes the suite; every mutant
must fail it.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from dit_long_sequence_gb300 import workloads as wl

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "dropped_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "lse_without_max": ("lse_out[r] = m + log(l);", "lse_out[r] = log(l);"),
    "k_used_as_v": ("const float *vj = vh + (int64_t)j * D;", "const float *vj = kh + (int64_t)j * D;"),
    "mask_off_by_one": ("const int nj = key_valid_len;",
                        "const int nj = key_valid_len < Nkv ? key_valid_len + 1 : key_valid_len;"),
    "no_normalisation": ("o_out[(int64_t)r * D + d] = acc[d] / l;", "o_out[(int64_t)r * D + d] = acc[d];"),
    "swapped_k_strides": ("(int64_t)j * k_s[1] + (int64_t)h * k_s[2]",
                          "(int64_t)j * k_s[2] + (int64_t)h * k_s[1]"),
    "exponent_sign": ("const double p = exp(s[j] - m);", "const double p = exp(m - s[j]);"),
    "channel_index_slip": ("dot += qd[d] * (double)kj[d];", "dot += qd[d] * (double)kj[(d + 1) % D];"),
    "log2_instead_of_ln": ("lse_out[r] = m + log(l);", "lse_out[r] = m + log2(l);"),
    "allow_mask_ignored": ("if (al && !al[j]) { s[j] = -INFINITY; continue; }", "if (0) { continue; }"),
    "allow_mask_inverted": ("if (al && !al[j])", "if (al && al[j])"),
    "allow_mask_wrong_row": ("(int64_t)i * allow_si", "(int64_t)(i + 1 < Nq ? i + 1 : i) * allow_si"),
    "empty_row_not_zero": ("if (m == -INFINITY) {          /* no allowed key */", "if (0) {"),
}


def _pin_suite(lib):
    """Returns the names of the pins that fail for the given compiled oracle."""
    failures = []

    def bits(t):
        return wl.bf16_bits(t.contiguous())

    # library special case: fp64 SDPA with a key mask, fused strided views
    B, N, H, D = 1, 40, 2, 64
    q, k, v, buf = wl.make_qkv(B, N, H, D, seed=21, fused=True)
    kvl, scale = 29, 0.125
    raw = wl.bf16_bits(buf)
    try:
        O, L = oracle.attn(raw[:, :, 0], raw[:, :, 1], raw[:, :, 2], key_valid_len=kvl,
                           scale=scale, lib=lib)
    except Exception:
        return ["raised"]
    qt, kt, vt = (x.to(torch.float64).permute(0, 2, 1, 3) for x in (q, k, v))
    mask = torch.zeros(1, N, dtype=torch.bool)
    mask[:, :kvl] = True
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    lref = torch.logsumexp(scale * torch.einsum("bhid,bhjd->bhij", qt, kt[:, :, :kvl]), -1)
    if not (np.allclose(O, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
            and np.allclose(L, lref.numpy(), rtol=0, atol=1e-12)):
        failures.append("sdpa_fp64")

    # library special case: a general boolean mask (fp64 SDPA), one row fully masked
    g = torch.Generator().manual_seed(5)
    Bm, Nm, Hm, Dm = 2, 24, 2, 32
    qm, km, vm, _ = wl.make_qkv(Bm, Nm, Hm, Dm, seed=33)
    allow = torch.rand((Bm, Nm, Nm), generator=g) < 0.4
    allow[:, :, 0] = True
    allow[1, 5, :] = False
    try:
        Om, Lm = oracle.attn(bits(qm), bits(km), bits(vm), scale=0.2, allow=allow.numpy(), lib=lib)
    except Exception:
        return failures + ["raised_mask"]
    qt, kt, vt = (x.to(torch.float64).permute(0, 2, 1, 3) for x in (qm, km, vm))
    am = allow[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=am, scale=0.2)
    s_ = 0.2 * torch.einsum("bhid,bhjd->bhij", qt, kt)
    lref = torch.logsumexp(s_.masked_fill(~am, -float("inf")), -1)
    ref = ref.permute(0, 2, 1, 3).numpy()
    ok_rows = np.ones((Bm, Nm), dtype=bool)
    ok_rows[1, 5] = False
    if not (np.allclose(Om[ok_rows], ref[ok_rows], rtol=0, atol=1e-12)
            and np.allclose(Lm.transpose(0, 2, 1)[ok_rows], lref.permute(0, 2, 1).numpy()[ok_rows], rtol=0,
                            atol=1e-12)
            and np.all(Om[1, 5] == 0) and np.all(np.isneginf(Lm[1, :, 5]))):
        failures.append("sdpa_fp64_general_mask")

    # closed form: weights 1:2:4 -> O = (5, 6), LSE = ln 7
    def exact(arr):
        return torch.tensor(arr, dtype=torch.float64).to(torch.bfloat16)
    q1 = exact([[[[1.0, 0.0]]]])
    k1 = exact([[[[0.0, 0.0]], [[1.0, 0.0]], [[2.0, 0.0]]]])
    v1 = exact([[[[7.0, 0.0]], [[0.0, 7.0]], [[7.0, 7.0]]]])
    O, L = oracle.attn(bits(q1), bits(k1), bits(v1), scale=math.log(2.0), lib=lib)
    if not (np.allclose(O[0, 0, 0], [5.0, 6.0], atol=1e-12) and abs(L[0, 0, 0] - math.log(7.0)) < 1e-12):
        failures.append("closed_form_124")
    return failures


def test_real_oracle_passes_the_suite():
    assert _pin_suite(oracle._load()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    c = tmp_path / f"mutant_{name}.c"
    so = tmp_path / f"libmutant_{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", str(so), str(c), "-lm"],
                   check=True)
    lib = oracle.bind_library(str(so))
    assert _pin_suite(lib), f"mutant {name} slipped through every pin"

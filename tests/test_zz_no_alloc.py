"""dit_attn_fwd_masked_noalloc: the masked attention with its occupancy
scratch in the library's fixed per-device array.  Collected last; the GPU test
runs the call twice in a row and compares each result with
dit_attn_fwd_masked (caller workspace) within the parity tolerances, and with
the oracle.  (Its size refusal is checked with the other host-side argument
checks in test_abi_cpu.py.)"""

import numpy as np
import pytest
import torch

import oracle
from dit_long_sequence_gb300 import workloads as wl

from parity import compare, host_bits

DEV = torch.device("cuda:0")


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_twice_in_a_row():
    import dit_long_sequence_gb300 as dl
    B, T, Tp, H, D = 2, 2900, 3072, 2, 128
    q, k, v, _ = wl.make_qkv(B, Tp, H, D, seed=51, device=DEV)
    idx = torch.arange(T)
    m = ((idx[:, None] // 500) == (idx[None, :] // 500)) | ((idx[:, None] + 3 * idx[None, :]) % 97 == 0)
    m = m[None].repeat(B, 1, 1)
    m[1, 256:512] = False
    bits = wl.pack_mask_bits(m).to(DEV)
    O_ref, L_ref = dl.attn_fwd_masked(q, k, v, bits, key_valid_len=T)
    runs = []
    for _ in range(2):
        out = torch.empty_like(O_ref)
        lse = torch.empty_like(L_ref)
        dl.attn_fwd_masked_noalloc(q, k, v, bits, key_valid_len=T, out=out, lse=lse)
        torch.cuda.synchronize()
        runs.append((out, lse))
    Oo, Lo = oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=T,
                         allow=oracle.expand_mask(m.numpy(), Tp))

    def full(O, L):
        return O.to(torch.float64).permute(0, 2, 1, 3).cpu().numpy(), L.double().cpu().numpy()
    ref = full(O_ref, L_ref)
    for out, lse in runs:
        got = full(out, lse)
        compare(*got, *ref)                                   # against the workspace entry point
        compare(*got, Oo.transpose(0, 2, 1, 3), Lo)           # and against the oracle
    assert torch.all(runs[0][0][1, 256:512] == 0)
    np.testing.assert_array_equal(runs[0][0].cpu().numpy(), runs[1][0].cpu().numpy())

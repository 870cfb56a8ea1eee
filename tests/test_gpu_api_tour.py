"""Every Python entry point shown in the README's usage section, called the
way a user calls it on an LTX-2-sized fused buffer: each returns without error,
gives finite results where rows have keys, and the workspace form agrees with
the plain call (the split items differ only by P's bf16 rounding)."""
import pytest
import torch

import dit_long_sequence_gb300 as dl
from dit_long_sequence_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_every_python_entry_point_runs_on_a_fused_buffer():
    B, N, H, D, T = 1, 24576, 32, 128, 24200
    qkv = wl.randn_bf16((B, N, 3, H, D), 91, "cuda")
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]

    out, lse = dl.attn_fwd(q, k, v, key_valid_len=T)
    ws = torch.empty(dl.attn_fwd_workspace_bytes(B, N, H, D, T), dtype=torch.uint8, device="cuda")
    out_ws, _ = dl.attn_fwd_ws(q, k, v, key_valid_len=T, workspace=ws)

    parts = torch.empty(2, B, N, H, D, device="cuda")
    lses = torch.empty(2, B, H, N, device="cuda")
    dl.attn_fwd(q, k[:, :12000], v[:, :12000], out=parts[0], lse=lses[0])
    dl.attn_fwd(q, k[:, 12000:T], v[:, 12000:T], out=parts[1], lse=lses[1])
    merged, merged_lse = dl.lse_merge(parts, lses)

    run_o = torch.zeros(B, N, H, D, device="cuda")
    run_l = torch.full((B, H, N), -float("inf"), device="cuda")
    dl.attn_fwd_accumulate(q, k[:, :12000], v[:, :12000], run_o, run_l)
    dl.attn_fwd_accumulate(q, k[:, 12000:T], v[:, 12000:T], run_o, run_l)

    qh, kh, vh = dl.qkv_to_head_major(qkv)
    cos, sin = wl.rope_tables_3d((16, 32, 48), D, device="cuda")
    qn, kn, vn = dl.qkv_norm_rope_to_head_major(qkv, q_weight=torch.ones(D, device="cuda"),
                                                k_weight=torch.ones(D, device="cuda"), rope_cos=cos, rope_sin=sin)

    qkv8 = dl.qkv_cast_fp8(qkv, scales=(64.0, 64.0, 64.0))
    out8, _ = dl.attn_fwd_fp8(*dl.split_stacked_fp8(qkv8), descales=(1 / 64, 1 / 64, 1 / 64), key_valid_len=T)

    allow = torch.rand(1, 2000, 2000, generator=torch.Generator().manual_seed(3)) < 0.1
    out_m, _ = dl.attn_fwd_masked(q[:, :2048], k[:, :2048], v[:, :2048], wl.pack_mask_bits(allow).cuda(),
                                  key_valid_len=2000)
    torch.cuda.synchronize()

    for name, t in (("out", out), ("out_ws", out_ws), ("merged", merged), ("run_o", run_o), ("qn", qn),
                    ("out8", out8), ("out_m", out_m)):
        assert torch.isfinite(t.float()).all(), name
    assert (out_ws - out).abs().max().item() <= 2e-3
    # the key-chunked forms agree with the single pass within the bf16 parity gates
    assert (merged - out).abs().max().item() <= 2e-2 and (run_o - out).abs().max().item() <= 2e-2
    assert (merged_lse - lse).abs().max().item() <= 1e-3 and (run_l - lse).abs().max().item() <= 1e-3
    # the plain split is the permute, bit for bit
    assert torch.equal(qh, q.permute(0, 2, 1, 3)) and torch.equal(vh, v.permute(0, 2, 1, 3))
    assert torch.equal(vn, v.permute(0, 2, 1, 3))
    rc, info = dl.check_watchdog()
    assert rc == 0, info

"""Placement checks of every entry point, on the GPU.

A buffer that is not memory of the current device, or a stream of another
device, is refused on the host with DIT_ERR_INVALID_ARG before anything is
enqueued.  The refused buffers here are pinned host memory filled with a NaN
(or 0xAB) canary: the test checks that the call raised and that the canary is
intact, i.e. no kernel ran.  (Pinned memory is reachable from the device, so
even a regressed check could not fault the GPU.)  Device memory from every
allocator torch uses, including the virtual-memory one behind expandable
segments, is accepted and gives the same results.
"""
import os
import subprocess
import sys

import pytest
import torch

from dit_long_sequence_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dl():
    import dit_long_sequence_gb300 as m
    return m


def _pinned(shape, dtype, fill):
    t = torch.empty(shape, dtype=dtype, pin_memory=True)
    if dtype == torch.uint8:
        t.fill_(fill)
    else:
        t.fill_(float(fill))
    return t


def _refused(dl, fn):
    from dit_long_sequence_gb300 import binding
    with pytest.raises(dl.DitError) as ei:
        fn()
    assert ei.value.status == binding.DIT_ERR_INVALID_ARG
    torch.cuda.synchronize()


def test_attention_refuses_host_outputs(dl):
    B, N, H, D = 1, 300, 2, 128
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed=80, device=DEV)
    out_h = _pinned((B, N, H, D), torch.float32, float("nan"))
    lse_h = _pinned((B, H, N), torch.float32, float("nan"))
    _refused(dl, lambda: dl.attn_fwd(q, k, v, out=out_h))
    _refused(dl, lambda: dl.attn_fwd(q, k, v, lse=lse_h))
    _refused(dl, lambda: dl.attn_fwd_ws(q, k, v, out=out_h))
    _refused(dl, lambda: dl.attn_fwd_masked(q, k, v, wl.pack_mask_bits(torch.ones(1, N, N, dtype=torch.bool)).to(DEV),
                                            out=out_h))
    ws_h = _pinned((dl.attn_fwd_workspace_bytes(B, N, H, D, N) + 16,), torch.uint8, 0xAB)
    _refused(dl, lambda: dl.attn_fwd_ws(q, k, v, workspace=ws_h))
    assert torch.isnan(out_h).all() and torch.isnan(lse_h).all() and (ws_h == 0xAB).all()
    rc, info = dl.check_watchdog()
    assert rc == 0, info


def test_fp8_cast_merge_and_layouts_refuse_host_outputs(dl):
    B, N, H, D = 1, 64, 2, 128
    qkv = wl.randn_bf16((B, N, 3, H, D), 81, DEV)
    out8 = _pinned((B, N, 3, H, D), torch.uint8, 0xAB)
    _refused(dl, lambda: dl.qkv_cast_fp8(qkv, (64.0, 64.0, 64.0), out=out8))
    assert (out8 == 0xAB).all()
    outs = [torch.empty((B, H, N, D), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    host_plane = _pinned((B, H, N, D), torch.bfloat16, float("nan"))
    _refused(dl, lambda: dl.qkv_to_head_major(qkv, outs=(outs[0], outs[1], host_plane)))
    _refused(dl, lambda: dl.qkv_norm_rope_to_head_major(qkv, q_weight=_pinned((D,), torch.float32, 1.0),
                                                         k_weight=torch.ones(D, device=DEV)))
    _refused(dl, lambda: dl.qkv_norm_rope_to_head_major(qkv, outs=(host_plane, outs[0], outs[1])))
    assert torch.isnan(host_plane).all()
    parts = torch.randn(2, B, N, H, D, device=DEV)
    lses = torch.randn(2, B, H, N, device=DEV)
    out_h = _pinned((B, N, H, D), torch.float32, float("nan"))
    _refused(dl, lambda: dl.lse_merge(parts, lses, out=out_h))
    _refused(dl, lambda: dl.lse_merge(parts.cpu().pin_memory(), lses))
    assert torch.isnan(out_h).all()


def test_side_streams_are_accepted(dl):
    B, N, H, D = 1, 300, 2, 128
    q, k, v, _ = wl.make_qkv(B, N, H, D, seed=82, device=DEV)
    O0, L0 = dl.attn_fwd(q, k, v)
    s = torch.cuda.Stream(device=DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        O1, L1 = dl.attn_fwd(q, k, v, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(O0, O1) and torch.equal(L0, L1)


_VMM_CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import dit_long_sequence_gb300 as dl
from dit_long_sequence_gb300 import workloads as wl
dev = torch.device("cuda:0")
q, k, v, _ = wl.make_qkv(1, 300, 2, 128, seed=83, device=dev)
O, L = dl.attn_fwd_ws(q, k, v)
parts = torch.stack([O, O]); lses = torch.stack([L, L])
M, LM = dl.lse_merge(parts, lses)
torch.cuda.synchronize()
assert torch.allclose(M, O, atol=1e-6) and torch.allclose(LM, L + 0.6931471805599453, atol=1e-5)
torch.save({"O": O.cpu(), "L": L.cpu()}, sys.argv[2])
print("ok")
"""


def test_virtual_memory_allocations_are_device_memory(dl, tmp_path):
    # torch's expandable segments map their memory with the virtual-memory calls
    q, k, v, _ = wl.make_qkv(1, 300, 2, 128, seed=83, device=DEV)
    O, L = dl.attn_fwd_ws(q, k, v)
    torch.cuda.synchronize()
    env = dict(os.environ, PYTORCH_CUDA_ALLOC_CONF="expandable_segments:True")
    res = tmp_path / "vmm.pt"
    r = subprocess.run([sys.executable, "-c", _VMM_CHILD, ROOT, str(res)], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr
    got = torch.load(res)
    assert torch.equal(got["O"], O.cpu()) and torch.equal(got["L"], L.cpu())

"""The debug library (libditattn_debug.so, include/dit_attn_debug.h) on the GPU.

Wind-down of the attention kernels themselves.  One CTA withholds one producer
signal (dit_debug_configure): the TMA thread skips a K/V load, the MMA thread
skips the completion signal of an S tile, or one softmax warp skips its
"P ready" arrive.  The warps waiting on it give up after the wait limit (20 ms
here), the first records DIT_ERR_TIMEOUT with its block, role and wait site,
the CTA's abort flag stops the other roles, copies and products in flight are
waited for with a limit, tensor memory is released and the kernel returns --
no trap, no fault, no wait without a limit.  Checked: the call returns well
inside the default two-second limit; the report names the faulted block and a
role/site that waits on the withheld signal; every other CTA's rows are
correct; and the next calls on the same context, through the debug and the
product library, match the oracle with a clean status word.  (The pages'
counterpart is the LTX-2 all2all barrier that doubles as deadlock detection
with a timeout: "8 卡怎么分 token：LTX-2 序列并行的 all2all 到底搬了什么",
"注意力怎么跨 rank 交换".)

In-kernel bounds checks.  With the O extent the checks allow shrunk by one
row, the last row's stores fail their check and are skipped (DIT_ERR_BOUNDS,
site BND_OUT) while every other element is written; no access outside the
caller's buffer happens either way.  And the parity suite's small shapes run
through the debug library with every check live (a child pytest with
DIT_ATTN_DEBUG=1) and leave the status word clean after each test.
"""
import ctypes
import os
import subprocess
import sys
import time

import numpy as np
import pytest
import torch

import oracle
from dit_long_sequence_gb300 import binding as bd
from dit_long_sequence_gb300 import workloads as wl

from parity import compare, compare_fp8, host_bits, host_u8

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEV = torch.device("cuda:0")

ROLE_SOFTMAX, ROLE_MMA, ROLE_LOAD = 1, 2, 3
SITE_Q_FULL, SITE_KV_FULL, SITE_KV_EMPTY, SITE_S_FULL, SITE_P_FULL, SITE_O_FINAL = 1, 2, 3, 4, 5, 6
BND_OUT = 105
LIMIT_US = 20000

# who can be waiting on the withheld signal when the first limit runs out
WAITERS = {
    bd.DIT_FAULT_SKIP_LOAD: {(ROLE_MMA, SITE_KV_FULL), (ROLE_SOFTMAX, SITE_S_FULL), (ROLE_LOAD, SITE_KV_EMPTY)},
    bd.DIT_FAULT_SKIP_S_COMMIT: {(ROLE_SOFTMAX, SITE_S_FULL), (ROLE_MMA, SITE_P_FULL), (ROLE_MMA, SITE_KV_FULL),
                                 (ROLE_LOAD, SITE_KV_EMPTY)},
    bd.DIT_FAULT_SKIP_P_ARRIVE: {(ROLE_MMA, SITE_P_FULL), (ROLE_SOFTMAX, SITE_S_FULL), (ROLE_LOAD, SITE_KV_EMPTY)},
}


@pytest.fixture(scope="module")
def dbg():
    lib = bd.load_debug_library()
    assert lib.dit_debug_build() == 1
    lib.dit_check_watchdog(None, None)           # start from a clean status word
    yield lib
    lib.dit_debug_configure(0, 0, 0, 0, 0)


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _check(lib):
    info = (ctypes.c_uint32 * 4)()
    rc = lib.dit_check_watchdog(_stream(), info)
    return rc, list(info)


def _attn(lib, q, k, v, out, lse, kvl, descales=None):
    B, Nq, H, D = q.shape
    st = bd.AttnStrides(bd.Strides4(*q.stride()), bd.Strides4(*k.stride()), bd.Strides4(*v.stride()),
                        bd.Strides4(*out.stride()))
    if descales is None:
        return lib.dit_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(st), B, Nq, k.shape[1], H, D,
                                kvl, D ** -0.5, out.data_ptr(), bd.DIT_F32, lse.data_ptr(), _stream())
    return lib.dit_attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(st), B, Nq, k.shape[1], H, D,
                                kvl, D ** -0.5, *descales, out.data_ptr(), bd.DIT_F32, lse.data_ptr(), _stream())


def _inputs(fp8, B=1, Nq=512, Nkv=1024, H=2, D=128, seed=61):
    if not fp8:
        q, k, v, _ = wl.make_qkv(B, Nq, H, D, seed, device=DEV, Nkv=Nkv)
        return (q, k, v), None
    q, k, v = (wl.randn_e4m3((B, n, H, D), seed + i, 64.0, DEV) for i, n in enumerate((Nq, Nkv, Nkv)))
    return (q, k, v), (1 / 64, 1 / 64, 1 / 64)


def _reference(qkv, desc, kvl):
    q, k, v = qkv
    if desc is None:
        O, L = oracle.attn(host_bits(q), host_bits(k), host_bits(v), key_valid_len=kvl)
    else:
        O, L = oracle.attn_fp8(host_u8(q), host_u8(k), host_u8(v), scale=q.shape[3] ** -0.5, descale_q=desc[0],
                               descale_k=desc[1], descale_v=desc[2], key_valid_len=kvl)
    return O.transpose(0, 2, 1, 3), L


def _cmp(desc, Og, Lg, Or, Lr, v):
    if desc is None:
        return compare(Og, Lg, Or, Lr)
    vmax = float(torch.from_numpy(oracle.e4m3_decode(host_u8(v))).abs().max()) * desc[2]
    return compare_fp8(Og, Lg, Or, Lr, vmax)


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
@pytest.mark.parametrize("fault,index", [
    (bd.DIT_FAULT_SKIP_LOAD, 2),        # K of key tile 1
    (bd.DIT_FAULT_SKIP_LOAD, 5),        # V of key tile 2
    (bd.DIT_FAULT_SKIP_S_COMMIT, 3),    # S_0 of key tile 3
    (bd.DIT_FAULT_SKIP_P_ARRIVE, 4),    # P_0 of key tile 4
])
def test_withheld_signal_winds_the_cta_down(dbg, fp8, fault, index):
    """Grid (2, 2, 1): block 1 (second query block of head 0) withholds one
    signal; blocks 0, 2 and 3 must finish normally."""
    qkv, desc = _inputs(fp8)
    q, k, v = qkv
    kvl = 1000
    B, Nq, H, D = q.shape
    Or, Lr = _reference(qkv, desc, kvl)
    out = torch.full((B, Nq, H, D), float("nan"), device=DEV)
    lse = torch.full((B, H, Nq), float("nan"), device=DEV)
    assert dbg.dit_debug_configure(fault, 1, index, LIMIT_US, 0) == bd.DIT_OK
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    try:
        assert _attn(dbg, q, k, v, out, lse, kvl, desc) == bd.DIT_OK
        rc, info = _check(dbg)                       # synchronises
    finally:
        dbg.dit_debug_configure(0, 0, 0, 0, 0)
    elapsed = time.perf_counter() - t0
    assert rc == bd.DIT_ERR_TIMEOUT, (rc, info)
    assert info[0] == bd.DIT_ERR_TIMEOUT and info[1] == 1, info
    assert (info[2], info[3]) in WAITERS[fault], info
    assert elapsed < 1.0, f"wind-down took {elapsed:.3f} s with a {LIMIT_US} us limit"
    # every CTA but the faulted one (rows 256-511 of head 0) is complete and right
    Og = out.double().permute(0, 2, 1, 3).cpu().numpy()
    Lg = lse.double().cpu().numpy()
    keep = np.ones((H, Nq), dtype=bool)
    keep[0, 256:512] = False
    _cmp(desc, Og[0][keep][None, None], Lg[0][keep][None, None], Or[0][keep][None, None], Lr[0][keep][None, None], v)
    # the context is intact: the same call again, debug library and product library
    for lib in (dbg, bd.raw()):
        out2 = torch.full_like(out, float("nan"))
        lse2 = torch.full_like(lse, float("nan"))
        assert _attn(lib, q, k, v, out2, lse2, kvl, desc) == bd.DIT_OK
        assert _check(lib)[0] == bd.DIT_OK
        _cmp(desc, out2.double().permute(0, 2, 1, 3).cpu().numpy(), lse2.double().cpu().numpy(), Or, Lr, v)


def test_default_limit_is_untouched_after_reconfiguring(dbg):
    """Out-of-range settings are refused on the host; a clean call after a
    fault test reports nothing."""
    assert dbg.dit_debug_configure(4, 0, 0, 0, 0) == bd.DIT_ERR_INVALID_ARG
    assert dbg.dit_debug_configure(1, -1, 0, 0, 0) == bd.DIT_ERR_INVALID_ARG
    assert dbg.dit_debug_configure(0, 0, 0, 999, 0) == bd.DIT_ERR_INVALID_ARG
    assert dbg.dit_debug_configure(0, 0, 0, 2000001, 0) == bd.DIT_ERR_INVALID_ARG
    assert dbg.dit_debug_configure(0, 0, 0, 0, -1) == bd.DIT_ERR_INVALID_ARG
    qkv, _ = _inputs(False)
    q, k, v = qkv
    out = torch.empty(q.shape, device=DEV)
    lse = torch.empty((1, 2, 512), device=DEV)
    assert _attn(dbg, q, k, v, out, lse, 1024) == bd.DIT_OK
    assert _check(dbg) == (bd.DIT_OK, [0, 0, 0, 0])


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_bounds_check_skips_the_store_it_refuses(dbg, fp8):
    """O extent shrunk by D elements: the last (b, row, head) row of O fails
    its check (its stores are skipped and keep the NaN canary); every other
    element and every LSE is written and right."""
    qkv, desc = _inputs(fp8, Nq=300, Nkv=555)
    q, k, v = qkv
    B, Nq, H, D = q.shape
    Or, Lr = _reference(qkv, desc, 555)
    out = torch.full((B, Nq, H, D), float("nan"), device=DEV)
    lse = torch.full((B, H, Nq), float("nan"), device=DEV)
    assert dbg.dit_debug_configure(0, 0, 0, 0, D) == bd.DIT_OK
    try:
        assert _attn(dbg, q, k, v, out, lse, 555, desc) == bd.DIT_OK
        rc, info = _check(dbg)
    finally:
        dbg.dit_debug_configure(0, 0, 0, 0, 0)
    assert rc == bd.DIT_ERR_BOUNDS and info[0] == bd.DIT_ERR_BOUNDS, (rc, info)
    assert info[2] == ROLE_SOFTMAX and info[3] == BND_OUT, info
    Og = out.double().permute(0, 2, 1, 3).cpu().numpy()
    assert np.isnan(Og[B - 1, H - 1, Nq - 1]).all()
    Og[B - 1, H - 1, Nq - 1] = Or[B - 1, H - 1, Nq - 1]
    _cmp(desc, Og, lse.double().cpu().numpy(), Or, Lr, v)


def test_parity_suite_small_shapes_through_the_debug_library():
    """The GPU parity tests of small shapes, run once more with the binding
    on the debug library (DIT_ATTN_DEBUG=1): every bounds check live, results
    within the same tolerances, and (tests/conftest.py) a clean status word
    after every test."""
    files = ["tests/test_gpu_attn.py", "tests/test_gpu_fuzz.py", "tests/test_gpu_mask_cross.py",
             "tests/test_gpu_fp8.py", "tests/test_gpu_tail_split.py", "tests/test_gpu_merge_layout.py",
             "tests/test_gpu_norm_rope.py"]
    sel = "not (workload or full_size or ltx or cosmos or ring9 or sampled)"
    env = dict(os.environ, DIT_ATTN_DEBUG="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu", "-k", sel,
                        *files], cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = r.stdout[-4000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    import re
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 60, tail

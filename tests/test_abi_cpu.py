"""Host-side checks of the C ABI that need no GPU.

The library loads and exports every entry point include/dit_attn.h declares,
and every argument check returns its status before anything touches a device.
The argument checks pass made-up device addresses, so they run only in a
process that sees no CUDA device: there a check that ever stopped returning
first could not launch anything.  Where a device is visible (an unfiltered
pytest on a GPU machine), one test re-runs them in a child process with
CUDA_VISIBLE_DEVICES="".
"""
import ctypes
import os
import re
import subprocess
import sys

import pytest


def _device_visible() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


DEVICE_VISIBLE = _device_visible()
# made-up device addresses: only where no device can be reached
deviceless = pytest.mark.skipif(DEVICE_VISIBLE, reason="passes made-up device addresses; re-run in a "
                                                      "deviceless child by test_argument_checks_in_a_deviceless_child")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from dit_long_sequence_gb300 import build
    build.build()
    from dit_long_sequence_gb300 import binding
    return binding


def _declared(header="dit_attn.h"):
    src = open(os.path.join(ROOT, "include", header)).read()
    # declarations start a line with their return type (comment lines start with " *")
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(dit_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"dit_attn_fwd", "dit_attn_lse_merge", "dit_qkv_to_head_major"} <= set(names)
    for n in names:
        assert hasattr(lib.raw(), n), n
    assert set(lib.EXPORTS) <= set(names)


def test_debug_library_exports_both_headers_and_product_none_of_the_debug_calls(lib):
    dbg = lib.load_debug_library()
    debug_names = _declared("dit_attn_debug.h")
    assert set(debug_names) == {"dit_debug_configure", "dit_debug_build"}
    for n in _declared() + debug_names:
        assert hasattr(dbg, n), n
    for n in debug_names:
        assert not hasattr(lib.raw(), n), n
    assert dbg.dit_debug_build() == 1


def test_status_strings(lib):
    for s in range(7):
        assert lib.raw().dit_status_string(s).startswith(b"DIT_")
    assert lib.raw().dit_version() >= 1


FAKE = 0x1000_0000  # 16-byte aligned, never dereferenced


def _fwd(lib, **kw):
    st = lib.AttnStrides(lib.Strides4(8 * 128 * 4, 4 * 128, 128, 1), lib.Strides4(8 * 128 * 4, 4 * 128, 128, 1),
                         lib.Strides4(8 * 128 * 4, 4 * 128, 128, 1), lib.Strides4(8 * 128 * 4, 4 * 128, 128, 1))
    args = dict(q=FAKE, k=FAKE, v=FAKE, st=st, B=1, Nq=8, Nkv=8, H=4, D=128, kvl=8, scale=0.088, out=FAKE,
                dt=lib.DIT_F32, lse=FAKE)
    args.update(kw)
    s = args["st"]
    return lib.raw().dit_attn_fwd(args["q"], args["k"], args["v"], ctypes.byref(s), args["B"], args["Nq"],
                                  args["Nkv"], args["H"], args["D"], args["kvl"], args["scale"], args["out"],
                                  args["dt"], args["lse"], None)


@deviceless
def test_attn_fwd_argument_checks(lib):
    E = lib
    assert _fwd(lib, D=96) == E.DIT_ERR_UNSUPPORTED
    assert _fwd(lib, D=256) == E.DIT_ERR_UNSUPPORTED
    assert _fwd(lib, kvl=9) == E.DIT_ERR_INVALID_ARG
    assert _fwd(lib, kvl=-1) == E.DIT_ERR_INVALID_ARG
    assert _fwd(lib, scale=0.0) == E.DIT_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == E.DIT_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("inf")) == E.DIT_ERR_INVALID_ARG
    assert _fwd(lib, B=-1) == E.DIT_ERR_INVALID_ARG
    assert _fwd(lib, out=None) == E.DIT_ERR_INVALID_ARG
    assert _fwd(lib, lse=None) == E.DIT_ERR_INVALID_ARG
    assert _fwd(lib, q=None) == E.DIT_ERR_INVALID_ARG
    assert _fwd(lib, dt=7) == E.DIT_ERR_INVALID_ARG
    assert _fwd(lib, q=FAKE + 8) == E.DIT_ERR_ALIGNMENT
    assert _fwd(lib, out=FAKE + 4) == E.DIT_ERR_ALIGNMENT
    bad = lib.Strides4(8 * 128 * 4, 4 * 128 + 4, 128, 1)   # n stride not 16-byte aligned
    good = lib.Strides4(8 * 128 * 4, 4 * 128, 128, 1)
    assert _fwd(lib, st=lib.AttnStrides(bad, good, good, good)) == E.DIT_ERR_ALIGNMENT
    nd = lib.Strides4(8 * 128 * 4, 4 * 128, 128, 2)      # d not contiguous
    assert _fwd(lib, st=lib.AttnStrides(good, good, nd, good)) == E.DIT_ERR_UNSUPPORTED
    # zero-size problems are a no-op that succeeds without touching memory
    assert _fwd(lib, B=0, q=None, out=None, lse=None) == E.DIT_OK
    assert _fwd(lib, Nq=0) == E.DIT_OK


@deviceless
def test_merge_argument_checks(lib):
    f = lib.raw().dit_attn_lse_merge
    ok_args = (FAKE, 1 * 8 * 4 * 128, 128, FAKE, 1 * 4 * 8, 2, 1, 8, 4, 128, FAKE, lib.DIT_F32, FAKE, None)

    def call(**kw):
        a = list(ok_args)
        names = ["o", "ocs", "ors", "l", "lcs", "n", "B", "Nq", "H", "D", "out", "dt", "lo", "s"]
        for k_, v_ in kw.items():
            a[names.index(k_)] = v_
        return f(*a)
    assert call(n=0) == lib.DIT_ERR_INVALID_ARG
    assert call(n=65) == lib.DIT_ERR_INVALID_ARG
    assert call(D=32) == lib.DIT_ERR_UNSUPPORTED
    assert call(ocs=8) == lib.DIT_ERR_INVALID_ARG      # chunks would overlap
    assert call(ocs=64, ors=256) == lib.DIT_ERR_INVALID_ARG   # interleaved chunks overlap within a row
    assert call(ors=64) == lib.DIT_ERR_INVALID_ARG     # row stride below D
    assert call(ocs=100000, ors=130) == lib.DIT_ERR_ALIGNMENT
    assert call(o=None) == lib.DIT_ERR_INVALID_ARG
    assert call(o=FAKE + 4) == lib.DIT_ERR_ALIGNMENT
    assert call(B=0) == lib.DIT_OK


@deviceless
def test_layout_argument_checks(lib):
    f = lib.raw().dit_qkv_to_head_major
    assert f(FAKE, 0, 3 * 4 * 12, 1, 8, 4, 12, FAKE, FAKE, FAKE, None) == lib.DIT_ERR_UNSUPPORTED  # D % 8
    assert f(FAKE, 0, 3 * 4 * 64 + 4, 1, 8, 4, 64, FAKE, FAKE, FAKE, None) == lib.DIT_ERR_ALIGNMENT
    assert f(None, 0, 3 * 4 * 64, 1, 8, 4, 64, FAKE, FAKE, FAKE, None) == lib.DIT_ERR_INVALID_ARG
    assert f(FAKE, 0, 3 * 4 * 64, 1, 8, 4, 64, FAKE + 2, FAKE, FAKE, None) == lib.DIT_ERR_ALIGNMENT
    assert f(FAKE, 0, 3 * 4 * 64, 1, 0, 4, 64, FAKE, FAKE, FAKE, None) == lib.DIT_OK


def test_product_path_never_imports_oracle():
    pkg = os.path.join(ROOT, "dit_long_sequence_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "attn_oracle" not in text, fn


def _fwd8(lib, **kw):
    g = lib.Strides4(8 * 3 * 4 * 128, 3 * 4 * 128, 128, 1)       # views of a stacked E4M3 buffer
    o = lib.Strides4(8 * 128 * 4, 4 * 128, 128, 1)
    args = dict(q=FAKE, k=FAKE + 512, v=FAKE + 1024, st=lib.AttnStrides(g, g, g, o), B=1, Nq=8, Nkv=8, H=4, D=128,
                kvl=8, scale=0.088, dq=0.01, dk=0.01, dv=0.02, out=FAKE, dt=lib.DIT_BF16, lse=FAKE)
    args.update(kw)
    return lib.raw().dit_attn_fwd_fp8(args["q"], args["k"], args["v"], ctypes.byref(args["st"]), args["B"],
                                      args["Nq"], args["Nkv"], args["H"], args["D"], args["kvl"], args["scale"],
                                      args["dq"], args["dk"], args["dv"], args["out"], args["dt"], args["lse"], None)


@deviceless
def test_attn_fwd_fp8_argument_checks(lib):
    E = lib
    assert _fwd8(lib, D=64) == E.DIT_ERR_UNSUPPORTED            # head dim 128 only
    assert _fwd8(lib, dq=0.0) == E.DIT_ERR_INVALID_ARG
    assert _fwd8(lib, dk=-1.0) == E.DIT_ERR_INVALID_ARG
    assert _fwd8(lib, dv=float("inf")) == E.DIT_ERR_INVALID_ARG
    assert _fwd8(lib, dv=float("nan")) == E.DIT_ERR_INVALID_ARG
    assert _fwd8(lib, dq=1e-20, dk=1e-20) == E.DIT_ERR_INVALID_ARG   # folded exponent scale underflows
    assert _fwd8(lib, kvl=9) == E.DIT_ERR_INVALID_ARG
    assert _fwd8(lib, q=FAKE + 8) == E.DIT_ERR_ALIGNMENT
    g8 = lib.Strides4(8 * 3 * 4 * 128, 3 * 4 * 128 + 8, 128, 1)   # 8 bytes: fine for bf16, not for E4M3 TMA
    g = lib.Strides4(8 * 3 * 4 * 128, 3 * 4 * 128, 128, 1)
    o = lib.Strides4(8 * 128 * 4, 4 * 128, 128, 1)
    assert _fwd8(lib, st=lib.AttnStrides(g, g8, g, o)) == E.DIT_ERR_ALIGNMENT
    assert _fwd8(lib, B=0, q=None, out=None, lse=None) == E.DIT_OK


@deviceless
def test_cast_fp8_argument_checks(lib):
    f = lib.raw().dit_qkv_cast_fp8
    ok = (FAKE, 0, 3 * 4 * 64, 1, 8, 4, 64, 1.0, 2.0, 3.0, FAKE, None)

    def call(**kw):
        a = list(ok)
        names = ["qkv", "sb", "sn", "B", "N", "H", "D", "sq", "sk", "sv", "out", "s"]
        for k_, v_ in kw.items():
            a[names.index(k_)] = v_
        return f(*a)
    assert call(D=8, sn=3 * 4 * 8) == lib.DIT_ERR_UNSUPPORTED       # D % 16
    assert call(sq=0.0) == lib.DIT_ERR_INVALID_ARG
    assert call(sv=float("inf")) == lib.DIT_ERR_INVALID_ARG
    assert call(sk=float("nan")) == lib.DIT_ERR_INVALID_ARG
    assert call(sn=3 * 4 * 64 + 4) == lib.DIT_ERR_ALIGNMENT
    assert call(out=FAKE + 8) == lib.DIT_ERR_ALIGNMENT
    assert call(qkv=None) == lib.DIT_ERR_INVALID_ARG
    assert call(N=-1) == lib.DIT_ERR_INVALID_ARG
    assert call(B=4, N=1 << 20, H=64, D=128, sn=3 * 64 * 128) == lib.DIT_ERR_UNSUPPORTED   # >= 2^32 chunks
    assert call(N=0) == lib.DIT_OK


@deviceless
def test_norm_rope_argument_checks(lib):
    f = lib.raw().dit_qkv_norm_rope_to_head_major
    ok = [FAKE, 0, 3 * 4 * 64, 1, 8, 4, 64, FAKE, FAKE, 1e-6, FAKE, FAKE + 4096, FAKE, FAKE, FAKE, None]
    names = ["qkv", "sb", "sn", "B", "N", "H", "D", "wq", "wk", "eps", "cos", "sin", "q", "k", "v", "s"]

    def call(**kw):
        a = list(ok)
        for k_, v_ in kw.items():
            a[names.index(k_)] = v_
        return f(*a)
    assert call(D=32, sn=3 * 4 * 32) == lib.DIT_ERR_UNSUPPORTED
    assert call(eps=-1.0) == lib.DIT_ERR_INVALID_ARG
    assert call(eps=float("nan")) == lib.DIT_ERR_INVALID_ARG
    assert call(sin=None) == lib.DIT_ERR_INVALID_ARG            # one table without the other
    assert call(wq=FAKE + 4) == lib.DIT_ERR_ALIGNMENT
    assert call(cos=FAKE + 8) == lib.DIT_ERR_ALIGNMENT
    assert call(sn=3 * 4 * 64 + 4) == lib.DIT_ERR_ALIGNMENT
    assert call(v=None) == lib.DIT_ERR_INVALID_ARG
    assert call(N=0) == lib.DIT_OK


@deviceless
def test_masked_argument_checks(lib):
    st = lib.AttnStrides(*(lib.Strides4(8 * 128 * 4, 4 * 128, 128, 1) for _ in range(4)))
    f = lib.raw().dit_attn_fwd_masked

    def call(mask=FAKE, sb=0, si=4, rows=8, kvl=8, B=1, ws=None, wsb=0):
        return f(FAKE, FAKE, FAKE, ctypes.byref(st), B, 8, 8, 4, 128, kvl, mask, sb, si, rows, 0.088, FAKE,
                 lib.DIT_F32, FAKE, ws, wsb, None)
    assert call(rows=9) == lib.DIT_ERR_INVALID_ARG          # more mask rows than queries
    assert call(rows=-1) == lib.DIT_ERR_INVALID_ARG
    assert call(mask=None) == lib.DIT_ERR_INVALID_ARG
    assert call(si=2) == lib.DIT_ERR_INVALID_ARG             # fewer words than one key tile reads
    assert call(si=6) == lib.DIT_ERR_ALIGNMENT
    assert call(sb=2) == lib.DIT_ERR_ALIGNMENT
    assert call(mask=FAKE + 4) == lib.DIT_ERR_ALIGNMENT
    assert call(sb=-4) == lib.DIT_ERR_INVALID_ARG
    assert call(ws=FAKE, wsb=2) == lib.DIT_ERR_INVALID_ARG     # smaller than the occupancy map
    assert call(ws=FAKE + 4, wsb=4096) == lib.DIT_ERR_ALIGNMENT
    assert call(B=0) == lib.DIT_OK
    ws = lib.raw().dit_attn_masked_workspace_bytes
    assert ws(1, 24576, 24200) == 96 * 6 * 4                   # 96 row blocks x 190 tiles -> 6 words
    assert ws(2, 256, 128) == 8 and ws(0, 10, 10) == 0 and ws(1, 10, 0) == 0


@deviceless
def test_attn_fwd_ws_argument_checks(lib):
    st = lib.AttnStrides(*(lib.Strides4(8 * 128 * 4, 4 * 128, 128, 1) for _ in range(4)))
    f = lib.raw().dit_attn_fwd_ws

    def call(D=128, kvl=8, scale=0.088, out=FAKE, B=1):
        return f(FAKE, FAKE, FAKE, ctypes.byref(st), B, 8, 8, 4, D, kvl, scale, out, lib.DIT_F32, FAKE,
                 FAKE, 1 << 20, None)
    # the checks shared with dit_attn_fwd run first, whatever the workspace
    assert call(D=96) == lib.DIT_ERR_UNSUPPORTED
    assert call(kvl=9) == lib.DIT_ERR_INVALID_ARG
    assert call(scale=0.0) == lib.DIT_ERR_INVALID_ARG
    assert call(out=None) == lib.DIT_ERR_INVALID_ARG
    assert call(out=FAKE + 4) == lib.DIT_ERR_ALIGNMENT
    assert call(B=0) == lib.DIT_OK
    # more than 2^31 - 1 work items (b, h, 256-row block): refused before any device call
    big = f(FAKE, FAKE, FAKE, ctypes.byref(st), 65535, 256 * 1000, 8, 65535, 128, 8, 0.088, FAKE, lib.DIT_F32,
            FAKE, None, 0, None)
    assert big == lib.DIT_ERR_UNSUPPORTED
    wsb = lib.raw().dit_attn_fwd_workspace_bytes
    assert wsb(1, 24576, 32, 96, 24200) == 0          # unsupported D
    assert wsb(0, 24576, 32, 128, 24200) == 0 and wsb(1, 24576, 32, 128, 0) == 0


@deviceless
def test_noalloc_rejects_maps_beyond_its_array_before_launching(lib):
    st = lib.AttnStrides(*(lib.Strides4(8 * 128 * 4, 4 * 128, 128, 1) for _ in range(4)))
    # B=64, 65,536 rows, 65,536 keys: 64 * 256 blocks * 16 words * 4 B = 1 MiB > 256 KiB
    rc = lib.raw().dit_attn_fwd_masked_noalloc(FAKE, FAKE, FAKE, ctypes.byref(st), 64, 65536, 65536, 4, 128, 65536,
                                               FAKE, 0, 2048, 65536, 0.088, FAKE, lib.DIT_F32, FAKE, None)
    assert rc == lib.DIT_ERR_UNSUPPORTED


def test_argument_checks_in_a_deviceless_child():
    """Where this process sees a CUDA device, the made-up-address checks run in
    a child process that sees none."""
    if not DEVICE_VISIBLE:
        pytest.skip("no device visible: the checks above ran in this process")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                        os.path.abspath(__file__)], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    m = re.search(r"(\d+) passed", r.stdout)
    n_checks = sum(1 for line in open(os.path.abspath(__file__)) if line.startswith("@deviceless"))
    assert m and int(m.group(1)) >= n_checks, r.stdout[-2000:]

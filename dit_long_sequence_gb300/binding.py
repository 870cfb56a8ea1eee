"""ctypes binding of libditattn.so (include/dit_attn.h).

Argument marshalling only: tensors are passed as device pointers with their
element strides and the current CUDA stream; every step of the computation
runs in the library's kernels.  PyTorch supplies device memory and streams.
There is no fallback: if the library is missing or a call fails, an exception
is raised.

With the environment variable DIT_ATTN_DEBUG=1 at import, the binding loads
the debug library instead (libditattn_debug.so: the same kernels with
in-kernel bounds checks, include/dit_attn_debug.h); load_debug_library()
gives a handle to it beside the product library.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import DEBUG_LIB as _DEBUG_LIB_PATH
from .build import LIB as _PRODUCT_LIB_PATH

is_debug_library = os.environ.get("DIT_ATTN_DEBUG", "") == "1"
_LIB_PATH = _DEBUG_LIB_PATH if is_debug_library else _PRODUCT_LIB_PATH
library_path = _LIB_PATH

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{os.path.basename(_LIB_PATH)} not found at {_LIB_PATH}; build it first with "
        "`python -m dit_long_sequence_gb300.build` (or __graft_entry__.build())")

DIT_OK, DIT_ERR_INVALID_ARG, DIT_ERR_UNSUPPORTED, DIT_ERR_ALIGNMENT, DIT_ERR_CUDA, DIT_ERR_TIMEOUT, DIT_ERR_BOUNDS = \
    range(7)
DIT_BF16, DIT_F32 = 0, 1
DIT_FAULT_NONE, DIT_FAULT_SKIP_LOAD, DIT_FAULT_SKIP_S_COMMIT, DIT_FAULT_SKIP_P_ARRIVE = range(4)


class Strides4(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("n", ctypes.c_int64), ("h", ctypes.c_int64), ("d", ctypes.c_int64)]


class AttnStrides(ctypes.Structure):
    _fields_ = [("q", Strides4), ("k", Strides4), ("v", Strides4), ("o", Strides4)]


_vp, _i, _i64, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float


def _declare(lib):
    """Argument and result types of the C ABI on a loaded library handle."""
    lib.dit_attn_fwd.restype = _i
    lib.dit_attn_fwd.argtypes = [_vp, _vp, _vp, ctypes.POINTER(AttnStrides), _i, _i, _i, _i, _i, _i, _f,
                                  _vp, _i, _vp, _vp]
    lib.dit_attn_fwd_ws.restype = _i
    lib.dit_attn_fwd_ws.argtypes = [_vp, _vp, _vp, ctypes.POINTER(AttnStrides), _i, _i, _i, _i, _i, _i, _f,
                                     _vp, _i, _vp, _vp, ctypes.c_size_t, _vp]
    lib.dit_attn_fwd_workspace_bytes.restype = ctypes.c_size_t
    lib.dit_attn_fwd_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
    lib.dit_attn_fwd_accumulate.restype = _i
    lib.dit_attn_fwd_accumulate.argtypes = [_vp, _vp, _vp, ctypes.POINTER(AttnStrides), _i, _i, _i, _i, _i, _i, _f,
                                             _vp, _vp, _vp]
    lib.dit_attn_fwd_masked.restype = _i
    lib.dit_attn_fwd_masked.argtypes = [_vp, _vp, _vp, ctypes.POINTER(AttnStrides), _i, _i, _i, _i, _i, _i, _vp, _i64,
                                         _i64, _i, _f, _vp, _i, _vp, _vp, ctypes.c_size_t, _vp]
    lib.dit_attn_fwd_masked_noalloc.restype = _i
    lib.dit_attn_fwd_masked_noalloc.argtypes = [_vp, _vp, _vp, ctypes.POINTER(AttnStrides), _i, _i, _i, _i, _i, _i, _vp,
                                                 _i64, _i64, _i, _f, _vp, _i, _vp, _vp]
    lib.dit_attn_masked_workspace_bytes.restype = ctypes.c_size_t
    lib.dit_attn_masked_workspace_bytes.argtypes = [_i, _i, _i]
    lib.dit_attn_masked_split_workspace_bytes.restype = ctypes.c_size_t
    lib.dit_attn_masked_split_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
    lib.dit_attn_fwd_fp8.restype = _i
    lib.dit_attn_fwd_fp8.argtypes = [_vp, _vp, _vp, ctypes.POINTER(AttnStrides), _i, _i, _i, _i, _i, _i, _f, _f, _f, _f,
                                      _vp, _i, _vp, _vp]
    lib.dit_attn_fwd_fp8_ws.restype = _i
    lib.dit_attn_fwd_fp8_ws.argtypes = [_vp, _vp, _vp, ctypes.POINTER(AttnStrides), _i, _i, _i, _i, _i, _i, _f, _f, _f,
                                         _f, _vp, _i, _vp, _vp, ctypes.c_size_t, _vp]
    lib.dit_qkv_cast_fp8.restype = _i
    lib.dit_qkv_cast_fp8.argtypes = [_vp, _i64, _i64, _i, _i, _i, _i, _f, _f, _f, _vp, _vp]
    lib.dit_qkv_norm_rope_to_head_major.restype = _i
    lib.dit_qkv_norm_rope_to_head_major.argtypes = [_vp, _i64, _i64, _i, _i, _i, _i, _vp, _vp, _f, _vp, _vp, _vp, _vp,
                                                     _vp, _vp]
    lib.dit_watchdog_selftest.restype = _i
    lib.dit_watchdog_selftest.argtypes = [ctypes.c_uint32, _vp]
    lib.dit_attn_lse_merge.restype = _i
    lib.dit_attn_lse_merge.argtypes = [_vp, _i64, _i64, _vp, _i64, _i, _i, _i, _i, _i, _vp, _i, _vp, _vp]
    lib.dit_qkv_to_head_major.restype = _i
    lib.dit_qkv_to_head_major.argtypes = [_vp, _i64, _i64, _i, _i, _i, _i, _vp, _vp, _vp, _vp]
    lib.dit_status_string.restype = ctypes.c_char_p
    lib.dit_status_string.argtypes = [_i]
    lib.dit_check_watchdog.restype = _i
    lib.dit_check_watchdog.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.dit_version.restype = ctypes.c_uint32
    if hasattr(lib, "dit_debug_configure"):
        lib.dit_debug_configure.restype = _i
        lib.dit_debug_configure.argtypes = [ctypes.c_uint32, _i, _i, ctypes.c_uint32, _i64]
        lib.dit_debug_build.restype = ctypes.c_uint32
    return lib


_lib = _declare(ctypes.CDLL(_LIB_PATH))


def load_debug_library():
    """ctypes handle of libditattn_debug.so with the C ABI declared: every
    dit_attn.h entry point plus dit_debug_configure / dit_debug_build.  Its
    kernels and device status word are its own (check it with its own
    dit_check_watchdog)."""
    if not os.path.exists(_DEBUG_LIB_PATH):
        raise ImportError(f"libditattn_debug.so not found at {_DEBUG_LIB_PATH}; build it first")
    return _declare(ctypes.CDLL(_DEBUG_LIB_PATH))


EXPORTS = ("dit_attn_fwd", "dit_attn_fwd_ws", "dit_attn_fwd_workspace_bytes", "dit_attn_fwd_masked", "dit_attn_fwd_masked_noalloc", "dit_attn_masked_workspace_bytes",
           "dit_attn_masked_split_workspace_bytes",
           "dit_attn_fwd_accumulate", "dit_attn_lse_merge", "dit_qkv_to_head_major",
           "dit_qkv_norm_rope_to_head_major", "dit_qkv_cast_fp8", "dit_attn_fwd_fp8", "dit_attn_fwd_fp8_ws", "dit_status_string",
           "dit_check_watchdog",
           "dit_watchdog_selftest", "dit_version")


class DitError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.dit_status_string(status).decode()}")


def _check(status: int, where: str):
    if status != DIT_OK:
        raise DitError(status, where)


def raw():
    """The ctypes library handle (for callers that marshal pointers themselves)."""
    return _lib


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _strides4(t: torch.Tensor) -> Strides4:
    return Strides4(*t.stride())


def _attn_args(q, k, v, key_valid_len, scale, out, lse, out_dtype):
    B, Nq, H, D = q.shape
    Nkv = k.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a bf16 CUDA tensor")
    if k.shape != (B, Nkv, H, D) or v.shape != (B, Nkv, H, D):
        raise ValueError("k and v must be [B, Nkv, H, D] matching q")
    kvl = Nkv if key_valid_len is None else int(key_valid_len)
    sc = float(D) ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Nq, H, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if out.dtype not in (torch.float32, torch.bfloat16) or tuple(out.shape) != (B, Nq, H, D):
        raise ValueError("out must be a [B, Nq, H, D] fp32 or bf16 tensor")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    st = AttnStrides(_strides4(q), _strides4(k), _strides4(v), _strides4(out))
    return B, Nq, Nkv, H, D, kvl, sc, out, lse, st


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, key_valid_len: int | None = None,
             scale: float | None = None, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
             out_dtype: torch.dtype = torch.float32, stream=None):
    """O = softmax(scale Q K^T) V and LSE, through `dit_attn_fwd`.

    q [B, Nq, H, D], k/v [B, Nkv, H, D]: bf16 CUDA tensors with any strides whose
    last dimension is contiguous (strided views of a fused QKV buffer work as is).
    Returns (out [B, Nq, H, D] in out_dtype, lse [B, H, Nq] fp32).
    """
    B, Nq, Nkv, H, D, kvl, sc, out, lse, st = _attn_args(q, k, v, key_valid_len, scale, out, lse, out_dtype)
    rc = _lib.dit_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(st), B, Nq, Nkv, H, D, kvl,
                           sc, out.data_ptr(), DIT_F32 if out.dtype == torch.float32 else DIT_BF16,
                           lse.data_ptr(), _stream_ptr(stream))
    _check(rc, "dit_attn_fwd")
    return out, lse


def attn_fwd_workspace_bytes(B: int, Nq: int, H: int, D: int, key_valid_len: int) -> int:
    """Workspace that lets attn_fwd_ws balance the grid's last wave (current device; 0: no split)."""
    return int(_lib.dit_attn_fwd_workspace_bytes(int(B), int(Nq), int(H), int(D), int(key_valid_len)))


def attn_fwd_ws(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, key_valid_len: int | None = None,
                scale: float | None = None, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                out_dtype: torch.dtype = torch.float32, workspace: torch.Tensor | None = None, stream=None):
    """attn_fwd through `dit_attn_fwd_ws`: the items of the grid's last partial
    wave are split over key ranges and merged.  The workspace (a uint8 CUDA
    tensor of attn_fwd_workspace_bytes) is allocated here unless given."""
    B, Nq, Nkv, H, D, kvl, sc, out, lse, st = _attn_args(q, k, v, key_valid_len, scale, out, lse, out_dtype)
    if workspace is None:
        nbytes = attn_fwd_workspace_bytes(B, Nq, H, D, kvl)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _lib.dit_attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(st), B, Nq, Nkv, H, D, kvl,
                              sc, out.data_ptr(), DIT_F32 if out.dtype == torch.float32 else DIT_BF16,
                              lse.data_ptr(), ws_ptr, ws_bytes, _stream_ptr(stream))
    _check(rc, "dit_attn_fwd_ws")
    return out, lse


def masked_workspace_bytes(B: int, Nq: int, key_valid_len: int) -> int:
    """Workspace that lets attn_fwd_masked skip key tiles the mask leaves empty."""
    return int(_lib.dit_attn_masked_workspace_bytes(int(B), int(Nq), int(key_valid_len)))


def masked_split_workspace_bytes(B: int, Nq: int, H: int, D: int, key_valid_len: int) -> int:
    """Workspace that lets attn_fwd_masked skip empty key tiles and split the
    grid's last partial wave (current device)."""
    return int(_lib.dit_attn_masked_split_workspace_bytes(int(B), int(Nq), int(H), int(D), int(key_valid_len)))


def attn_fwd_masked(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask_bits: torch.Tensor, *,
                    mask_rows: int | None = None, key_valid_len: int | None = None, scale: float | None = None,
                    out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                    out_dtype: torch.dtype = torch.float32, workspace: torch.Tensor | None = None,
                    skip_empty_tiles: bool = True, stream=None):
    """Attention with a general bit mask through `dit_attn_fwd_masked`.

    mask_bits: int32 CUDA tensor [B or 1, R, W] of packed bits (bit j&31 of word
    j>>5 of row i: query i may attend key j), W a multiple of 4 with
    W >= 4*ceil(key_valid_len/128); a leading dimension of 1 shares the mask
    across the batch.  Rows i >= mask_rows (default R) attend every valid key.
    With skip_empty_tiles (default) a workspace (allocated here unless given,
    of masked_split_workspace_bytes) lets the kernel skip key tiles the mask
    leaves empty and split the grid's last partial wave over key ranges; a
    given workspace of only masked_workspace_bytes skips without splitting.
    """
    B, Nq, H, D = q.shape
    Nkv = k.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a bf16 CUDA tensor")
    if k.shape != (B, Nkv, H, D) or v.shape != (B, Nkv, H, D):
        raise ValueError("k and v must be [B, Nkv, H, D] matching q")
    if mask_bits.dtype != torch.int32 or mask_bits.dim() != 3 or mask_bits.stride(2) != 1 or not mask_bits.is_cuda:
        raise ValueError("mask_bits must be an int32 CUDA tensor [B or 1, rows, words], words contiguous")
    if mask_bits.shape[0] not in (1, B):
        raise ValueError("mask_bits must have B or 1 batch entries")
    rows = mask_bits.shape[1] if mask_rows is None else int(mask_rows)
    if rows > mask_bits.shape[1]:
        raise ValueError("mask_rows exceeds the mask's rows")
    kvl = Nkv if key_valid_len is None else int(key_valid_len)
    sc = float(D) ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Nq, H, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if out.dtype not in (torch.float32, torch.bfloat16) or tuple(out.shape) != (B, Nq, H, D):
        raise ValueError("out must be a [B, Nq, H, D] fp32 or bf16 tensor")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    sb = 0 if mask_bits.shape[0] == 1 else mask_bits.stride(0)
    ws_ptr, ws_bytes = None, 0
    if skip_empty_tiles:
        need = masked_split_workspace_bytes(B, Nq, H, D, kvl)
        if workspace is None and need > 0:
            workspace = torch.empty((need + 15) // 16 * 16, dtype=torch.uint8, device=q.device)
        if workspace is not None:
            ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = AttnStrides(_strides4(q), _strides4(k), _strides4(v), _strides4(out))
    rc = _lib.dit_attn_fwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(st), B, Nq, Nkv, H, D, kvl,
                                  mask_bits.data_ptr(), sb, mask_bits.stride(1), rows, sc, out.data_ptr(),
                                  DIT_F32 if out.dtype == torch.float32 else DIT_BF16, lse.data_ptr(),
                                  ws_ptr, ws_bytes, _stream_ptr(stream))
    _check(rc, "dit_attn_fwd_masked")
    return out, lse


def attn_fwd_masked_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask_bits: torch.Tensor, *,
                            mask_rows: int | None = None, key_valid_len: int | None = None,
                            scale: float | None = None, out: torch.Tensor | None = None,
                            lse: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32, stream=None):
    """attn_fwd_masked through `dit_attn_fwd_masked_noalloc`: the tile-occupancy
    scratch is the library's fixed per-device array, no workspace is passed.
    out and lse must be given (or are allocated here by PyTorch, not by the
    library)."""
    B, Nq, H, D = q.shape
    Nkv = k.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a bf16 CUDA tensor")
    if mask_bits.dtype != torch.int32 or mask_bits.dim() != 3 or mask_bits.stride(2) != 1 or not mask_bits.is_cuda:
        raise ValueError("mask_bits must be an int32 CUDA tensor [B or 1, rows, words], words contiguous")
    rows = mask_bits.shape[1] if mask_rows is None else int(mask_rows)
    kvl = Nkv if key_valid_len is None else int(key_valid_len)
    sc = float(D) ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Nq, H, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    sb = 0 if mask_bits.shape[0] == 1 else mask_bits.stride(0)
    st = AttnStrides(_strides4(q), _strides4(k), _strides4(v), _strides4(out))
    rc = _lib.dit_attn_fwd_masked_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(st), B, Nq, Nkv, H,
                                          D, kvl, mask_bits.data_ptr(), sb, mask_bits.stride(1), rows, sc,
                                          out.data_ptr(), DIT_F32 if out.dtype == torch.float32 else DIT_BF16,
                                          lse.data_ptr(), _stream_ptr(stream))
    _check(rc, "dit_attn_fwd_masked_noalloc")
    return out, lse


def attn_fwd_accumulate(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, lse: torch.Tensor, *,
                        key_valid_len: int | None = None, scale: float | None = None, stream=None):
    """Fold attention of q over this key chunk into the running fp32 (out, lse)
    in place, through `dit_attn_fwd_accumulate`.  Start from lse = -inf."""
    B, Nq, H, D = q.shape
    Nkv = k.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a bf16 CUDA tensor")
    if k.shape != (B, Nkv, H, D) or v.shape != (B, Nkv, H, D):
        raise ValueError("k and v must be [B, Nkv, H, D] matching q")
    if out.dtype != torch.float32 or tuple(out.shape) != (B, Nq, H, D):
        raise ValueError("out must be an fp32 [B, Nq, H, D] tensor")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    kvl = Nkv if key_valid_len is None else int(key_valid_len)
    sc = float(D) ** -0.5 if scale is None else float(scale)
    st = AttnStrides(_strides4(q), _strides4(k), _strides4(v), _strides4(out))
    rc = _lib.dit_attn_fwd_accumulate(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(st), B, Nq, Nkv, H, D,
                                      kvl, sc, out.data_ptr(), lse.data_ptr(), _stream_ptr(stream))
    _check(rc, "dit_attn_fwd_accumulate")
    return out, lse


def lse_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, *, out: torch.Tensor | None = None,
              lse_out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32, stream=None):
    """Merge n partials through `dit_attn_lse_merge`.

    o_parts [n, B, Nq, H, D] fp32: any view whose (B, Nq, H) dims collapse to one
    row index with a common row stride and d contiguous -- chunk-major
    (contiguous [n, B, Nq, H, D]) or interleaved (a [B, Nq, H, n, D] buffer seen
    through .permute(3, 0, 1, 2, 4)); lse_parts [n, B, H, Nq] fp32 with every
    chunk contiguous.  Returns (out [B, Nq, H, D], lse_out [B, H, Nq]).
    """
    n, B, Nq, H, D = o_parts.shape
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
        raise TypeError("partials must be fp32")
    if tuple(lse_parts.shape) != (n, B, H, Nq):
        raise ValueError("lse_parts must be [n, B, H, Nq]")
    rs = o_parts.stride(3)
    if o_parts.stride(4) != 1 or o_parts.stride(2) != H * rs or o_parts.stride(1) != Nq * H * rs:
        raise ValueError("o_parts rows must share one stride with d contiguous")
    if not lse_parts[0].is_contiguous():
        raise ValueError("each LSE chunk must be contiguous")
    if out is None:
        out = torch.empty((B, Nq, H, D), dtype=out_dtype, device=o_parts.device)
    if lse_out is None:
        lse_out = torch.empty((B, H, Nq), dtype=torch.float32, device=o_parts.device)
    if not out.is_contiguous() or not lse_out.is_contiguous():
        raise ValueError("outputs must be contiguous")
    rc = _lib.dit_attn_lse_merge(o_parts.data_ptr(), o_parts.stride(0), rs, lse_parts.data_ptr(),
                                 lse_parts.stride(0), n, B, Nq, H, D, out.data_ptr(),
                                 DIT_F32 if out.dtype == torch.float32 else DIT_BF16, lse_out.data_ptr(),
                                 _stream_ptr(stream))
    _check(rc, "dit_attn_lse_merge")
    return out, lse_out


def qkv_to_head_major(qkv: torch.Tensor, *, outs=None, stream=None):
    """Split a fused [B, N, 3, H, D] bf16 buffer (b and n strides free, inner
    [3, H, D] contiguous) into three contiguous [B, H, N, D] tensors."""
    B, N, three, H, D = qkv.shape
    if three != 3 or qkv.dtype != torch.bfloat16:
        raise ValueError("expected a bf16 [B, N, 3, H, D] tensor")
    if qkv.stride(4) != 1 or qkv.stride(3) != D or qkv.stride(2) != H * D:
        raise ValueError("the [3, H, D] block of every sequence row must be contiguous")
    if outs is None:
        outs = tuple(torch.empty((B, H, N, D), dtype=torch.bfloat16, device=qkv.device) for _ in range(3))
    for o in outs:
        if not o.is_contiguous() or tuple(o.shape) != (B, H, N, D):
            raise ValueError("outputs must be contiguous [B, H, N, D]")
    rc = _lib.dit_qkv_to_head_major(qkv.data_ptr(), qkv.stride(0), qkv.stride(1), B, N, H, D,
                                    outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(),
                                    _stream_ptr(stream))
    _check(rc, "dit_qkv_to_head_major")
    return outs


def qkv_norm_rope_to_head_major(qkv: torch.Tensor, *, q_weight: torch.Tensor | None = None,
                                k_weight: torch.Tensor | None = None, eps: float = 1e-6,
                                rope_cos: torch.Tensor | None = None, rope_sin: torch.Tensor | None = None,
                                outs=None, stream=None):
    """dit_qkv_to_head_major with Q/K RMSNorm (fp32 [D] weights; None skips)
    and RoPE on consecutive pairs (fp32 [N, D/2] cos/sin tables; None skips)
    fused in, through `dit_qkv_norm_rope_to_head_major`."""
    B, N, three, H, D = qkv.shape
    if three != 3 or qkv.dtype != torch.bfloat16 or not qkv.is_cuda:
        raise ValueError("expected a bf16 CUDA [B, N, 3, H, D] tensor")
    if qkv.stride(4) != 1 or qkv.stride(3) != D or qkv.stride(2) != H * D:
        raise ValueError("the [3, H, D] block of every sequence row must be contiguous")
    for name, w in (("q_weight", q_weight), ("k_weight", k_weight)):
        if w is not None and (w.dtype != torch.float32 or tuple(w.shape) != (D,) or not w.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous fp32 [D] tensor")
    if (rope_cos is None) != (rope_sin is None):
        raise ValueError("pass both rope tables or neither")
    for name, tb in (("rope_cos", rope_cos), ("rope_sin", rope_sin)):
        if tb is not None and (tb.dtype != torch.float32 or tuple(tb.shape) != (N, D // 2) or not tb.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous fp32 [N, D/2] tensor")
    if outs is None:
        outs = tuple(torch.empty((B, H, N, D), dtype=torch.bfloat16, device=qkv.device) for _ in range(3))
    for o in outs:
        if not o.is_contiguous() or tuple(o.shape) != (B, H, N, D) or o.dtype != torch.bfloat16:
            raise ValueError("outputs must be contiguous bf16 [B, H, N, D]")

    def ptr(t):
        return None if t is None else t.data_ptr()
    rc = _lib.dit_qkv_norm_rope_to_head_major(qkv.data_ptr(), qkv.stride(0), qkv.stride(1), B, N, H, D,
                                              ptr(q_weight), ptr(k_weight), float(eps), ptr(rope_cos),
                                              ptr(rope_sin), outs[0].data_ptr(), outs[1].data_ptr(),
                                              outs[2].data_ptr(), _stream_ptr(stream))
    _check(rc, "dit_qkv_norm_rope_to_head_major")
    return outs


_FP8_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def qkv_cast_fp8(qkv: torch.Tensor, scales, *, out: torch.Tensor | None = None, stream=None):
    """One-pass E4M3 cast of a stacked [B, N, 3, H, D] bf16 buffer (b and n
    strides free, inner [3, H, D] contiguous), q/k/v scaled by scales[0..2],
    through `dit_qkv_cast_fp8`.  Returns the contiguous [B, N, 3, H, D] result
    (uint8 codes unless `out` is given as float8_e4m3fn)."""
    B, N, three, H, D = qkv.shape
    if three != 3 or qkv.dtype != torch.bfloat16 or not qkv.is_cuda:
        raise ValueError("expected a bf16 CUDA [B, N, 3, H, D] tensor")
    if qkv.stride(4) != 1 or qkv.stride(3) != D or qkv.stride(2) != H * D:
        raise ValueError("the [3, H, D] block of every sequence row must be contiguous")
    sq, sk, sv = (float(x) for x in scales)
    if out is None:
        out = torch.empty((B, N, 3, H, D), dtype=torch.uint8, device=qkv.device)
    if out.dtype not in _FP8_DTYPES or tuple(out.shape) != (B, N, 3, H, D) or not out.is_contiguous():
        raise ValueError("out must be a contiguous uint8 / float8_e4m3fn [B, N, 3, H, D] tensor")
    rc = _lib.dit_qkv_cast_fp8(qkv.data_ptr(), qkv.stride(0), qkv.stride(1), B, N, H, D, sq, sk, sv,
                               out.data_ptr(), _stream_ptr(stream))
    _check(rc, "dit_qkv_cast_fp8")
    return out


def _attn_fp8_args(q, k, v, descales, key_valid_len, scale, out, lse, out_dtype):
    B, Nq, H, D = q.shape
    Nkv = k.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype not in _FP8_DTYPES or not t.is_cuda:
            raise TypeError(f"{name} must be a uint8 / float8_e4m3fn CUDA tensor")
    if k.shape != (B, Nkv, H, D) or v.shape != (B, Nkv, H, D):
        raise ValueError("k and v must be [B, Nkv, H, D] matching q")
    dq, dk, dv = (float(x) for x in descales)
    kvl = Nkv if key_valid_len is None else int(key_valid_len)
    sc = float(D) ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Nq, H, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if out.dtype not in (torch.float32, torch.bfloat16) or tuple(out.shape) != (B, Nq, H, D):
        raise ValueError("out must be a [B, Nq, H, D] fp32 or bf16 tensor")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    st = AttnStrides(_strides4(q), _strides4(k), _strides4(v), _strides4(out))
    return B, Nq, Nkv, H, D, kvl, sc, dq, dk, dv, out, lse, st


def attn_fwd_fp8(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, descales, *, key_valid_len: int | None = None,
                 scale: float | None = None, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                 out_dtype: torch.dtype = torch.float32, stream=None):
    """Attention on E4M3 codes through `dit_attn_fwd_fp8`: q, k, v [B, N, H, D]
    uint8 / float8_e4m3fn views (e.g. of qkv_cast_fp8's output) standing for
    q * descales[0], k * descales[1], v * descales[2].  Returns (out, lse)."""
    B, Nq, Nkv, H, D, kvl, sc, dq, dk, dv, out, lse, st = _attn_fp8_args(q, k, v, descales, key_valid_len, scale,
                                                                         out, lse, out_dtype)
    rc = _lib.dit_attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(st), B, Nq, Nkv, H, D, kvl,
                               sc, dq, dk, dv, out.data_ptr(), DIT_F32 if out.dtype == torch.float32 else DIT_BF16,
                               lse.data_ptr(), _stream_ptr(stream))
    _check(rc, "dit_attn_fwd_fp8")
    return out, lse


def attn_fwd_fp8_ws(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, descales, *,
                    key_valid_len: int | None = None, scale: float | None = None, out: torch.Tensor | None = None,
                    lse: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32,
                    workspace: torch.Tensor | None = None, stream=None):
    """attn_fwd_fp8 through `dit_attn_fwd_fp8_ws`: the grid's last partial wave
    split over key ranges and merged.  The workspace (a uint8 CUDA tensor of
    attn_fwd_workspace_bytes) is allocated here unless given."""
    B, Nq, Nkv, H, D, kvl, sc, dq, dk, dv, out, lse, st = _attn_fp8_args(q, k, v, descales, key_valid_len, scale,
                                                                         out, lse, out_dtype)
    if workspace is None:
        nbytes = attn_fwd_workspace_bytes(B, Nq, H, D, kvl)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _lib.dit_attn_fwd_fp8_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(st), B, Nq, Nkv, H, D, kvl,
                                  sc, dq, dk, dv, out.data_ptr(), DIT_F32 if out.dtype == torch.float32 else DIT_BF16,
                                  lse.data_ptr(), ws_ptr, ws_bytes, _stream_ptr(stream))
    _check(rc, "dit_attn_fwd_fp8_ws")
    return out, lse


def split_stacked_fp8(qkv8: torch.Tensor):
    """The q, k, v [B, N, H, D] views of a stacked [B, N, 3, H, D] FP8 buffer."""
    return qkv8[:, :, 0], qkv8[:, :, 1], qkv8[:, :, 2]


def watchdog_selftest(limit_us: int = 100_000, stream=None):
    """Enqueue the library's watchdog self-test (a bounded wait that must run
    out); read the outcome with check_watchdog()."""
    _check(_lib.dit_watchdog_selftest(int(limit_us), _stream_ptr(stream)), "dit_watchdog_selftest")


def check_watchdog(stream=None):
    """Synchronise and read/clear the device status word: (status, info[4])."""
    info = (ctypes.c_uint32 * 4)()
    rc = _lib.dit_check_watchdog(_stream_ptr(stream), info)
    return rc, list(info)

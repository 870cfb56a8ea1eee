"""Plain fp64 CPU oracle for the attention / LSE-merge / QKV-layout path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The product path (the CUDA library
and its Python binding) never imports, links or runs anything here, and this
package never imports the product path: the two share no code.

Contents
--------
``attn``                 dense bidirectional attention + LSE, fp64, in C
                         (``attn_oracle.c``), on whole heads or on sampled rows.
``lse_merge``            batched (O, LSE) combine, fp64, numpy.
``lse_merge_streaming``  the same combine as a streaming pairwise recurrence.
``qkv_to_head_major``    the fused-QKV split/permute, numpy indexing.
``e4m3_encode`` / ``e4m3_decode``  the FP8 E4M3 format (round to nearest even,
                         saturating), numpy, from the format's definition.
``qkv_cast_fp8``         the one-pass scaled cast of a stacked QKV buffer.
``attn_fp8``             attention on E4M3 inputs with per-tensor descales.

Citations (page title, section):
  * "Scaling Video Generation Across NVL72 rack with TensorRT-LLM":
    - "The Scaling Challenge in Video Generation": dense, unmasked,
      bidirectional N x N attention every step.
    - "Ring Attention", paragraph "Online-softmax merge": each partial pass
      yields an output and an LSE; they are merged in fp32 by a streaming
      softmax recurrence until the result equals one global pass.
    - "Attention2D Parallelism", paragraphs "Local Attention" and "Merge phase":
      partial O is [B,S,H,D], LSE is [B,H,S]; a batched combine merges the
      col_size partials over disjoint key spans; the "Difference from Ring"
      table names Ring's recurrence the sigmoid / logsigmoid form.
    - "Ulysses Parallelism", paragraph "Fused vs. unfused QKV all-to-all":
      the stacked buffer is [B, S, 3, H, D].
  * "8 卡怎么分 token：LTX-2 序列并行的 all2all 到底搬了什么", "数据流拆解",
    paragraph "构造 padding mask": key-only (1,1,T) mask, pads at the tail.
  * "CUDA IPC Ulysses：在 H100 上重叠 Attention 通信", "基线与瓶颈": V of a fused
    QKV projection is a legal strided view; no packing copy.
  * NVL72 blog, "Ulysses Parallelism", paragraph on the stacked buffer: one
    single-pass FP8 cast over the contiguous [B, S, 3, H, D] QKV buffer before
    an FP8 attention kernel, whose result feeds the kernel without a copy.

Parity status: every function here is pinned by the CPU tests (brute force,
closed forms, library special cases and invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, IEEE fp64, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC",
           "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind_library(path: str):
    """ctypes handle for a compiled oracle library at ``path``."""
    lib = ctypes.CDLL(path)
    f = lib.oracle_attn_head_rows
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                  ctypes.POINTER(ctypes.c_int64),
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_double, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64]
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = bind_library(_LIB_PATH)
    return _lib


def max_threads() -> int:
    """OpenMP threads the C oracle runs with."""
    return int(_load().oracle_max_threads())


def _bf16_view_strides(a: np.ndarray, name: str):
    """Element strides (b, n, h) of a [B, N, H, D] uint16 view with d contiguous."""
    if a.dtype != np.uint16 or a.ndim != 4:
        raise TypeError(f"{name}: expected a 4-D uint16 array of bf16 bits, got {a.dtype} {a.shape}")
    st = [s // 2 for s in a.strides]
    if any(s % 2 for s in a.strides) or (a.shape[3] > 1 and st[3] != 1):
        raise ValueError(f"{name}: the head dimension must be contiguous")
    return (ctypes.c_int64 * 3)(st[0], st[1], st[2])


def attn(q: np.ndarray, k: np.ndarray, v: np.ndarray, *, key_valid_len: int | None = None,
         scale: float | None = None, rows: np.ndarray | None = None, threads: int = 0,
         lib=None, allow: np.ndarray | None = None):
    """fp64 attention with LSE on bf16 inputs given as uint16 bit arrays.

    q: [B, Nq, H, D], k/v: [B, Nkv, H, D] -- any numpy views (strided views
    of a fused buffer included) whose last axis is contiguous.

    rows None  -> every query row; returns O [B, Nq, H, D], LSE [B, H, Nq].
    rows given -> an int array [B, H, R] of query rows per head; returns
                  O [B, H, R, D] and LSE [B, H, R] for those rows.
    Keys j >= key_valid_len are masked (default: none).  ``allow`` (optional,
    [B, Nq, >= key_valid_len], bool or uint8, last axis contiguous): query i
    may attend key j only where allow[b, i, j]; rows left with no key give
    O = 0, LSE = -inf.  ``lib`` selects another compiled copy of the oracle
    (the mutation tests use it).
    """
    lib = _load() if lib is None else lib
    B, Nq, H, D = q.shape
    Nkv = k.shape[1]
    if k.shape != (B, Nkv, H, D) or v.shape != (B, Nkv, H, D):
        raise ValueError("k and v must be [B, Nkv, H, D] with q's B, H, D")
    kvl = Nkv if key_valid_len is None else int(key_valid_len)
    sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
    qs, ks, vs = _bf16_view_strides(q, "q"), _bf16_view_strides(k, "k"), _bf16_view_strides(v, "v")
    full = rows is None
    if full:
        rows = np.broadcast_to(np.arange(Nq, dtype=np.int32), (B, H, Nq))
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    R = rows.shape[2]
    o = np.empty((B, H, R, D), dtype=np.float64)
    lse = np.empty((B, H, R), dtype=np.float64)
    al_ptr, al_sb, al_si = None, 0, 0
    if allow is not None:
        allow = np.asarray(allow)
        if allow.dtype == np.bool_:
            allow = allow.view(np.uint8)
        if allow.dtype != np.uint8 or allow.ndim != 3 or allow.shape[0] != B or allow.shape[1] != Nq \
                or allow.shape[2] < kvl or allow.strides[2] != 1:
            raise ValueError("allow must be a [B, Nq, >= key_valid_len] byte array, last axis contiguous")
        al_ptr, al_sb, al_si = allow.ctypes.data, allow.strides[0], allow.strides[1]
    for b in range(B):
        for h in range(H):
            r_bh = np.ascontiguousarray(rows[b, h])
            o_bh = np.empty((R, D), dtype=np.float64)
            l_bh = np.empty((R,), dtype=np.float64)
            rc = lib.oracle_attn_head_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, qs, ks, vs,
                                           Nq, Nkv, D, kvl, sc, b, h, r_bh.ctypes.data, R,
                                           o_bh.ctypes.data, l_bh.ctypes.data, int(threads),
                                           al_ptr, al_sb, al_si)
            if rc != 0:
                raise ValueError(f"oracle_attn_head_rows failed with {rc}")
            o[b, h] = o_bh
            lse[b, h] = l_bh
    if full:
        return np.ascontiguousarray(o.transpose(0, 2, 1, 3)), lse
    return o, lse


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Batched combine of n partial passes over disjoint key spans (fp64).

    o_parts [n, B, S, H, D], lse_parts [n, B, H, S] -> O [B, S, H, D], LSE [B, H, S].
    With M = max_k L_k and w_k = exp(L_k - M):  O = sum_k w_k O_k / sum_k w_k,
    LSE = M + ln sum_k w_k.  A chunk with L_k = -inf has weight 0; if every
    chunk is -inf the row is O = 0, LSE = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    M = lse_parts.max(axis=0)                                   # [B,H,S]
    empty = np.isneginf(M)
    Ms = np.where(empty, 0.0, M)
    w = np.exp(lse_parts - Ms[None])                            # [n,B,H,S], 0 for -inf
    lam = w.sum(axis=0)                                         # [B,H,S]
    wt = np.transpose(w, (0, 1, 3, 2))[..., None]               # [n,B,S,H,1]
    num = (wt * np.where(wt > 0, o_parts, 0.0)).sum(axis=0)     # [B,S,H,D]
    lam_t = np.transpose(lam, (0, 2, 1))[..., None]
    o = np.where(lam_t > 0, num / np.where(lam_t > 0, lam_t, 1.0), 0.0)
    lse = np.where(empty, -np.inf, Ms + np.log(np.where(empty, 1.0, lam)))
    return o, lse


def lse_merge_streaming(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Ring's streaming form of the same combine, one partial at a time (fp64).

    Running (O, L) absorbs (O_b, L_b) by
        O <- O - sigmoid(L_b - L) * (O - O_b)
        L <- L - log sigmoid(L - L_b)
    The sigmoid weight is evaluated as exp(L_b - L_new) with
    L_new = logaddexp(L, L_b); an all -inf pair leaves the state unchanged.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    O = np.zeros(o_parts.shape[1:], dtype=np.float64)
    L = np.full(lse_parts.shape[1:], -np.inf)
    for kk in range(o_parts.shape[0]):
        Lb = lse_parts[kk]
        Ob = o_parts[kk]
        both_empty = np.isneginf(L) & np.isneginf(Lb)
        with np.errstate(invalid="ignore"):
            Lnew = np.where(both_empty, -np.inf, np.logaddexp(L, Lb))
            sig = np.where(both_empty, 0.0, np.exp(Lb - np.where(both_empty, 0.0, Lnew)))
        sig_t = np.transpose(sig, (0, 2, 1))[..., None]
        Obs = np.where(sig_t > 0, Ob, 0.0)
        O = O - sig_t * (O - Obs)
        L = Lnew
    return O, L


def qkv_to_head_major(qkv: np.ndarray):
    """Split a fused [B, N, 3, H, D] buffer into three [B, H, N, D] arrays.

    out_t[b, h, n, d] = qkv[b, n, t, h, d] for t in (q, k, v): a pure copy.
    """
    if qkv.ndim != 5 or qkv.shape[2] != 3:
        raise ValueError("expected a [B, N, 3, H, D] array")
    return tuple(np.ascontiguousarray(qkv[:, :, t].transpose(0, 2, 1, 3)) for t in range(3))


# ------------------------------------------------------------------ FP8 E4M3
# E4M3 (the "fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
# bits; no infinities; S.1111.111 is NaN; largest finite 448 = 1.75 * 2^8;
# smallest normal 2^-6; subnormals m/8 * 2^-6, the smallest 2^-9.

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 bytes -> exact float64 values (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


def e4m3_encode(x) -> np.ndarray:
    """float64 -> E4M3 bytes: round to nearest, ties to even; magnitudes beyond
    448 saturate to +-448; NaN -> 0x7F; the sign of zero is kept."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    out = np.zeros(a.shape, dtype=np.int64)
    finite = np.isfinite(a)
    # normal range: exponent from frexp (a = f * 2^k, f in [0.5, 1))
    f, k = np.frexp(np.where(finite & (a > 0), a, 1.0))
    e = k - 1                                    # a = (2f) * 2^e, 2f in [1, 2)
    normal = finite & (a >= 2.0 ** -6)
    mant = np.rint((2.0 * f - 1.0) * 8.0)        # ties to even
    carry = mant >= 8
    e = np.where(carry, e + 1, e)
    mant = np.where(carry, 0, mant)
    code_n = ((e + 7) << 3) + mant.astype(np.int64)
    over = normal & ((e > 8) | ((e == 8) & (mant >= 7)))
    code_n = np.where(over, 0x7E, code_n)
    # subnormal range: multiples of 2^-9, ties to even (8 * 2^-9 is the smallest normal)
    code_s = np.rint(np.where(finite, a, 0.0) / 2.0 ** -9).astype(np.int64)
    out = np.where(normal, code_n, np.where(finite, code_s, 0x7E))
    out = np.where(np.isnan(x), 0x7F, out)
    out = np.where(neg, out | 0x80, out)
    return out.astype(np.uint8)


def qkv_cast_fp8(qkv_bits: np.ndarray, scales) -> np.ndarray:
    """One-pass cast of a stacked [B, N, 3, H, D] bf16 buffer (uint16 bits) to
    E4M3: out[b, n, t] = e4m3(x[b, n, t] * scales[t]) for t in (q, k, v)."""
    bits = np.asarray(qkv_bits, dtype=np.uint16)
    sc = np.asarray(scales, dtype=np.float32).reshape(1, 1, 3, 1, 1)
    out = np.empty(bits.shape, dtype=np.uint8)
    step = max(1, (1 << 22) // max(1, int(np.prod(bits.shape[2:]))))   # rows per slice, bounds the temporaries
    for n0 in range(0, bits.shape[1], step):
        x = bf16_bits_to_f64(bits[:, n0:n0 + step]).astype(np.float32)
        # the scaled value is formed in fp32 on the device: one fp32 rounding of
        # the product, then one E4M3 rounding; the same two roundings here
        out[:, n0:n0 + step] = e4m3_encode((x * sc).astype(np.float64))
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def e4m3_to_bf16_bits(codes: np.ndarray) -> np.ndarray:
    """Every finite E4M3 value is exactly a bf16 value (3 <= 7 mantissa bits,
    exponents 2^-9 .. 2^8); returns those bf16 bit patterns."""
    v = e4m3_decode(codes).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def attn_fp8(q8: np.ndarray, k8: np.ndarray, v8: np.ndarray, *, scale: float, descale_q: float,
             descale_k: float, descale_v: float, key_valid_len: int | None = None,
             rows: np.ndarray | None = None, threads: int = 0):
    """Attention on E4M3 inputs q8, k8, v8 ([B, N, H, D] uint8 views) that stand
    for Q = q8 * descale_q, K = k8 * descale_k, V = v8 * descale_v:
    softmax(scale * Q K^T) V and its LSE, in fp64, through ``attn``."""
    lut = e4m3_to_bf16_bits(np.arange(256, dtype=np.uint8))
    qb, kb, vb = (lut[np.asarray(a, dtype=np.uint8)] for a in (q8, k8, v8))
    O, L = attn(qb, kb, vb, key_valid_len=key_valid_len, scale=scale * descale_q * descale_k, rows=rows,
                threads=threads)
    return O * descale_v, L


# ------------------------------------------------- Q/K normalisation + RoPE
# "CUDA IPC Ulysses：在 H100 上重叠 Attention 通信", "基线与瓶颈": Q and K are
# normalised and rotated (RoPE) before attention, V is not; the pages give
# neither formula.  Reading taken here: RMSNorm over the head dimension,
#     y_d = x_d / sqrt(mean_d(x_d^2) + eps) * w_d,
# then the RoFormer rotation of consecutive pairs by per-position angles whose
# cosines and sines the caller tabulates ([N, D/2]; 1-D or 3-D positions alike):
#     (y_2i, y_2i+1) -> (y_2i c - y_2i+1 s,  y_2i s + y_2i+1 c),  c, s = cos/sin[n, i].

def rms_norm(x: np.ndarray, weight, eps: float) -> np.ndarray:
    """RMSNorm over the last axis in fp64; weight None = no scaling."""
    x = np.asarray(x, dtype=np.float64)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return y if weight is None else y * np.asarray(weight, dtype=np.float64)


def rope_pairs(y: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate consecutive pairs of the last axis; cos/sin broadcast against
    y[..., 0::2] (e.g. [N, 1, D/2] against [N, H, D/2])."""
    y = np.asarray(y, dtype=np.float64)
    c = np.asarray(cos, dtype=np.float64)
    s = np.asarray(sin, dtype=np.float64)
    out = np.empty_like(y)
    a, b = y[..., 0::2], y[..., 1::2]
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def qkv_norm_rope_to_head_major(qkv_bits: np.ndarray, q_weight, k_weight, eps: float, rope_cos, rope_sin):
    """Fused [B, N, 3, H, D] bf16 (uint16 bits) -> fp64 head-major q, k, v
    [B, H, N, D]: q and k RMS-normalised (weight None = no norm for that tensor)
    and rotated (tables None = no rotation), v copied."""
    x = bf16_bits_to_f64(qkv_bits)
    outs = []
    for t, w in ((0, q_weight), (1, k_weight), (2, None)):
        y = x[:, :, t]                                    # [B, N, H, D]
        if t < 2:
            if w is not None:
                y = rms_norm(y, w, eps)
            if rope_cos is not None:
                c = np.asarray(rope_cos, dtype=np.float64)[None, :, None, :]
                s = np.asarray(rope_sin, dtype=np.float64)[None, :, None, :]
                y = rope_pairs(y, c, s)
        outs.append(np.ascontiguousarray(np.transpose(y, (0, 2, 1, 3))))
    return tuple(outs)


def expand_mask(mask: np.ndarray, n_padded: int) -> np.ndarray:
    """The padding rule of "8 卡怎么分 token", "构造 padding mask", for a user
    (B, T, T) mask (True = may attend): expanded to (B, Tp, Tp), pad key
    columns j >= T are masked and pad query rows i >= T attend every valid key."""
    mask = np.asarray(mask, dtype=bool)
    B, T, T2 = mask.shape
    if T != T2 or n_padded < T:
        raise ValueError("mask must be (B, T, T) with T <= n_padded")
    out = np.zeros((B, n_padded, n_padded), dtype=bool)
    out[:, :T, :T] = mask
    out[:, T:, :T] = True
    return out

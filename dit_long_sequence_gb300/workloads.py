"""Workload shapes and seeded synthetic inputs.

This module only draws inputs and names shapes; it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle may use it.

Input recipe (the pages are silent on it): a ``torch.Generator`` on the target
device seeded with the workload's seed draws fp32 N(0, 1) values, rounded to
bf16 (round-to-nearest-even) -- q, then k, then v, or the whole fused
[B, N, 3, H, D] projection buffer in one draw.  The oracle reads the very same
bf16 bits copied to the host.

Shapes are model-shaped stand-ins for the pages' workloads (no weights or
datasets exist here): LTX-2 sequence-parallel padding, Cosmos 3 Nano's 44,160
video tokens, Wan 2.2 A14B's 21 x 45 x 80 latent grid, and a ring-style key
split into 9 chunks.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    D: int
    N: int                       # query and key rows (self-attention)
    seed: int
    key_valid_len: int | None = None   # None: no key mask
    fused: bool = False          # Q/K/V are strided views of one [B,N,3,H,D] buffer
    kv_chunks: int = 1           # >1: keys split into equal chunks, merged afterwards
    fp8: bool = False            # stacked bf16 buffer cast to E4M3, then FP8 attention
    description: str = ""

    @property
    def kv_len(self) -> int:
        return self.N if self.key_valid_len is None else self.key_valid_len

    @property
    def scale(self) -> float:
        return float(self.D) ** -0.5

    def flops(self) -> float:
        """Algorithmic attention FLOPs 4*B*H*Nq*Nkv*D over valid rows: with a
        tail key mask the pad query rows are cut after the gather, so both Nq
        and Nkv count the valid tokens only."""
        return 4.0 * self.B * self.H * self.kv_len * self.kv_len * self.D

    def executed_flops(self) -> float:
        """FLOPs the kernel actually performs: every query row, valid keys."""
        return 4.0 * self.B * self.H * self.N * self.kv_len * self.D


WORKLOADS = {
    "tiny": Workload("tiny", B=1, H=2, D=64, N=1024, seed=0,
                     description="tiny self-attention, whole-oracle parity case"),
    "ltx2_padded": Workload("ltx2_padded", B=1, H=32, D=128, N=24576, seed=1, key_valid_len=24200,
                            description="LTX-2-shaped padded sequence-parallel attention, "
                                        "24,200 valid tokens padded to 24,576, key-only mask"),
    "cosmos3_nano": Workload("cosmos3_nano", B=2, H=16, D=128, N=44160, seed=2, fused=True,
                             description="Cosmos-3-Nano-shaped, CFG batch 2, Q/K/V strided views "
                                         "of one fused [B,N,3*H*D] projection buffer"),
    "wan22_a14b": Workload("wan22_a14b", B=2, H=40, D=128, N=75600, seed=3,
                           description="Wan-2.2-A14B-shaped, CFG batch 2, 21x45x80 latent grid"),
    "ltx2_padded_fp8": Workload("ltx2_padded_fp8", B=1, H=32, D=128, N=24576, seed=1, key_valid_len=24200,
                                fused=True, fp8=True,
                                description="the LTX-2-shaped padded case on the FP8 path: one-pass E4M3 "
                                            "cast of the stacked [B,N,3,H,D] buffer, FP8 attention on it"),
    "wan22_a14b_fp8": Workload("wan22_a14b_fp8", B=2, H=40, D=128, N=75600, seed=3, fused=True, fp8=True,
                               description="the Wan-2.2-A14B-shaped case on the FP8 path"),
    "ring9": Workload("ring9", B=1, H=64, D=128, N=147456, seed=4, kv_chunks=9,
                      description="ring-style: keys split into 9 chunks of 16,384, "
                                  "(O, LSE) partials merged"),
}


# Per-tensor cast factors for N(0, 1) inputs: |x| stays below ~6.3 over 10^9
# draws, so 64 * |x| < 448, and 1/64 is an exact descale.
FP8_SCALES = (64.0, 64.0, 64.0)


def generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, seed: int, device="cpu", gen: torch.Generator | None = None) -> torch.Tensor:
    """fp32 N(0,1) from a seeded generator, rounded to bf16."""
    g = gen if gen is not None else generator(device, seed)
    return torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def randn_e4m3(shape, seed: int, scale: float, device="cpu") -> torch.Tensor:
    """E4M3 codes (uint8) of fp32 N(0,1) * scale from a seeded generator,
    clamped to +-448 and converted by torch's float8_e4m3fn: random FP8 inputs
    shaped like a calibrated cast's output, for both the kernels and the oracle."""
    x = torch.randn(tuple(shape), generator=generator(device, seed), device=device, dtype=torch.float32) * scale
    return x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def pack_mask_bits(mask, n_keys: int | None = None) -> torch.Tensor:
    """Bit-pack a boolean [B, R, Nk] mask (True = may attend; torch or numpy)
    into int32 words [B, R, W] on the host: bit (j & 31) of word j >> 5;
    W = 4 * ceil(n_keys / 128) (whole 128-key tiles, zero bits past Nk).  Input
    marshalling for the masked kernel."""
    m = mask.cpu().numpy() if isinstance(mask, torch.Tensor) else np.asarray(mask)
    B, R, Nk = m.shape
    nk = Nk if n_keys is None else max(int(n_keys), Nk)
    W = 4 * ((nk + 127) // 128)
    out = np.zeros((B, R, W), dtype=np.uint32)
    step = 4096
    for r0 in range(0, R, step):
        blk = np.zeros((B, min(step, R - r0), W * 32), dtype=bool)
        blk[:, :, :Nk] = m[:, r0:r0 + step]
        out[:, r0:r0 + step] = np.packbits(blk, axis=-1, bitorder="little").view("<u4")
    return torch.from_numpy(out.view(np.int32))


def rope_tables_3d(grid, D: int, base: float = 10000.0, device="cpu"):
    """Rotary angle tables for a flattened (T, Hh, W) latent grid: the D/2
    channel pairs are split over the three axes (1/4 time, 3/8 height, 3/8
    width), pair i of an axis with d_a pairs turning at base^(-i/d_a) per grid
    step.  Returns fp32 cos, sin [T*Hh*W, D/2] (angles formed in fp64).  An
    input generator for the rotary step, shaped like a video DiT's 3-D RoPE."""
    T, Hh, W = grid
    half = D // 2
    dt = half // 4
    dh = (half - dt) // 2
    dw = half - dt - dh
    t, h, w = torch.meshgrid(torch.arange(T, dtype=torch.float64), torch.arange(Hh, dtype=torch.float64),
                             torch.arange(W, dtype=torch.float64), indexing="ij")
    parts = []
    for pos, d in ((t, dt), (h, dh), (w, dw)):
        freq = base ** (-torch.arange(d, dtype=torch.float64) / d)
        parts.append(pos.reshape(-1, 1) * freq[None, :])
    ang = torch.cat(parts, dim=1)
    return ang.cos().to(torch.float32).to(device), ang.sin().to(torch.float32).to(device)


def make_qkv(B: int, N: int, H: int, D: int, seed: int, device="cpu", fused: bool = False,
             Nkv: int | None = None):
    """Seeded bf16 q, k, v as [B, N, H, D] tensors.

    fused=True: one [B, N, 3, H, D] buffer drawn in a single call; q, k, v are
    strided views into it (stride_n = 3*H*D), returned with the buffer.
    """
    if fused:
        if Nkv not in (None, N):
            raise ValueError("a fused buffer has one sequence length")
        buf = randn_bf16((B, N, 3, H, D), seed, device)
        return buf[:, :, 0], buf[:, :, 1], buf[:, :, 2], buf
    nkv = N if Nkv is None else Nkv
    g = generator(device, seed)
    q = randn_bf16((B, N, H, D), seed, device, g)
    k = randn_bf16((B, nkv, H, D), seed, device, g)
    v = randn_bf16((B, nkv, H, D), seed, device, g)
    return q, k, v, None


def make_workload_inputs(w: Workload, device="cpu"):
    return make_qkv(w.B, w.N, w.H, w.D, w.seed, device=device, fused=w.fused)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The bf16 bit patterns of a tensor as a host numpy uint16 view (strides kept)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    base = t if t.device.type == "cpu" else None
    if base is None:
        raise ValueError("copy the tensor to the host first")
    return t.view(torch.int16).numpy().view(np.uint16)


def host_bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a (possibly strided, possibly device) bf16 tensor's bits.

    Strided views of a larger buffer are copied together with their base so
    that the strides survive; the returned array is a numpy view with the same
    element strides as ``t``.
    """
    if t.device.type == "cpu":
        return bf16_bits(t)
    storage_elems = t.untyped_storage().nbytes() // 2
    base = torch.empty(0, dtype=torch.bfloat16, device=t.device).set_(
        t.untyped_storage(), 0, (storage_elems,), (1,))
    host = base.cpu()
    view = host.as_strided(t.shape, t.stride(), t.storage_offset())
    return bf16_bits(view)


def sample_rows(B: int, H: int, Nq: int, n_rows: int, seed: int, must=()) -> np.ndarray:
    """Distinct query rows per (b, h): [B, H, R] int32, R = min(n_rows, Nq).

    Rows 0 and Nq-1 and every row in ``must`` are always included; the rest are
    drawn with numpy's default_rng(1000 + seed).
    """
    rng = np.random.default_rng(1000 + int(seed))
    R = min(int(n_rows), Nq)
    forced = sorted({0, Nq - 1, *[int(m) for m in must if 0 <= int(m) < Nq]})[:R]
    out = np.empty((B, H, R), dtype=np.int32)
    pool = np.setdiff1d(np.arange(Nq, dtype=np.int64), np.asarray(forced, dtype=np.int64))
    for b in range(B):
        for h in range(H):
            extra = rng.choice(pool, size=R - len(forced), replace=False) if R > len(forced) else []
            out[b, h] = np.sort(np.concatenate([np.asarray(forced, dtype=np.int64),
                                                np.asarray(extra, dtype=np.int64)]))
    return out

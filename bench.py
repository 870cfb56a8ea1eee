"""Benchmark: attention TFLOP/s (4*B*H*Nq*Nkv*D) on one GB300, and its
fraction of the measured dense-bf16 peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the hot path over one batch of synthetic input.  The
default workload is ring9, the largest single-GPU configuration: B=1, H=64,
D=128, 147,456 tokens, the keys split into 9 chunks of 16,384.  Its step is 9
attention calls with LSE (dit_attn_fwd_ws: dit_attn_fwd with a workspace that
splits the grid's last partial wave over key ranges, plus the small kernel that
merges those pieces), each on one key chunk, writing its (O, LSE) partial
straight into a per-row interleaved buffer, then one dit_attn_lse_merge of the
9 partials.  Other workloads: ltx2_padded (split of the fused
[B, T, 3, H, D] projection into head-major Q/K/V by dit_qkv_to_head_major,
then attention with the key-only mask), cosmos3_nano (attention straight on
strided views of the fused buffer), wan22_a14b (separate Q/K/V),
ltx2_padded_fp8 / wan22_a14b_fp8 (one-pass E4M3 cast of the stacked buffer,
then dit_attn_fwd_fp8_ws).

Printed (rank 0, one JSON line): value = algorithmic FLOPs of all ranks / max
over ranks of the device time of K steps; e2e = the same metric through the
C ABI with the step's inputs copied from pinned host memory and O + LSE copied
back inside the timed region; roofline = the attention kernel timed with CUDA
events on its own stream inside the timed region, against the measured bf16
peak that matches how it ran (the sustained figure when the timed region saw
the power cap, else the burst figure); cpu_baseline = the fp64
oracle on a bounded row sample on the host cores.  Inputs exceed the 129 MB
L2, so no flush runs between steps.  N > 1 runs independent replicas (weak
scaling); the path has no cross-GPU exchange.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s (4*B*H*Nq*Nkv*D) and % of GB300 dense BF16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------- helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def choose_bf16_peak(peaks: dict, clocks: dict):
    """The bf16 denominator for the timed kernel: the sustained figure when the
    timed region ran under the power cap (sw_power_cap seen in the clock
    samples, as in the seconds-long GEMM loop that figure comes from), else the
    burst figure of a kernel timed alone.  Returns (peak TFLOP/s, kind)."""
    capped = "sw_power_cap" in (clocks or {}).get("reasons", [])
    if capped and peaks.get("bf16_tflops_sustained"):
        return float(peaks["bf16_tflops_sustained"]), "sustained (sw_power_cap active in the timed region)"
    return float(peaks["bf16_tflops"]), "burst"


def code_only(text: str) -> str:
    """C/C++ source with its comments removed and its whitespace collapsed
    (string and character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(main: str = "attn_fwd.cu") -> str:
    """Hash of the code an attention kernel is compiled from (its .cu, the PTX
    wrappers, the debug-check helpers and the kernel-argument header), comments
    and layout left out; host-only files are left out too."""
    h = hashlib.sha256()
    for fn in (main, "ptx.cuh", "debug.cuh", "internal.h"):
        with open(os.path.join(ROOT, "dit_long_sequence_gb300", "csrc", fn), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per attention call for this workload from the ncu record
    (profiles/dram_traffic.json), if it was taken on the current kernel
    source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path, encoding="utf-8") as f:
        rec = json.load(f)
    main = "attn_fwd_fp8.cu" if workload.endswith("_fp8") else "attn_fwd.cu"
    for e in rec.get("entries", []):
        if e.get("workload") == workload and e.get("kernel_source_sha256_16") == kernel_source_hash(main):
            return float(e["dram_bytes_per_call"])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples (every 50 ms); only samples taken
    inside [mark_start, mark_stop] count."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    _count = 0   # one file per sampler in this process

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None
        ClockSampler._count += 1
        self.path = os.path.join(tempfile.gettempdir(), f"dit_bench_clocks_{os.getpid()}_{ClockSampler._count}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.6)   # let the sampler start producing before the timed region
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        import datetime
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, cmax = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            if self.t0 is not None and not (self.t0 - 0.05 <= ts <= self.t1 + 0.05):
                continue
            sm.append(clk)
            smax = cmax
            for name, val in zip(names, parts[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": ["no sample inside the timed region"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "window_s": (self.t1 - self.t0) if self.t0 else None}


def dist_setup(n_gpus: int):
    """torchrun environment -> (rank, world, local_rank); N = 1 needs no process group."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def reduce_max(value: float) -> float:
    """Max over ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------------- the step

class Step:
    """Device buffers and the launch sequence of one step for a workload."""

    def __init__(self, w, dev):
        import torch
        import dit_long_sequence_gb300 as dl
        from dit_long_sequence_gb300 import workloads as wl
        self.w, self.dev, self.dl = w, dev, dl
        self.stream = torch.cuda.current_stream(dev)
        B, N, H, D = w.B, w.N, w.H, w.D
        base = w.name.split("_h")[0]
        self.mode = "cast+attn_fp8" if w.fp8 else ("layout+attn" if base in ("ltx2_padded", "tiny") else (
            "chunked+merge" if w.kv_chunks > 1 else "attn"))
        if self.mode == "layout+attn" or w.fused:
            # one fused [B, N, 3, H, D] projection buffer is the step's input
            self.inputs = [wl.randn_bf16((B, N, 3, H, D), w.seed, dev)]
        else:
            q, k, v, _ = wl.make_qkv(B, N, H, D, w.seed, device=dev)
            self.inputs = [q, k, v]
        if self.mode == "layout+attn":
            self.planes = tuple(torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev) for _ in range(3))
        if self.mode == "cast+attn_fp8":
            self.qkv8 = torch.empty((B, N, 3, H, D), dtype=torch.uint8, device=dev)
            self.descales = tuple(1.0 / x for x in wl.FP8_SCALES)
        if self.mode == "chunked+merge":
            n = w.kv_chunks
            # per-row interleaved partials [B, N, H, n, D]: the merge reads one stream
            self.o_buf = torch.empty((B, N, H, n, D), dtype=torch.float32, device=dev)
            self.o_parts = self.o_buf.permute(3, 0, 1, 2, 4)
            self.l_parts = torch.empty((n, B, H, N), dtype=torch.float32, device=dev)
        self.out = torch.empty((B, N, H, D), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        # attention calls get the tail-split workspace (none when the plan has no split)
        kvl_call = w.N // w.kv_chunks if self.mode == "chunked+merge" else w.kv_len
        nb = dl.attn_fwd_workspace_bytes(B, N, H, D, kvl_call)
        self.ws = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None
        # attention kernel (+ the split items' piece launch and the tail merge)
        per_attn = 3 if self.ws is not None else 1
        self.launches_per_step = {"layout+attn": 1 + per_attn, "attn": per_attn,
                                  "chunked+merge": w.kv_chunks * per_attn + 1, "cast+attn_fp8": 1 + per_attn}[self.mode]
        self.attn_events = []

    def qkv_of(self, inputs):
        """The [B, N, H, D] q, k, v views the attention reads for these inputs."""
        if self.mode == "layout+attn":
            return tuple(p.permute(0, 2, 1, 3) for p in self.planes)
        if self.mode == "cast+attn_fp8":
            return self.qkv8[:, :, 0], self.qkv8[:, :, 1], self.qkv8[:, :, 2]
        if len(inputs) == 1:
            f = inputs[0]
            return f[:, :, 0], f[:, :, 1], f[:, :, 2]
        return tuple(inputs)

    @property
    def q(self):
        return self.qkv_of(self.inputs)[0]

    @property
    def k(self):
        return self.qkv_of(self.inputs)[1]

    @property
    def v(self):
        return self.qkv_of(self.inputs)[2]

    def launch(self, inputs, out, lse, stream, record=False):
        """Enqueue one step reading `inputs` and writing (out, lse) on `stream`."""
        import torch
        dl, w = self.dl, self.w
        if self.mode == "layout+attn":
            dl.qkv_to_head_major(inputs[0], outs=self.planes, stream=stream)
        if self.mode == "cast+attn_fp8":
            from dit_long_sequence_gb300 import workloads as wl
            dl.qkv_cast_fp8(inputs[0], wl.FP8_SCALES, out=self.qkv8, stream=stream)
        q, k, v = self.qkv_of(inputs)
        ev = None
        if record:
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            ev[0].record(stream)
        if self.mode == "chunked+merge":
            n = w.kv_chunks
            cl = w.N // n
            for c in range(n):
                dl.attn_fwd_ws(q, k[:, c * cl:(c + 1) * cl], v[:, c * cl:(c + 1) * cl],
                               out=self.o_parts[c], lse=self.l_parts[c], workspace=self.ws, stream=stream)
        elif self.mode == "cast+attn_fp8":
            dl.attn_fwd_fp8_ws(q, k, v, self.descales, key_valid_len=w.key_valid_len, out=out, lse=lse,
                               workspace=self.ws, stream=stream)
        else:
            dl.attn_fwd_ws(q, k, v, key_valid_len=w.key_valid_len, out=out, lse=lse, workspace=self.ws,
                           stream=stream)
        if record:
            ev[1].record(stream)
            self.attn_events.append(ev)
        if self.mode == "chunked+merge":
            dl.lse_merge(self.o_parts, self.l_parts, out=out, lse_out=lse, stream=stream)

    def run(self, record=False):
        self.launch(self.inputs, self.out, self.lse, self.stream, record=record)

    def input_tensor(self):
        return self.inputs[0] if len(self.inputs) == 1 else None

    def attn_ms_per_launch(self):
        import torch
        torch.cuda.synchronize()
        times = [a.elapsed_time(b) for a, b in self.attn_events]
        per = self.w.kv_chunks if self.mode == "chunked+merge" else 1
        return statistics.mean(times) / per if times else float("nan")

    def attn_ms_median(self):
        import torch
        torch.cuda.synchronize()
        times = [a.elapsed_time(b) for a, b in self.attn_events]
        per = self.w.kv_chunks if self.mode == "chunked+merge" else 1
        return statistics.median(times) / per if times else float("nan")


def time_merge_kernel(dev, B, N, H, D, n_chunks=9, reps=5, interleaved=True):
    """HBM roofline of dit_attn_lse_merge on ring-style partials of this shape
    (chunks interleaved per row, or chunk-major)."""
    import torch
    import dit_long_sequence_gb300 as dl
    from dit_long_sequence_gb300 import workloads as wl
    g = wl.generator(dev, 77)
    if interleaved:
        o = torch.randn((B, N, H, n_chunks, D), generator=g, device=dev).permute(3, 0, 1, 2, 4)
    else:
        o = torch.randn((n_chunks, B, N, H, D), generator=g, device=dev)
    l = torch.randn((n_chunks, B, H, N), generator=g, device=dev) + 10.0
    out = torch.empty((B, N, H, D), device=dev)
    lo = torch.empty((B, H, N), device=dev)
    for _ in range(3):
        dl.lse_merge(o, l, out=out, lse_out=lo)
    s = torch.cuda.current_stream(dev)
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        dl.lse_merge(o, l, out=out, lse_out=lo)
        b.record(s)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    nbytes = (n_chunks + 1) * (B * N * H * D * 4 + B * H * N * 4)
    ms = statistics.median(ts)
    del o, l, out, lo
    return nbytes, ms


def time_layout_kernel(step, reps=5):
    """HBM roofline of the step's layout kernel: the QKV split (2 + 2 bytes per
    element) or the FP8 cast (2 + 1 bytes per element)."""
    import torch
    from dit_long_sequence_gb300 import workloads as wl
    if step.mode not in ("layout+attn", "cast+attn_fp8"):
        return None
    s = step.stream
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        if step.mode == "layout+attn":
            step.dl.qkv_to_head_major(step.inputs[0], outs=step.planes, stream=s)
        else:
            step.dl.qkv_cast_fp8(step.inputs[0], wl.FP8_SCALES, out=step.qkv8, stream=s)
        b.record(s)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    nbytes = step.inputs[0].numel() * (4 if step.mode == "layout+attn" else 3)
    return nbytes, statistics.median(ts)


def time_norm_rope_kernel(step, reps=5):
    """HBM roofline of the split with Q/K RMSNorm + 3-D RoPE fused in (2 + 2
    bytes per element; the fp32 angle tables are read from L2)."""
    import torch
    from dit_long_sequence_gb300 import workloads as wl
    if step.mode != "layout+attn":
        return None
    w = step.w
    grid = {24576: (16, 32, 48), 1024: (4, 16, 16)}.get(w.N)
    if grid is None:
        return None
    cos, sin = wl.rope_tables_3d(grid, w.D, device=step.dev)
    wq = torch.ones((w.D,), device=step.dev)
    wk = torch.ones((w.D,), device=step.dev)
    s = step.stream
    ts = []
    for i in range(reps + 2):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        step.dl.qkv_norm_rope_to_head_major(step.inputs[0], q_weight=wq, k_weight=wk, rope_cos=cos, rope_sin=sin,
                                            outs=step.planes, stream=s)
        b.record(s)
        b.synchronize()
        if i >= 2:
            ts.append(a.elapsed_time(b))
    return 2 * step.inputs[0].numel() * 2, statistics.median(ts)


def time_masked_attention(step, reps=3):
    """The general-mask variant (dit_attn_fwd_masked) on the step's q/k/v with
    (T, T) user masks over the valid tokens -- frame-local blocks of 1,512
    tokens plus ~5% hashed long-range links (no empty key tile), and the
    frame-local blocks alone (most key tiles empty: with and without the
    occupancy workspace) -- against the unmasked kernel, every call with the
    workspace that also splits the grid's last partial wave.  TFLOP/s counts
    the unmasked FLOPs, i.e. it is an equivalent rate."""
    import numpy as np
    import torch
    from dit_long_sequence_gb300 import workloads as wl
    w = step.w
    T = w.kv_len
    words = np.zeros((1, T, 4 * ((T + 127) // 128)), dtype=np.int32)
    cols = np.arange(T, dtype=np.int64)
    for r0 in range(0, T, 2048):
        r = np.arange(r0, min(T, r0 + 2048), dtype=np.int64)[:, None]
        m = ((r // 1512) == (cols[None, :] // 1512)) | (((r * 1103515245 + cols[None, :] * 12345 + 7) >> 9) % 20 == 0)
        words[0, r0:r0 + m.shape[0]] = wl.pack_mask_bits(m[None]).numpy()[0]
    bits = torch.from_numpy(words).to(step.dev)
    # frame-local blocks only (no long-range links): most key tiles are empty
    local = np.zeros_like(words)
    for r0 in range(0, T, 2048):
        r = np.arange(r0, min(T, r0 + 2048), dtype=np.int64)[:, None]
        local[0, r0:r0 + r.shape[0]] = wl.pack_mask_bits(((r // 1512) == (cols[None, :] // 1512))[None]).numpy()[0]
    local_bits = torch.from_numpy(local).to(step.dev)
    # the workspace holds the occupancy map and the tail split, as the unmasked call's does
    ws = torch.empty(max(16, step.dl.masked_split_workspace_bytes(w.B, w.N, w.H, w.D, T)), dtype=torch.uint8,
                     device=step.dev)
    ws_u = torch.empty(max(16, step.dl.attn_fwd_workspace_bytes(w.B, w.N, w.H, w.D, T)), dtype=torch.uint8,
                       device=step.dev)
    q, k, v = step.q, step.k, step.v
    s = step.stream
    out = {}
    for name, fn in (("masked", lambda: step.dl.attn_fwd_masked(q, k, v, bits, key_valid_len=T, out=step.out,
                                                                   lse=step.lse, workspace=ws, stream=s)),
                     ("masked_frame_local_skip", lambda: step.dl.attn_fwd_masked(
                         q, k, v, local_bits, key_valid_len=T, out=step.out, lse=step.lse, workspace=ws, stream=s)),
                     ("masked_frame_local_no_skip", lambda: step.dl.attn_fwd_masked(
                         q, k, v, local_bits, key_valid_len=T, out=step.out, lse=step.lse,
                         skip_empty_tiles=False, stream=s)),
                     ("unmasked", lambda: step.dl.attn_fwd_ws(q, k, v, key_valid_len=T, out=step.out, lse=step.lse,
                                                              workspace=ws_u, stream=s))):
        fn()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        out[name] = {"ms": ms, "TFLOP/s": w.flops() / (ms * 1e-3) / 1e12}
    density = float(np.unpackbits(words[0, :2048].view(np.uint8), bitorder="little").mean()) * \
        (words.shape[2] * 32) / T
    out["mask_density"] = density
    del bits
    return out


# --------------------------------------------------------------- cpu baseline

def cpu_baseline(w, dev_inputs=None, target_s=12.0):
    """The fp64 oracle as it stands, on a bounded sample of query rows of the
    workload (all keys), on the host cores.  Returns a dict in the metric's unit.
    FP8 workloads: dev_inputs are the E4M3 code views and the oracle's FP8
    attention runs on them."""
    import numpy as np
    import oracle
    from dit_long_sequence_gb300 import workloads as wl
    if dev_inputs is None:
        dev_inputs = baseline_inputs(w)
    q, k, v = dev_inputs
    if w.fp8:
        qb, kb, vb = (u8_host(t) for t in (q, k, v))
        d = tuple(1.0 / x for x in wl.FP8_SCALES)
    else:
        qb, kb, vb = wl.host_bf16_bits(q), wl.host_bf16_bits(k), wl.host_bf16_bits(v)
    kvl = w.key_valid_len
    per_row = 4.0 * w.kv_len * w.D

    def run(rows_per_head, heads):
        rows = wl.sample_rows(1, heads, w.N, rows_per_head, seed=w.seed)
        qs, ks, vs = qb[:1, :, :heads], kb[:1, :, :heads], vb[:1, :, :heads]
        t0 = time.perf_counter()
        if w.fp8:
            oracle.attn_fp8(qs, ks, vs, scale=w.scale, descale_q=d[0], descale_k=d[1], descale_v=d[2],
                            key_valid_len=kvl, rows=rows)
        else:
            oracle.attn(qs, ks, vs, key_valid_len=kvl, rows=rows)
        return time.perf_counter() - t0, rows.size

    heads = min(w.H, 8)
    rows_per_head = 4
    t, n = run(rows_per_head, heads)
    while t < 0.25 * target_s and rows_per_head < w.N:
        grow = 4 if t < 0.05 * target_s else max(1.2, 0.5 * target_s / max(t, 1e-6))
        rows_per_head = int(min(w.N, max(rows_per_head + 1, rows_per_head * grow)))
        t, n = run(rows_per_head, heads)
    if t < 0.6 * target_s and rows_per_head < w.N:
        rows_per_head = int(min(w.N, rows_per_head * target_s / max(t, 1e-6)))
        t, n = run(rows_per_head, heads)
    tflops = n * per_row / t / 1e12
    return {"value": tflops, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{n} query rows ({rows_per_head} per head, heads 0-{heads - 1} of batch 0) "
                      f"x all {w.kv_len} valid keys, fp64, {t:.1f} s",
            "rows_per_s": n / t, "seconds": t,
            "extrapolated_full_step_s": (w.flops() / per_row) / (n / t)}


def baseline_inputs(w, heads=8):
    """Host inputs of the CPU baseline: the workload's bf16 q, k, v; for FP8
    workloads the oracle's E4M3 cast of batch 0, heads < `heads` of the same
    seeded stacked buffer (all the sample reads)."""
    import torch
    import oracle
    from dit_long_sequence_gb300 import workloads as wl
    if not w.fp8:
        return wl.make_workload_inputs(w, device="cpu")[:3]
    buf = wl.randn_bf16((w.B, w.N, 3, w.H, w.D), w.seed, "cpu")[:1, :, :, :heads]
    codes = oracle.qkv_cast_fp8(wl.host_bf16_bits(buf.contiguous()), wl.FP8_SCALES)
    return tuple(torch.from_numpy(codes[:, :, t]) for t in range(3))


def u8_host(t):
    """Host numpy copy of a (possibly strided) uint8 view, strides kept."""
    import torch
    if t.device.type == "cpu":
        return t.numpy()
    n = t.untyped_storage().nbytes()
    base = torch.empty(0, dtype=torch.uint8, device=t.device).set_(t.untyped_storage(), 0, (n,), (1,))
    return base.cpu().as_strided(t.shape, t.stride(), t.storage_offset()).numpy()


# ------------------------------------------------------------------------ main

def run_reference(args, w):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    q, k, v = baseline_inputs(w)
    for _ in range(args.warmup):
        cpu_baseline(w, (q, k, v), target_s=1.0)
    if args.steps is None:
        args.steps = 5
    vals = [cpu_baseline(w, (q, k, v), target_s=max(2.0, 60.0 / max(args.steps, 1))) for _ in range(args.steps)]
    value = statistics.mean(v_["value"] for v_ in vals)
    secs = sum(v_["seconds"] for v_ in vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded bf16 N(0,1)" + (", cast to E4M3 by the oracle)" if w.fp8 else ")"),
            "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": vals[-1]["cores"], "kind": "oracle",
                             "sample": vals[-1]["sample"] + " per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def config_of(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "D": w.D, "seq_len": w.N,
            "key_valid_len": w.kv_len, "kv_chunks": w.kv_chunks, "fused_qkv": w.fused,
            "inputs": "e4m3 (one-pass cast of the stacked bf16 buffer, scales 64)" if w.fp8 else "bf16",
            "out_dtype": "fp32", "global_batch": w.B, "l2": "inputs larger than the 129 MB L2, no flush",
            "description": w.description}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about 1.5 s of timed work)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="ring9")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the head count (small profiling cases of the same kernel)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-kernel-legs", action="store_true",
                    help="skip the secondary HBM-kernel timing legs (small device footprint for profiling runs)")
    ap.add_argument("--masked", action="store_true",
                    help="also time the general-mask attention variant on this workload (bf16 workloads)")
    args = ap.parse_args(argv)
    from dit_long_sequence_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    if args.heads is not None:
        import dataclasses
        w = dataclasses.replace(w, H=args.heads, name=f"{w.name}_h{args.heads}")
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import dit_long_sequence_gb300 as dl

    step = Step(w, dev)
    t_warm = time.perf_counter()
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if args.steps is None:
        per = (time.perf_counter() - t_warm) / args.warmup
        args.steps = int(max(5, min(400, math.ceil(1.5 / max(per, 1e-4)))))
    rc, info = dl.check_watchdog()
    if rc != 0:
        raise RuntimeError(f"watchdog: {rc} {info}")

    # ---------------- device-timed region
    step.attn_events.clear()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        clk.mark_start()
        start.record(step.stream)
        for _ in range(args.steps):
            step.run(record=True)
        stop.record(step.stream)
        torch.cuda.synchronize()
        clk.mark_stop()
    barrier()
    ms_total = start.elapsed_time(stop)
    ms_total = reduce_max(ms_total)
    ms_per_step = ms_total / args.steps
    flops_step = w.flops()
    value = world * flops_step * args.steps / (ms_total * 1e-3) / 1e12
    attn_ms = step.attn_ms_per_launch()
    per_launch_flops = flops_step / (w.kv_chunks if w.kv_chunks > 1 else 1)
    peaks, peak_kind = load_peaks()
    bf16_peak = float(peaks["bf16_tflops"])
    clocks = clk.summary()
    bf16_use, use_kind = choose_bf16_peak(peaks, clocks)
    # FP8 contraction: the measured bf16 peak x the nominal fp8 / bf16 ratio (4.5 / 2.25)
    mult = 2.0 if w.fp8 else 1.0
    peak = mult * bf16_use
    achieved = per_launch_flops / (attn_ms * 1e-3) / 1e12
    traffic = profiled_traffic(w.name)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "kernel": "attn_fwd_fp8_kernel<false,false>" if w.fp8 else "attn_fwd_kernel<128,false,false,false,false>",
                "peak_kind": (f"{peak_kind} dense bf16 {use_kind} x 2 (nominal fp8/bf16 ratio)" if w.fp8
                              else f"{peak_kind} dense bf16 {use_kind}"),
                "frac_of_burst": achieved / (mult * bf16_peak),
                "frac_of_sustained": (achieved / (mult * float(peaks["bf16_tflops_sustained"]))
                                      if peaks.get("bf16_tflops_sustained") else None),
                "flops_per_launch": per_launch_flops, "ms_per_launch": attn_ms,
                "ms_per_launch_median": step.attn_ms_median()}
    ws_bytes = 0 if step.ws is None else step.ws.numel()
    call, kern = ("dit_attn_fwd_fp8_ws", "attn_fwd_fp8_kernel") if w.fp8 else ("dit_attn_fwd_ws", "attn_fwd_kernel")
    roofline["timed"] = (f"the {call} call: {kern}" +
                         (" (whole items and the split items' pieces) and attn_tail_merge_kernel" if ws_bytes
                          else " (no tail split for this shape)"))
    roofline["tail_split_workspace_bytes"] = ws_bytes

    # ---------------- secondary HBM-bound kernels
    extra = {}
    lay = None if args.no_kernel_legs else time_layout_kernel(step)
    if lay is not None:
        gbs = lay[0] / (lay[1] * 1e-3) / 1e9
        extra["cast_fp8" if w.fp8 else "layout"] = {"bytes": lay[0], "ms": lay[1], "GB/s": gbs, "frac_hbm": gbs / float(peaks["hbm_gbs"])}
    nr = None if args.no_kernel_legs else time_norm_rope_kernel(step)
    if nr is not None:
        gbs = nr[0] / (nr[1] * 1e-3) / 1e9
        extra["layout_norm_rope"] = {"bytes": nr[0], "ms": nr[1], "GB/s": gbs,
                                     "frac_hbm": gbs / float(peaks["hbm_gbs"])}
    for il, key in (() if args.no_kernel_legs else ((True, "merge_n9_interleaved"), (False, "merge_n9_chunk_major"))):
        mb, mms = time_merge_kernel(dev, w.B, w.N, w.H, w.D, n_chunks=9, interleaved=il)
        mgbs = mb / (mms * 1e-3) / 1e9
        extra[key] = {"bytes": mb, "ms": mms, "GB/s": mgbs, "frac_hbm": mgbs / float(peaks["hbm_gbs"])}

    if args.masked and not w.fp8:
        extra["attn_masked"] = time_masked_attention(step)

    # ---------------- end-to-end through host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(step, args, world)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3" if w.fp8 else "bf16",
            "data": "synthetic (seeded bf16 N(0,1), no weights)",
            "config": config_of(w), "roofline": roofline, "clocks": clocks,
            "gpu_launches": step.launches_per_step * args.steps, "e2e": e2e, "kernels": extra,
            "pct_of_bf16_peak": 100.0 * value / world / bf16_peak}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, (step.q, step.k, step.v))
    if rank == 0:
        print(json.dumps(line))
    return 0


def run_e2e(step, args, world):
    """Same metric through the C ABI with host buffers.  Every step copies its
    inputs from pinned host memory, runs, and copies O and LSE back; copies run
    on their own streams so that step i+1's upload and step i-1's download
    overlap step i's kernels (two device buffer sets, ordered by events)."""
    import torch
    dev = step.dev
    host_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in step.inputs]
    for h, d in zip(host_in, step.inputs):
        h.copy_(d)
    dev_in = [step.inputs, [torch.empty_like(t) for t in step.inputs]]
    dev_out = [(step.out, step.lse), (torch.empty_like(step.out), torch.empty_like(step.lse))]
    host_out = [(torch.empty(step.out.shape, dtype=step.out.dtype, pin_memory=True),
                 torch.empty(step.lse.shape, dtype=step.lse.dtype, pin_memory=True)) for _ in range(2)]
    s_comp = step.stream
    s_h2d = torch.cuda.Stream(device=dev)
    s_d2h = torch.cuda.Stream(device=dev)

    def pipeline(n_steps, t_start=None, t_end=None):
        comp_done, d2h_done = {}, {}
        if t_start is not None:
            t_start.record(s_h2d)
        for i in range(n_steps):
            slot = i & 1
            h2d_done = torch.cuda.Event()
            with torch.cuda.stream(s_h2d):
                if i >= 2:
                    s_h2d.wait_event(comp_done[i - 2])      # the inputs of step i-2 were consumed
                for h, d in zip(host_in, dev_in[slot]):
                    d.copy_(h, non_blocking=True)
                h2d_done.record(s_h2d)
            s_comp.wait_event(h2d_done)
            if i >= 2:
                s_comp.wait_event(d2h_done[i - 2])          # step i-2's result has been read back
            o, l = dev_out[slot]
            step.launch(dev_in[slot], o, l, s_comp)
            comp_done[i] = torch.cuda.Event()
            comp_done[i].record(s_comp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(comp_done[i])
                host_out[slot][0].copy_(o, non_blocking=True)
                host_out[slot][1].copy_(l, non_blocking=True)
                d2h_done[i] = torch.cuda.Event()
                d2h_done[i].record(s_d2h)
        if t_end is not None:
            s_d2h.wait_event(comp_done[n_steps - 1])
            t_end.record(s_d2h)

    pipeline(3)
    torch.cuda.synchronize()
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # No nvidia-smi sampling in this window: its polling slowed this three-stream
    # pipeline (9.35 vs 6.71 ms per step over 40 LTX-2 steps), while the
    # single-stream device window above shows no such effect.
    pipeline(args.steps, a, b)
    torch.cuda.synchronize()
    barrier()
    ms = reduce_max(a.elapsed_time(b))
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = host_out[0][0].numel() * host_out[0][0].element_size() + host_out[0][1].numel() * host_out[0][1].element_size()
    return {"value": world * step.w.flops() * args.steps / (ms * 1e-3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / args.steps,
            "pipelined": "uploads and downloads on copy streams overlap the neighbouring steps' kernels"}


if __name__ == "__main__":
    sys.exit(main())

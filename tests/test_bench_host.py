"""Host logic of bench.py, on the CPU: the multi-rank reduction (two gloo ranks),
the FLOP accounting, clock-sample filtering, the choice of the roofline's
peak, the profile-hash gate on the reported DRAM traffic, and a bounded
CPU-baseline sample."""
import json
import math
import os
import socket
import sys
import time

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from dit_long_sequence_gb300 import workloads as wl  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    r, w, _ = bench.dist_setup(world)
    bench.barrier()
    got = bench.reduce_max(1.5 + r)           # per-rank "elapsed time"
    bench.barrier()
    q.put((r, w, got))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(o[0] for o in out) == [0, 1]
    assert all(o[1] == world and o[2] == 2.5 for o in out)


def test_single_process_needs_no_group():
    os.environ.pop("WORLD_SIZE", None)
    assert bench.reduce_max(3.25) == 3.25
    with pytest.raises(SystemExit):
        os.environ["WORLD_SIZE"] = "2"
        try:
            bench.dist_setup(1)
        finally:
            os.environ.pop("WORLD_SIZE", None)


def test_flops_and_config():
    w = wl.WORKLOADS["ltx2_padded"]
    assert w.flops() == 4.0 * 1 * 32 * 24200 * 24200 * 128
    assert w.executed_flops() == 4.0 * 1 * 32 * 24576 * 24200 * 128
    c = bench.config_of(w)
    assert c["workload"] == "ltx2_padded" and c["key_valid_len"] == 24200 and c["seq_len"] == 24576
    assert "larger than" in c["l2"]
    # every workload's inputs exceed the 129 MB L2 except the tiny parity case
    for name, wk in wl.WORKLOADS.items():
        if name != "tiny":
            assert 3 * wk.B * wk.N * wk.H * wk.D * 2 > 129e6


def test_clock_samples_outside_the_window_are_ignored(tmp_path):
    clk = bench.ClockSampler(0)
    clk.path = str(tmp_path / "clocks.csv")
    t0 = time.time()
    rows = [
        (t0 - 5.0, 900, "Active"),     # before the window: ignored
        (t0 + 0.10, 2000, "Not Active"),
        (t0 + 0.20, 2070, "Not Active"),
        (t0 + 0.30, 1990, "Active"),   # sw_power_cap active inside the window
        (t0 + 9.00, 500, "Active"),    # after the window: ignored
    ]
    with open(clk.path, "w") as f:
        for ts, mhz, cap in rows:
            stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(ts)) + f".{int((ts % 1) * 1000):03d}"
            f.write(f"{stamp}, 0, {mhz}, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, {cap}\n")
    clk.proc = object()            # pretend the sampler ran
    clk.t0, clk.t1 = t0, t0 + 0.5
    s = clk.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2000 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_traffic_only_reported_for_the_profiled_kernel_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "dit_long_sequence_gb300" / "csrc")
    for fn in ("attn_fwd.cu", "ptx.cuh", "debug.cuh", "internal.h"):
        (tmp_path / "dit_long_sequence_gb300" / "csrc" / fn).write_text(f"int {fn.replace('.', '_')};")
    h = bench.kernel_source_hash()
    rec = {"entries": [{"workload": "w", "kernel_source_sha256_16": h, "dram_bytes_per_call": 1.5e9}]}
    (prof / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench.profiled_traffic("w") == 1.5e9
    assert bench.profiled_traffic("other") is None
    # a comment or a layout change keeps the capture valid; a code change voids it
    src = tmp_path / "dit_long_sequence_gb300" / "csrc" / "attn_fwd.cu"
    src.write_text("// a note\nint   attn_fwd_cu; /* more */\n")
    assert bench.profiled_traffic("w") == 1.5e9
    src.write_text("int attn_fwd_cu = 1;")
    assert bench.profiled_traffic("w") is None
    src.write_text("int attn_fwd_cu;")
    rec["entries"][0]["kernel_source_sha256_16"] = "0000000000000000"
    (prof / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench.profiled_traffic("w") is None


def test_code_only_drops_comments_but_keeps_literals():
    src = 'int a = 1; // x "y"\n/* multi\n line */ const char* s = "p // q /* r */"; char c = \'"\';'
    assert bench.code_only(src) == 'int a = 1; const char* s = "p // q /* r */"; char c = \'"\';'
    assert bench.code_only("a  \n\t b") == "a b"


def test_peak_is_the_sustained_figure_only_under_the_power_cap():
    peaks = {"bf16_tflops": 1896.7, "bf16_tflops_sustained": 1693.2}
    assert bench.choose_bf16_peak(peaks, {"reasons": []}) == (1896.7, "burst")
    v, kind = bench.choose_bf16_peak(peaks, {"reasons": ["sw_power_cap"]})
    assert v == 1693.2 and kind.startswith("sustained")
    assert bench.choose_bf16_peak({"bf16_tflops": 1900.0}, {"reasons": ["sw_power_cap"]})[0] == 1900.0
    assert bench.choose_bf16_peak(peaks, {"reasons": ["clock sampling unavailable"]})[0] == 1896.7


def test_cpu_baseline_is_bounded_and_in_the_metric_unit():
    w = wl.WORKLOADS["tiny"]
    t0 = time.perf_counter()
    cb = bench.cpu_baseline(w, target_s=0.5)
    assert time.perf_counter() - t0 < 30
    assert cb["kind"] == "oracle" and cb["unit"] == "TFLOP/s" and cb["cores"] >= 1
    assert cb["value"] > 0 and math.isfinite(cb["value"])
    json.dumps(cb)

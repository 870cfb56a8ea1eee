"""Host-side checks of the tail-split plan (plan_tail_split and
split_workspace_bytes in csrc/split_plan.h), compiled into a small host
program with g++ -- no GPU needed.

The plan cuts the last partial wave of work items (items mod SMs of them)
into f key ranges.  Checked here: the properties it must have for any input
(no split for a whole number of waves, f in [2, 8], every range at least 16
key tiles, at most one wave of pieces when the grid is a single partial
wave, the workspace holding every piece's partial O and LSE), and the plans
of the benchmark's shapes on a 152-SM GB300.
"""
import itertools
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dit_long_sequence_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include "split_plan.h"
int main() {
    long long items; int tiles, sms, D;
    while (std::scanf("%lld %d %d %d", &items, &tiles, &sms, &D) == 4) {
        const dit::SplitPlan p = dit::plan_tail_split(items, tiles, sms);
        std::printf("%lld %d %lld %lld\n", (long long)p.first, p.f, (long long)p.n_ctas,
                    (long long)dit::split_workspace_bytes(p, D));
    }
    return 0;
}
"""


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda.h")):
            return os.path.join(d, "include")
    return None


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    inc = _cuda_include()
    if shutil.which("g++") is None or inc is None:
        pytest.skip("needs g++ and the CUDA headers")
    d = tmp_path_factory.mktemp("plan")
    src, exe = d / "plan.cpp", d / "plan"
    src.write_text(HARNESS)
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, "-I", inc, str(src), "-o", str(exe)], check=True)

    def run(cases):
        text = "".join(f"{i} {t} {s} {D}\n" for i, t, s, D in cases)
        out = subprocess.run([str(exe)], input=text, capture_output=True, text=True, check=True).stdout.split("\n")
        return [tuple(int(x) for x in line.split()) for line in out if line.strip()]
    return run


def test_properties_over_a_grid_of_inputs(plan):
    cases = [(items, tiles, sms, D)
             for items, tiles, sms, D in itertools.product(
                 [1, 7, 8, 64, 151, 152, 153, 200, 303, 304, 3072, 5536, 23680, 36864],
                 [0, 1, 15, 16, 31, 32, 47, 63, 128, 190, 345, 591],
                 [148, 152], [64, 128])]
    for (items, tiles, sms, D), (first, f, n_ctas, nbytes) in zip(cases, plan(cases)):
        tail = items % sms
        if f == 1:
            assert (first, n_ctas, nbytes) == (items, 0, 0)
            # no split only when there is nothing to gain or too few keys
            assert tail == 0 or tiles < 32 or (items < sms and 2 * tail > sms)
            continue
        assert 2 <= f <= 8
        assert first == items - tail and n_ctas == tail * f
        assert tiles // f >= 16                                   # every range >= 16 key tiles
        if items < sms:
            assert n_ctas <= sms                                  # one wave of pieces
        o_bytes = n_ctas * 256 * D * 4
        assert nbytes >= o_bytes + n_ctas * 256 * 4 and nbytes % 256 == 0
        assert nbytes - o_bytes - n_ctas * 256 * 4 < 256          # LSE part padded to 256 bytes only


def test_benchmark_shapes_on_152_sms(plan):
    def items(B, N, H):
        return B * H * ((N + 255) // 256)
    cases = [
        (items(1, 24576, 32), (24200 + 127) // 128, 152, 128),   # LTX-2: 3,072 items, 32 left over
        (items(2, 44160, 16), 345, 152, 128),                    # Cosmos: 64 left over
        (items(2, 75600, 40), 591, 152, 128),                    # Wan: 120 left over
        (items(1, 147456, 64), 128, 152, 128),                   # a ring-9 chunk: 80 left over
        (items(1, 1024, 2), 8, 152, 64),                         # tiny: too few key tiles
    ]
    got = plan(cases)
    assert got[0][:3] == (3040, 4, 128) and got[0][3] == 128 * 256 * 128 * 4 + 128 * 256 * 4
    assert got[1][:3] == (5472, 2, 128)
    assert got[2][:3] == (23560, 2, 240)
    assert got[3][:3] == (36784, 2, 160)
    assert got[4][:3] == (8, 1, 0)

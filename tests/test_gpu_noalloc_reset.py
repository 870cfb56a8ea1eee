"""dit_attn_fwd_masked_noalloc across cudaDeviceReset, from a plain C program.

The entry point takes its tile-occupancy scratch from a fixed array in the
library's module and caches the array's device address per CUDA context.
After cudaDeviceReset the runtime loads the module into a new primary context
where the array has a new address; a cache keyed only on the device would hand
the kernel a stale address.  tests/harness/noalloc_after_reset.c (no PyTorch,
its own cudaMalloc'd buffers) runs the call, resets the device and runs it
again: the two results must be bit-identical and the watchdog clean.

libditattn.so carries the CUDA runtime statically, so a reset issued through
another runtime instance would not reach the library's own module.  The test
therefore links the already-built objects of the library once more against the
shared runtime, into a temporary copy, so that the program and the library
share one runtime and the reset is the library's own.
"""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime.h")):
            return d
    pytest.skip("no CUDA toolkit headers")


def test_noalloc_call_is_right_after_a_device_reset(tmp_path):
    from dit_long_sequence_gb300 import build
    build.build()
    cuda = _cuda_home()
    cc = shutil.which("gcc") or "gcc"
    exe = tmp_path / "noalloc_after_reset"
    lib_dir = str(tmp_path)
    objs = [os.path.join(build.BUILD, os.path.splitext(s)[0] + ".o") for s in build.SOURCES]
    subprocess.run([build.nvcc()] + build.ARCH + ["-shared", "-cudart", "shared", "-o",
                                                  os.path.join(lib_dir, "libditattn.so")] + objs, check=True)
    cmd = [cc, "-O2", "-std=c11", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "harness", "noalloc_after_reset.c"), "-o", str(exe),
           "-L", lib_dir, "-lditattn", "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    subprocess.run(cmd, check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr

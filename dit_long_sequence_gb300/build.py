"""Builds libditattn.so in-tree with nvcc for sm_103a (no cmake, no torch).

    python -m dit_long_sequence_gb300.build [--force] [--verbose]

Each .cu under csrc/ compiles to an object in parallel, then one shared-library
link: dit_long_sequence_gb300/_build/libditattn.so.  The same sources compiled
with -DDIT_DEBUG (in-kernel bounds checks and fault injection,
include/dit_attn_debug.h) give _build/debug/libditattn_debug.so, built in the
same parallel pass.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libditattn.so")
DEBUG_BUILD = os.path.join(BUILD, "debug")
DEBUG_LIB = os.path.join(DEBUG_BUILD, "libditattn_debug.so")
SOURCES = ["api.cu", "attn_fwd.cu", "attn_fwd_fp8.cu", "qkv_cast_fp8.cu", "lse_merge.cu", "qkv_layout.cu",
           "qkv_norm_rope.cu", "mask_occupancy.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (CUDA toolkit required to build libditattn.so)")
    return cand


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool = True) -> str:
    """Builds libditattn.so (and, with debug=True, libditattn_debug.so) if
    a source is newer; returns the product library's path."""
    targets = [(LIB, BUILD, [])]
    if debug:
        targets.append((DEBUG_LIB, DEBUG_BUILD, ["-DDIT_DEBUG"]))
    targets = [t for t in targets if force or not up_to_date(t[0])]
    if not targets:
        return LIB
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(job):
        src, out_dir, defs = job
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + common + defs + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src} {' '.join(defs)}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(f"== {src} {' '.join(defs)}\n" + r.stderr)
        return obj

    jobs = []
    for lib, out_dir, defs in targets:
        os.makedirs(out_dir, exist_ok=True)
        jobs += [(src, out_dir, defs) for src in SOURCES]
    with ThreadPoolExecutor(max_workers=min(len(jobs), max(4, os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, jobs))
    for lib, out_dir, _ in targets:
        mine = [o for o in objs if os.path.dirname(o) == out_dir]
        tmp = lib + f".tmp{os.getpid()}"
        r = subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + mine, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ns = ap.parse_args()
    print(build(force=ns.force, verbose=ns.verbose))

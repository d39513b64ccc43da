"""Compile liblora.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into
``segmented_gemm_gb300/liblora.so``; the same sources compiled with
``-DLORA_DEBUG`` (segment-table checks before every use, kernels that test
table-derived row indices) are linked into ``liblora_debug.so`` beside it.
The CUDA runtime is linked statically so the library only needs the driver
at run time.  Usage: ``python -m segmented_gemm_gb300.build [--force]
[--verbose]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "liblora.so")
DEBUG_LIB_PATH = os.path.join(PKG, "liblora_debug.so")

SOURCES = ["lora_api.cu", "seg_build.cu", "fused_tc.cu", "fused_splitk.cu", "fused_cluster.cu",
           "lora_noalloc.cu", "moe.cu", "widen.cu", "seg_check.cu", "stage.cu", "moe_pair.cu"]
VARIANTS = ((LIB_PATH, "", []), (DEBUG_LIB_PATH, "debug", ["-DLORA_DEBUG"]))
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "lora.h"))
    return files


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in _deps() + [src, __file__])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile both variants (all translation units in one pool) and link
    each library whose objects changed; returns the normal library's path."""
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                     "--expt-relaxed-constexpr"]
    if verbose:
        common += ["-Xptxas", "-v"]
    jobs, objs, relink = [], {}, {}
    for lib, sub, defs in VARIANTS:
        odir = os.path.join(BUILD_DIR, sub) if sub else BUILD_DIR
        os.makedirs(odir, exist_ok=True)
        objs[lib] = [os.path.join(odir, s.replace(".cu", ".o")) for s in SOURCES]
        relink[lib] = force or not os.path.exists(lib)
        for src, o in zip(SOURCES, objs[lib]):
            s = os.path.join(CSRC, src)
            if force or _stale(o, s):
                jobs.append([nvcc, "-c", s, "-o", o] + common + defs)
                relink[lib] = True

    def run(cmd):
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        return cmd, r.returncode, r.stdout

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for cmd, rc, out in ex.map(run, jobs):
            if verbose or rc:
                sys.stdout.write(out)
            if rc:
                raise RuntimeError(f"nvcc failed ({rc}) for {cmd[2]}")
    for lib, _, _ in VARIANTS:
        if not relink[lib]:
            continue
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, "-shared", "-o", tmp] + objs[lib] + ARCH + ["-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode:
            sys.stdout.write(r.stdout)
            raise RuntimeError("nvcc link failed")
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv)
    print(LIB_PATH)

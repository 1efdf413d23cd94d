"""Build libdspark.so in-tree with nvcc for sm_103a (no GPU needed).

    python -m semi_autoregressive_speculative_gb300.build [--force] [--trace]

Each translation unit compiles in parallel; the objects link into
``semi_autoregressive_speculative_gb300/lib/libdspark.so`` with a static CUDA
runtime, so the library loads on any host with the NVIDIA driver.
``--trace`` builds ``lib/libdspark_trace.so`` instead: the same sources with
the draft kernel's phase stamps compiled in (-DDSPARK_DRAFT_TRACE), for the
``draft_trace`` tool; the product library never carries them.
"""
from __future__ import annotations

import argparse
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libdspark.so")
OBJDIR = os.path.join(PKG, "_build")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


TRACE_LIB = os.path.join(LIBDIR, "libdspark_trace.so")


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    lib = TRACE_LIB if trace else LIB
    objdir = os.path.join(OBJDIR, "trace") if trace else OBJDIR
    defines = ["-DDSPARK_DRAFT_TRACE"] if trace else []
    if not force and up_to_date(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    procs = []
    objs = []
    for src in _sources():
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [NVCC, *ARCH, *FLAGS, *defines, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(f) for f in failed))
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([NVCC, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--trace", action="store_true", help="build lib/libdspark_trace.so (draft phase stamps)")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose, trace=args.trace))

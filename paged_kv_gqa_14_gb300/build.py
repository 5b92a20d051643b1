"""Build the CUDA library in-tree: paged_kv_gqa_14_gb300/_build/libpkv.so (sm_103a only).

Each translation unit is compiled by its own nvcc process in parallel, then linked into a
shared library against the shared CUDA runtime.  Rebuilds only when a source or header is
newer than the library.  ``python -m paged_kv_gqa_14_gb300.build [--force] [--verbose]``.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpkv.so")

# (source, object name, extra flags): decode_tc.cu is built once per pool block size
SOURCES = [("abi.cu", "abi.o", []), ("kv_append.cu", "kv_append.o", []), ("attention.cu", "attention.o", []),
           ("noalloc.cu", "noalloc.o", []), ("copy.cu", "copy.o", [])] + [
    ("decode_tc.cu", f"decode_tc_bs{bs}.o", [f"-DPKV_DECODE_TC_BS={bs}"]) for bs in (8, 16, 32, 64, 128)]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# No --use_fast_math: sincosf in the RoPE kernel stays the accurate library routine; the
# kernels call fast approximations (ex2.approx) explicitly where they want them.
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _inputs():
    files = [os.path.join(INCLUDE, "pkv.h")]
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")):
            files.append(os.path.join(CSRC, f))
    return files


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link; returns the library path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src, oname, extra in SOURCES:
        obj = os.path.join(BUILD, oname)
        cmd = [cc, *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((oname, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_info or p.returncode):
            print(f"--- {src}\n{out}", flush=True)
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv, ptxas_info="--ptxas" in sys.argv)
    print(LIB)

"""Build libkt.so (CUDA, sm_103a) in-tree with nvcc.

Each translation unit is compiled in parallel to an object file under _build/,
then linked into block_sparse_long_quest_gb300/libkt.so.  Objects are rebuilt
when their source, the internal header or the public header changed.
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
LIB = os.path.join(PKG, "libkt.so")
SOURCES = ["kt_api.cu", "attn.cu", "select.cu", "reps.cu", "dynamic.cu", "preselect.cu",
           "quant.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas: bool):
    f = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-I", INCLUDE,
         "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, "kt_internal.cuh"), os.path.join(INCLUDE, "kt.h")]
    hdr_time = max(os.path.getmtime(h) for h in headers)
    objs, procs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        stale = (force or verbose_ptxas or not os.path.exists(o)
                 or os.path.getmtime(o) < max(os.path.getmtime(s), hdr_time))
        if stale:
            cmd = [nvcc(), *_flags(verbose_ptxas), "-c", s, "-o", o]
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out.strip():
            sys.stderr.write(f"[nvcc {src}]\n{out}\n")
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    if procs or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        # nvcc links the CUDA runtime statically by default
        subprocess.check_call([nvcc(), *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)

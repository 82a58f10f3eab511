"""Builds libdit_attn.so in-tree for sm_103a (nvcc, no cmake).

Each translation unit compiles in parallel into ``_build/``; the objects link into
``video_dit_attention_gb300/libdit_attn.so`` with the CUDA runtime linked statically, so the
library loads on a machine without a GPU driver (it only needs one to run kernels).

The same objects, with the attention kernels compiled again under DIT_TEST_HOOKS, also link
into ``libdit_attn_testhooks.so``: a test-only library whose bounded waits a test can shorten
and make run out (include/dit_attn_test_hooks.h). The product code never loads it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdit_attn.so")
TEST_LIB = os.path.join(HERE, "libdit_attn_testhooks.so")
TEST_HOOK_SOURCES = ["attn_fwd.cu", "cross_attn.cu"]   # recompiled with -DDIT_TEST_HOOKS for the test library
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_SOURCES = ["attn_fwd.cu", "cross_attn.cu", "elementwise.cu", "fp8.cu", "api.cu"]
CXX_SOURCES = ["rope_table.cpp"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdit_attn.so")


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compiles and links the library; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC"]
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        cmd = [nvcc, *ARCH, "-lineinfo", *common, "--expt-relaxed-constexpr", "-c",
               os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append((cmd, obj))
    test_objs = {}
    for src in TEST_HOOK_SOURCES:
        obj = os.path.join(BUILD, src + ".testhooks.o")
        cmd = [nvcc, *ARCH, "-lineinfo", *common, "--expt-relaxed-constexpr", "-DDIT_TEST_HOOKS", "-c",
               os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, obj))
        test_objs[src + ".o"] = obj
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        jobs.append(([nvcc, *common, "-x", "c++", "-c", os.path.join(CSRC, src), "-o", obj], obj))
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(lambda j: _run(j[0]), jobs))
    if verbose:
        for o in outs:
            if o.strip():
                print(o)
    product = [o for _, o in jobs if not o.endswith(".testhooks.o")]
    tmp = LIB + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *product])
    os.replace(tmp, LIB)
    test = [test_objs.get(os.path.basename(o), o) for o in product]
    tmp = TEST_LIB + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *test])
    os.replace(tmp, TEST_LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))

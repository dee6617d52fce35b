"""Build libdflash.so in-tree from csrc/*.cu for sm_103a.

Each translation unit compiles in parallel with nvcc; the objects link into one
shared library next to this file. Rebuilds only what changed. Usable as
``python -m block_diffusion_speculative_fusion_gb300.build``.

``build(debug=True)`` makes libdflash_debug.so from the same sources with
DFLASH_DEBUG defined: the kernels then also record, in the workspace error
word, the inputs that release builds clamp without a record (context and
commit lengths out of range, committed rows without a pool slot).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdflash.so")
LIB_DEBUG = os.path.join(HERE, "libdflash_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdflash")
    return cand


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def build(verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    objdir = OBJDIR + "_debug" if debug else OBJDIR
    lib = LIB_DEBUG if debug else LIB
    os.makedirs(objdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_mtime = max([os.path.getmtime(h) for h in _headers()] + [os.path.getmtime(__file__)])
    flags = NVCC_FLAGS + (["-DDFLASH_DEBUG"] if debug else []) + list(extra_flags or [])
    procs = []
    objs = []
    for src in srcs:
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_mtime):
            continue
        cmd = [nvcc()] + ARCH + flags + ["-I", INCLUDE, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose and text.strip():
            print(text, flush=True)
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    newest = max(os.path.getmtime(o) for o in objs)
    if procs or not os.path.exists(lib) or os.path.getmtime(lib) < newest:
        tmp = lib + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(tmp, lib)
    if not debug:
        _build_tools(verbose)
    return lib


TOOLS = os.path.join(HERE, "tools")
HOST_COST = os.path.join(OBJDIR, "abi_host_cost")


def _build_tools(verbose: bool = False) -> None:
    """The C harness that times the ABI's per-call host cost (bench.py runs it)."""
    src = os.path.join(TOOLS, "abi_host_cost.c")
    if not os.path.exists(src):
        return
    newest = max(os.path.getmtime(src), os.path.getmtime(LIB), os.path.getmtime(os.path.join(INCLUDE, "dflash.h")))
    if os.path.exists(HOST_COST) and os.path.getmtime(HOST_COST) >= newest:
        return
    cmd = [nvcc(), "-O2", "-o", HOST_COST, src, "-I", INCLUDE, "-L", HERE, "-ldflash", "-lcudart",
           "-Xlinker", f"-rpath={HERE}"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("abi_host_cost build failed:\n" + r.stdout.decode(errors="replace"))


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))

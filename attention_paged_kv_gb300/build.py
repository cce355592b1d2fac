"""Build ``libpagedattn.so`` in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel; the CUDA runtime is linked
statically and only the ``pagedattn_*`` symbols of include/pagedattn.h are
exported, so the library can share a process with PyTorch's own runtime.
``python -m attention_paged_kv_gb300.build`` runs it from the command line.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import time

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedattn.so")
SOURCES = ["api.cu", "plan.cpp", "prefill.cu", "decode.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libpagedattn")


def _common_flags():
    return ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
            "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"] + ARCH


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile every source and link the shared library; returns its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = nvcc_path()
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in ("common.cuh", "internal.h", "layout.h")] + \
        [os.path.join(ROOT, "include", "pagedattn.h")]
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(d) for d in deps)
        if os.path.getmtime(LIB) >= newest:
            return LIB
    t0 = time.time()
    procs = []
    objs = []
    for s in srcs:
        obj = os.path.join(OUT_DIR, os.path.basename(s) + ".o")
        objs.append(obj)
        cmd = [nvcc, "-c", s, "-o", obj] + _common_flags() + ["-Xptxas", "-v"]
        log = open(obj + ".log", "w")
        procs.append((subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log, cmd, obj))
    failed = []
    for p, log, cmd, obj in procs:
        rc = p.wait()
        log.close()
        if rc != 0:
            failed.append((cmd, open(obj + ".log").read()))
    if failed:
        msg = "\n\n".join(" ".join(c) + "\n" + out[-6000:] for c, out in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    vs = os.path.join(OUT_DIR, "exports.map")
    with open(vs, "w") as f:
        f.write("{ global: pagedattn_*; local: *; };\n")
    tmp = LIB + ".tmp"
    link = [nvcc, "-shared", "-o", tmp] + objs + ARCH + [
        "--cudart", "static", "-Xlinker", "--version-script=" + vs, "-Xlinker", "--exclude-libs,ALL"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB} in {time.time() - t0:.1f}s")
    return LIB


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv)

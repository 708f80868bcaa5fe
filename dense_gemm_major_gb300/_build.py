"""In-tree build of the CUDA library (libdense_gemm.so) for sm_103a.

Each translation unit under csrc/ is compiled by its own nvcc process, in
parallel, then linked into one shared library next to this file.  A unit is
recompiled only when it or a header it may include is newer than its object.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(ROOT, "_build", "obj")
LIB = os.path.join(PKG, "libdense_gemm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
# Extra nvcc flags for measurement builds (for example
# -DDENSE_GEMM_L2_HINT=1); a change of them rebuilds every unit.
EXTRA_FLAGS = os.environ.get("DENSE_GEMM_NVCC_FLAGS", "").split()
FLAGS_STAMP = os.path.join(OBJ_DIR, "flags.txt")


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def build(verbose: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(OBJ_DIR, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest_header = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    flags_text = " ".join(EXTRA_FLAGS)
    try:
        with open(FLAGS_STAMP) as f:
            flags_changed = f.read() != flags_text
    except OSError:
        flags_changed = bool(EXTRA_FLAGS)
    procs = []
    objs = []
    for src in sources:
        obj = os.path.join(OBJ_DIR, os.path.basename(src) + ".o")
        objs.append(obj)
        stale = (flags_changed or not os.path.exists(obj)
                 or os.path.getmtime(obj) < os.path.getmtime(src)
                 or os.path.getmtime(obj) < newest_header)
        if not stale and not ptxas_verbose:
            continue
        cmd = [nvcc()] + NVCC_FLAGS + EXTRA_FLAGS + (["-Xptxas", "-v"] if ptxas_verbose else []) + \
            ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif text.strip() and (verbose or ptxas_verbose):
            print(f"--- {os.path.basename(src)}\n{text}", file=sys.stderr)
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    with open(FLAGS_STAMP, "w") as f:
        f.write(flags_text)
    if procs or not os.path.exists(LIB) or any(os.path.getmtime(LIB) < os.path.getmtime(o) for o in objs):
        cmd = [nvcc()] + ARCH + ["-shared", "-o", LIB] + objs + ["-lcuda"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.check_call(cmd)
    return LIB


if __name__ == "__main__":
    build(verbose=True, ptxas_verbose="-v" in sys.argv)

"""Builds the FLARE++ CUDA library in-tree with nvcc for sm_103a.

Produces ``rank_latent_routing_gb300/_lib/libflarepp.so`` (a plain C-ABI
shared library; the CUDA runtime is linked statically). Translation units are
compiled in parallel, then linked.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
# FLAREPP_TRACE=1 selects the pipeline-trace build, kept in a folder of its own
# so that it never stands in for the normal library
TRACE = os.environ.get("FLAREPP_TRACE") == "1"
LIBDIR = os.path.join(PKG, "_lib_trace" if TRACE else "_lib")
LIB = os.path.join(LIBDIR, "libflarepp.so")
SOURCES = ["flarepp.cu", "tc.cu", "proj.cu", "backward.cu", "flarepp_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: the FLARE++ library needs the CUDA toolkit to build")
    return p


def _flags() -> list[str]:
    trace = ["-DFLAREPP_TRACE"] if TRACE else []
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                   "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"] + trace


def _deps() -> list[str]:
    files = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile (if sources changed) and return the library path."""
    if not force and not ptxas_info and up_to_date():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    objs = []

    def compile_one(src: str) -> str:
        obj = os.path.join(LIBDIR, os.path.splitext(src)[0] + ".o")
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + _flags()
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or ptxas_info or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}")
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(len(SOURCES), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [cc, "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)

"""Build the vc_* shared libraries in-tree with nvcc for sm_103a.

    python -m verify_compressed_kv_gb300.build [--jobs N] [--verbose]

Outputs ``verify_compressed_kv_gb300/lib/libvc_*.so``.  libvc_core is built
first; the four compute libraries link against it with an $ORIGIN rpath, and
are compiled in parallel.
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
LIBDIR = os.path.join(PKG, "lib")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]

LIBS = {
    "vc_quant_kv": ["vc_quant_kv.cu"],
    "vc_draft_attn": ["vc_draft_attn.cu"],
    "vc_verify_attn": ["vc_verify_attn.cu"],
    "vc_accept": ["vc_accept.cu"],
}


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the vc_* libraries")


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout, r.stderr, flush=True)
    return r


def build(jobs: int = 4, verbose: bool = False, extra_flags=None) -> list[str]:
    os.makedirs(LIBDIR, exist_ok=True)
    nv = nvcc()
    extra = list(extra_flags or [])
    core = os.path.join(LIBDIR, "libvc_core.so")
    _run([nv, *ARCH, *COMMON, *extra, "-shared", os.path.join(CSRC, "vc_core.cpp"), "-o", core], verbose)

    def one(item):
        name, srcs = item
        out = os.path.join(LIBDIR, f"lib{name}.so")
        cmd = [nv, *ARCH, *COMMON, *extra, "-shared", *[os.path.join(CSRC, s) for s in srcs],
               "-L", LIBDIR, "-lvc_core", "-Xlinker", "-rpath,$ORIGIN", "-o", out]
        _run(cmd, verbose)
        return out

    with ThreadPoolExecutor(max(1, jobs)) as ex:
        outs = list(ex.map(one, LIBS.items()))
    return [core, *outs]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--jobs", type=int, default=4)
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-v", action="store_true", help="print register / smem usage")
    a = ap.parse_args(argv)
    flags = ["-Xptxas", "-v"] if a.ptxas_v else []
    for p in build(a.jobs, a.verbose or a.ptxas_v, flags):
        print(p)


if __name__ == "__main__":
    sys.exit(main())

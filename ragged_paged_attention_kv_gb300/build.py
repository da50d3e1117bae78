"""Builds librpa.so (the C-ABI CUDA library) in-tree for sm_103a.

    python -m ragged_paged_attention_kv_gb300.build [--force] [--verbose]

Each translation unit under csrc/ is compiled by nvcc in parallel, then
linked into ragged_paged_attention_kv_gb300/librpa.so.  Sources are rebuilt
only when they (or a header) are newer than their object.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "librpa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=(), defines=None):
    # RPA_NVCC_DEFINES: extra -D options (e.g. "-DRPA_DECODE_UNITS_TARGET=2048") for tuning builds
    if defines is None:
        defines = os.environ.get("RPA_NVCC_DEFINES", "").split()
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr", *defines, *extra]


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(obj, deps):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, obj, verbose, ptxas_verbose, defines=None):
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    cmd = [_nvcc(), *_flags(extra, defines), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
    if verbose:
        print(" ".join(cmd))
    return r.stderr


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          variant: str = None, defines=None) -> str:
    """Builds librpa.so; with `variant` (a name) and `defines` (-D options), a
    separate copy built with those options under _build/variants/<name>/ --
    for tests that need a build-time setting the product never uses (a
    short wait limit, say).  Returns the library's path."""
    obj_dir, lib = OBJ_DIR, LIB
    if variant is not None:
        obj_dir = os.path.join(OBJ_DIR, "variants", variant)
        lib = os.path.join(obj_dir, "librpa.so")
        defines = list(defines or [])
    os.makedirs(obj_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = _headers()
    jobs = []
    objs = []
    for src in sources:
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or ptxas_verbose or _stale(obj, [src, *headers]):
            jobs.append((src, obj))
    logs = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            futs = [ex.submit(_compile, s, o, verbose, ptxas_verbose, defines) for s, o in jobs]
            for f in futs:
                logs.append(f.result())
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)
    if ptxas_verbose:
        print("\n".join(logs))
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas", action="store_true", help="print -Xptxas -v resource usage")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose, ptxas_verbose=args.ptxas))


if __name__ == "__main__":
    sys.exit(main())

"""Build libflashsinkhorn.so for sm_103a in-tree (no cmake, no pip install).

Each ``csrc/*.cu`` translation unit is compiled by its own nvcc process, in
parallel, then linked into ``streaming_sinkhorn_solver_gb300/libflashsinkhorn.so``.
Objects go to ``streaming_sinkhorn_solver_gb300/_build/``.  A unit is rebuilt
when it or any header it may include is newer than its object.

    python -m streaming_sinkhorn_solver_gb300.build [--force] [--verbose] [--debug-bounds]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libflashsinkhorn.so")
# debug build: global-memory index checks of the FMA, prep and block-sparse
# kernels (-DFS_DEBUG_BOUNDS), reported by fs_debug_bounds()
OUT_DBG = os.path.join(PKG, "_build_dbg")
LIB_DBG = os.path.join(PKG, "libflashsinkhorn_dbg.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(src: str, obj: str, newest_header: float) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return os.path.getmtime(src) > t or newest_header > t


def build(force: bool = False, verbose: bool = False, extra_flags=None,
          debug_bounds: bool = False) -> str:
    out_dir, lib_path = (OUT_DBG, LIB_DBG) if debug_bounds else (OUT, LIB)
    os.makedirs(out_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdrs = _headers()
    newest = max((os.path.getmtime(h) for h in hdrs), default=0.0)
    flags = NVCC_FLAGS + list(extra_flags or []) + (["-DFS_DEBUG_BOUNDS"] if debug_bounds else [])
    jobs = []
    for src in sources:
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        if force or _stale(src, obj, newest):
            jobs.append((src, obj))

    def compile_one(job):
        src, obj = job
        cmd = [nvcc()] + ARCH + flags + ["-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(compile_one, jobs))
    objs = [os.path.join(out_dir, os.path.basename(s)[:-3] + ".o") for s in sources]
    if force or jobs or not os.path.exists(lib_path) or any(
            os.path.getmtime(o) > os.path.getmtime(lib_path) for o in objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print register/spill report")
    ap.add_argument("--debug-bounds", action="store_true",
                    help="build libflashsinkhorn_dbg.so with global-memory index checks")
    args = ap.parse_args()
    extra = ["-Xptxas", "-v"] if args.ptxas_info else []
    print(build(force=args.force or args.ptxas_info, verbose=args.verbose or args.ptxas_info,
                extra_flags=extra, debug_bounds=args.debug_bounds))


if __name__ == "__main__":
    main()

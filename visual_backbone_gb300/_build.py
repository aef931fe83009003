"""Build of libvh.so: every CUDA source compiled for sm_103a, in parallel, then linked.

The library links the CUDA runtime statically and needs no driver library at
link time, so it loads (and exports its symbols) on machines without a GPU.
``build(debug=True)`` makes libvh_dbg.so instead: the same sources with VH_DEBUG_BOUNDS
defined, so the scan kernels check their indices (counted in stats[VH_STAT_BOUNDS]).
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libvh.so")
LIB_DEBUG = os.path.join(HERE, "libvh_dbg.so")
SOURCES = ["vh_api.cu", "vh_scan_simt.cu", "vh_scan_tc.cu", "vh_scan_tc64.cu", "vh_scan_bwd.cu",
           "vh_qproj.cu", "vh_qproj_tc.cu", "vh_block.cu", "vh_gemm_tc.cu", "vh_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            f"-I{INCLUDE}", f"-I{CSRC}", *extra]


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "vh.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False,
          debug: bool = False) -> str:
    """Compile csrc/*.cu to objects in parallel and link libvh.so (libvh_dbg.so with
    debug=True) in place."""
    lib = LIB_DEBUG if debug else LIB
    if not force and not _stale(lib):
        return lib
    bdir = BUILD_DIR + ("_dbg" if debug else "")
    os.makedirs(bdir, exist_ok=True)
    procs = []
    extra = ["-Xptxas", "-v"] if ptxas_v else []
    if debug:
        extra.append("-DVH_DEBUG_BOUNDS")
    for src in SOURCES:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [NVCC, *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                  stderr=subprocess.STDOUT, text=True)))
    objs, errors = [], []
    for src, obj, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"{src}:\n{out}")
        elif (verbose or ptxas_v) and out:
            print(out, file=sys.stderr)
        objs.append(obj)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.check_call([NVCC, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_v="--ptxas-v" in sys.argv,
          debug="--debug" in sys.argv)

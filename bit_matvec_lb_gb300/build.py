"""Build liblb.so (the C-ABI library) in-tree with nvcc for sm_103a only.

    python -m bit_matvec_lb_gb300.build          # or bit_matvec_lb_gb300.build.build()

Each .cu under csrc/ is compiled in parallel to an object, then linked with the static CUDA
runtime into bit_matvec_lb_gb300/_build/liblb.so.  Only the lb_* entry points are exported.
The instruction-rate probes under probe/ (a measurement library the bench loads, not part of
the C ABI) are linked the same way into _build/liblbprobe.so.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "liblb.so")
PROBE = os.path.join(HERE, "probe")
PROBE_LIB = os.path.join(BUILD, "liblbprobe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
              "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the GB300 library cannot be built")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "lb.h")]


def _probe_sources():
    return sorted(glob.glob(os.path.join(PROBE, "*.cu")))


def up_to_date() -> bool:
    for lib, deps in ((LIB, _deps()), (PROBE_LIB, _deps() + _probe_sources())):
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if not all(os.path.getmtime(p) <= t for p in deps):
            return False
    return True


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every csrc/*.cu for sm_103a and link liblb.so; returns its path."""
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    psrcs = _probe_sources()
    srcs = _sources() + psrcs
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(src, obj):
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        list(ex.map(lambda p: compile_one(*p), zip(srcs, objs)))
    nprobe = len(psrcs)
    for lib, lobjs in ((LIB, objs[:len(objs) - nprobe]), (PROBE_LIB, objs[len(objs) - nprobe:])):
        if not lobjs:
            continue
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *lobjs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

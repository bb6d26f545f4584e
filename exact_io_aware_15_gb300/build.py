"""Builds the in-tree shared library ``_lib/libfa_gb300.so`` from ``csrc/``.

Each translation unit is compiled for sm_103a in parallel with nvcc, then the
objects are linked into one shared library (CUDA runtime linked statically,
driver API reached through the runtime's entry-point query, so the library has
no libcuda link dependency).  Outputs go under ``_lib/`` next to this file and
are not committed.

A second library, ``_lib/libfa_gb300_debug.so``, is linked from the same
objects except the tensor-core forward, which is compiled with -DFA_DEBUG:
its kernels then check every shared-memory, tensor-memory and output index
range before use and report a failed check as FA_ERR_DEVICE_BOUNDS (the
binding loads it when FA_GB300_LIBRARY names it; the tests use it to run the
odd-shaped forward cases under those checks).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT, "libfa_gb300.so")
DEBUG_LIB = os.path.join(OUT, "libfa_gb300_debug.so")
DEBUG_SOURCES = ["fwd_tc.cu"]  # compiled a second time with -DFA_DEBUG
SOURCES = ["fa_api.cu", "fwd_tc.cu", "fwd_f32.cu", "decode.cu", "combine.cu",
           "decode_noalloc.cu", "bwd_tc.cu", "rowstats.cu", "scan.cu",
           "decode_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I" + os.path.join(ROOT, "include"), "-I" + CSRC,
                   "--expt-relaxed-constexpr", *extra]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
               if f.endswith((".cuh", ".h"))] + [
        os.path.join(ROOT, "include", "fa_gb300.h")]
    cc = nvcc()
    objs = []
    debug_objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, *headers]):
            extra = ["-Xptxas", "-v"] if ptxas_info else []
            jobs.append([cc, *_flags(extra), "-c", s, "-o", o])
        if src in DEBUG_SOURCES:
            od = os.path.join(OUT, src.replace(".cu", ".debug.o"))
            debug_objs.append(od)
            if force or _stale(od, [s, *headers]):
                jobs.append([cc, *_flags(["-DFA_DEBUG"]), "-c", s, "-o", od])
        else:
            debug_objs.append(o)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or ptxas_info or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError("nvcc failed: " + " ".join(cmd))
    for lib, lib_objs in ((LIB, objs), (DEBUG_LIB, debug_objs)):
        if force or jobs or _stale(lib, lib_objs):
            cmd = [cc, *ARCH, "-shared", "-o", lib + ".tmp", *lib_objs]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
                raise RuntimeError("link failed")
            os.replace(lib + ".tmp", lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv, force="-f" in sys.argv))

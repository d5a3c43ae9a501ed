"""Build libmla.so (the CUDA library behind include/mla.h) in-tree with nvcc.

    python -m mla_latent_kv_71_b300.build [--force] [--verbose] [--checks]

Compiles csrc/mla_lib.cu (one translation unit) for sm_103a only and writes
mla_latent_kv_71_b300/libmla.so.  The CUDA runtime is linked statically; the
driver's tensor-map encoder is looked up at run time, so the library needs
no link against libcuda.  --checks builds libmla_checks.so instead, with
MLA_CHECKS=1: the kernels also check their work split (page ranges, partial
slots, GEMM items) against the shapes, raising the device status word on a
violation, and fill their shared memory with NaN before use, so that a read
of a byte no copy wrote shows up in the results.  The binding loads it when
the environment variable MLA_CHECKS is 1.
"""

from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmla.so")
LIB_CHECKS = os.path.join(HERE, "libmla_checks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmla.so")
    return cand


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + [os.path.join(ROOT, "include", "mla.h")])


def stale(checks: bool = False) -> bool:
    lib = LIB_CHECKS if checks else LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False, extra=(), checks: bool = False) -> str:
    lib = LIB_CHECKS if checks else LIB
    if not force and not stale(checks):
        return lib
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
           *(["-DMLA_CHECKS=1"] if checks else []),
           *(["-Xptxas", "-v"] if verbose else []), *extra,
           os.path.join(CSRC, "mla_lib.cu"), "-o", lib + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose:
        sys.stderr.write(r.stdout + r.stderr)
    os.replace(lib + ".tmp", lib)
    return lib


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas resource usage")
    ap.add_argument("--checks", action="store_true", help="build libmla_checks.so (MLA_CHECKS=1)")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, checks=a.checks))


if __name__ == "__main__":
    main()

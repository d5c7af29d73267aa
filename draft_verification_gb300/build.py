"""Build libspecverify.so in-tree for sm_103a (GB300) with nvcc.

    python -m draft_verification_gb300.build          # or build() from Python

Each translation unit is compiled in parallel, then linked into one shared
library next to this file (draft_verification_gb300/lib/).  Only nvcc and
the host compiler are needed; no CMake, no torch extension machinery.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "lib")
LIB_NAME = "libspecverify.so"
SOURCES = ["verify.cu", "api.cu", "noalloc.cu", "compact.cu", "clasp.cu", "pipeline_async.cu", "lm_head.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-Xptxas", "-v"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: set CUDA_HOME or put nvcc on PATH")


DEBUG_DIR = os.path.join(PKG, "lib_debug")


def lib_path(debug_checks: bool | None = None) -> str:
    """The library to load: the debug-checks build when debug_checks is true,
    or (None) when the environment variable SPEC_VERIFY_DEBUG_CHECKS is 1."""
    if debug_checks is None:
        debug_checks = os.environ.get("SPEC_VERIFY_DEBUG_CHECKS") == "1"
    return os.path.join(DEBUG_DIR if debug_checks else OUT_DIR, LIB_NAME)


def _newer(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(verbose: bool = False, force: bool = False, debug_checks: bool = False) -> str:
    """Compile every translation unit and link the library; returns its path.
    debug_checks builds the variant whose vector loads and bulk copies check
    their alignment preconditions (-DSPEC_DEBUG_CHECKS) into lib_debug/."""
    nvcc = nvcc_path()
    out_dir = DEBUG_DIR if debug_checks else OUT_DIR
    os.makedirs(out_dir, exist_ok=True)
    extra = ["-DSPEC_DEBUG_CHECKS"] if debug_checks else []
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "spec_verify.h"))
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or not _newer(o, [s] + headers):
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", s, "-o", o]
            jobs.append((src, cmd))

    def run(job):
        name, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return name, cmd, r

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for name, cmd, r in ex.map(run, jobs):
            if r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
                raise RuntimeError(f"nvcc failed on {name}: {' '.join(cmd)}")
            if verbose:
                sys.stderr.write(f"[build] {name}\n{r.stderr}")
    lib = lib_path(debug_checks)
    if force or jobs or not os.path.exists(lib):
        cmd = [nvcc, *ARCH, "-shared", "-o", lib, *objs, "-lcudart", "-lcublas"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed: " + " ".join(cmd))
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug_checks="--debug-checks" in sys.argv))

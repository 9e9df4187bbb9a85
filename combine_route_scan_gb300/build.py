"""Build the CUDA library libcrs_moe.so (sm_103a) in-tree.

Each .cu file compiles to its own object in parallel with nvcc, then nvcc links
them into combine_route_scan_gb300/_build/libcrs_moe.so. The CUDA runtime is
linked statically. No cmake.

``build(observer=True)`` builds the flag-observer test variant
(_build/observer/libcrs_moe.so, ``-DMOE_FLAG_OBSERVER``): the dispatch payload
grid's last CTA watches the ready flags and copies each segment the moment its
flag is set, so that a test can check that no flag is visible before its rows.
The binding loads it when the environment variable CRS_MOE_OBSERVER is 1.

``build(phase=True)`` builds the phase-time test variant
(_build/phase/libcrs_moe.so, ``-DMOE_PHASE_TIMES``): every kernel records its
earliest CTA start, its CTAs' passage of the wait for the previous kernel and
its latest CTA end (%globaltimer) for tests/test_phase_times_gpu.py; loaded
when CRS_MOE_PHASE is 1.

``build(checked=True)`` builds the bounds-checked variant
(_build/checked/libcrs_moe.so, ``-DMOE_BOUNDS_CHECK``): every index a kernel
derives from data is checked against its buffer, and a miss records
MOE_ERR_OUT_OF_BOUNDS and skips the access. The binding loads it when the
environment variable CRS_MOE_CHECKED is 1.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libcrs_moe.so")
CHECKED_DIR = os.path.join(OUT_DIR, "checked")
CHECKED_LIB = os.path.join(CHECKED_DIR, "libcrs_moe.so")
OBSERVER_DIR = os.path.join(OUT_DIR, "observer")
OBSERVER_LIB = os.path.join(OBSERVER_DIR, "libcrs_moe.so")
PHASE_DIR = os.path.join(OUT_DIR, "phase")
PHASE_LIB = os.path.join(PHASE_DIR, "libcrs_moe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs_mtime() -> float:
    files = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files.append(os.path.join(os.path.dirname(HERE), "include", "moe.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra_flags=None, checked: bool = False,
          observer: bool = False, phase: bool = False) -> str:
    out_dir, lib = ((CHECKED_DIR, CHECKED_LIB) if checked else (OBSERVER_DIR, OBSERVER_LIB) if observer else
                    (PHASE_DIR, PHASE_LIB) if phase else (OUT_DIR, LIB))
    os.makedirs(out_dir, exist_ok=True)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _inputs_mtime():
        return lib
    cc = nvcc()
    flags = (NVCC_FLAGS + list(extra_flags or []) + (["-DMOE_BOUNDS_CHECK"] if checked else []) +
             (["-DMOE_FLAG_OBSERVER"] if observer else []) + (["-DMOE_PHASE_TIMES"] if phase else []))
    if verbose:
        flags = flags + ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv, checked="--checked" in sys.argv))

"""Builds libfp4moe.so (the CUDA library behind include/fp4moe.h) in-tree.

nvcc compiles each translation unit for sm_103a in parallel and links a
shared library next to this file.  Rebuilds only when a source is newer than
the library.  Usable as ``python -m block_scaled_fp4_02_gb300.build``
(``--checked`` for the bounds-checked variant).

Two variants come from the same sources: "release" (libfp4moe.so) and
"checked" (libfp4moe_checked.so, compiled with FP4MOE_BOUNDS_CHECK: every
data-dependent index is checked before its access and a failure records
FP4MOE_ERR_BOUNDS in the device status word).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfp4moe.so")
VARIANTS = {
    "release": (LIB, BUILD, []),
    "checked": (os.path.join(HERE, "libfp4moe_checked.so"),
                os.path.join(BUILD, "checked"), ["-DFP4MOE_BOUNDS_CHECK"]),
}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-O2", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required")
    return cand


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(CSRC, "*.h"))
            + [os.path.join(ROOT, "include", "fp4moe.h"), __file__])


def lib_path(variant: str = "release") -> str:
    return VARIANTS[variant][0]


def up_to_date(variant: str = "release") -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False,
          extra_flags: list[str] | None = None, variant: str = "release") -> str:
    lib, bdir, vflags = VARIANTS[variant]
    if not force and up_to_date(variant):
        return lib
    nvcc = _nvcc()
    os.makedirs(bdir, exist_ok=True)
    flags = NVCC_FLAGS + vflags + (extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *flags, "-I", os.path.join(ROOT, "include"),
               "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(max(1, len(sources()))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if v else None
    variant = "checked" if "--checked" in sys.argv else "release"
    print(build(force=True, verbose=v, extra_flags=extra, variant=variant))

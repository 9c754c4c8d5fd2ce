"""Build libkivi.so (the CUDA library behind include/kivi.h) in-tree with nvcc.

Each translation unit is compiled in parallel for sm_103a only, then linked
into a shared library next to this file.  IEEE division and denormals are kept
(no --use_fast_math): the encode kernels must reproduce fp32 IEEE quotients.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkivi.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-prec-div=true", "-ftz=false", "-prec-sqrt=true",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libkivi")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__])


# Variants: "" (the library) and "checked" (KIVI_CHECKS defined: the streamed
# decode checks every copy range, tile and output row on the device and
# reports a failed check as KIVI_ECHECK in its workspace status word).
VARIANT_FLAGS = {"": [], "checked": ["-DKIVI_CHECKS"]}


def lib_path(variant: str = "") -> str:
    return LIB if not variant else os.path.join(HERE, f"libkivi_{variant}.so")


def needs_build(variant: str = "") -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          variant: str = "") -> str:
    """Compile libkivi.so (or the variant's library) if missing or stale;
    return its path."""
    lib = lib_path(variant)
    if not (force or needs_build(variant)):
        return lib
    bdir = BUILD if not variant else BUILD + "_" + variant
    os.makedirs(bdir, exist_ok=True)
    nv = nvcc()
    flags = NVCC_FLAGS + VARIANT_FLAGS[variant] + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nv, *ARCH, *flags, "-c", src, "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nv, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))

"""Build of libspecverify.so with nvcc for sm_103a (GB300), in-tree."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(PKG, "libspecverify.so")
# the debug build: device-side bounds and alignment checks (-DSV_CHECKS)
LIBRARY_CHECKS = os.path.join(PKG, "libspecverify_checks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cuh")))


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libspecverify")


def compile_flags(nvtx: bool = False, extra_flags=(), checks: bool = False) -> list[str]:
    """nvcc flags of the library build; nvtx adds the NVTX ranges around the
    entry points (-DSV_NVTX), checks the device-side bounds and alignment
    checks of the debug build (-DSV_CHECKS)."""
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
            "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64", f"-I{INCLUDE}",
            *(["-DSV_NVTX"] if nvtx else []), *(["-DSV_CHECKS"] if checks else []),
            *extra_flags]


def build_library(force: bool = False, verbose: bool = False, extra_flags=(),
                  nvtx: bool | None = None, checks: bool = False) -> str:
    """Compile csrc/specverify.cu into libspecverify.so (one translation
    unit, -O3, IEEE division and sqrt, no fast-math).  nvtx (default: the
    environment variable SV_NVTX=1) builds the traced variant; a change of
    flags forces a rebuild.  checks builds the debug library,
    libspecverify_checks.so, instead."""
    if nvtx is None:
        nvtx = os.environ.get("SV_NVTX", "") == "1"
    flags = compile_flags(nvtx, extra_flags, checks)
    out = LIBRARY_CHECKS if checks else LIBRARY
    stamp = out + ".flags"
    newest = max(os.path.getmtime(p) for p in sources() + [os.path.join(INCLUDE, "specverify.h")])
    same_flags = os.path.exists(stamp) and open(stamp).read() == " ".join(flags)
    if (not force and same_flags and os.path.exists(out)
            and os.path.getmtime(out) >= newest):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *flags, "-o", tmp, os.path.join(CSRC, "specverify.cu")]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    with open(stamp, "w") as f:
        f.write(" ".join(flags))
    return out

"""Builds the CUDA library ``libssscan.so`` in-tree for sm_103a with nvcc.

Run ``python -m selective_state_space_138_b300.build`` (or call ``build()``).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "ss_scan.cu")
HEADER = os.path.join(ROOT, "include", "ss_scan.h")
LIB = os.path.join(PKG, "libssscan.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMPILE_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--use_fast_math", "-Xcompiler", "-fPIC,-O2"]
LINK_FLAGS = ["-shared", "-cudart", "shared"]
# the parts of ss_scan.cu compiled as separate objects in parallel (SS_PART):
# 0 shared entry points, 1 forward scan, 2 backward pass, 3 decode and conv, 4 SSD
PARTS = (1, 2, 3, 4, 0)


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    """Every file the library is compiled from (one source and its parts)."""
    d = os.path.dirname(SRC)
    return sorted(os.path.join(d, f) for f in os.listdir(d) if f.endswith((".cu", ".cuh")))


# the files each part is compiled from besides ss_scan.cu, the shared headers and the C header
COMMON = ("ss_scan.cu", "device_common.cuh", "host_common.cuh")
PART_FILES = {0: (), 1: ("scan_fwd.cuh", "scan_fwd_host.cuh", "fault_probe.cuh"), 2: ("scan_bwd.cuh",), 3: ("decode.cuh", "conv.cuh"), 4: ("ssd.cuh", "ssd_host.cuh")}
OBJDIR = os.path.join(PKG, "_build")


def part_inputs(part: int) -> list[str]:
    d = os.path.dirname(SRC)
    return [os.path.join(d, f) for f in (*COMMON, *PART_FILES[part])] + [HEADER, __file__]


def part_object(part: int) -> str:
    return os.path.join(OBJDIR, "part%d.o" % part)


def stale_parts(force: bool = False) -> list[int]:
    out = []
    for part in PARTS:
        obj = part_object(part)
        if force or not os.path.exists(obj) or any(os.path.getmtime(f) > os.path.getmtime(obj)
                                                   for f in part_inputs(part)):
            out.append(part)
    return out


def needs_build() -> bool:
    """The library is missing or older than a file it is compiled from (the
    part objects need not be present: a copy of the tree with a fresh library
    does not rebuild)."""
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in (*sources(), HEADER, __file__))


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile the stale parts of ss_scan.cu in parallel (objects kept in
    _build/) and link every part into LIB."""
    if not force and not needs_build():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    procs = []
    for part in stale_parts(force or bool(extra)):
        obj = part_object(part)
        tmpobj = obj + ".tmp%d" % os.getpid()
        cmd = [nvcc(), *ARCH, *COMPILE_FLAGS, "-DSS_PART=%d" % part, "-I", os.path.join(ROOT, "include"),
               "-c", "-o", tmpobj, SRC, *(extra or [])]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((cmd, tmpobj, obj, subprocess.Popen(cmd)))
    failed = []
    for cmd, tmpobj, obj, pr in procs:
        if pr.wait() != 0:
            failed.append(cmd)
        else:
            os.replace(tmpobj, obj)
    if failed:
        raise subprocess.CalledProcessError(1, failed[0])
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, *LINK_FLAGS, "-o", tmp, *[part_object(p) for p in PARTS]]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None)

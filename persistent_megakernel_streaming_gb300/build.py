"""Build libcp.so in-tree with nvcc for sm_103a.

The sources compile in parallel (one nvcc per translation unit), then link
into ``_lib/libcp.so`` beside this file. The CUDA runtime is linked
statically, so the library needs only the driver at run time.
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
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libcp.so")
# (source, object, extra flags): the frame kernel is built three times, once
# reading every size at run time and twice with the Qwen3-TTS 1.7B
# CodePredictor's sizes fixed (CP_SHAPE_1P7B), for handles of up to 64 rows and
# (CP_ROWS_128) of more; the host picks the build per handle.
SOURCES = [
    ("cp_kernel.cu", "cp_kernel.cu.o", []),
    ("cp_kernel.cu", "cp_kernel_1p7b.cu.o", ["-DCP_SHAPE_1P7B"]),
    ("cp_kernel.cu", "cp_kernel_1p7b_r128.cu.o", ["-DCP_SHAPE_1P7B", "-DCP_ROWS_128"]),
    ("cp_host.cu", "cp_host.cu.o", []),
    ("cp_plan.cpp", "cp_plan.cpp.o", []),
]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(src: str) -> list:
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if src.endswith(".cu"):
        return common + ARCH + ["-lineinfo"]
    return common


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(ROOT, "include", "cp.h"))
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, extra: list | None = None) -> str:
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    objs = []
    jobs = []
    for s, o, defs in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(LIBDIR, o)
        objs.append(obj)
        if force or extra or _stale(obj, src):
            jobs.append([cc, "-c", src, "-o", obj] + _flags(s) + defs + list(extra or []))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {cmd[2]}")

    with ThreadPoolExecutor(max_workers=len(jobs) or 1) as ex:
        list(ex.map(run, jobs))
    if jobs or not os.path.exists(LIB):
        run([cc, "-shared", "-o", LIB] + objs + ARCH + ["-Xcompiler", "-fPIC", "-cudart", "static"])
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))

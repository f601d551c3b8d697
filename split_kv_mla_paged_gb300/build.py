"""Build libmla_decode.so in-tree with nvcc for sm_103a (no cmake, one step)."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB_NAME = "libmla_decode.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
SOURCES = [os.path.join(CSRC, "mla_decode.cu"), os.path.join(CSRC, "mla_decode_bf16.cu"),
           os.path.join(CSRC, "mla_merge.cu"), os.path.join(CSRC, "kv_append.cu"),
           os.path.join(CSRC, "plan.cpp")]
OBJ_DIR = os.path.join(HERE, "_build")
DEPENDS = SOURCES + [
    os.path.join(CSRC, "mla_internal.h"),
    os.path.join(CSRC, "sm103_ptx.cuh"),
    os.path.join(CSRC, "mla_device.cuh"),
    os.path.join(os.path.dirname(HERE), "include", "mla_decode.h"),
]
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the C-ABI library if it is missing or stale; return its path."""
    if not force and not needs_build():
        return LIB_PATH
    # One nvcc per translation unit, all at once, then one link.
    os.makedirs(OBJ_DIR, exist_ok=True)
    tag = f"{os.getpid()}"
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(OBJ_DIR, os.path.basename(src) + f".{tag}.o")
        cmd = [_nvcc(), *NVCC_FLAGS, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        objs.append(obj)
        procs.append((src, subprocess.Popen(cmd)))
    failed = [src for src, pr in procs if pr.wait() != 0]
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB_PATH + f".tmp{tag}"
    cmd = [_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", *objs, "-o", tmp]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    for obj in objs:
        os.remove(obj)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

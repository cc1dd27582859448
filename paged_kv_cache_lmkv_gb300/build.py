"""Build liblmkv.so (the C-ABI library) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "liblmkv.so")
SOURCES = [os.path.join(CSRC, "lmkv_api.cu"), os.path.join(CSRC, "lmkv_cachegen.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "lmkv_kernels.cuh"), os.path.join(CSRC, "lmkv_fp8.cuh"),
                  os.path.join(CSRC, "lmkv_internal.h"),
                  os.path.join(INCLUDE, "lmkv.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblmkv.so")
    return cand


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not is_stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    nvcc = nvcc_path()
    # one object per translation unit, compiled in parallel, then one link
    objs, procs = [], []
    for src in SOURCES:
        obj = f"{tmp}.{os.path.basename(src)}.o"
        cmd = [nvcc, ARCH, "-O3", "-lineinfo", "-std=c++17", "-c", "-Xcompiler", "-fPIC",
               "-I", INCLUDE, "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        procs.append((subprocess.Popen(cmd), cmd))
    try:
        for proc, cmd in procs:
            if proc.wait() != 0:
                raise subprocess.CalledProcessError(proc.returncode, cmd)
        subprocess.run([nvcc, ARCH, "-shared", "-o", tmp] + objs, check=True)
    finally:
        for proc, _ in procs:
            if proc.poll() is None:
                proc.kill()
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

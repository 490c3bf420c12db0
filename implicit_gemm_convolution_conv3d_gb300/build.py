"""Build libconv3d.so in-tree with nvcc for sm_103a.

Each .cu under csrc/ is compiled in parallel (-gencode arch=compute_103a,
code=sm_103a, -O3 -lineinfo, IEEE division: no fast-math) and linked into a
shared library beside this file.  cudart is linked statically; the driver's
tensor-map encoders are fetched at run time, so the library loads on hosts
without a GPU.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libconv3d.so")
BUILD_DIR = os.path.join(ROOT, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["conv_igemm.cu", "aux_kernels.cu", "conv3d_api.cu", "conv_noalloc.cu", "conv_fused_q.cu"]
HEADERS = ["ptx.cuh", "internal.h", "tile_table.h", "kernel_common.cuh"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas: bool):
    f = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", f"-I{INCLUDE}",
         f"-I{CSRC}"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "conv3d.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int = 0) -> str:
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs = []
    todo = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD_DIR, s.replace(".cu", ".o"))
        objs.append(obj)
        if force or verbose_ptxas or _stale(obj, src):
            todo.append((src, obj))

    def compile_one(item):
        src, obj = item
        cmd = [nvcc, "-c", src, "-o", obj + ".tmp", *_flags(verbose_ptxas)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return r.stderr

    if todo:
        n = jobs or min(len(todo), os.cpu_count() or 1)
        with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
            for log in ex.map(compile_one, todo):
                if verbose_ptxas and log:
                    sys.stderr.write(log)
    if todo or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, "-shared", *ARCH, "-o", tmp, *objs, "-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

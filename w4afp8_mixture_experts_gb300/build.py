"""Builds libw4a8moe.so (the CUDA library) in-tree with nvcc for sm_103a.

Translation units are compiled in parallel and linked with the static CUDA
runtime; the result lands in w4afp8_mixture_experts_gb300/_lib/.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libw4a8moe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                "-diag-suppress", "177"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest(paths) -> float:
    return max(os.path.getmtime(p) for p in paths)


def _compile(nvcc, src, obj, deps, extra):
    if os.path.exists(obj) and os.path.getmtime(obj) >= _newest([src] + deps):
        return obj
    cmd = [nvcc] + FLAGS + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build_shared(srcs, out, deps, extra=(), jobs=None) -> str:
    nvcc = nvcc_path()
    os.makedirs(os.path.dirname(out), exist_ok=True)
    objs = [os.path.join(os.path.dirname(out), os.path.basename(s)[:-3] + ".o") for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, os.cpu_count() or 4)) as ex:
        list(ex.map(lambda so: _compile(nvcc, so[0], so[1], deps, list(extra)), zip(srcs, objs)))
    if not (os.path.exists(out) and os.path.getmtime(out) >= _newest(objs)):
        cmd = [nvcc] + ARCH + ["-shared", "-o", out] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return out


def build() -> str:
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return build_shared(srcs, LIB, deps)


if __name__ == "__main__":
    print(build())

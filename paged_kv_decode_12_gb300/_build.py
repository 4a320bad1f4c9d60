"""Build ``libpkv.so`` in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel to an object file, then linked
into one shared library next to this file.  The CUDA runtime is linked as a
shared library so that the process uses one runtime instance with PyTorch.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libpkv.so")
BUILD_DIR = os.path.join(ROOT, "_build")

SOURCES = ["pkv_host.cpp", "pkv_sched.cpp", "pkv_layers.cpp", "pkv_append.cu", "pkv_decode.cu", "pkv_step.cu",
           "pkv_fp8.cu", "pkv_probe.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _stale(outputs, inputs) -> bool:
    if not all(os.path.exists(o) for o in outputs):
        return True
    newest_in = max(os.path.getmtime(i) for i in inputs)
    return min(os.path.getmtime(o) for o in outputs) < newest_in


TIMELINE_LIB = os.path.join(HERE, "libpkv_timeline.so")


def build(force: bool = False, verbose: bool = False, extra_flags=None, timeline: bool = False) -> str:
    """Compile every source and link the library; returns its path.  With ``timeline``
    the sources are compiled with -DPKV_TIMELINE into libpkv_timeline.so (the per-CTA
    timeline of include/pkv_timeline.h), in a build folder of their own."""
    nvcc = _nvcc()
    lib_path = TIMELINE_LIB if timeline else LIB
    build_dir = os.path.join(BUILD_DIR, "timeline") if timeline else BUILD_DIR
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers += [os.path.join(INCLUDE, h) for h in os.listdir(INCLUDE) if h.endswith(".h")]
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    objs = [os.path.join(build_dir, os.path.basename(s) + ".o") for s in srcs]
    if not force and not _stale([lib_path], srcs + headers + [__file__]):
        return lib_path
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "--expt-relaxed-constexpr"]
    common += list(extra_flags or [])
    if timeline:
        common += ["-DPKV_TIMELINE"]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [nvcc] + ARCH + common + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0 or verbose:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        list(ex.map(compile_one, zip(srcs, objs)))
    tmp = lib_path + f".tmp{os.getpid()}"
    link = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
        "-Xlinker", "-rpath," + _cuda_lib_dir(nvcc)]
    if verbose:
        print(" ".join(link), file=sys.stderr)
    subprocess.run(link, check=True)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

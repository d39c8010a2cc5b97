"""Build ``libmxfp4_gb300.so`` in-tree with nvcc for sm_103a.

Each CUDA translation unit compiles in parallel; the objects link into one
shared library next to this file.  Run ``python -m mxfp4_quantized_gemm_gb300.build``.
``build(variant="timeline")`` builds the same sources with the decode
kernel's timeline stamps compiled in (``libmxfp4_gb300_timeline.so``), for
``bench.py --timeline``; the product library never carries them.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
INCLUDE_DIR = os.path.join(os.path.dirname(PKG_DIR), "include")
LIB_NAME = "libmxfp4_gb300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
SOURCES = ("quant.cu", "norm_quant.cu", "gemm.cu", "decode.cu", "bmm.cu", "capi.cu", "noalloc.cu", "tc_rate.cu")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, variant: str = "default") -> str:
    if variant not in ("default", "timeline"):
        raise ValueError(f"unknown build variant {variant!r}")
    nvcc = _nvcc()
    build_dir = BUILD_DIR if variant == "default" else BUILD_DIR + "_" + variant
    lib_path = LIB_PATH if variant == "default" else LIB_PATH.replace(".so", f"_{variant}.so")
    extra = [] if variant == "default" else ["-DMXFP4_STAMPS"]
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers += [os.path.join(INCLUDE_DIR, f) for f in os.listdir(INCLUDE_DIR) if f.endswith(".h")]

    def compile_one(src: str) -> str:
        s = os.path.join(CSRC, src)
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        if force or _stale(obj, [s] + headers):
            cmd = [nvcc, *NVCC_FLAGS, *extra, "-I", INCLUDE_DIR, "-c", s, "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr}")
            if verbose and res.stderr:
                print(res.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(lib_path, objs):
        cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", lib_path]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stderr}")
    return lib_path


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv))

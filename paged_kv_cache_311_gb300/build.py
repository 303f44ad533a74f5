"""Builds libpkv.so in-tree for sm_103a with nvcc (no cmake).

The translation units compile in parallel; the CUDA runtime is linked
statically, so the library depends only on the driver at run time.
Usage: python -m paged_kv_cache_311_gb300.build [--verbose-ptxas]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB_DIR = os.path.join(HERE, "_lib")
SOURCES = ["pkv_abi.cu", "pa_decode_f32.cu", "pa_decode_f16.cu", "pa_decode_bf16.cu",
           "pkv_static_ws.cu", "pkv_plan.cu", "pkv_usage.cu", "pkv_block_pool.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpkv.so")
    return path


def library_path() -> str:
    return os.path.join(LIB_DIR, "libpkv.so")


def build(extra_flags=(), out_path: str | None = None, verbose_ptxas: bool = False) -> str:
    out = out_path or library_path()
    obj_dir = os.path.join(os.path.dirname(out), "obj")
    os.makedirs(obj_dir, exist_ok=True)
    flags = [*ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
             "-I", os.path.join(ROOT, "include"), *extra_flags]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [nvcc(), *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose_ptxas:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = f"{out}.{os.getpid()}.tmp"
    subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose_ptxas="--verbose-ptxas" in sys.argv))

"""Build libpkv.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel; the shared library links the CUDA
runtime statically and exports only the PKV_API symbols of include/pkv.h.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpkv.so")
SOURCES = ["api.cpp", "gqa_decode.cu", "gqa_noalloc.cu", "mla_verify.cu", "mla_verify_native.cu",
           "mla_verify_pair.cu", "kv_append.cu"]
HEADERS = ["pkv_internal.h", "ptx.cuh", "tcgen05.cuh", "mla_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpkv")
    return exe


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compile every kernel and the C ABI into paged_kv_cache_30_gb300/_build/libpkv.so."""
    os.makedirs(BUILD, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "pkv.h")]
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    objs = [os.path.join(BUILD, os.path.basename(s) + ".o") for s in srcs]
    flags = NVCC_FLAGS + (extra_flags or [])
    exe = nvcc()

    def compile_one(i):
        if not force and not _stale(objs[i], [srcs[i], *hdrs, __file__]):
            return None
        cmd = [exe, *ARCH, *flags, "-c", srcs[i], "-o", objs[i] + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {srcs[i]}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        os.replace(objs[i] + ".tmp", objs[i])
        return srcs[i]

    with ThreadPoolExecutor(len(srcs)) as ex:
        list(ex.map(compile_one, range(len(srcs))))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [exe, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None))

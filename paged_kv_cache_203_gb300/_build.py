"""Builds libpkv.so, the sm_103a CUDA library behind the C ABI in include/pkv.h.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library next to this file (git-ignored).  No cmake, no torch
extension machinery: the library has no torch dependency at all.
"""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

_HERE = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(os.path.dirname(_HERE), "include")
_BUILD = os.path.join(_HERE, "_build")

SOURCES = [
    "pkv_abi.cu",
    "pkv_pagetable.cu",
    "pkv_merge.cu",
    "pkv_decode.cu",
    "pkv_extend.cu",
    "pkv_mla.cu",
    "pkv_noalloc.cu",
    "pkv_append.cu",
]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", "-I", _INCLUDE]


def lib_path() -> str:
    return os.path.join(_HERE, "libpkv.so")


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _compile(src: str, extra: list[str], verbose: bool) -> str:
    obj = os.path.join(_BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), *ARCH_FLAGS, *NVCC_FLAGS, *extra, "-c",
           os.path.join(_CSRC, src), "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout + res.stderr, flush=True)
    return obj


def build_library(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link libpkv.so."""
    os.makedirs(_BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose), SOURCES))
    out = lib_path()
    tmp = out + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def sources_newer_than_library() -> bool:
    lib = lib_path()
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    files = [os.path.join(_CSRC, f) for f in os.listdir(_CSRC)]
    files.append(os.path.join(_INCLUDE, "pkv.h"))
    return any(os.path.getmtime(f) > t for f in files)

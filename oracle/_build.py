"""Builds the float64 CPU oracle (``pkv_oracle.c``) with the host C compiler.

Test infrastructure: compiling the checker is not using it.  The library is
plain C99 + OpenMP, with no architecture-specific flags, so it builds the same
way on x86-64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def oracle_lib_path() -> str:
    return os.path.join(_HERE, "libpkv_oracle.so")


def build_oracle(verbose: bool = False) -> str:
    out = oracle_lib_path()
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-o", tmp, os.path.join(_HERE, "pkv_oracle.c"), "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out

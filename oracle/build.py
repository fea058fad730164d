"""Compile the CPU oracle (test infrastructure) into oracle/_build/libccv_oracle.so.

Plain gcc, no target-specific flags, so the same source builds on x86-64 and
aarch64 hosts.  -ffp-contract=off keeps every multiply and add separately
rounded, which is the arithmetic the oracle documents.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ccv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libccv_oracle.so")


def compile_to(src: str, lib: str) -> None:
    """Compile one oracle source file into a shared library at ``lib``."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", lib, src, "-lm"]
    subprocess.run(cmd, check=True)


def build(force: bool = False) -> str:
    """Build the oracle shared library if it is missing or stale; return its path.

    ``CCV_ORACLE_LIB`` names a prebuilt library to use instead; the mutation
    test points it at deliberately broken copies of the oracle.
    """
    override = os.environ.get("CCV_ORACLE_LIB")
    if override:
        return override
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    compile_to(SRC, tmp)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

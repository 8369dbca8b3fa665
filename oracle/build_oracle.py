"""Compile the C oracle into oracle/liboracle.so (test infrastructure only).

Plain gcc, no architecture-specific flags, so the same source builds on x86-64
and aarch64 hosts.  Called by ``__graft_entry__.build()`` and, lazily, by
``oracle/oracle.py``.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "tffn_oracle.c")
HDR = os.path.join(HERE, "tffn_oracle.h")
LIB = os.path.join(HERE, "liboracle.so")


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    lib_t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > lib_t for p in (SRC, HDR))


def build(force: bool = False) -> str:
    if force or needs_build():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c99", "-D_GNU_SOURCE", "-O2", "-fno-fast-math",
               "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

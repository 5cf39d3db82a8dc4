"""Compile the CPU oracle (test infrastructure) into oracle/libkivi_oracle.so.

Plain gcc, portable flags only (the same source builds on x86-64 and aarch64).
-ffp-contract=off keeps every fp32 multiply and add separately rounded, which
the bit-exact quantiser comparison relies on; -ffast-math is never used.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kivi_oracle.c")
HDR = os.path.join(HERE, "kivi_oracle.h")
LIB = os.path.join(HERE, "libkivi_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-pthread", "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(force: bool = False) -> str:
    """Build the oracle library if missing or older than its sources."""
    stale = (not os.path.exists(LIB) or
             os.path.getmtime(LIB) < max(os.path.getmtime(SRC), os.path.getmtime(HDR)))
    if force or stale:
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))

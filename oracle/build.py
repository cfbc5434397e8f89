"""Build the CPU oracle (plain C11) into oracle/_build/libbq_oracle.so.

Test infrastructure: the oracle is compiled with no fast-math and no
floating-point contraction, so each float operation in bq_oracle.c is a single
IEEE operation in program order on both x86-64 and aarch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libbq_oracle.so")
LIB_OMP = os.path.join(OUT_DIR, "libbq_oracle_omp.so")
SRC = os.path.join(HERE, "bq_oracle.c")
HDR = os.path.join(HERE, "bq_oracle.h")

CFLAGS = ["-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off",
          "-fno-strict-aliasing", "-fPIC", "-shared", "-Wall", "-Wextra"]


def _compile(out: str, extra, force: bool) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR), os.path.getmtime(__file__))
        if os.path.getmtime(out) >= newest:
            return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, *extra, "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle if it is missing or older than its sources; return its path."""
    return _compile(LIB, [], force)


def build_omp(force: bool = False) -> str:
    """The same source built with OpenMP (row-parallel GEMV, for the all-core
    CPU baseline timing); the per-row arithmetic is unchanged."""
    return _compile(LIB_OMP, ["-fopenmp"], force)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
    print(build_omp(force="--force" in sys.argv))

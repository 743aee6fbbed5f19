"""Build the CPU oracle's shared library (test infrastructure).

Compiles ``nvfp4_oracle.c`` with gcc into ``oracle/_build/libnvfp4_oracle.so``:
``-O2 -ffp-contract=off`` keeps every binary32 step a separately rounded
operation; no ISA-specific flags, so the same source builds on x86-64 and
aarch64 hosts and gives the same results on both.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nvfp4_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libnvfp4_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    compile_source(SRC, tmp)
    os.replace(tmp, LIB)
    return LIB


def compile_source(src: str, out: str) -> None:
    """gcc with the oracle's flags: `src` (a C file) -> shared library `out`."""
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

"""Build the CPU oracle's shared library (test infrastructure only).

The oracle is plain C compiled with -ffp-contract=off so that no product and
add fuse; it shares no source with the CUDA library.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pdattn_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile oracle/pdattn_oracle.c into oracle/_build/liboracle.so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    # OpenMP only spreads independent rows over threads; without it the
    # same code runs serially.
    r = subprocess.run(base + ["-fopenmp", SRC, "-o", tmp, "-lm"], capture_output=True, text=True)
    if r.returncode != 0:
        subprocess.run(base + [SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

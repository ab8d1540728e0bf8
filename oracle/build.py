"""Compile the CPU oracle (moe_oracle.c) into oracle/_build/liboracle.so.

Test infrastructure: the oracle is built so that the test suite, the package's
smoke check and the benchmark's CPU-baseline leg can call it.  The product
library never links or loads it.

Flags: -ffp-contract=off keeps the compiler from fusing multiplies and adds on
its own (the oracle spells out every fused multiply-add it performs), and no
fast-math option is given, so IEEE semantics hold on x86-64 and aarch64 alike.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


FLAGS = ["-std=gnu99", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-Wall"]


def build_source(text: str, out: str) -> str:
    """Compile C source text (a variant of moe_oracle.c, for the tests that
    plant mistakes in the oracle) with the oracle's own flags into `out`."""
    src = out + ".c"
    with open(src, "w") as f:
        f.write(text)
    res = subprocess.run(["gcc", *FLAGS, src, "-o", out, "-lm"], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("oracle variant build failed:\n" + res.stderr)
    return out


def build(force: bool = False, quiet: bool = True) -> str:
    """Build liboracle.so if it is missing or older than its source; return its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *FLAGS, SRC, "-o", tmp, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + " ".join(cmd) + "\n" + res.stderr)
    if not quiet and res.stderr:
        sys.stderr.write(res.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, quiet=False))

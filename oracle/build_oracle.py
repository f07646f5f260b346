"""Compile the CPU oracle (pkv_oracle.c) into libpkv_oracle.so beside it.

Test infrastructure: the oracle is the checker, never part of the product.
Run as a script (``python oracle/build_oracle.py``) or call ``build()``.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkv_oracle.c")
LIB = os.path.join(HERE, "libpkv_oracle.so")

# -ffp-contract=off: the fp8 encoder's fp32 product must be one rounded
# multiply on x86-64 and on aarch64 alike (gcc fuses a*b+c by default on
# aarch64).  No -march/-ffast-math: results must not depend on the host.
FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread"]


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *FLAGS, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


def build_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (used by the tests that
    plant a mistake in the oracle and check that a pin catches it)."""
    src_path = out_path[:-3] + ".c"
    with open(src_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *FLAGS, src_path, "-o", out_path, "-lm"], check=True)
    return out_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

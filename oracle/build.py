"""Build the CPU oracle (plain C, gcc) into oracle/_build/libmxq_oracle.so.

Test infrastructure: see the package docstring. Portable flags only (the
same source builds on x86-64 and aarch64); floating-point contraction is
disabled so that results do not depend on the host's FMA units.
"""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "_build", "libmxq_oracle.so")


def build_oracle(verbose: bool = False) -> str:
    out = library_path()
    os.makedirs(os.path.dirname(out), exist_ok=True)
    src = os.path.join(_HERE, "mxq_oracle.c")
    base = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
            "-fvisibility=hidden", "-Wall", "-Wextra", "-Wno-unused-parameter", src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=not verbose)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=not verbose)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build_oracle(verbose=True))

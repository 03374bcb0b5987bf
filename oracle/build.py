"""Builds the C oracle ``libmsa_oracle.so`` with the host C compiler.

Test infrastructure: it compiles ``oracle/msa_oracle.c`` only (no CUDA, no
code shared with the library under test). Flags: -O2, no fast-math and
-ffp-contract=off (no fused multiply-add), so x86 and Arm hosts compute the
same bits; OpenMP across independent units.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "msa_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmsa_oracle.so")
FLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math"]


def cc() -> str:
    for cand in (os.environ.get("CC"), shutil.which("gcc"), shutil.which("cc")):
        if cand:
            return cand
    raise RuntimeError("no C compiler found")


def build(force: bool = False) -> str:
    """Compile the oracle if its source is newer than the library; returns the path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC),
                                                                          os.path.getmtime(__file__)):
        return LIB
    tmp = f"{LIB}.{os.getpid()}.tmp"
    r = subprocess.run([cc(), *FLAGS, SRC, "-o", tmp, "-lm"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the C oracle failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="-f" in sys.argv))

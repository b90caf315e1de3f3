"""Builds the plain C++ oracle (oracle/dsa_oracle_ref.cpp) into
oracle/_build/liboracle_ref.so with the host C++ compiler. Test
infrastructure: only the tests and the benchmark's CPU legs load it."""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dsa_oracle_ref.cpp")
OUT = os.path.join(HERE, "_build", "liboracle_ref.so")


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    if not force and os.path.exists(OUT) and os.path.getmtime(OUT) >= os.path.getmtime(SRC):
        return OUT
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("no C++ compiler found for the oracle")
    tmp = OUT + ".tmp"
    r = subprocess.run([cxx, "-O2", "-std=c++17", "-pthread", "-shared", "-fPIC", "-o", tmp, SRC],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force=True))

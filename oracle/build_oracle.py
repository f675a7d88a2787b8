"""Builds the C++ oracle (oracle/moe_oracle_ref.cpp) into
oracle/_build/libmoe_oracle.so with g++ (OpenMP when the compiler has it).

Test infrastructure: __graft_entry__.build() compiles it beside the CUDA
library (building the checker is not using it); only tests/, smoke() and
bench.py's cpu_baseline / reference legs load it."""

from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle_ref.cpp")
OUT = os.path.join(HERE, "_build", "libmoe_oracle.so")
# -ffp-contract=off: no fused multiply-adds, so the sums round the same way
# on every host (x86-64 here, aarch64 on the GPU machine)
FLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared"]


def build() -> str:
    if os.path.exists(OUT) and os.path.getmtime(OUT) >= os.path.getmtime(SRC):
        return OUT
    cxx = os.environ.get("CXX") or shutil.which("g++") or "g++"
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    for extra in (["-fopenmp"], []):
        r = subprocess.run([cxx] + FLAGS + extra + [SRC, "-o", OUT], stdout=subprocess.PIPE,
                           stderr=subprocess.STDOUT, text=True)
        if r.returncode == 0:
            return OUT
    raise RuntimeError("oracle build failed:\n" + r.stdout)


if __name__ == "__main__":
    print(build())

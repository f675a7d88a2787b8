"""Builds the package's shared libraries in-tree with nvcc, for sm_103a only.

  _build/libmoe_gb300.so   the MoE layer library (C ABI of include/moe.h)
  _build/libmoe_synth.so   the seeded device-side input generator

Translation units compile in parallel; a library is rebuilt only when one of
its sources or headers is newer than it.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                     "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE]

LIBS = {
    "libmoe_gb300.so": ["api.cu", "router.cu", "router_tc.cu", "permute.cu", "combine.cu", "gemm_simt.cu",
                        "gemm_tc.cu", "gemm_tc2.cu", "gemm_tc_bwd.cu", "bwd.cu", "permute_noalloc.cu",
                        "aux_loss.cu", "gemm_mxfp8.cu"],
    "libmoe_synth.so": ["synth.cu"],
}


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def _headers():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(verbose: bool = False, extra_flags=None) -> dict:
    """Compile every library that is out of date; returns {name: path}."""
    os.makedirs(OUT, exist_ok=True)
    nv = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])
    headers = _headers()
    out = {}
    jobs = []
    for lib, srcs in LIBS.items():
        target = os.path.join(OUT, lib)
        out[lib] = target
        deps = [os.path.join(CSRC, s) for s in srcs] + headers
        if not _stale(target, deps):
            continue
        objs = []
        for s in srcs:
            obj = os.path.join(OUT, s.replace(".cu", ".o"))
            objs.append(obj)
            if _stale(obj, [os.path.join(CSRC, s)] + headers):
                jobs.append([nv] + flags + ["-c", os.path.join(CSRC, s), "-o", obj])
        out[lib] = (target, objs)
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        for log in ex.map(_run, jobs):
            if verbose and log:
                print(log)
    for lib, v in list(out.items()):
        if isinstance(v, tuple):
            target, objs = v
            _run([nv] + ARCH + ["-shared", "-o", target] + objs +
                 ["-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64"])
            out[lib] = target
    return out


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv))

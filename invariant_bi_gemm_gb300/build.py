"""Build the CUDA libraries in-tree with nvcc for sm_103a.

Produces, under ``invariant_bi_gemm_gb300/_build/``:
  libbi_gemm.so           the product (C ABI of include/bi_gemm.h, bi_rmsnorm.h, bi_attention.h,
                          bi_prenorm.h)
  libbi_gemm_controls.so  test-only negative controls and failure injection

Both are compiled in parallel; a library is rebuilt when any source is newer.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

TARGETS = {
    "libbi_gemm.so": ("bi_gemm.cu", "bi_rmsnorm.cu", "bi_attention.cu", "bi_prenorm.cu"),
    "libbi_gemm_controls.so": ("bi_gemm_controls.cu",),
}


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _sources():
    return (glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(ROOT, "include", "*.h")) +
            glob.glob(os.path.join(ROOT, "tests", "include", "*.h")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in _sources())


def lib_path(name: str = "libbi_gemm.so") -> str:
    return os.path.join(OUT, name)


def build(force: bool = False, verbose: bool = False) -> dict:
    """Compile every stale library; returns {name: path}.  Raises on a compiler error."""
    os.makedirs(OUT, exist_ok=True)
    procs = []
    for name, srcs in TARGETS.items():
        out = lib_path(name)
        if not force and not _stale(out):
            continue
        tmp = out + f".tmp{os.getpid()}"
        cmd = [
            nvcc(), "-std=c++17", "-O3", ARCH, "-lineinfo",
            "-Xcompiler", "-fPIC,-fvisibility=hidden",
            "-Xlinker", "-Bsymbolic",
            "-shared", "-o", tmp, *[os.path.join(CSRC, s) for s in srcs],
        ]
        if verbose:
            cmd.insert(4, "-Xptxas=-v")
        procs.append((name, out, tmp, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for name, out, tmp, p in procs:
        log, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(log.decode(errors="replace"))
        if p.returncode:
            errors.append(name)
            if os.path.exists(tmp):
                os.remove(tmp)
        else:
            os.replace(tmp, out)
    if errors:
        raise RuntimeError(f"nvcc failed for {errors}")
    return {name: lib_path(name) for name in TARGETS}


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

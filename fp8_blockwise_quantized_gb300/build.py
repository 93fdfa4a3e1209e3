"""Build the CUDA library in-tree: csrc/*.cu -> libgmm_gb300.so (sm_103a only).

Each translation unit is compiled by its own nvcc process in parallel, then
linked into one shared library next to this file.  No fast-math: the
quantization scales must be IEEE fp32 divisions.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgmm_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _flags(verbose_ptxas: bool) -> list[str]:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True) -> str:
    if (not force and not verbose_ptxas and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= _deps_mtime()):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    procs = []
    objs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [NVCC, "-c", src, "-o", obj] + _flags(verbose_ptxas)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif text.strip() and (verbose_ptxas or not quiet):
            sys.stderr.write(f"== {os.path.basename(src)}\n{text}")
    if failed:
        msg = "\n".join(f"== {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = LIB + ".tmp"
    subprocess.run([NVCC] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs,
                   check=True, capture_output=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="-v" in sys.argv, quiet=False))

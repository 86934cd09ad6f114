"""Build ``libmgattn.so`` in-tree with nvcc for sm_103a (one translation unit, static cudart)."""

from __future__ import annotations

import os
import shutil
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(_HERE)
SOURCES = [os.path.join(_HERE, "csrc", "mg_attn.cu")]
DEPS = SOURCES + [os.path.join(_HERE, "csrc", "mg_attn_kernels.cuh"), os.path.join(_HERE, "csrc", "ptx.cuh"),
                  os.path.join(ROOT, "include", "mg_attn.h")]
OUT = os.path.join(_HERE, "libmgattn.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise FileNotFoundError("nvcc not found")
    return p


def command(out: str = OUT, extra=()) -> list:
    return [nvcc_path(), *ARCH_FLAGS, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
            "-I", os.path.join(ROOT, "include"), *extra, "-o", out, *SOURCES]


def build(force: bool = False, verbose: bool = False, out: str = OUT) -> str:
    """Compile when the library is missing or older than any source; returns its path."""
    stale = not os.path.exists(out) or any(os.path.getmtime(out) < os.path.getmtime(s) for s in DEPS)
    if force or stale:
        cmd = command(out, ("-Xptxas", "-v") if verbose else ())
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if verbose:
            print(r.stdout + r.stderr)
    return out


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""Build ``libmgattn.so`` in-tree with nvcc for sm_103a (static cudart).

Two translation units: ``mg_attn.cu`` (the attention path) and ``mg_diag.cu`` (the launch-floor
and exponential-rate measurements), compiled in parallel to objects and linked into one library."""

from __future__ import annotations

import os
import shutil
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(_HERE)
SOURCES = [os.path.join(_HERE, "csrc", "mg_attn.cu"), os.path.join(_HERE, "csrc", "mg_diag.cu")]
DEPS = SOURCES + [os.path.join(_HERE, "csrc", "mg_attn_kernels.cuh"), os.path.join(_HERE, "csrc", "mg_combine.cuh"),
                  os.path.join(_HERE, "csrc", "mg_attn_pair.cuh"), os.path.join(_HERE, "csrc", "mg_attn_swap.cuh"),
                  os.path.join(_HERE, "csrc", "ptx.cuh"),
                  os.path.join(ROOT, "include", "mg_attn.h"), os.path.join(ROOT, "include", "mg_diag.h")]
OUT = os.path.join(_HERE, "libmgattn.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise FileNotFoundError("nvcc not found")
    return p


def compile_command(src: str, obj: str, extra=()) -> list:
    return [nvcc_path(), *ARCH_FLAGS, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
            "-I", os.path.join(ROOT, "include"), *extra, "-c", "-o", obj, src]


def link_command(objs, out: str = OUT) -> list:
    return [nvcc_path(), *ARCH_FLAGS, "-shared", "-o", out, *objs]


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, out: str = OUT) -> str:
    """Compile when the library is missing or older than any source; returns its path."""
    stale = not os.path.exists(out) or any(os.path.getmtime(out) < os.path.getmtime(s) for s in DEPS)
    if force or stale:
        from concurrent.futures import ThreadPoolExecutor

        objs = [out + "." + os.path.splitext(os.path.basename(s))[0] + ".o" for s in SOURCES]
        extra = ("-Xptxas", "-v") if verbose else ()
        with ThreadPoolExecutor(len(SOURCES)) as pool:
            logs = list(pool.map(lambda so: _run(compile_command(so[0], so[1], extra)), zip(SOURCES, objs)))
        logs.append(_run(link_command(objs, out)))
        for o in objs:
            os.remove(o)
        if verbose:
            print("".join(logs))
    return out


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

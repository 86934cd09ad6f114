"""fp64 CPU oracle for Mirage's exp-normalised GQA kernel graph.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's ``cpu_baseline`` / ``--impl reference`` legs may import this package.
The CUDA product path (``attention_mugraph_gb300``) never imports, links or
falls back to it, and the two share no code: the only module both sides use is
the seeded input generator, which holds none of the method's arithmetic.

The oracle is the graph of the Mirage GQA tutorial (documentation,
tutorials/group-query-attention, "Define GQA Computation Graph") written out
as a plain double-precision loop in ``mg_oracle.c``:
``A = matmul(Q,K); E = exp(A); S = reduction(E,2); D = div(E,S); O = matmul(D,V)``.
Every function here is pinned by the ``-m "not gpu"`` tests (closed forms,
brute force, a library special case, invariants, mutation checks).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mg_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmgoracle.so")
_lock = threading.Lock()
_lib = None


def compile_library(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile an oracle C source into a shared library (gcc, OpenMP, -O2).

    No fast-math: the loops keep IEEE double semantics in the order written.
    """
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           src, "-o", out, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build(force: bool = False) -> str:
    """Build ``libmgoracle.so`` next to its source when missing or stale."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            compile_library()
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.mg_oracle_attention.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64,
                                        ctypes.c_int, f64p]
    lib.mg_oracle_attention.restype = ctypes.c_int
    lib.mg_oracle_attention_rows.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64,
                                             ctypes.POINTER(ctypes.c_int64), i64,
                                             ctypes.c_int, f64p]
    lib.mg_oracle_attention_rows.restype = ctypes.c_int
    lib.mg_oracle_attention_qknorm_rows.argtypes = [u16p, u16p, u16p, i64, i64, i64, i64, ctypes.c_double,
                                                    ctypes.POINTER(ctypes.c_int64), i64, ctypes.c_int, f64p]
    lib.mg_oracle_attention_qknorm_rows.restype = ctypes.c_int
    lib.mg_oracle_max_threads.argtypes = []
    lib.mg_oracle_max_threads.restype = ctypes.c_int
    return lib


def load_library(path: str | None = None):
    """Load (building first if needed) the oracle library; ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(path)
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _as_half_bits(x) -> np.ndarray:
    """Contiguous uint16 view of an fp16 array or tensor (bit patterns, no rounding)."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(x)
    if a.dtype != np.float16:
        raise TypeError(f"oracle inputs must be fp16, got {a.dtype}")
    return a.view(np.uint16)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def max_threads(lib=None) -> int:
    return int((lib or load_library()).mg_oracle_max_threads())


def attention(Q, K, V, threads: int = 0, lib=None) -> np.ndarray:
    """O = (exp(Q.K) / rowsum(exp(Q.K))) . V in double; returns (B, M, d) float64.

    Q (B,M,d), K (B,d,N), V (B,N,d), all fp16. ``threads`` <= 0 uses every core.
    """
    q, k, v = _as_half_bits(Q), _as_half_bits(K), _as_half_bits(V)
    if q.ndim != 3 or k.ndim != 3 or v.ndim != 3:
        raise ValueError("Q, K, V must be 3-D")
    B, M, d = q.shape
    if k.shape[0] != B or k.shape[1] != d or v.shape[0] != B or v.shape[2] != d:
        raise ValueError(f"shape mismatch: Q{q.shape} K{k.shape} V{v.shape}")
    N = k.shape[2]
    if v.shape[1] != N:
        raise ValueError(f"shape mismatch: K{k.shape} V{v.shape}")
    out = np.empty((B, M, d), dtype=np.float64)
    lib = lib or load_library()
    rc = lib.mg_oracle_attention(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                 _ptr(v, ctypes.c_uint16), B, M, N, d, int(threads),
                                 _ptr(out, ctypes.c_double))
    if rc != 0:
        raise RuntimeError(f"mg_oracle_attention failed with code {rc}")
    return out


def attention_rows(Q, K, V, rows, threads: int = 0, lib=None) -> np.ndarray:
    """Selected output rows only: ``rows`` are flat indices b*M + m; returns (len(rows), d)."""
    q, k, v = _as_half_bits(Q), _as_half_bits(K), _as_half_bits(V)
    B, M, d = q.shape
    N = k.shape[2]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((r.size, d), dtype=np.float64)
    lib = lib or load_library()
    rc = lib.mg_oracle_attention_rows(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                      _ptr(v, ctypes.c_uint16), B, M, N, d,
                                      _ptr(r, ctypes.c_int64), r.size, int(threads),
                                      _ptr(out, ctypes.c_double))
    if rc != 0:
        raise RuntimeError(f"mg_oracle_attention_rows failed with code {rc}")
    return out


QKNORM_EPS = 1e-6  # the library's fixed epsilon of rms_norm (MG_QKNORM_EPS in include/mg_attn.h)


def attention_qknorm(Q, K, V, eps: float = QKNORM_EPS, rows=None, threads: int = 0, lib=None) -> np.ndarray:
    """QK-norm attention: Q and K each rms-normalised over d (x / sqrt(mean(x^2) + eps)), then the
    graph (documentation, tutorials/attention-with-kv-norm). Returns (B, M, d) float64, or
    (len(rows), d) for the listed flat rows b*M + m."""
    q, k, v = _as_half_bits(Q), _as_half_bits(K), _as_half_bits(V)
    B, M, d = q.shape
    N = k.shape[2]
    if k.shape != (B, d, N) or v.shape != (B, N, d):
        raise ValueError(f"shape mismatch: Q{q.shape} K{k.shape} V{v.shape}")
    r = np.arange(B * M, dtype=np.int64) if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((len(r), d), dtype=np.float64)
    lib = lib or load_library()
    rc = lib.mg_oracle_attention_qknorm_rows(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                             _ptr(v, ctypes.c_uint16), B, M, N, d, float(eps),
                                             _ptr(r, ctypes.c_int64), len(r), int(threads),
                                             _ptr(out, ctypes.c_double))
    if rc != 0:
        raise RuntimeError(f"mg_oracle_attention_qknorm_rows failed with code {rc}")
    return out.reshape(B, M, d) if rows is None else out

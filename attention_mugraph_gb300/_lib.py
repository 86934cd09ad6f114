"""ctypes binding of ``libmgattn.so`` (declared in ``include/mg_attn.h``).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels. The names mirror the C ABI (``mg_attn_plan``, ``mg_attn_run``, ...). PyTorch is
used for device memory and streams; there is no CPU fallback, and every call fails loudly
when the library is missing or returns an error.
"""

from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmgattn.so")

MG_OK = 0
MG_ERR_INSUFFICIENT_SMEM = 1
MG_ERR_LAYOUT = 2
MG_ERR_CONFIG = 3
MG_ERR_INVALID_ARG = 4
MG_ERR_UNSUPPORTED = 5
MG_ERR_CUDA = 6
MG_ERR_TIMEOUT = 7

MG_FLAG_NO_PDL = 0x1
MG_FLAG_INJECT_TIMEOUT = 0x2
MG_FLAG_NO_CLUSTER = 0x4
MG_FLAG_SAFE_SOFTMAX = 0x8
MG_FLAG_QK_NORM = 0x10
MG_FLAG_Q_PAIRS = 0x20
MG_FLAG_NO_Q_PAIRS = 0x40
MG_FLAG_STREAM_K = 0x80
MG_FLAG_NO_STREAM_K = 0x100
MG_FLAG_SWAP_AB = 0x200
MG_FLAG_NO_SWAP_AB = 0x400
MG_FLAG_PUSH_COMBINE = 0x800
MG_FLAG_NO_EARLY_LOADS = 0x1000
MG_FLAG_ISOLATED = 0x2000
MG_QKNORM_EPS = 1e-6

# Every function include/mg_attn.h declares.
EXPORTS = ("mg_attn_plan", "mg_attn_plan_ex", "mg_attn_run", "mg_attn_run_host", "mg_attn_destroy",
           "mg_attn_get_status", "mg_attn_get_info", "mg_attn_query", "mg_attn_status_string",
           "mg_attn_last_error", "mg_attn_version", "mg_attn_set_timing_events", "mg_attn_run_noalloc")
# Every function include/mg_diag.h declares.
DIAG_EXPORTS = ("mg_diag_launch_floor", "mg_diag_exp_rate", "mg_diag_last_error")


class MgAttnOptions(ctypes.Structure):
    _fields_ = [("n_split", ctypes.c_int32), ("stages", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("timeout_ns", ctypes.c_int64)]


class MgAttnPlanInfo(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("d", ctypes.c_int64),
                ("block_m", ctypes.c_int32), ("block_n", ctypes.c_int32), ("m_tiles", ctypes.c_int32),
                ("n_tiles", ctypes.c_int32), ("n_split", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("grid_ctas", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("tmem_cols", ctypes.c_int32), ("kernels_per_run", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("cluster_ctas", ctypes.c_int32),
                ("q_tiles_per_cta", ctypes.c_int32), ("schedule", ctypes.c_int32), ("swap_ab", ctypes.c_int32),
                ("xchg_push", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class MgAttnError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        text = _status_text(status)
        super().__init__(f"{where}: {text} (status {status})" + (f": {detail}" if detail else ""))


_lock = threading.Lock()
_lib = None


def _status_text(status: int) -> str:
    if _lib is None:
        return "error"
    return _lib.mg_attn_status_string(status).decode()


def _bind(lib):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    st = ctypes.c_int
    lib.mg_attn_plan.argtypes = [i64, i64, i64, i64, ctypes.POINTER(vp)]
    lib.mg_attn_plan.restype = st
    lib.mg_attn_plan_ex.argtypes = [i64, i64, i64, i64, ctypes.POINTER(MgAttnOptions), ctypes.POINTER(vp)]
    lib.mg_attn_plan_ex.restype = st
    lib.mg_attn_run.argtypes = [vp, vp, vp, vp, vp, vp]
    lib.mg_attn_run.restype = st
    lib.mg_attn_run_host.argtypes = [vp, vp, vp, vp, vp, vp]
    lib.mg_attn_run_host.restype = st
    lib.mg_attn_destroy.argtypes = [vp]
    lib.mg_attn_destroy.restype = st
    lib.mg_attn_get_status.argtypes = [vp]
    lib.mg_attn_get_status.restype = st
    lib.mg_attn_get_info.argtypes = [vp, ctypes.POINTER(MgAttnPlanInfo)]
    lib.mg_attn_get_info.restype = st
    lib.mg_attn_query.argtypes = [i64, i64, i64, i64, ctypes.POINTER(MgAttnOptions), i32, i32,
                                  ctypes.POINTER(MgAttnPlanInfo)]
    lib.mg_attn_query.restype = st
    lib.mg_attn_status_string.argtypes = [st]
    lib.mg_attn_status_string.restype = ctypes.c_char_p
    lib.mg_attn_last_error.argtypes = []
    lib.mg_attn_last_error.restype = ctypes.c_char_p
    lib.mg_attn_set_timing_events.argtypes = [vp, vp, vp]
    lib.mg_attn_set_timing_events.restype = st
    lib.mg_attn_run_noalloc.argtypes = [i64, i64, i64, i64, vp, vp, vp, vp, vp]
    lib.mg_attn_run_noalloc.restype = st
    lib.mg_attn_version.argtypes = []
    lib.mg_attn_version.restype = i32
    lib.mg_diag_launch_floor.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_float)]
    lib.mg_diag_launch_floor.restype = st
    lib.mg_diag_exp_rate.argtypes = [i32, i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    lib.mg_diag_exp_rate.restype = st
    lib.mg_diag_last_error.argtypes = []
    lib.mg_diag_last_error.restype = ctypes.c_char_p
    return lib


def load_library(path: str = LIB_PATH):
    """Load ``libmgattn.so`` (built by ``attention_mugraph_gb300.build``). Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise ImportError(f"{path} is missing: build it with attention_mugraph_gb300.build.build() "
                                  "(there is no CPU fallback)")
            _lib = _bind(ctypes.CDLL(path))
    return _lib


def _check(status: int, where: str):
    if status != MG_OK:
        raise MgAttnError(status, where, load_library().mg_attn_last_error().decode())


def _options(n_split=0, stages=0, flags=0, timeout_ns=0) -> MgAttnOptions:
    return MgAttnOptions(int(n_split), int(stages), int(flags), 0, int(timeout_ns))


def mg_attn_query(B, M, N, d, num_sms, max_smem_optin=232448, n_split=0, stages=0, flags=0, timeout_ns=0) -> dict:
    """The plan's decisions for a device with ``num_sms`` SMs, without a GPU."""
    lib = load_library()
    info = MgAttnPlanInfo()
    opts = _options(n_split, stages, flags, timeout_ns)
    _check(lib.mg_attn_query(B, M, N, d, ctypes.byref(opts), num_sms, max_smem_optin, ctypes.byref(info)),
           "mg_attn_query")
    return info.as_dict()


def _stream_handle(stream):
    if stream is None:
        import torch

        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def run_noalloc(Q, K, V, O, stream=None):
    """mg_attn_run_noalloc: O = attention(Q, K, V) with no plan and no device allocation (the split
    partials go to the library's fixed 8 MiB array; calls that overlap on the GPU share it and
    must be serialised). Q (B,M,d), K (B,d,N), V (B,N,d), O (B,M,d): contiguous fp16 CUDA tensors."""
    import torch

    B, M, d = (int(x) for x in Q.shape)
    N = int(K.shape[2])
    for t, shape, name in ((Q, (B, M, d), "Q"), (K, (B, d, N), "K"), (V, (B, N, d), "V"), (O, (B, M, d), "O")):
        if t.dtype != torch.float16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be a contiguous fp16 CUDA tensor of shape {shape}")
    lib = load_library()
    _check(lib.mg_attn_run_noalloc(B, M, N, d, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                                   _stream_handle(stream)), "mg_attn_run_noalloc")
    return O


class Plan:
    """Owns one ``mg_attn_plan_t`` for a fixed (B, M, N, d) on the current CUDA device."""

    def __init__(self, B, M, N, d, n_split=0, stages=0, flags=0, timeout_ns=0):
        self._lib = load_library()
        self._h = ctypes.c_void_p()
        opts = _options(n_split, stages, flags, timeout_ns)
        _check(self._lib.mg_attn_plan_ex(B, M, N, d, ctypes.byref(opts), ctypes.byref(self._h)), "mg_attn_plan")
        info = MgAttnPlanInfo()
        _check(self._lib.mg_attn_get_info(self._h, ctypes.byref(info)), "mg_attn_get_info")
        self.info = info.as_dict()
        self.shape = (int(B), int(M), int(N), int(d))

    def _expect(self, t, shape, name):
        import torch

        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != torch.float16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be a contiguous CUDA fp16 tensor of shape {shape}, got "
                             f"{tuple(t.shape)} {t.dtype} {t.device} contiguous={t.is_contiguous()}")

    def run(self, Q, K, V, O, stream=None):
        """Enqueue O = attention(Q, K, V) on ``stream`` (default: torch's current stream)."""
        B, M, N, d = self.shape
        self._expect(Q, (B, M, d), "Q")
        self._expect(K, (B, d, N), "K")
        self._expect(V, (B, N, d), "V")
        self._expect(O, (B, M, d), "O")
        _check(self._lib.mg_attn_run(self._h, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                                     _stream_handle(stream)), "mg_attn_run")
        return O

    def run_ptr(self, q_ptr, k_ptr, v_ptr, o_ptr, stream=None):
        """Raw-pointer form of run(); the caller vouches for shapes and placement."""
        _check(self._lib.mg_attn_run(self._h, q_ptr, k_ptr, v_ptr, o_ptr, _stream_handle(stream)), "mg_attn_run")

    def run_host(self, hQ, hK, hV, hO, stream=None):
        """Host-buffer variant: hQ/hK/hV/hO are CPU fp16 tensors (pinned for async copies)."""
        import torch

        B, M, N, d = self.shape
        for t, shape, name in ((hQ, (B, M, d), "hQ"), (hK, (B, d, N), "hK"), (hV, (B, N, d), "hV"),
                               (hO, (B, M, d), "hO")):
            if t.dtype != torch.float16 or t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shape:
                raise ValueError(f"{name} must be a contiguous CPU fp16 tensor of shape {shape}")
        _check(self._lib.mg_attn_run_host(self._h, hQ.data_ptr(), hK.data_ptr(), hV.data_ptr(), hO.data_ptr(),
                                          _stream_handle(stream)), "mg_attn_run_host")
        return hO

    def set_timing_events(self, ev_begin=None, ev_end=None):
        """Record two torch.cuda.Event objects around the fused kernel of later runs (None: off).
        The events must already exist on the CUDA side (torch creates them on their first record)."""
        b = ctypes.c_void_p(ev_begin.cuda_event) if ev_begin is not None else None
        e = ctypes.c_void_p(ev_end.cuda_event) if ev_end is not None else None
        if (ev_begin is not None and not b.value) or (ev_end is not None and not e.value):
            raise ValueError("record the events once before handing them to the library")
        _check(self._lib.mg_attn_set_timing_events(self._h, b, e), "mg_attn_set_timing_events")

    def status(self) -> int:
        """Sticky device status (synchronises the device): MG_OK or MG_ERR_TIMEOUT."""
        return int(self._lib.mg_attn_get_status(self._h))

    def destroy(self):
        if self._h:
            _check(self._lib.mg_attn_destroy(self._h), "mg_attn_destroy")
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            if self._h:
                self._lib.mg_attn_destroy(self._h)
        except Exception:
            pass


def _check_diag(status: int, where: str):
    if status != MG_OK:
        raise MgAttnError(status, where, load_library().mg_diag_last_error().decode())


def diag_launch_floor(ctas, cluster=1, smem_bytes=215296, pdl=True, launches=1000) -> float:
    """µs per launch of a no-work kernel with this launch shape (``mg_diag_launch_floor``)."""
    out = ctypes.c_float()
    _check_diag(load_library().mg_diag_launch_floor(int(ctas), int(cluster), int(smem_bytes), 1 if pdl else 0,
                                                    int(launches), ctypes.byref(out)), "mg_diag_launch_floor")
    return float(out.value)


def diag_exp_rate(iters=2000, poly=False) -> tuple:
    """(exponentials per SM clock, per SM ns) of the fused kernel's exp (``mg_diag_exp_rate``)."""
    clk, ns = ctypes.c_double(), ctypes.c_double()
    _check_diag(load_library().mg_diag_exp_rate(int(iters), 1 if poly else 0, ctypes.byref(clk), ctypes.byref(ns)),
                "mg_diag_exp_rate")
    return float(clk.value), float(ns.value)


def mg_attn_plan(B, M, N, d, **opts) -> Plan:
    return Plan(B, M, N, d, **opts)


_plans: dict = {}


def attention(Q, K, V, out=None, stream=None):
    """O = (exp(Q.K) / rowsum(exp(Q.K))) . V for fp16 CUDA tensors Q (B,M,d), K (B,d,N), V (B,N,d).

    Plans are cached per (shape, device)."""
    import torch

    B, M, d = Q.shape
    N = K.shape[2]
    key = (int(B), int(M), int(N), int(d), Q.device.index)
    plan = _plans.get(key)
    if plan is None:
        with torch.cuda.device(Q.device):
            plan = _plans[key] = Plan(B, M, N, d)
    if out is None:
        out = torch.empty((B, M, d), dtype=torch.float16, device=Q.device)
    return plan.run(Q, K, V, out, stream)

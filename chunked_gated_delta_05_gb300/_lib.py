"""ctypes view of libgdn's C ABI (include/gdn.h): struct layouts, loading and error mapping."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

GDN_OK, GDN_EINVAL, GDN_EUNSUPPORTED, GDN_ECUDA, GDN_ETIMEOUT, GDN_ERANGE = 0, 1, 2, 3, 4, 5

c_int, c_float, c_size_t, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p


class Desc(ctypes.Structure):
    _fields_ = [("B", c_int), ("T", c_int), ("H", c_int), ("K", c_int), ("V", c_int),
                ("chunk_size", c_int), ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)),
                ("num_seqs", c_int), ("scale", c_float), ("use_qk_l2norm", c_int),
                ("use_beta_sigmoid", c_int), ("output_final_state", c_int), ("num_k_heads", c_int),
                ("use_gate_in_kernel", c_int), ("lower_bound", c_float)]


class FwdArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("g", c_void_p),
                ("beta", c_void_p), ("initial_state", c_void_p), ("o", c_void_p),
                ("final_state", c_void_p), ("workspace", c_void_p), ("workspace_bytes", c_size_t),
                ("status", c_void_p), ("saved", c_void_p), ("saved_bytes", c_size_t),
                ("A_log", c_void_p), ("dt_bias", c_void_p)]


class BwdArgs(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("g", c_void_p),
                ("beta", c_void_p), ("initial_state", c_void_p), ("dO", c_void_p),
                ("dht", c_void_p), ("dq", c_void_p), ("dk", c_void_p), ("dv", c_void_p),
                ("dbeta", c_void_p), ("dg", c_void_p), ("dh0", c_void_p),
                ("workspace", c_void_p), ("workspace_bytes", c_size_t), ("status", c_void_p),
                ("saved", c_void_p), ("saved_bytes", c_size_t), ("A_log", c_void_p), ("dt_bias", c_void_p),
                ("dA_log", c_void_p), ("ddt_bias", c_void_p)]


class ConvDesc(ctypes.Structure):
    _fields_ = [("B", c_int), ("T", c_int), ("C", c_int), ("W", c_int), ("dilation", c_int),
                ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)), ("num_seqs", c_int), ("activation", c_int)]


class ConvFwdArgs(ctypes.Structure):
    _fields_ = [("x", c_void_p), ("weight", c_void_p), ("bias", c_void_p), ("halo", c_void_p),
                ("y", c_void_p), ("workspace", c_void_p), ("workspace_bytes", c_size_t)]


class ConvBwdArgs(ctypes.Structure):
    _fields_ = [("x", c_void_p), ("weight", c_void_p), ("bias", c_void_p), ("halo", c_void_p),
                ("dy", c_void_p), ("dx", c_void_p), ("dweight", c_void_p), ("dbias", c_void_p),
                ("dhalo", c_void_p), ("workspace", c_void_p), ("workspace_bytes", c_size_t)]


# Every symbol include/gdn.h declares, with its ctypes signature.
SIGNATURES = {
    "gdn_strerror": ([c_int], ctypes.c_char_p),
    "gdn_last_error": ([], ctypes.c_char_p),
    "gdn_device_supported": ([c_int], c_int),
    "gdn_fwd_workspace_size": ([ctypes.POINTER(Desc)], c_size_t),
    "gdn_bwd_workspace_size": ([ctypes.POINTER(Desc)], c_size_t),
    "kda_fwd_workspace_size": ([ctypes.POINTER(Desc)], c_size_t),
    "kda_bwd_workspace_size": ([ctypes.POINTER(Desc)], c_size_t),
    "gdn_saved_size": ([ctypes.POINTER(Desc)], c_size_t),
    "kda_saved_size": ([ctypes.POINTER(Desc)], c_size_t),
    "gdn_fwd": ([ctypes.POINTER(Desc), ctypes.POINTER(FwdArgs), c_void_p], c_int),
    "gdn_bwd": ([ctypes.POINTER(Desc), ctypes.POINTER(BwdArgs), c_void_p], c_int),
    "kda_fwd": ([ctypes.POINTER(Desc), ctypes.POINTER(FwdArgs), c_void_p], c_int),
    "kda_bwd": ([ctypes.POINTER(Desc), ctypes.POINTER(BwdArgs), c_void_p], c_int),
    "gdn_fwd_noalloc": ([ctypes.POINTER(Desc), ctypes.POINTER(FwdArgs), c_void_p], c_int),
    "gdn_fwd_noalloc_capacity": ([], c_size_t),
    "gdn_set_chain_segment": ([c_int], c_int),
    "gdn_chain_plan": ([ctypes.POINTER(Desc), ctypes.POINTER(c_int), ctypes.POINTER(c_int)], c_int),
    "gdn_set_head_groups": ([c_int], c_int),
    "gdn_conv_fwd_workspace_size": ([ctypes.POINTER(ConvDesc)], c_size_t),
    "gdn_conv_bwd_workspace_size": ([ctypes.POINTER(ConvDesc)], c_size_t),
    "gdn_conv_fwd": ([ctypes.POINTER(ConvDesc), ctypes.POINTER(ConvFwdArgs), c_void_p], c_int),
    "gdn_conv_bwd": ([ctypes.POINTER(ConvDesc), ctypes.POINTER(ConvBwdArgs), c_void_p], c_int),
    "gdn_timing_enable": ([c_int], c_int),
    "gdn_timing_kinds": ([], c_int),
    "gdn_timing_name": ([c_int], ctypes.c_char_p),
    "gdn_timing_read": ([c_int, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(c_int)], c_int),
    "gdn_wait_selftest": ([c_void_p, ctypes.c_longlong, c_void_p, c_void_p], c_int),
}

_lock = threading.Lock()
_lib = None


def load(build_if_missing: bool = True):
    """Load libgdn.so (building it first when missing or stale). Raises if it cannot."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing:
                path = _build.build()
            else:
                path = _build.LIB
                if not os.path.exists(path):
                    raise RuntimeError("libgdn.so is not built; run chunked_gated_delta_05_gb300.build")
            lib = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


class GdnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


def check(code: int) -> None:
    if code == GDN_OK:
        return
    lib = load()
    detail = lib.gdn_last_error().decode() or lib.gdn_strerror(code).decode()
    if code == GDN_EINVAL:
        raise ValueError(detail)
    raise GdnError(code, f"{lib.gdn_strerror(code).decode()}: {detail}")


def timing_enable(on: bool = True) -> None:
    """Bracket every library kernel launch with CUDA events (profiling aid)."""
    check(load().gdn_timing_enable(int(bool(on))))


def timing_read() -> dict:
    """Per-kernel {name: (total_ms, launches)} since the last read; synchronizes the events."""
    lib = load()
    out = {}
    for kind in range(lib.gdn_timing_kinds()):
        ms = ctypes.c_double()
        n = c_int()
        check(lib.gdn_timing_read(kind, ctypes.byref(ms), ctypes.byref(n)))
        out[lib.gdn_timing_name(kind).decode()] = (ms.value, n.value)
    return out

"""CPU oracle for the chunked gated delta rule (Gated DeltaNet and Kimi Delta Attention).

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` leg (and its ``--impl reference`` arm) may import this package. The CUDA
library never calls it and shares no code with it.

Two independent implementations live here:

* ``recurrent.cpp``: the token-by-token recurrence in fp64, forward and adjoint backward,
  scalar (GDN) or per-channel (KDA) gate, dense or packed documents, threaded over
  (sequence, head) chains. It is the oracle the GPU path is judged against.
* ``chunked.py``: the naive chunked form the eager reference on the pages computes (GDN),
  used to cross-check the recurrence and to expose chunk intermediates.

``build()`` compiles ``recurrent.cpp`` with the host C++ compiler into ``_build/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "recurrent.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the fp64 recurrence into a shared library; return its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            common = [ctypes.c_int, ip, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                      dp, dp, dp, dp, dp, dp]
            lib.oracle_gdr_fwd.argtypes = common + [dp, dp, ctypes.c_int]
            lib.oracle_gdr_fwd.restype = ctypes.c_int
            lib.oracle_gdr_bwd.argtypes = common + [dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
            lib.oracle_gdr_bwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _sequences(B, T, cu_seqlens):
    """Return (starts, lens) of the independent sequences over the flattened B*T rows."""
    if cu_seqlens is None:
        starts = np.arange(B, dtype=np.int64) * T
        lens = np.full(B, T, dtype=np.int64)
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        if B != 1:
            raise ValueError("packed documents need batch size 1")
        starts = cu[:-1].copy()
        lens = np.diff(cu)
    return np.ascontiguousarray(starts), np.ascontiguousarray(lens)


def _dims(q, v, g):
    B, T, _, K = q.shape
    H, V = v.shape[2], v.shape[-1]
    per_channel = int(g.ndim == 4)
    return B, T, H, K, V, per_channel


def _repeat_heads(x, H):
    """Grouped q/k heads: ``x [B,T,Hk,K]`` repeated to the ``H`` value heads, each q/k head
    ``H // Hk`` times in a row (``repeat_interleave`` of the hyper-parallel GDN and KDA pages,
    value head h reading q/k head h // (H // Hk))."""
    Hk = x.shape[2]
    if H % Hk:
        raise ValueError("the value heads must be a multiple of the q/k heads")
    return np.repeat(x, H // Hk, axis=2) if Hk != H else x


def _sum_groups(dx, Hk):
    """Gradient of a repeated q/k head: the sum over the value heads that read it."""
    B, T, H, K = dx.shape
    return dx.reshape(B, T, Hk, H // Hk, K).sum(axis=3) if Hk != H else dx


def gdr_fwd(q, k, v, g, beta, *, scale=None, initial_state=None, output_final_state=True,
            use_qk_l2norm=False, use_beta_sigmoid=False, cu_seqlens=None, threads=0):
    """Token recurrence forward in fp64.

    q, k ``[B,T,Hk,K]`` (Hk dividing H: grouped q/k heads, see ``_repeat_heads``); v ``[B,T,H,V]``;
    g ``[B,T,H]`` (GDN) or ``[B,T,H,K]`` (KDA), natural
    log decay; beta ``[B,T,H]``; initial_state ``[N,H,K,V]`` (N = B, or the number of
    documents when ``cu_seqlens`` is given). Returns ``(o [B,T,H,V], final [N,H,K,V] or None)``.
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    h0 = _f64(initial_state)
    B, T, H, K, V, per_channel = _dims(q, v, g)
    q, k = np.ascontiguousarray(_repeat_heads(q, H)), np.ascontiguousarray(_repeat_heads(k, H))
    starts, lens = _sequences(B, T, cu_seqlens)
    N = len(lens)
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    o = np.zeros((B, T, H, V))
    hT = np.zeros((N, H, K, V)) if output_final_state else None
    rc = _load().oracle_gdr_fwd(
        N, starts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, K, V, per_channel,
        int(bool(use_qk_l2norm)), int(bool(use_beta_sigmoid)), float(scale),
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(hT), int(threads))
    if rc != 0:
        raise ValueError("oracle_gdr_fwd rejected its arguments")
    return o, hT


def gdr_bwd(q, k, v, g, beta, dO, *, dht=None, scale=None, initial_state=None,
            use_qk_l2norm=False, use_beta_sigmoid=False, cu_seqlens=None, threads=0):
    """Adjoint of :func:`gdr_fwd`: gradients of ``<dO, o> + <dht, final>``.

    Returns a dict with dq, dk, dv, dbeta (w.r.t. beta as passed), dg (w.r.t. the raw
    per-token gate, same shape as g) and dh0 (``[N,H,K,V]``).
    """
    q, k, v, g, beta, dO = (_f64(x) for x in (q, k, v, g, beta, dO))
    h0, dht = _f64(initial_state), _f64(dht)
    B, T, H, K, V, per_channel = _dims(q, v, g)
    Hk = q.shape[2]
    q, k = np.ascontiguousarray(_repeat_heads(q, H)), np.ascontiguousarray(_repeat_heads(k, H))
    starts, lens = _sequences(B, T, cu_seqlens)
    N = len(lens)
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dbeta=np.zeros_like(beta), dg=np.zeros_like(g), dh0=np.zeros((N, H, K, V)))
    rc = _load().oracle_gdr_bwd(
        N, starts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, K, V, per_channel,
        int(bool(use_qk_l2norm)), int(bool(use_beta_sigmoid)), float(scale),
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(dO), _ptr(dht),
        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["dg"]),
        _ptr(out["dh0"]), int(threads))
    if rc != 0:
        raise ValueError("oracle_gdr_bwd rejected its arguments")
    out["dq"], out["dk"] = _sum_groups(out["dq"], Hk), _sum_groups(out["dk"], Hk)
    return out

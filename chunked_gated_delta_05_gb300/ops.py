"""PyTorch-facing wrappers of libgdn. Argument marshalling only: torch allocates device memory
and provides the stream; every step of the computation runs in the library's CUDA kernels.
There is no fallback path: without the built library or a GB300 these functions raise."""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib

K_DIM = 128
CHUNK = 64


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_tensor(name, t, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _offsets(cu_seqlens, T):
    """Host int32 copy of packed document offsets (CPU tensor or sequence of ints)."""
    if cu_seqlens is None:
        return None
    if isinstance(cu_seqlens, torch.Tensor):
        if cu_seqlens.device.type != "cpu" or cu_seqlens.dim() != 1 or \
                cu_seqlens.dtype not in (torch.int32, torch.int64):
            raise ValueError("cu_seqlens must be a one-dimensional CPU int32/int64 tensor or a sequence")
        vals = [int(x) for x in cu_seqlens.tolist()]
    else:
        if any(isinstance(x, bool) or not isinstance(x, int) for x in cu_seqlens):
            raise ValueError("cu_seqlens entries must be ints")
        vals = [int(x) for x in cu_seqlens]
    if len(vals) < 2:
        raise ValueError("cu_seqlens needs at least two entries")
    return (ctypes.c_int32 * len(vals))(*vals), len(vals) - 1


def _desc(B, T, H, scale, l2, sig, final, offsets, Hk=None, gate=None):
    d = _lib.Desc()
    d.B, d.T, d.H, d.K, d.V, d.chunk_size = B, T, H, K_DIM, K_DIM, CHUNK
    d.num_k_heads = 0 if Hk is None or Hk == H else int(Hk)
    if offsets is not None:
        arr, n = offsets
        d.cu_seqlens = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
        d.num_seqs = n
    else:
        d.num_seqs = B
    d.scale = 0.0 if scale is None else float(scale)
    d.use_qk_l2norm, d.use_beta_sigmoid, d.output_final_state = int(bool(l2)), int(bool(sig)), int(bool(final))
    if gate is not None:
        d.use_gate_in_kernel, d.lower_bound = 1, float(gate[2])
    return d


def _gate_checks(gate, H, dev):
    """``gate = (A_log [H], dt_bias [H,128] or [H*128], lower_bound)`` of the in-kernel KDA gate,
    or None. Returns fp32 contiguous parameter tensors (or Nones)."""
    if gate is None:
        return None, None
    A_log, dt_bias, lb = gate
    if lb is None:
        raise ValueError("lower_bound is required with the in-kernel gate")
    _check_tensor("A_log", A_log, torch.float32, (H,), dev)
    if not isinstance(dt_bias, torch.Tensor) or dt_bias.numel() != H * K_DIM or dt_bias.dtype != torch.float32 \
            or dt_bias.device != dev or not dt_bias.is_contiguous():
        raise ValueError(f"dt_bias must be a contiguous fp32 tensor of {H}*{K_DIM} elements on {dev}")
    return A_log, dt_bias


def _common_checks(q, k, v, g, beta, per_channel, offsets):
    """Shapes: q, k [B,T,Hk,K]; v [B,T,H,V] with Hk dividing H (grouped q/k heads when
    Hk < H); g [B,T,H] or [B,T,H,K]; beta [B,T,H]. Returns (B, T, H, Hk, N, device)."""
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q and v must have shape [B,T,H,D]")
    B, T, Hk, K = q.shape
    H = v.shape[2]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if H % Hk != 0:
        raise ValueError("the value heads must be a multiple of the q/k heads")
    _check_tensor("q", q, torch.bfloat16, (B, T, Hk, K), dev)
    _check_tensor("k", k, torch.bfloat16, (B, T, Hk, K), dev)
    _check_tensor("v", v, torch.bfloat16, (B, T, H, v.shape[-1]), dev)
    gshape = (B, T, H, K) if per_channel else (B, T, H)
    _check_tensor("g", g, torch.float32, gshape, dev)
    _check_tensor("beta", beta, torch.bfloat16, (B, T, H), dev)
    N = B if offsets is None else offsets[1]
    return B, T, H, Hk, N, dev


def _fwd(per_channel, q, k, v, g, beta, initial_state, output_final_state, use_qk_l2norm,
         use_beta_sigmoid, cu_seqlens, scale, status, save=False, gate=None):
    lib = _lib.load()
    offsets = _offsets(cu_seqlens, q.shape[1] if q.dim() == 4 else 0)
    B, T, H, Hk, N, dev = _common_checks(q, k, v, g, beta, per_channel, offsets)
    if initial_state is not None:
        _check_tensor("initial_state", initial_state, torch.float32, (N, H, K_DIM, K_DIM), dev)
    A_log, dt_bias = _gate_checks(gate, H, dev)
    desc = _desc(B, T, H, scale, use_qk_l2norm, use_beta_sigmoid, output_final_state, offsets, Hk, gate)
    if save:
        size_fn = lib.kda_saved_size if per_channel else lib.gdn_saved_size
    else:
        size_fn = lib.kda_fwd_workspace_size if per_channel else lib.gdn_fwd_workspace_size
    ws_bytes = size_fn(ctypes.byref(desc))
    if ws_bytes == 0:
        _lib.check(_lib.GDN_EINVAL)
    o = torch.empty((B, T, H, K_DIM), dtype=torch.bfloat16, device=dev)  # value heads
    final = torch.empty((N, H, K_DIM, K_DIM), dtype=torch.float32, device=dev) if output_final_state else None
    buf = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    a = _lib.FwdArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), g=_ptr(g), beta=_ptr(beta),
                     initial_state=_ptr(initial_state), o=_ptr(o), final_state=_ptr(final),
                     workspace=None if save else _ptr(buf), workspace_bytes=0 if save else ws_bytes,
                     status=_ptr(status), saved=_ptr(buf) if save else None, saved_bytes=ws_bytes if save else 0,
                     A_log=_ptr(A_log), dt_bias=_ptr(dt_bias))
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    fn = lib.kda_fwd if per_channel else lib.gdn_fwd
    _lib.check(fn(ctypes.byref(desc), ctypes.byref(a), stream))
    if save:
        return o, final, buf
    return o, final


def _bwd(per_channel, q, k, v, g, beta, dO, dht, initial_state, use_qk_l2norm, use_beta_sigmoid,
         cu_seqlens, scale, status, saved=None, gate=None):
    lib = _lib.load()
    offsets = _offsets(cu_seqlens, q.shape[1] if q.dim() == 4 else 0)
    B, T, H, Hk, N, dev = _common_checks(q, k, v, g, beta, per_channel, offsets)
    _check_tensor("dO", dO, torch.bfloat16, (B, T, H, K_DIM), dev)
    if initial_state is not None:
        _check_tensor("initial_state", initial_state, torch.float32, (N, H, K_DIM, K_DIM), dev)
    if dht is not None:
        _check_tensor("dht", dht, torch.float32, (N, H, K_DIM, K_DIM), dev)
    A_log, dt_bias = _gate_checks(gate, H, dev)
    desc = _desc(B, T, H, scale, use_qk_l2norm, use_beta_sigmoid, False, offsets, Hk, gate)
    size_fn = lib.kda_bwd_workspace_size if per_channel else lib.gdn_bwd_workspace_size
    ws_bytes = size_fn(ctypes.byref(desc))
    if ws_bytes == 0:
        _lib.check(_lib.GDN_EINVAL)
    saved_bytes = 0
    if saved is not None:
        saved_bytes = (lib.kda_saved_size if per_channel else lib.gdn_saved_size)(ctypes.byref(desc))
        if not isinstance(saved, torch.Tensor) or saved.device != dev or saved.numel() < saved_bytes:
            raise ValueError("saved must be the buffer returned by the forward with save=True")
        ws_bytes -= saved_bytes
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dbeta = torch.empty_like(beta)
    dg = torch.empty_like(g)
    dh0 = torch.empty((N, H, K_DIM, K_DIM), dtype=torch.float32, device=dev) if initial_state is not None else None
    dA_log = torch.empty_like(A_log) if gate is not None else None
    ddt_bias = torch.empty_like(dt_bias) if gate is not None else None
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    a = _lib.BwdArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), g=_ptr(g), beta=_ptr(beta),
                     initial_state=_ptr(initial_state), dO=_ptr(dO), dht=_ptr(dht), dq=_ptr(dq),
                     dk=_ptr(dk), dv=_ptr(dv), dbeta=_ptr(dbeta), dg=_ptr(dg), dh0=_ptr(dh0),
                     workspace=_ptr(ws), workspace_bytes=ws_bytes, status=_ptr(status),
                     saved=_ptr(saved), saved_bytes=saved_bytes, A_log=_ptr(A_log), dt_bias=_ptr(dt_bias),
                     dA_log=_ptr(dA_log), ddt_bias=_ptr(ddt_bias))
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    fn = lib.kda_bwd if per_channel else lib.gdn_bwd
    _lib.check(fn(ctypes.byref(desc), ctypes.byref(a), stream))
    if gate is not None:
        return dq, dk, dv, dbeta, dg, dh0, dA_log, ddt_bias
    return dq, dk, dv, dbeta, dg, dh0


def set_chain_segment(chunks: int) -> None:
    """Force the segment length (in chunks) of the segmented state chain for every later call
    of the process; 0 restores the automatic choice. Workspace and saved sizes depend on it."""
    _lib.check(_lib.load().gdn_set_chain_segment(int(chunks)))


def set_head_groups(groups: int) -> None:
    """Force 1 or 2 head groups (the second on the library's side stream) for every later call
    of the process; 0 restores the automatic choice. Results do not depend on it."""
    _lib.check(_lib.load().gdn_set_head_groups(int(groups)))


def chain_plan(B: int, T: int, H: int, cu_seqlens: Optional[Sequence[int]] = None):
    """``(chunks per segment, most segments of any sequence)`` the library picks for a shape."""
    offsets = _offsets(cu_seqlens, T)
    desc = _desc(B, T, H, None, True, False, False, offsets)
    L, S = ctypes.c_int(), ctypes.c_int()
    _lib.check(_lib.load().gdn_chain_plan(ctypes.byref(desc), ctypes.byref(L), ctypes.byref(S)))
    return L.value, S.value


def gdn_fwd(q, k, v, g, beta, *, initial_state=None, output_final_state=False, use_qk_l2norm=True,
            use_beta_sigmoid=False, cu_seqlens: Optional[Sequence[int]] = None, scale=None, status=None,
            save=False):
    """Gated DeltaNet forward. Returns ``(o [B,T,H,128] bf16, final_state [N,H,128,128] fp32 or
    None)``; with ``save=True`` also the saved-intermediates buffer to hand to :func:`gdn_bwd`."""
    return _fwd(False, q, k, v, g, beta, initial_state, output_final_state, use_qk_l2norm,
                use_beta_sigmoid, cu_seqlens, scale, status, save)


def kda_fwd(q, k, v, g, beta, *, initial_state=None, output_final_state=False, use_qk_l2norm=True,
            use_beta_sigmoid=True, cu_seqlens: Optional[Sequence[int]] = None, scale=None, status=None,
            save=False, A_log=None, dt_bias=None, lower_bound=None):
    """Kimi Delta Attention forward (per-channel gate g [B,T,H,128]). With ``A_log`` [H],
    ``dt_bias`` [H,128] and ``lower_bound`` in [-5, 0), g holds gate logits x and the kernels
    use the safe gate lower_bound * sigmoid(exp(A_log) (x + dt_bias))."""
    gate = None if A_log is None else (A_log, dt_bias, lower_bound)
    return _fwd(True, q, k, v, g, beta, initial_state, output_final_state, use_qk_l2norm,
                use_beta_sigmoid, cu_seqlens, scale, status, save, gate)


def gdn_bwd(q, k, v, g, beta, dO, *, dht=None, initial_state=None, use_qk_l2norm=True,
            use_beta_sigmoid=False, cu_seqlens=None, scale=None, status=None, saved=None):
    """Gated DeltaNet backward. Returns ``(dq, dk, dv, dbeta, dg, dh0 or None)``. ``saved`` is the
    buffer of a ``save=True`` forward on the same inputs (else the forward is recomputed)."""
    return _bwd(False, q, k, v, g, beta, dO, dht, initial_state, use_qk_l2norm, use_beta_sigmoid,
                cu_seqlens, scale, status, saved)


def kda_bwd(q, k, v, g, beta, dO, *, dht=None, initial_state=None, use_qk_l2norm=True,
            use_beta_sigmoid=True, cu_seqlens=None, scale=None, status=None, saved=None,
            A_log=None, dt_bias=None, lower_bound=None):
    """Kimi Delta Attention backward. Returns ``(dq, dk, dv, dbeta, dg, dh0 or None)``; with the
    in-kernel gate (``A_log``, ``dt_bias``, ``lower_bound`` as in :func:`kda_fwd`) dg is w.r.t.
    the gate logits and ``dA_log [H]``, ``ddt_bias`` (dt_bias's shape) follow."""
    gate = None if A_log is None else (A_log, dt_bias, lower_bound)
    return _bwd(True, q, k, v, g, beta, dO, dht, initial_state, use_qk_l2norm, use_beta_sigmoid,
                cu_seqlens, scale, status, saved, gate)


class ChunkGatedDeltaRule(torch.autograd.Function):
    """Autograd wrapper: forward through gdn_fwd/kda_fwd in save mode, backward through
    gdn_bwd/kda_bwd with the saved intermediates. With the KDA in-kernel gate, g holds the gate
    logits and A_log, dt_bias receive gradients too."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, initial_state, A_log, dt_bias, per_channel, use_qk_l2norm,
                use_beta_sigmoid, cu_seqlens, scale, output_final_state, lower_bound):
        gate = None if A_log is None else (A_log, dt_bias, lower_bound)
        o, final, saved = _fwd(per_channel, q, k, v, g, beta, initial_state, output_final_state,
                               use_qk_l2norm, use_beta_sigmoid, cu_seqlens, scale, None, save=True, gate=gate)
        ctx.save_for_backward(q, k, v, g, beta, initial_state, A_log, dt_bias, saved)
        ctx.cfg = (per_channel, use_qk_l2norm, use_beta_sigmoid, cu_seqlens, scale, lower_bound)
        return o, final

    @staticmethod
    def backward(ctx, dO, dfinal):
        q, k, v, g, beta, h0, A_log, dt_bias, saved = ctx.saved_tensors
        per_channel, l2, sig, cu, scale, lower_bound = ctx.cfg
        gate = None if A_log is None else (A_log, dt_bias, lower_bound)
        out = _bwd(per_channel, q, k, v, g, beta, dO.contiguous(), None if dfinal is None else dfinal.contiguous(),
                   h0, l2, sig, cu, scale, None, saved, gate)
        dq, dk, dv, dbeta, dg, dh0 = out[:6]
        dA, ddt = (out[6], out[7]) if gate is not None else (None, None)
        return dq, dk, dv, dg, dbeta, dh0, dA, ddt, None, None, None, None, None, None, None


def chunk_gated_delta_rule(q, k, v, g, beta, *, initial_state=None, output_final_state=False,
                           use_qk_l2norm=True, use_beta_sigmoid=None, cu_seqlens=None, scale=None,
                           A_log=None, dt_bias=None, lower_bound=None):
    """Differentiable entry point; the gate's rank selects GDN ([B,T,H]) or KDA ([B,T,H,K]).
    For KDA, ``A_log``, ``dt_bias`` and ``lower_bound`` select the in-kernel safe gate (g then
    holds the gate logits; see :func:`kda_fwd`)."""
    per_channel = g.dim() == 4
    if use_beta_sigmoid is None:
        use_beta_sigmoid = per_channel
    if A_log is not None and not per_channel:
        raise ValueError("the in-kernel gate is a KDA option (g must be [B,T,H,K])")
    return ChunkGatedDeltaRule.apply(q, k, v, g, beta, initial_state, A_log, dt_bias, per_channel, use_qk_l2norm,
                                     use_beta_sigmoid, cu_seqlens, scale, output_final_state, lower_bound)


# ---------------------------------------------------------------- short convolution

def _conv_desc(x, weight, dilation, activation, offsets):
    if x.dim() != 3 or weight.dim() != 2 or weight.shape[0] != x.shape[2]:
        raise ValueError("x must be [B,T,C] and weight [C,W]")
    d = _lib.ConvDesc()
    d.B, d.T, d.C = x.shape
    d.W, d.dilation, d.activation = weight.shape[1], int(dilation), int(bool(activation))
    if offsets is not None:
        arr, n = offsets
        d.cu_seqlens = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
        d.num_seqs = n
    else:
        d.num_seqs = d.B
    return d


def _conv_checks(x, weight, bias, halo, N, HW):
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    B, T, C = x.shape
    _check_tensor("x", x, torch.bfloat16, (B, T, C), dev)
    _check_tensor("weight", weight, torch.float32, (C, weight.shape[1]), dev)
    if bias is not None:
        _check_tensor("bias", bias, torch.float32, (C,), dev)
    if halo is not None:
        _check_tensor("halo", halo, torch.bfloat16, (N, HW, C), dev)
    return dev


def causal_conv1d_fwd(x, weight, bias=None, *, dilation=1, activation=True, cu_seqlens=None, halo=None):
    """Causal depthwise Conv1d (+ SiLU) over the token axis of ``x [B,T,C]`` (bf16) with
    ``weight [C,W]`` (fp32), optional ``bias [C]`` and ``halo [N,(W-1)*dilation,C]``, per packed
    document when ``cu_seqlens`` is given. Returns ``y [B,T,C]`` (bf16)."""
    lib = _lib.load()
    offsets = _offsets(cu_seqlens, x.shape[1] if x.dim() == 3 else 0)
    desc = _conv_desc(x, weight, dilation, activation, offsets)
    N = desc.num_seqs
    dev = _conv_checks(x, weight, bias, halo, N, (weight.shape[1] - 1) * dilation)
    ws_bytes = lib.gdn_conv_fwd_workspace_size(ctypes.byref(desc))
    if ws_bytes == 0:
        _lib.check(_lib.GDN_EINVAL)
    y = torch.empty_like(x)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    a = _lib.ConvFwdArgs(x=_ptr(x), weight=_ptr(weight), bias=_ptr(bias), halo=_ptr(halo), y=_ptr(y),
                         workspace=_ptr(ws), workspace_bytes=ws_bytes)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    _lib.check(lib.gdn_conv_fwd(ctypes.byref(desc), ctypes.byref(a), stream))
    return y


def causal_conv1d_bwd(x, weight, bias, dy, *, dilation=1, activation=True, cu_seqlens=None, halo=None):
    """Gradients of ``<dy, causal_conv1d_fwd(...)>``: ``(dx bf16, dweight fp32, dbias fp32 or
    None, dhalo fp32 or None)``."""
    lib = _lib.load()
    offsets = _offsets(cu_seqlens, x.shape[1] if x.dim() == 3 else 0)
    desc = _conv_desc(x, weight, dilation, activation, offsets)
    N = desc.num_seqs
    HW = (weight.shape[1] - 1) * dilation
    dev = _conv_checks(x, weight, bias, halo, N, HW)
    _check_tensor("dy", dy, torch.bfloat16, tuple(x.shape), dev)
    ws_bytes = lib.gdn_conv_bwd_workspace_size(ctypes.byref(desc))
    if ws_bytes == 0:
        _lib.check(_lib.GDN_EINVAL)
    dx = torch.empty_like(x)
    dw = torch.empty_like(weight)
    db = torch.empty_like(bias) if bias is not None else None
    dh = torch.empty((N, HW, x.shape[2]), dtype=torch.float32, device=dev) if halo is not None else None
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    a = _lib.ConvBwdArgs(x=_ptr(x), weight=_ptr(weight), bias=_ptr(bias), halo=_ptr(halo), dy=_ptr(dy),
                         dx=_ptr(dx), dweight=_ptr(dw), dbias=_ptr(db), dhalo=_ptr(dh), workspace=_ptr(ws),
                         workspace_bytes=ws_bytes)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    _lib.check(lib.gdn_conv_bwd(ctypes.byref(desc), ctypes.byref(a), stream))
    return dx, dw, db, dh


class CausalConv1d(torch.autograd.Function):
    """Autograd wrapper of the short convolution."""

    @staticmethod
    def forward(ctx, x, weight, bias, halo, dilation, activation, cu_seqlens):
        ctx.save_for_backward(x, weight, bias, halo)
        ctx.cfg = (dilation, activation, cu_seqlens)
        return causal_conv1d_fwd(x, weight, bias, dilation=dilation, activation=activation,
                                 cu_seqlens=cu_seqlens, halo=halo)

    @staticmethod
    def backward(ctx, dy):
        x, weight, bias, halo = ctx.saved_tensors
        dilation, activation, cu = ctx.cfg
        dx, dw, db, dh = causal_conv1d_bwd(x, weight, bias, dy.contiguous(), dilation=dilation,
                                           activation=activation, cu_seqlens=cu, halo=halo)
        return dx, dw, db, (None if dh is None else dh.to(halo.dtype)), None, None, None


def causal_conv1d(x, weight, bias=None, *, dilation=1, activation=True, cu_seqlens=None, halo=None):
    """Differentiable short convolution (see :func:`causal_conv1d_fwd`)."""
    return CausalConv1d.apply(x, weight, bias, halo, dilation, activation, cu_seqlens)

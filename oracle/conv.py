"""Short convolution oracle (test infrastructure: only the tests, the smoke check and the
benchmark's CPU baseline use it; the product path never does).

Causal depthwise Conv1d over the token axis with optional bias and SiLU, per sequence, in
fp64 (the ShortConv ahead of the delta rule on the hyper-parallel GDN Diff Coverage page:
`_causal_conv1d_with_cp_halo` runs `conv1d` with causal zero padding, keeps the first T
outputs and applies `F.silu`; packed documents are convolved independently; a halo of the
previous (W-1) dilation tokens may stand in for the zero padding):

    z[t][c] = bias[c] + sum_{i<W} w[c][i] x[t - (W-1-i) d][c],    y = z * sigmoid(z)

Reading for dilation d > 1 (the pages require padding W-1 with the eager module but pass a
dilation to the fused backend): the causal form above, i.e. padding (W-1) d.
"""
from __future__ import annotations

import numpy as np


def _sequences(B, T, cu_seqlens):
    if cu_seqlens is None:
        return [(b * T, T, b) for b in range(B)]
    cu = [int(x) for x in cu_seqlens]
    return [(cu[n], cu[n + 1] - cu[n], n) for n in range(len(cu) - 1)]


def _extended(x_rows, halo_n, HW):
    """The sequence's inputs with its HW preceding rows (halo, or zeros) in front."""
    C = x_rows.shape[1]
    front = np.zeros((HW, C)) if halo_n is None else np.asarray(halo_n, np.float64)
    return np.concatenate([front, x_rows], axis=0)


def causal_conv1d(x, weight, bias=None, *, dilation=1, activation=True, cu_seqlens=None, halo=None):
    """x ``[B,T,C]``, weight ``[C,W]``, bias ``[C]`` or None, halo ``[N,(W-1)d,C]`` or None.
    Returns y ``[B,T,C]`` in fp64."""
    x = np.asarray(x, np.float64)
    w = np.asarray(weight, np.float64)
    B, T, C = x.shape
    W = w.shape[1]
    HW = (W - 1) * dilation
    flat = x.reshape(B * T, C)
    y = np.zeros_like(flat)
    for start, length, n in _sequences(B, T, cu_seqlens):
        ext = _extended(flat[start:start + length], None if halo is None else halo[n], HW)
        for t in range(length):
            z = np.zeros(C) if bias is None else np.asarray(bias, np.float64).copy()
            for i in range(W):
                z += w[:, i] * ext[HW + t - (W - 1 - i) * dilation]
            y[start + t] = z / (1.0 + np.exp(-z)) if activation else z
    return y.reshape(B, T, C)


def causal_conv1d_bwd(x, weight, bias, dy, *, dilation=1, activation=True, cu_seqlens=None, halo=None):
    """Adjoint of :func:`causal_conv1d`: gradients of ``<dy, y>``. Returns a dict with dx
    ``[B,T,C]``, dweight ``[C,W]``, dbias ``[C]`` and dhalo ``[N,(W-1)d,C]`` (zeros when no
    halo was given)."""
    x = np.asarray(x, np.float64)
    w = np.asarray(weight, np.float64)
    dy = np.asarray(dy, np.float64)
    B, T, C = x.shape
    W = w.shape[1]
    HW = (W - 1) * dilation
    flat, dflat = x.reshape(B * T, C), dy.reshape(B * T, C)
    seqs = _sequences(B, T, cu_seqlens)
    dx = np.zeros_like(flat)
    dw = np.zeros((C, W))
    db = np.zeros(C)
    dhalo = np.zeros((len(seqs), HW, C))
    for start, length, n in seqs:
        ext = _extended(flat[start:start + length], None if halo is None else halo[n], HW)
        dext = np.zeros_like(ext)
        for t in range(length):
            z = np.zeros(C) if bias is None else np.asarray(bias, np.float64).copy()
            for i in range(W):
                z += w[:, i] * ext[HW + t - (W - 1 - i) * dilation]
            if activation:
                s = 1.0 / (1.0 + np.exp(-z))
                dz = dflat[start + t] * s * (1.0 + z * (1.0 - s))   # d/dz of z sigmoid(z)
            else:
                dz = dflat[start + t]
            db += dz
            for i in range(W):
                u = HW + t - (W - 1 - i) * dilation
                dw[:, i] += dz * ext[u]
                dext[u] += w[:, i] * dz
        dx[start:start + length] = dext[HW:]
        dhalo[n] = dext[:HW]
    return dict(dx=dx.reshape(B, T, C), dweight=dw, dbias=db, dhalo=dhalo)

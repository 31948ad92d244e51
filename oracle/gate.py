"""Oracle of the in-kernel gate activation of Kimi Delta Attention (the "safe gate").

TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and the benchmark's CPU legs may
import it. It shares no code with the CUDA library.

What the pages fix. The KDA native prepare is called with ``use_gate_in_kernel=True``,
``safe_gate=True``, ``lower_bound``, ``A_log`` and ``dt_bias`` (kimi_delta_attention_ascendc.py
coverage page, ``_prepare_kda``); ``ascendc_chunk_kda`` documents the shapes and range: gate
logits with the query's shape ``[B,T,H,128]``, ``a_log`` with H elements, ``dt_bias`` with
H*128 elements, ``lower_bound`` in [-5, 0); and ``chunk_kda_bwd_finalize`` returns the
gradients ``da_log`` and ``ddt_bias`` with the gate's gradient. The fused KDA backends reject
a gate without the lower bound ("requires the lower-bounded gate").

What the pages leave open, and the reading taken. The formula itself is not on the pages. The
plainest reading consistent with a lower bound in [-5, 0), a per-head decay parameter kept as
a logarithm and a per-channel bias added to the logits is a sigmoid squashed into
(lower_bound, 0):

    g[b,t,h,k] = lower_bound * sigmoid(exp(A_log[h]) * (x[b,t,h,k] + dt_bias[h,k]))

(natural-log decay: the state row k is multiplied by exp(g)). Every g lies strictly between
lower_bound and 0, so the decay per token stays in (exp(lower_bound), 1). Parity tests of the
gate pin this reading, not the pages.
"""
from __future__ import annotations

import numpy as np


def _sigmoid(z):
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def kda_safe_gate(x, A_log, dt_bias, lower_bound):
    """Activated per-channel log-decay from the gate logits.

    x ``[B,T,H,K]``; A_log ``[H]``; dt_bias ``[H,K]`` (or H*K values); returns g ``[B,T,H,K]``
    in fp64."""
    x = np.asarray(x, np.float64)
    H, K = x.shape[2], x.shape[3]
    a = np.exp(np.asarray(A_log, np.float64).reshape(H))[:, None]
    d = np.asarray(dt_bias, np.float64).reshape(H, K)
    return float(lower_bound) * _sigmoid(a * (x + d))


def kda_safe_gate_bwd(dg, x, A_log, dt_bias, lower_bound):
    """Chain rule through :func:`kda_safe_gate`: from the gradient ``dg`` w.r.t. the activated
    gate to ``(dx [B,T,H,K], dA_log [H], ddt_bias [H,K])``. With z = exp(A_log) (x + dt_bias)
    and s = sigmoid(z): dg/dx = dg/d dt_bias = lower_bound s (1 - s) exp(A_log), and
    dg/dA_log = lower_bound s (1 - s) z."""
    x = np.asarray(x, np.float64)
    dg = np.asarray(dg, np.float64)
    H, K = x.shape[2], x.shape[3]
    a = np.exp(np.asarray(A_log, np.float64).reshape(H))[:, None]
    d = np.asarray(dt_bias, np.float64).reshape(H, K)
    z = a * (x + d)
    s = _sigmoid(z)
    ds = float(lower_bound) * s * (1.0 - s)
    dx = dg * ds * a
    dA_log = (dg * ds * z).sum(axis=(0, 1, 3))
    ddt_bias = dx.sum(axis=(0, 1))
    return dx, dA_log, ddt_bias

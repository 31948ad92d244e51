"""Second oracle: the naive chunked form of Gated DeltaNet, in numpy fp64.

TEST INFRASTRUCTURE ONLY: used by the tests to cross-check the token recurrence in
``recurrent.cpp`` and to expose chunk intermediates. It shares nothing with the CUDA path.

It follows the eager PyTorch reference on the hyper-parallel "Diff Coverage" page
(``torch_chunk_gated_delta_rule`` and ``_prepare_gdn_chunks_for_summary`` /
``_run_prepared_gdn_chunks``), step by step and in the same order:

1. optional L2 norm of q and k along the head dim, eps 1e-6 inside the square root
   (``_l2norm``);
2. zero-pad the sequence to a multiple of the chunk size;
3. scale q (the page hard-codes 1/sqrt(K); here ``scale`` is a parameter, default 1/sqrt(K));
4. ``v_beta = v * beta``, ``k_beta = k * beta``; split into chunks;
5. chunk-local cumulative gate ``g = cumsum(g)``;
6. decay mask ``exp(g_i - g_j)`` on the lower triangle (diagonal included);
7. ``attn = -(k_beta @ k^T * decay)`` with the upper triangle *and* the diagonal zeroed;
8. the forward-substitution row loop, then ``+ I``: ``attn`` becomes ``(I + L)^-1``;
9. ``value = attn @ v_beta`` and ``k_cumdecay = attn @ (k_beta * exp(g))``;
10. the chunk loop: ``v_new = value - k_cumdecay @ S``;
    ``o = (q * exp(g)) @ S + (q k^T * decay) @ v_new``;
    ``S = S * exp(g_last) + (k * exp(g_last - g))^T @ v_new``.

The page's step 10 has one elided factor in the state update; it is restored from the
identical update printed in ``torch_chunk_gated_delta_rule`` on the same page
(``exp(g_last - g)`` on k).

Only the scalar gate is on the page; the per-channel variant is checked through the
recurrence oracle.
"""
from __future__ import annotations

import numpy as np


def l2norm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """``x * rsqrt(sum(x*x, -1) + eps)`` (the page's ``_l2norm``)."""
    return x * (1.0 / np.sqrt((x * x).sum(-1, keepdims=True) + eps))


def chunk_gated_delta_rule(q, k, v, g, beta, *, scale=None, initial_state=None,
                           output_final_state=False, use_qk_l2norm=False, chunk_size=64,
                           return_intermediates=False):
    """Chunked GDN forward for one dense batch.

    Shapes (float64): q, k ``[B,T,H,K]``; v ``[B,T,H,V]``; g, beta ``[B,T,H]``;
    initial_state ``[B,H,K,V]`` or None. Returns ``(o [B,T,H,V], final_state or None)``
    and, with ``return_intermediates``, a dict of per-chunk G, L, A, w, u, Aqk and the
    state entering each chunk (head-major ``[B,H,NT,...]``).
    """
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    C = int(chunk_size)
    if use_qk_l2norm:
        q = l2norm(q)
        k = l2norm(k)
    # (B,T,H,D) -> (B,H,T,D)
    q, k, v = (np.ascontiguousarray(x.transpose(0, 2, 1, 3)) for x in (q, k, v))
    g, beta = (np.ascontiguousarray(x.transpose(0, 2, 1)) for x in (g, beta))
    pad = (C - T % C) % C
    if pad:
        q, k, v = (np.pad(x, ((0, 0), (0, 0), (0, pad), (0, 0))) for x in (q, k, v))
        g, beta = (np.pad(x, ((0, 0), (0, 0), (0, pad))) for x in (g, beta))
    Tp = T + pad
    NT = Tp // C
    if scale is None:
        scale = 1.0 / np.sqrt(K)
    q = q * scale
    v_beta = v * beta[..., None]
    k_beta = k * beta[..., None]
    q, k, k_beta, v_beta = (x.reshape(B, H, NT, C, x.shape[-1]) for x in (q, k, k_beta, v_beta))
    g = g.reshape(B, H, NT, C).cumsum(-1)
    diff = g[..., :, None] - g[..., None, :]
    lower = np.tril(np.ones((C, C), dtype=bool))
    decay = np.where(lower, np.exp(np.where(lower, diff, 0.0)), 0.0)
    strict_upper_incl_diag = ~np.tril(np.ones((C, C), dtype=bool), -1)
    attn = -(k_beta @ np.swapaxes(k, -1, -2)) * decay
    attn[..., strict_upper_incl_diag] = 0.0
    L = -attn.copy()
    for i in range(1, C):
        row = attn[..., i, :i].copy()
        sub = attn[..., :i, :i].copy()
        attn[..., i, :i] = row + (row[..., :, None] * sub).sum(-2)
    A = attn + np.eye(C)
    u = A @ v_beta
    w = A @ (k_beta * np.exp(g)[..., None])

    S = np.zeros((B, H, K, V)) if initial_state is None else np.array(initial_state, dtype=np.float64)
    o = np.zeros((B, H, NT, C, V))
    entry = np.zeros((B, H, NT, K, V))
    Aqk = np.zeros((B, H, NT, C, C))
    for c in range(NT):
        qc, kc = q[:, :, c], k[:, :, c]
        gc = g[:, :, c]
        attn_qk = (qc @ np.swapaxes(kc, -1, -2)) * decay[:, :, c]
        Aqk[:, :, c] = attn_qk
        entry[:, :, c] = S
        v_new = u[:, :, c] - w[:, :, c] @ S
        o[:, :, c] = (qc * np.exp(gc)[..., None]) @ S + attn_qk @ v_new
        S = S * np.exp(gc[..., -1])[..., None, None] + \
            np.swapaxes(kc * np.exp(gc[..., -1:] - gc)[..., None], -1, -2) @ v_new
    o = o.reshape(B, H, Tp, V)[:, :, :T].transpose(0, 2, 1, 3)
    final = S if output_final_state else None
    if return_intermediates:
        return o, final, dict(G=g, L=L, A=A, w=w, u=u, Aqk=Aqk, entry=entry)
    return o, final

"""Seeded synthetic inputs for the gated delta rule (shared by tests, smoke check and bench).

This module draws random tensors only; it holds none of the method's arithmetic, so both
the CUDA path and the CPU oracle can consume what it produces.

Recipe: a torch CPU ``Generator`` seeded per workload draws, in this order, q, k, v, g,
beta, h0, dO, dht, each in fp32 and then cast. q, k, v ~ N(0,1) in bf16. g is a log-decay
-softplus(N(0,1)) in fp32 ([B,T,H] for the scalar gate, [B,T,H,K] for the per-channel gate).
beta is sigmoid(N(0,1)) in bf16, or the bf16 logit N(0,1) itself when the kernel applies
the sigmoid. h0 ~ N(0, std) fp32 (zeros when std is 0), dO ~ N(0,1) bf16, dht ~ N(0, std)
fp32 (absent when std is 0). Packed documents draw their lengths from numpy with the same
seed (see ``doc_lengths``).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int = 128
    V: int = 128
    per_channel: bool = False       # KDA gate [B,T,H,K]
    beta_logits: bool = False       # beta passed as a logit; sigmoid applied in kernel
    h0_std: float = 0.0
    dht_std: float = 0.0
    n_docs: int = 0                 # >0: packed documents (B must be 1)
    doc_min: int = 256
    doc_max: int = 3072
    backward: bool = True
    seed: int = 0
    use_qk_l2norm: bool = True
    num_k_heads: int = 0            # >0: grouped q/k heads (q, k drawn with this many heads)
    extra: dict = field(default_factory=dict)

    @property
    def tokens(self) -> int:
        return self.B * self.T


# The five workloads of the method's benchmark plan, the forward target shape, and a grouped-head
# variant of the training shape.
WORKLOADS = {
    "gdn_smoke_b1_t256_h2": Workload("gdn_smoke_b1_t256_h2", 1, 256, 2, backward=False, seed=0),
    "gdn_b2_t4096_h16": Workload("gdn_b2_t4096_h16", 2, 4096, 16, h0_std=0.02, seed=1),
    "gdn_b1_t32768_h16": Workload("gdn_b1_t32768_h16", 1, 32768, 16, dht_std=0.01, seed=2),
    "gdn_varlen_t16384_12docs_h16": Workload("gdn_varlen_t16384_12docs_h16", 1, 16384, 16,
                                             n_docs=12, seed=3),
    "kda_b1_t8192_h32": Workload("kda_b1_t8192_h32", 1, 8192, 32, per_channel=True,
                                 beta_logits=True, seed=4),
    "gdn_b1_t8192_h16": Workload("gdn_b1_t8192_h16", 1, 8192, 16, seed=5),
    # a smaller KDA case for kernel profiles (inputs still larger than L2)
    "kda_b1_t4096_h32": Workload("kda_b1_t4096_h32", 1, 4096, 32, per_channel=True, beta_logits=True, seed=7),
    # grouped q/k heads (next row of the plan): 16 value heads over 4 q/k heads
    "gdn_gqa_b2_t4096_h16_hk4": Workload("gdn_gqa_b2_t4096_h16_hk4", 2, 4096, 16, h0_std=0.02, seed=6,
                                         num_k_heads=4),
}


def doc_lengths(total: int, n_docs: int, lo: int, hi: int, seed: int) -> list[int]:
    """Document lengths: n_docs integers drawn from U[lo, hi], rescaled to sum exactly to
    ``total`` (floor, the remainder spread one token each over the first documents), redrawn
    until every length lies in [lo, hi]."""
    rs = np.random.RandomState(seed)
    for _ in range(10000):
        raw = rs.randint(lo, hi + 1, size=n_docs).astype(np.float64)
        lens = np.floor(raw * total / raw.sum()).astype(np.int64)
        rem = int(total - lens.sum())
        lens[:rem] += 1
        if lens.min() >= lo and lens.max() <= hi and lens.sum() == total:
            return [int(x) for x in lens]
    raise RuntimeError("could not draw document lengths in range")


def cu_seqlens_for(lengths) -> list[int]:
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return out


def make_inputs(w: Workload, *, seed: Optional[int] = None, lengths=None) -> dict:
    """Draw one batch for workload ``w`` on the CPU. Returns a dict of CPU tensors:
    q, k, v, g, beta, h0 (or None), dO, dht (or None), cu_seqlens (list or None)."""
    s = w.seed if seed is None else seed
    gen = torch.Generator(device="cpu")
    gen.manual_seed(s)
    B, T, H, K, V = w.B, w.T, w.H, w.K, w.V

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32)

    Hk = w.num_k_heads if w.num_k_heads > 0 else H
    q = randn(B, T, Hk, K).to(torch.bfloat16)
    k = randn(B, T, Hk, K).to(torch.bfloat16)
    v = randn(B, T, H, V).to(torch.bfloat16)
    gshape = (B, T, H, K) if w.per_channel else (B, T, H)
    g = -torch.nn.functional.softplus(randn(*gshape))
    b = randn(B, T, H)
    beta = (b if w.beta_logits else torch.sigmoid(b)).to(torch.bfloat16)
    cu = None
    if lengths is not None:
        cu = cu_seqlens_for(lengths)
    elif w.n_docs > 0:
        cu = cu_seqlens_for(doc_lengths(T, w.n_docs, w.doc_min, w.doc_max, s))
    N = B if cu is None else len(cu) - 1
    h0 = randn(N, H, K, V) * w.h0_std if w.h0_std > 0 else None
    dO = randn(B, T, H, V).to(torch.bfloat16)
    dht = randn(N, H, K, V) * w.dht_std if w.dht_std > 0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, dO=dO, dht=dht, cu_seqlens=cu)


def custom(B, T, H, *, K=128, V=128, per_channel=False, beta_logits=False, h0_std=0.0,
           dht_std=0.0, lengths=None, seed=0, g_scale=1.0) -> dict:
    """Small ad-hoc batch with the same distributions (``g_scale`` multiplies the softplus
    argument's spread, to widen or narrow the gate range)."""
    w = Workload("custom", B, T, H, K, V, per_channel=per_channel, beta_logits=beta_logits,
                 h0_std=h0_std, dht_std=dht_std, seed=seed)
    d = make_inputs(w, lengths=lengths)
    if g_scale != 1.0:
        gen = torch.Generator(device="cpu")
        gen.manual_seed(seed + 7919)
        shape = tuple(d["g"].shape)
        d["g"] = -torch.nn.functional.softplus(torch.randn(*shape, generator=gen) * g_scale)
    return d

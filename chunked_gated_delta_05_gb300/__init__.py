"""Chunkwise gated delta rule (Gated DeltaNet and Kimi Delta Attention) on one GB300.

The computation lives in ``libgdn.so`` (hand-written sm_103a CUDA behind the C ABI of
``include/gdn.h``); this package builds and loads it and marshals PyTorch tensors into it.
Importing the package does not touch the GPU; calling an op without the built library or
without a compute-capability 10.3 device raises.
"""
from .ops import (CausalConv1d, ChunkGatedDeltaRule, causal_conv1d, causal_conv1d_bwd, causal_conv1d_fwd,
                  chain_plan, chunk_gated_delta_rule, gdn_bwd, gdn_fwd, kda_bwd, kda_fwd, set_chain_segment,
                  set_head_groups)
from ._lib import GDN_EINVAL, GDN_ERANGE, GDN_ETIMEOUT, GdnError, load as load_library

__all__ = ["gdn_fwd", "gdn_bwd", "kda_fwd", "kda_bwd", "chunk_gated_delta_rule",
           "ChunkGatedDeltaRule", "GdnError", "GDN_EINVAL", "GDN_ETIMEOUT", "GDN_ERANGE", "load_library", "set_chain_segment", "set_head_groups", "chain_plan",
           "causal_conv1d", "causal_conv1d_fwd", "causal_conv1d_bwd", "CausalConv1d"]

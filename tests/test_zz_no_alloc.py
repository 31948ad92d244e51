"""The allocation-free forward entry point (gdn_fwd_noalloc), called through the C ABI.

It serves callers that cannot allocate device memory when they run the layer (for example
code running under CUDA graph capture, or an embedder whose memory belongs to another
allocator): it takes no workspace and uses a fixed static scratch array inside the library.
This file is collected last so that a run stopping at the first failure has already run
everything else; it passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from chunked_gated_delta_05_gb300 import _lib, gdn_fwd, synth
from tests._util import assert_output, assert_state

pytestmark = pytest.mark.gpu


def _noalloc_call(lib, d, dc, status):
    B, T, H, K = dc["q"].shape
    desc = _lib.Desc()
    desc.B, desc.T, desc.H, desc.K, desc.V, desc.chunk_size = B, T, H, 128, 128, 64
    desc.num_seqs = B
    desc.scale = 0.0
    desc.use_qk_l2norm, desc.use_beta_sigmoid, desc.output_final_state = 1, 0, 1
    o = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty((B, H, 128, 128), dtype=torch.float32, device="cuda")
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    a = _lib.FwdArgs(q=p(dc["q"]), k=p(dc["k"]), v=p(dc["v"]), g=p(dc["g"]), beta=p(dc["beta"]),
                     initial_state=p(dc["h0"]), o=p(o), final_state=p(hT), workspace=None,
                     workspace_bytes=0, status=p(status))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.gdn_fwd_noalloc(ctypes.byref(desc), ctypes.byref(a), stream)
    assert rc == 0, lib.gdn_last_error().decode()
    return o, hT


def test_noalloc_matches_allocating_forward_twice():
    lib = _lib.load()
    assert lib.gdn_fwd_noalloc_capacity() == 32 << 20
    d = synth.custom(1, 200, 2, h0_std=0.02, seed=31)
    dc = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_o, ref_h = gdn_fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                           output_final_state=True)
    torch.cuda.synchronize()
    ref_o, ref_h = ref_o.float().cpu().numpy(), ref_h.cpu().numpy()
    for _ in range(2):
        o, hT = _noalloc_call(lib, d, dc, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_output("o (no-alloc vs gdn_fwd)", o.float().cpu().numpy(), ref_o)
        assert_state("final_state (no-alloc vs gdn_fwd)", hT.cpu().numpy(), ref_h)


def test_noalloc_rejects_oversized_problem_and_workspace():
    lib = _lib.load()
    desc = _lib.Desc()
    desc.B, desc.T, desc.H, desc.K, desc.V, desc.chunk_size = 1, 65536, 16, 128, 128, 64
    desc.num_seqs = 1
    a = _lib.FwdArgs()
    a.q = a.k = a.v = a.g = a.beta = 0x1000
    a.o = 0x10000000
    rc = lib.gdn_fwd_noalloc(ctypes.byref(desc), ctypes.byref(a), None)
    assert rc == _lib.GDN_EINVAL and "32 MiB" in lib.gdn_last_error().decode()
    desc.T = 128
    a.workspace = 0x20000000
    a.workspace_bytes = 1 << 20
    assert lib.gdn_fwd_noalloc(ctypes.byref(desc), ctypes.byref(a), None) == _lib.GDN_EINVAL

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

from chunked_gated_delta_05_gb300 import _lib, gdn_fwd, set_chain_segment, synth

pytestmark = pytest.mark.gpu


def _outputs(dc):
    B, T, H, K = dc["q"].shape
    return (torch.empty((B, T, H, 128), dtype=torch.bfloat16, device="cuda"),
            torch.empty((B, H, 128, 128), dtype=torch.float32, device="cuda"))


def _noalloc_call(lib, d, dc, status, out=None):
    B, T, H, K = dc["q"].shape
    desc = _lib.Desc()
    desc.B, desc.T, desc.H, desc.K, desc.V, desc.chunk_size = B, T, H, 128, 128, 64
    desc.num_seqs = B
    desc.scale = 0.0
    desc.use_qk_l2norm, desc.use_beta_sigmoid, desc.output_final_state = 1, 0, 1
    o, hT = _outputs(dc) if out is None else out
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    a = _lib.FwdArgs(q=p(dc["q"]), k=p(dc["k"]), v=p(dc["v"]), g=p(dc["g"]), beta=p(dc["beta"]),
                     initial_state=p(dc["h0"]), o=p(o), final_state=p(hT), workspace=None,
                     workspace_bytes=0, status=p(status))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.gdn_fwd_noalloc(ctypes.byref(desc), ctypes.byref(a), stream)
    assert rc == 0, lib.gdn_last_error().decode()
    return o, hT


def _reference(dc):
    o, h = gdn_fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                   output_final_state=True)
    torch.cuda.synchronize()
    return o, h


def _inputs(B, T, H, seed, h0_std=0.02, lengths=None):
    d = synth.custom(B, T, H, h0_std=h0_std, seed=seed, lengths=lengths)
    return d, {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


@pytest.mark.parametrize("segment", [0, 2])
def test_noalloc_matches_allocating_forward(segment):
    """Two calls on problem A with a call on a different problem B between them, each against
    gdn_fwd on the same inputs. The two entry points run the same kernels, so the results must
    be bit-identical; a stale value left in the shared array by an earlier call would show up
    as a difference. Segment length 2 makes the forward use the segmented chain's buffers in
    the array as well. Device free memory must not change across the calls."""
    lib = _lib.load()
    assert lib.gdn_fwd_noalloc_capacity() == 32 << 20
    set_chain_segment(segment)
    try:
        dA, dcA = _inputs(1, 200, 2, seed=31)
        dB, dcB = _inputs(1, 333, 3, seed=32, h0_std=0.5)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        refA, refB = _reference(dcA), _reference(dcB)
        _noalloc_call(lib, dA, dcA, status)  # first call on the device: looks the array up
        torch.cuda.synchronize()
        seq = (dcA, dcB, dcA)
        outs = [_outputs(dc) for dc in seq]
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for dc, out in zip(seq, outs):
            _noalloc_call(lib, None, dc, status, out)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert int(status.item()) == 0
        for (o, hT), (ro, rh) in zip(outs, (refA, refB, refA)):
            assert torch.equal(o, ro), "o differs from gdn_fwd"
            assert torch.equal(hT, rh), "final_state differs from gdn_fwd"
        assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    finally:
        set_chain_segment(0)


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

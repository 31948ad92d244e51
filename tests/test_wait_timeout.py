"""The failure path of the bounded in-kernel waits, on the GPU and without a fault: a wait that
nothing completes gives up after its limit, the status word reports the timeout, and the
context and stream stay usable (the next forward on the same stream still matches the oracle)."""
import ctypes

import pytest
import torch

from chunked_gated_delta_05_gb300 import _lib, gdn_fwd, synth
from tests._util import assert_output, assert_state, oracle_fwd, to_cuda

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_reports_timeout():
    lib = _lib.load()
    src = torch.arange(1024, dtype=torch.int32, device="cuda")  # 4096 bytes for the copy in flight
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.gdn_wait_selftest(ctypes.c_void_p(src.data_ptr()), 1_000_000, ctypes.c_void_p(status.data_ptr()),
                               stream)
    assert rc == _lib.GDN_OK, lib.gdn_last_error().decode()
    torch.cuda.synchronize()
    assert int(status.item()) == 3  # a thread wait ran out
    # the next call on the same stream works and is correct
    d = synth.custom(1, 200, 2, h0_std=0.02, seed=90)
    dc = to_cuda(d)
    status.zero_()
    o, hT = gdn_fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                    output_final_state=True, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rT = oracle_fwd(d)
    assert_output("o", o.float().cpu().numpy(), ro)
    assert_state("final_state", hT.cpu().numpy(), rT)


def test_selftest_rejects_bad_arguments():
    lib = _lib.load()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.gdn_wait_selftest(None, 1000, ctypes.c_void_p(status.data_ptr()), None) == _lib.GDN_EINVAL

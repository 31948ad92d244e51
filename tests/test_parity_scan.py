"""GPU parity of the segmented state chain (chunk-parallel affine scan of the chain).

The segment length is forced through the library's override so that small problems run every
part of the scan: the fully-run first segment, the map runs (M from the identity, B from
zero), the compose kernel over several segments, the second pass and ragged last segments.
Weak decay keeps the state alive across many chunks, so a wrong map or a wrong composition
order shows up in the outputs. Every case is checked against the fp64 oracle and against the
plain serial chain on the same inputs.
"""
import numpy as np
import pytest
import torch

from chunked_gated_delta_05_gb300 import gdn_bwd, gdn_fwd, kda_bwd, kda_fwd, set_chain_segment, synth
from tests._util import assert_output, assert_state, oracle_bwd, oracle_fwd, rel_l2, to_cuda

pytestmark = pytest.mark.gpu

PLAIN = 1 << 20  # a segment longer than any sequence: the plain chain


@pytest.fixture(autouse=True)
def _restore_plan():
    yield
    set_chain_segment(0)


def weak_decay(d, factor=0.02):
    """Scale the log-decay towards 0 so the state carries over many chunks."""
    d["g"] = d["g"] * factor
    return d


def fwd(d, L, per_channel=False, **kw):
    set_chain_segment(L)
    dc = to_cuda(d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn = kda_fwd if per_channel else gdn_fwd
    o, hT = fn(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
               output_final_state=True, cu_seqlens=d["cu_seqlens"], status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o.float().cpu().numpy(), hT.cpu().numpy()


def bwd(d, L, per_channel=False, saved=False, **kw):
    set_chain_segment(L)
    dc = to_cuda(d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv = None
    if saved:
        ffn = kda_fwd if per_channel else gdn_fwd
        _, _, sv = ffn(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                       cu_seqlens=d["cu_seqlens"], status=status, save=True, **kw)
    fn = kda_bwd if per_channel else gdn_bwd
    out = fn(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"],
             initial_state=dc["h0"], cu_seqlens=d["cu_seqlens"], status=status, saved=sv, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return [None if x is None else x.float().cpu().numpy() for x in out]


def check_fwd(d, L, per_channel=False, **kw):
    o, hT = fwd(d, L, per_channel, **kw)
    ro, rT = oracle_fwd(d, per_channel=per_channel, **kw)
    r_o = assert_output("o", o, ro)
    r_s = assert_state("final_state", hT, rT)
    po, pT = fwd(d, PLAIN, per_channel, **kw)
    # the scan reassociates the chain's fp32 sums only: it stays close to the plain chain
    assert rel_l2(o, po) < 2e-3 and rel_l2(hT, pT) < 5e-4
    print(f"L={L}: o {r_o[0]:.2e}, state {r_s:.2e}; vs plain o {rel_l2(o, po):.1e} state {rel_l2(hT, pT):.1e}")


def check_bwd(d, L, per_channel=False, saved=False, **kw):
    got = bwd(d, L, per_channel, saved, **kw)
    ref = oracle_bwd(d, **kw)
    names = ("dq", "dk", "dv", "dbeta", "dg")
    msgs = []
    for name, x in zip(names, got[:5]):
        msgs.append(f"{name} {assert_output(name, x, ref[name])[0]:.1e}")
    if d["h0"] is not None:
        msgs.append(f"dh0 {assert_state('dh0', got[5], ref['dh0']):.1e}")
    plain = bwd(d, PLAIN, per_channel, saved, **kw)
    for name, x, p in zip(names, got[:5], plain[:5]):
        assert rel_l2(x, p) < 2e-3, name
    print(f"L={L}: " + ", ".join(msgs))


@pytest.mark.parametrize("L", [1, 2, 3, 5])
def test_fwd_dense_weak_decay(L):
    # 16 chunks, the last one partial: 16, 8, 6 (ragged) and 4 segments
    check_fwd(weak_decay(synth.custom(1, 1000, 2, h0_std=0.02, seed=40)), L)


def test_fwd_batch_and_strong_decay():
    check_fwd(synth.custom(2, 700, 3, h0_std=0.02, seed=41), 2)


def test_fwd_packed_documents():
    # documents of 1 .. 7 chunks: 1, 2, 3 and 4 segments of 2 chunks, some ragged
    lens = [64, 65, 200, 450, 7, 129, 300]
    check_fwd(weak_decay(synth.custom(1, sum(lens), 2, h0_std=0.02, lengths=lens, seed=42)), 2)


def test_fwd_kda():
    d = weak_decay(synth.custom(1, 600, 2, per_channel=True, beta_logits=True, seed=43))
    check_fwd(d, 2, per_channel=True, use_beta_sigmoid=True)


@pytest.mark.parametrize("L", [1, 3])
def test_bwd_dense_weak_decay(L):
    check_bwd(weak_decay(synth.custom(1, 1000, 2, h0_std=0.02, dht_std=0.01, seed=44)), L)


def test_bwd_packed_saved():
    lens = [64, 65, 200, 450, 7, 129]
    d = weak_decay(synth.custom(1, sum(lens), 2, h0_std=0.02, dht_std=0.01, lengths=lens, seed=45))
    check_bwd(d, 2, saved=True)


def test_bwd_kda():
    d = weak_decay(synth.custom(1, 600, 2, per_channel=True, beta_logits=True, dht_std=0.01, seed=46))
    check_bwd(d, 2, per_channel=True, use_beta_sigmoid=True)


def test_automatic_plan_matches_plain():
    """The automatic plan of a long single sequence (scan active) against the plain chain."""
    d = weak_decay(synth.custom(1, 64 * 48, 2, h0_std=0.02, seed=47))
    o, hT = fwd(d, 0)
    po, pT = fwd(d, PLAIN)
    assert rel_l2(o, po) < 2e-3 and rel_l2(hT, pT) < 5e-4
    np.testing.assert_array_equal(np.isfinite(o), True)

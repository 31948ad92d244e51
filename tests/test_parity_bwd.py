"""GPU backward parity: gradients from the CUDA path against the fp64 oracle's adjoint."""
import numpy as np
import pytest
import torch

from chunked_gated_delta_05_gb300 import gdn_bwd, synth
from tests._util import assert_output, assert_state, oracle_bwd, to_cuda

pytestmark = pytest.mark.gpu


def run_bwd(d, **kw):
    dc = to_cuda(d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gdn_bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"],
                  initial_state=dc["h0"], cu_seqlens=d["cu_seqlens"], status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return [None if x is None else x.float().cpu().numpy() for x in out]


def check(d, **kw):
    dq, dk, dv, db, dg, dh0 = run_bwd(d, **kw)
    ref_kw = {k: v for k, v in kw.items() if k in ("use_qk_l2norm", "use_beta_sigmoid", "scale")}
    ref = oracle_bwd(d, **ref_kw)
    msgs = []
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv), ("dbeta", db), ("dg", dg)):
        r = assert_output(name, x, ref[name])
        msgs.append(f"{name} {r[0]:.1e}")
    if d["h0"] is not None:
        msgs.append(f"dh0 {assert_state('dh0', dh0, ref['dh0']):.1e}")
    print("parity bwd rel-L2: " + ", ".join(msgs))


@pytest.mark.parametrize("T", [64, 100, 200])
def test_dense(T):
    check(synth.custom(1, T, 2, h0_std=0.02, dht_std=0.01, seed=10 + T))


def test_batch_two_no_state():
    check(synth.custom(2, 130, 2, seed=21))


def test_beta_logits_with_sigmoid():
    check(synth.custom(1, 150, 2, beta_logits=True, h0_std=0.02, seed=22), use_beta_sigmoid=True)


def test_packed_documents():
    lens = [1, 63, 64, 65, 130, 7]
    check(synth.custom(1, sum(lens), 2, h0_std=0.02, dht_std=0.01, lengths=lens, seed=23))


def test_no_l2norm():
    d = synth.custom(1, 128, 2, seed=24)
    d["k"] = (d["k"].float() * 0.08).to(torch.bfloat16)
    d["q"] = (d["q"].float() * 0.08).to(torch.bfloat16)
    check(d, use_qk_l2norm=False, scale=0.3)


def test_saved_mode_matches_recompute():
    """The backward on the forward's saved intermediates equals the recomputing backward."""
    from chunked_gated_delta_05_gb300 import gdn_fwd
    d = synth.custom(1, 200, 2, h0_std=0.02, dht_std=0.01, seed=25)
    dc = to_cuda(d)
    o1, h1, saved = gdn_fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                            output_final_state=True, save=True)
    o2, h2 = gdn_fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                     output_final_state=True)
    g1 = gdn_bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"],
                 initial_state=dc["h0"], saved=saved)
    g2 = gdn_bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"],
                 initial_state=dc["h0"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)

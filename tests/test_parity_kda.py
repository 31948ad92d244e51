"""GPU parity of the per-channel-gate (Kimi Delta Attention) path against the fp64 oracle."""
import numpy as np
import pytest
import torch

from chunked_gated_delta_05_gb300 import kda_fwd, synth
from tests._util import assert_output, assert_state, oracle_fwd, to_cuda

pytestmark = pytest.mark.gpu


def run_fwd(d, **kw):
    dc = to_cuda(d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, hT = kda_fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                    output_final_state=True, cu_seqlens=d["cu_seqlens"], status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o.float().cpu().numpy(), hT.cpu().numpy()


def check_fwd(d, **kw):
    o, hT = run_fwd(d, **kw)
    ro, rT = oracle_fwd(d, use_beta_sigmoid=kw.get("use_beta_sigmoid", True),
                        use_qk_l2norm=kw.get("use_qk_l2norm", True))
    r_o = assert_output("o", o, ro)
    r_s = assert_state("final_state", hT, rT)
    print(f"parity kda fwd o rel-L2 {r_o[0]:.2e} max-abs {r_o[1]:.2e}; state rel-L2 {r_s:.2e}")


@pytest.mark.parametrize("T", [1, 64, 100, 256])
def test_kda_fwd_dense(T):
    check_fwd(synth.custom(1, T, 2, per_channel=True, beta_logits=True, h0_std=0.02, seed=40 + T))


def test_kda_fwd_batch_and_packed():
    check_fwd(synth.custom(2, 130, 2, per_channel=True, beta_logits=True, seed=41))
    lens = [1, 63, 64, 65, 130, 7]
    check_fwd(synth.custom(1, sum(lens), 2, per_channel=True, beta_logits=True, h0_std=0.02,
                           lengths=lens, seed=42))


def test_kda_fwd_strong_gates():
    check_fwd(synth.custom(1, 192, 2, per_channel=True, beta_logits=True, seed=43, g_scale=2.0))


def check_bwd(d, **kw):
    from chunked_gated_delta_05_gb300 import kda_bwd
    from tests._util import oracle_bwd
    dc = to_cuda(d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kda_bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"],
                  initial_state=dc["h0"], cu_seqlens=d["cu_seqlens"], status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    dq, dk, dv, db, dg, dh0 = [None if x is None else x.float().cpu().numpy() for x in out]
    ref = oracle_bwd(d, use_beta_sigmoid=kw.get("use_beta_sigmoid", True), use_qk_l2norm=kw.get("use_qk_l2norm", True))
    msgs = []
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv), ("dbeta", db), ("dg", dg)):
        r = assert_output(name, x, ref[name])
        msgs.append(f"{name} {r[0]:.1e}")
    if d["h0"] is not None:
        msgs.append(f"dh0 {assert_state('dh0', dh0, ref['dh0']):.1e}")
    print("parity kda bwd rel-L2: " + ", ".join(msgs))


@pytest.mark.parametrize("T", [64, 100, 200])
def test_kda_bwd_dense(T):
    check_bwd(synth.custom(1, T, 2, per_channel=True, beta_logits=True, h0_std=0.02, dht_std=0.01, seed=50 + T))


def test_kda_bwd_packed():
    lens = [1, 63, 64, 65, 130, 7]
    check_bwd(synth.custom(1, sum(lens), 2, per_channel=True, beta_logits=True, h0_std=0.02, dht_std=0.01,
                           lengths=lens, seed=51))


def test_kda_bwd_strong_gates():
    # decays of up to several units per token: the pair sums' block factorisation must stay finite
    check_bwd(synth.custom(1, 192, 2, per_channel=True, beta_logits=True, h0_std=0.02, dht_std=0.01,
                           seed=52, g_scale=2.0))


def test_kda_bwd_saved_equals_recompute_and_repeats():
    """The backward on the forward's saved tiles equals the recomputing backward bit for bit, and
    a second call returns the same bits: the per-channel kernels reduce in a fixed order (the
    tensor-core pair sums included), so nothing depends on scheduling."""
    from chunked_gated_delta_05_gb300 import kda_bwd
    lens = [130, 7, 300, 64]
    d = synth.custom(1, sum(lens), 4, per_channel=True, beta_logits=True, h0_std=0.02, dht_std=0.01,
                     lengths=lens, seed=53)
    dc = to_cuda(d)
    kw = dict(initial_state=dc["h0"], cu_seqlens=d["cu_seqlens"])
    o, hT, saved = kda_fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], output_final_state=True,
                           save=True, **kw)
    runs = [kda_bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"], saved=saved, **kw),
            kda_bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"], saved=saved, **kw),
            kda_bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"], **kw)]
    torch.cuda.synchronize()
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert (a is None) == (b is None)
            if a is not None:
                assert torch.equal(a, b)

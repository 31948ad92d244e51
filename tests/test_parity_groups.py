"""Head groups: the library may split a problem's heads into two groups that run on two
streams (the second on a stream the library keeps per device, forked from and joined back into
the caller's stream). Every head is computed independently, so the split must not change a
single bit of any output; and the split path must match the fp64 oracle like the plain one."""
import pytest
import torch

from chunked_gated_delta_05_gb300 import (gdn_bwd, gdn_fwd, kda_bwd, kda_fwd, set_chain_segment,
                                          set_head_groups, synth)
from tests._util import assert_output, assert_state, oracle_bwd, oracle_fwd, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _restore():
    yield
    set_head_groups(0)
    set_chain_segment(0)


def _run(d, per_channel, sig, groups, saved):
    set_head_groups(groups)
    dc = to_cuda(d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fwd, bwd = (kda_fwd, kda_bwd) if per_channel else (gdn_fwd, gdn_bwd)
    kw = dict(use_beta_sigmoid=sig, cu_seqlens=d["cu_seqlens"], status=status)
    out = fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"], output_final_state=True,
              save=saved, **kw)
    o, hT = out[0], out[1]
    grads = bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"], initial_state=dc["h0"],
                saved=out[2] if saved else None, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return [o, hT] + [g for g in grads if g is not None]


@pytest.mark.parametrize("per_channel,saved,lengths,segment", [
    (False, True, None, 0),
    (False, False, [700, 1100, 248], 0),
    (True, True, None, 3),
])
def test_split_is_bit_identical(per_channel, saved, lengths, segment):
    T = 2048
    d = synth.custom(1, T, 8, per_channel=per_channel, beta_logits=per_channel, h0_std=0.02, dht_std=0.01,
                     lengths=lengths, seed=95)
    set_chain_segment(segment)
    one = _run(d, per_channel, per_channel, 1, saved)
    two = _run(d, per_channel, per_channel, 2, saved)
    for a, b in zip(one, two):
        assert torch.equal(a, b)
    # and the split run against the oracle
    ro, rT = oracle_fwd(d, use_beta_sigmoid=per_channel)
    assert_output("o", two[0].float().cpu().numpy(), ro)
    assert_state("final_state", two[1].cpu().numpy(), rT)
    ref = oracle_bwd(d, use_beta_sigmoid=per_channel)
    for name, x in zip(("dq", "dk", "dv", "dbeta", "dg"), two[2:7]):
        assert_output(name, x.float().cpu().numpy(), ref[name])
    assert_state("dh0", two[7].cpu().numpy(), ref["dh0"])


def test_automatic_choice_splits_large_problems():
    """At 8 heads x 64 chunks the automatic choice splits; the outputs equal the forced single
    group's."""
    d = synth.custom(1, 4096, 8, h0_std=0.02, seed=96)
    auto = _run(d, False, False, 0, True)
    one = _run(d, False, False, 1, True)
    for a, b in zip(auto, one):
        assert torch.equal(a, b)

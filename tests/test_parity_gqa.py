"""GPU parity of grouped q/k heads (num_v_heads > num_k_heads): value head h reads q/k head
h // G by indexing, and dq/dk are the group sums; checked against the fp64 oracle, whose
reading is the pages' repeat_interleave of q and k."""
import pytest
import torch

from chunked_gated_delta_05_gb300 import gdn_bwd, gdn_fwd, kda_bwd, kda_fwd, set_chain_segment, synth
from tests._util import assert_output, assert_state, oracle_bwd, oracle_fwd, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _restore_plan():
    yield
    set_chain_segment(0)


def grouped(d, Hk):
    """Keep the first Hk q/k heads of a seeded problem (the value-side tensors keep H)."""
    d = dict(d)
    d["q"] = d["q"][:, :, :Hk].contiguous()
    d["k"] = d["k"][:, :, :Hk].contiguous()
    return d


def check(d, per_channel=False, **kw):
    dc = to_cuda(d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fwd = kda_fwd if per_channel else gdn_fwd
    bwd = kda_bwd if per_channel else gdn_bwd
    o, hT = fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"], output_final_state=True,
                cu_seqlens=d["cu_seqlens"], status=status, **kw)
    grads = bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"], initial_state=dc["h0"],
                cu_seqlens=d["cu_seqlens"], status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rT = oracle_fwd(d, **kw)
    assert_output("o", o.float().cpu().numpy(), ro)
    assert_state("final_state", hT.cpu().numpy(), rT)
    ref = oracle_bwd(d, **kw)
    for name, x in zip(("dq", "dk", "dv", "dbeta", "dg"), grads[:5]):
        assert x.shape == dc[name[1:] if name != "dbeta" else "beta"].shape
        assert_output(name, x.float().cpu().numpy(), ref[name])
    if d["h0"] is not None:
        assert_state("dh0", grads[5].cpu().numpy(), ref["dh0"])


@pytest.mark.parametrize("H,Hk,T", [(4, 2, 200), (4, 1, 130), (6, 3, 64)])
def test_gdn_grouped(H, Hk, T):
    check(grouped(synth.custom(1, T, H, h0_std=0.02, dht_std=0.01, seed=60 + H + Hk + T), Hk))


def test_gdn_grouped_batch_and_packed():
    check(grouped(synth.custom(2, 150, 4, seed=61), 2))
    lens = [64, 7, 130, 65]
    check(grouped(synth.custom(1, sum(lens), 4, h0_std=0.02, lengths=lens, seed=62), 1))


def test_gdn_grouped_segmented_chain():
    set_chain_segment(2)
    d = synth.custom(1, 700, 4, h0_std=0.02, dht_std=0.01, seed=63)
    d["g"] = d["g"] * 0.02
    check(grouped(d, 2))


def test_kda_grouped():
    d = synth.custom(1, 200, 4, per_channel=True, beta_logits=True, dht_std=0.01, seed=64)
    check(grouped(d, 2), per_channel=True, use_beta_sigmoid=True)

"""GPU parity on the degenerate cases of the recurrence, against the fp64 oracle.

* Hard state reset: a log-decay of -inf (exp(g) = 0) at a token cuts the state there; -1e4
  does the same in every floating-point format. The GDN eager reference forms its decays as
  exp(g_i - g_j) from chunk-local cumulative gates (`torch_chunk_gated_delta_rule`, hyper-parallel
  GDN Diff Coverage page), which an infinite gate turns into NaN unless the kernel keeps the
  cumulative gate finite. Resets sit at sequence starts, mid-chunk, on chunk edges and at
  document starts; the rest of the gate is weak so the state would otherwise carry far.
* beta = 0 tokens: the token writes nothing into the state (pure decay step).
* KDA within its supported range: runs of tokens at the pages' safe-gate lower bound (-5 per
  token and channel) drive the state to zero without leaving the range; an infinite per-channel
  gate is outside the range and must be reported through the status word, not fault.

Every case runs dense and packed, on the plain chain and on the segmented chain.
"""
import math

import numpy as np
import pytest
import torch

from chunked_gated_delta_05_gb300 import (GDN_ERANGE, gdn_bwd, gdn_fwd, kda_bwd, kda_fwd,
                                          set_chain_segment, synth)
from tests._util import assert_output, assert_state, oracle_bwd, oracle_fwd, to_cuda

pytestmark = pytest.mark.gpu

PLAIN = 1 << 20  # a segment longer than any sequence: the plain chain


@pytest.fixture(autouse=True)
def _restore_plan():
    yield
    set_chain_segment(0)


def _edit(d, *, neg_inf=(), big=(), beta_zero=(), weak=0.05):
    """Weak gate everywhere, then hard resets and beta = 0 at the given (row, token) pairs."""
    d["g"] = d["g"] * weak
    for b, t in neg_inf:
        d["g"][b, t] = -math.inf
    for b, t in big:
        d["g"][b, t] = -1e4
    for b, t in beta_zero:
        d["beta"][b, t] = 0.0
    return d


def _run(d, L, per_channel, sig, backward=True):
    set_chain_segment(L)
    dc = to_cuda(d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(use_beta_sigmoid=sig, cu_seqlens=d["cu_seqlens"], status=status)
    fwd, bwd = (kda_fwd, kda_bwd) if per_channel else (gdn_fwd, gdn_bwd)
    o, hT, sv = fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                    output_final_state=True, save=True, **kw)
    grads = None
    if backward:
        grads = bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"],
                    initial_state=dc["h0"], saved=sv, **kw)
    torch.cuda.synchronize()
    return int(status.item()), o, hT, grads


def _check(d, L, per_channel=False, sig=False):
    st, o, hT, grads = _run(d, L, per_channel, sig)
    assert st == 0, f"device status {st}"
    ro, rT = oracle_fwd(d, per_channel=per_channel, use_beta_sigmoid=sig)
    msgs = [f"o {assert_output('o', o.float().cpu().numpy(), ro)[0]:.1e}",
            f"state {assert_state('final_state', hT.cpu().numpy(), rT):.1e}"]
    ref = oracle_bwd(d, use_beta_sigmoid=sig)
    for name, x in zip(("dq", "dk", "dv", "dbeta", "dg"), grads[:5]):
        msgs.append(f"{name} {assert_output(name, x.float().cpu().numpy(), ref[name])[0]:.1e}")
    if d["h0"] is not None:
        msgs.append(f"dh0 {assert_state('dh0', grads[5].cpu().numpy(), ref['dh0']):.1e}")
    print(f"L={L}: " + ", ".join(msgs))
    return grads


@pytest.mark.parametrize("L", [PLAIN, 2])
def test_gdn_hard_reset_dense(L):
    d = synth.custom(2, 300, 2, h0_std=0.02, dht_std=0.01, seed=70)
    d = _edit(d, neg_inf=[(0, 0), (0, 37), (0, 64), (1, 127), (1, 200)],
              big=[(0, 150), (1, 63), (1, 64), (1, 65)], beta_zero=[(0, 5), (0, 38), (1, 128), (1, 299)])
    grads = _check(d, L)
    dg = grads[4].cpu().numpy()
    # a reset gate has no gradient: exp(g) and every term that carries it are 0
    assert dg[0, 0].max() == 0 and dg[0, 37].max() == 0 and dg[1, 64].max() == 0


@pytest.mark.parametrize("L", [PLAIN, 2])
def test_gdn_hard_reset_packed(L):
    lens = [70, 130, 45, 190]
    d = synth.custom(1, sum(lens), 2, h0_std=0.02, dht_std=0.01, lengths=lens, seed=71)
    # a reset at a document's first token, in the middle of a document, on a chunk edge
    d = _edit(d, neg_inf=[(0, 70), (0, 100), (0, 245)], big=[(0, 64), (0, 200)],
              beta_zero=[(0, 0), (0, 69), (0, 71), (0, 300)])
    _check(d, L)


def test_gdn_all_beta_zero_is_pure_decay():
    """beta = 0 everywhere: nothing is written, the state only decays (final = exp(sum g) S0)."""
    d = synth.custom(1, 150, 2, h0_std=0.02, dht_std=0.01, seed=72)
    d["g"] = d["g"] * 0.02  # the state must survive 150 decays to be measurable in fp32
    d["beta"].zero_()
    _check(d, PLAIN)


@pytest.mark.parametrize("L", [PLAIN, 2])
def test_kda_lower_bound_runs_and_beta_zero(L):
    d = synth.custom(1, 300, 2, per_channel=True, h0_std=0.02, dht_std=0.01, seed=73)
    d["beta"] = torch.sigmoid(d["beta"].float()).to(torch.bfloat16)
    d = _edit(d, beta_zero=[(0, 3), (0, 64), (0, 190)])
    # 40 tokens at the safe-gate lower bound in half of the channels: exp(-200) resets them
    d["g"][0, 100:140, :, :64] = -5.0
    # a whole chunk at the bound in every channel
    d["g"][0, 192:256] = -5.0
    _check(d, L, per_channel=True, sig=False)


def test_kda_lower_bound_runs_packed():
    lens = [90, 64, 150]
    d = synth.custom(1, sum(lens), 2, per_channel=True, beta_logits=True, h0_std=0.02, lengths=lens,
                     seed=74)
    d["g"] = d["g"] * 0.05
    d["g"][0, 150:220] = -5.0
    _check(d, 2, per_channel=True, sig=True)


def test_kda_out_of_range_gate_is_reported():
    """An infinite per-channel gate lies outside what the per-channel kernels support: the call
    completes, and the status word reports GDN_ERANGE."""
    d = synth.custom(1, 200, 2, per_channel=True, beta_logits=True, seed=75)
    d["g"][0, 70, 1, 5] = -math.inf
    st, o, hT, _ = _run(d, PLAIN, True, True, backward=False)
    assert st == GDN_ERANGE
    # the next call on the same stream starts from a clean status and is correct again
    d2 = synth.custom(1, 200, 2, per_channel=True, beta_logits=True, seed=76)
    st2, o2, hT2, _ = _run(d2, PLAIN, True, True, backward=False)
    assert st2 == 0
    ro, rT = oracle_fwd(d2, per_channel=True, use_beta_sigmoid=True)
    assert_output("o", o2.float().cpu().numpy(), ro)
    assert_state("final_state", hT2.cpu().numpy(), rT)

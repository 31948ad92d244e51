"""GPU parity of the differentiable entry point (`chunk_gated_delta_rule`, a torch.autograd
Function over the save-mode forward and the backward on the saved intermediates): gradients from
loss.backward() against the fp64 oracle's backward for the same upstream gradients."""
import pytest
import torch

from chunked_gated_delta_05_gb300 import chunk_gated_delta_rule, synth
from tests._util import assert_output, assert_state, oracle_bwd, oracle_fwd

pytestmark = pytest.mark.gpu


def run(d, per_channel):
    leaf = lambda t: None if t is None else t.cuda().requires_grad_(True)
    q, k, v, g, beta, h0 = (leaf(d[n]) for n in ("q", "k", "v", "g", "beta", "h0"))
    o, final = chunk_gated_delta_rule(q, k, v, g, beta, initial_state=h0, output_final_state=True,
                                      use_beta_sigmoid=per_channel, cu_seqlens=d["cu_seqlens"])
    # loss whose gradients w.r.t. o and the final state are dO and dht
    loss = (o.float() * d["dO"].cuda().float()).sum() + (final * d["dht"].cuda()).sum()
    loss.backward()
    torch.cuda.synchronize()
    return o, final, {"dq": q.grad, "dk": k.grad, "dv": v.grad, "dg": g.grad, "dbeta": beta.grad,
                      "dh0": None if h0 is None else h0.grad}


@pytest.mark.parametrize("per_channel", [False, True])
def test_autograd_matches_oracle(per_channel):
    lens = [70, 130, 56]
    d = synth.custom(1, sum(lens), 2, per_channel=per_channel, beta_logits=per_channel, h0_std=0.02,
                     dht_std=0.01, lengths=lens, seed=80 + int(per_channel))
    o, final, grads = run(d, per_channel)
    ro, rT = oracle_fwd(d, use_beta_sigmoid=per_channel)
    assert_output("o", o.detach().float().cpu().numpy(), ro)
    assert_state("final_state", final.detach().cpu().numpy(), rT)
    ref = oracle_bwd(d, use_beta_sigmoid=per_channel)
    for name in ("dq", "dk", "dv", "dbeta", "dg"):
        assert_output(name, grads[name].float().cpu().numpy(), ref[name])
    assert_state("dh0", grads["dh0"].cpu().numpy(), ref["dh0"])


def test_autograd_with_in_kernel_gate():
    """KDA with the in-kernel safe gate through the autograd entry point: the gate logits and
    the gate parameters receive the oracle's gradients (gate reading of oracle/gate.py)."""
    import numpy as np
    from oracle import gate

    T, H = 150, 2
    d = synth.custom(1, T, H, per_channel=True, beta_logits=True, h0_std=0.02, dht_std=0.01, seed=83)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(84)
    x = torch.randn(1, T, H, 128, generator=gen)
    A_log = torch.randn(H, generator=gen) * 0.5
    dt_bias = torch.randn(H, 128, generator=gen) * 0.5
    leaf = lambda t: t.cuda().requires_grad_(True)
    q, k, v, beta, h0 = (leaf(d[n]) for n in ("q", "k", "v", "beta", "h0"))
    xg, ag, dg = leaf(x), leaf(A_log), leaf(dt_bias)
    o, final = chunk_gated_delta_rule(q, k, v, xg, beta, initial_state=h0, output_final_state=True,
                                      A_log=ag, dt_bias=dg, lower_bound=-5.0)
    loss = (o.float() * d["dO"].cuda().float()).sum() + (final * d["dht"].cuda()).sum()
    loss.backward()
    torch.cuda.synchronize()
    g_act = gate.kda_safe_gate(x.double().numpy(), A_log.double().numpy(), dt_bias.double().numpy(), -5.0)
    dref = dict(d)
    dref["g"] = torch.from_numpy(g_act)
    ro, rT = oracle_fwd(dref, use_beta_sigmoid=True)
    assert_output("o", o.detach().float().cpu().numpy(), ro)
    ref = oracle_bwd(dref, use_beta_sigmoid=True)
    dx, dA, ddt = gate.kda_safe_gate_bwd(ref["dg"], x.double().numpy(), A_log.double().numpy(),
                                         dt_bias.double().numpy(), -5.0)
    assert_output("dg", xg.grad.cpu().numpy(), dx)
    assert_output("da_log", ag.grad.cpu().numpy(), dA)
    assert_output("ddt_bias", dg.grad.cpu().numpy(), ddt)
    assert_output("dq", q.grad.float().cpu().numpy(), ref["dq"])
    assert_state("dh0", h0.grad.cpu().numpy(), ref["dh0"])

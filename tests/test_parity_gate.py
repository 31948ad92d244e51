"""GPU parity of KDA with the in-kernel safe gate (the KDA page's `_prepare_kda` with
use_gate_in_kernel and safe_gate; gradients da_log and ddt_bias as `chunk_kda_bwd_finalize`
returns them) against the oracle: the gate reading of oracle/gate.py followed by the fp64
recurrence. The comparison pins the library to that reading of the pages, which give the
gate's interface, range and gradients but not its formula."""
import numpy as np
import pytest
import torch

from chunked_gated_delta_05_gb300 import kda_bwd, kda_fwd, set_chain_segment, synth
from oracle import gate
from tests._util import assert_output, assert_state, oracle_bwd, oracle_fwd, to_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _restore_plan():
    yield
    set_chain_segment(0)


def _inputs(T, H, lengths, seed, h0_std=0.0):
    d = synth.custom(1, T, H, per_channel=True, beta_logits=True, h0_std=h0_std, dht_std=0.01,
                     lengths=lengths, seed=seed)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 1)
    x = torch.randn(1, T, H, 128, generator=gen)
    A_log = torch.randn(H, generator=gen) * 0.5
    dt_bias = torch.randn(H, 128, generator=gen) * 0.5
    return d, x, A_log, dt_bias


@pytest.mark.parametrize("lb,lengths,saved,segment", [
    (-5.0, None, True, 0),
    (-1.0, None, False, 0),
    (-5.0, [70, 130, 100], True, 2),
])
def test_kda_gate_in_kernel(lb, lengths, saved, segment):
    T, H = 300, 2
    d, x, A_log, dt_bias = _inputs(T, H, lengths, seed=80, h0_std=0.02)
    set_chain_segment(segment)
    dc = to_cuda(d)
    xc, ac, dtc = x.cuda(), A_log.cuda(), dt_bias.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gkw = dict(A_log=ac, dt_bias=dtc, lower_bound=lb, cu_seqlens=d["cu_seqlens"], status=status)
    out = kda_fwd(dc["q"], dc["k"], dc["v"], xc, dc["beta"], initial_state=dc["h0"], output_final_state=True,
                  save=saved, **gkw)
    o, hT = out[0], out[1]
    sv = out[2] if saved else None
    grads = kda_bwd(dc["q"], dc["k"], dc["v"], xc, dc["beta"], dc["dO"], dht=dc["dht"], initial_state=dc["h0"],
                    saved=sv, **gkw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert len(grads) == 8
    # oracle: the gate reading, then the recurrence and its adjoint, then the gate's chain rule
    g_act = gate.kda_safe_gate(x.double().numpy(), A_log.double().numpy(), dt_bias.double().numpy(), lb)
    dref = dict(d)
    dref["g"] = torch.from_numpy(g_act)
    ro, rT = oracle_fwd(dref, use_beta_sigmoid=True)
    ref = oracle_bwd(dref, use_beta_sigmoid=True)
    dx, dA, ddt = gate.kda_safe_gate_bwd(ref["dg"], x.double().numpy(), A_log.double().numpy(),
                                         dt_bias.double().numpy(), lb)
    msgs = [f"o {assert_output('o', o.float().cpu().numpy(), ro)[0]:.1e}",
            f"state {assert_state('final_state', hT.cpu().numpy(), rT):.1e}"]
    for name, x_, r_ in zip(("dq", "dk", "dv", "dbeta"), grads[:4], (ref["dq"], ref["dk"], ref["dv"], ref["dbeta"])):
        msgs.append(f"{name} {assert_output(name, x_.float().cpu().numpy(), r_)[0]:.1e}")
    msgs.append(f"dx {assert_output('dg', grads[4].cpu().numpy(), dx)[0]:.1e}")
    msgs.append(f"dh0 {assert_state('dh0', grads[5].cpu().numpy(), ref['dh0']):.1e}")
    msgs.append(f"dA_log {assert_output('da_log', grads[6].cpu().numpy(), dA)[0]:.1e}")
    msgs.append(f"ddt_bias {assert_output('ddt_bias', grads[7].cpu().numpy(), ddt)[0]:.1e}")
    print(f"lb={lb} saved={saved} segment={segment}: " + ", ".join(msgs))


def test_kda_gate_in_kernel_equals_explicit_gate():
    """The in-kernel activation feeds the same kernels as a gate activated by the caller: the
    outputs agree with a KDA call on the oracle's activated gate (rounded to fp32) up to the
    fp32 rounding of the activation."""
    T, H = 200, 2
    d, x, A_log, dt_bias = _inputs(T, H, None, seed=81)
    dc = to_cuda(d)
    g_act = torch.from_numpy(gate.kda_safe_gate(x.double().numpy(), A_log.double().numpy(),
                                                dt_bias.double().numpy(), -5.0)).float()
    o1, h1 = kda_fwd(dc["q"], dc["k"], dc["v"], x.cuda(), dc["beta"], output_final_state=True,
                     A_log=A_log.cuda(), dt_bias=dt_bias.cuda(), lower_bound=-5.0)
    o2, h2 = kda_fwd(dc["q"], dc["k"], dc["v"], g_act.cuda(), dc["beta"], output_final_state=True)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert ((h1 - h2).norm() / h2.norm()).item() <= 1e-4

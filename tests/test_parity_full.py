"""GPU parity at the benchmark plan's full sizes: every workload of the plan, run through the
entry points and launch configuration bench.py times (the training step: a save-mode forward,
then the backward on its saved intermediates; and the inference forward of the forward
target), against the fp64 oracle on all outputs (the oracle finishes each of these in seconds
on the host cores)."""
import numpy as np
import pytest
import torch

from chunked_gated_delta_05_gb300 import gdn_bwd, gdn_fwd, kda_bwd, kda_fwd, synth
from tests._util import assert_output, assert_state, oracle_bwd, oracle_fwd, to_cuda

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_full_size_workload(name):
    w = synth.WORKLOADS[name]
    d = synth.make_inputs(w)
    dc = to_cuda(d)
    fwd, bwd = (kda_fwd, kda_bwd) if w.per_channel else (gdn_fwd, gdn_bwd)
    kw = dict(use_qk_l2norm=w.use_qk_l2norm, use_beta_sigmoid=w.beta_logits, cu_seqlens=d["cu_seqlens"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # inference forward (no saves), as the forward-target measurement runs it
    o_inf, hT_inf = fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                        output_final_state=True, status=status, **kw)
    # training step, as the benchmark's timed step runs it
    o, hT, saved = fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                       output_final_state=True, status=status, save=True, **kw)
    grads = None
    if w.backward:
        grads = bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"],
                    initial_state=dc["h0"], status=status, saved=saved, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rT = oracle_fwd(d, use_qk_l2norm=w.use_qk_l2norm, use_beta_sigmoid=w.beta_logits)
    msgs = [f"o {assert_output('o', o.float().cpu().numpy(), ro)[0]:.1e}",
            f"state {assert_state('final_state', hT.cpu().numpy(), rT):.1e}",
            f"o(inference) {assert_output('o', o_inf.float().cpu().numpy(), ro)[0]:.1e}",
            f"state(inference) {assert_state('final_state', hT_inf.cpu().numpy(), rT):.1e}"]
    if grads is not None:
        ref = oracle_bwd(d, use_qk_l2norm=w.use_qk_l2norm, use_beta_sigmoid=w.beta_logits)
        for name_, x in zip(("dq", "dk", "dv", "dbeta", "dg"), grads[:5]):
            msgs.append(f"{name_} {assert_output(name_, x.float().cpu().numpy(), ref[name_])[0]:.1e}")
        if d["h0"] is not None:
            msgs.append(f"dh0 {assert_state('dh0', grads[5].cpu().numpy(), ref['dh0']):.1e}")
    print(f"full-size {name}: " + ", ".join(msgs))

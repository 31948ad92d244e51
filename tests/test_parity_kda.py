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

"""The library's calls inside a CUDA graph: a forward and a training step (save-mode forward,
backward on the saved buffer), both large enough to split their heads over the library's second
stream, are captured with torch.cuda.graph and replayed; the replayed results equal the eager
calls' bit for bit (the kernels are deterministic), and a replay on new input values matches
an eager call on those values."""
import pytest
import torch

from chunked_gated_delta_05_gb300 import gdn_bwd, gdn_fwd, synth

pytestmark = pytest.mark.gpu


def _step(dc, status):
    o, hT, sv = gdn_fwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], initial_state=dc["h0"],
                        output_final_state=True, status=status, save=True)
    grads = gdn_bwd(dc["q"], dc["k"], dc["v"], dc["g"], dc["beta"], dc["dO"], dht=dc["dht"],
                    initial_state=dc["h0"], status=status, saved=sv)
    return [o, hT] + list(grads)


def test_training_step_replays_from_a_graph():
    # 256 chunks x 16 heads: the forward and the backward both split their heads
    d = synth.custom(1, 16384, 16, h0_std=0.02, dht_std=0.01, seed=97)
    dc = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    eager = _step(dc, status)  # also creates the library's second stream before any capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(dc, status)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = _step(dc, status)
    graph.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for a, b in zip(eager, captured):
        assert torch.equal(a, b)
    # new values in the captured input buffers: the replay computes on them
    d2 = synth.custom(1, 16384, 16, h0_std=0.02, dht_std=0.01, seed=98)
    for k in ("q", "k", "v", "g", "beta", "h0", "dO", "dht"):
        dc[k].copy_(d2[k].cuda())
    graph.replay()
    torch.cuda.synchronize()
    eager2 = _step(dc, status)
    torch.cuda.synchronize()
    for a, b in zip(eager2, captured):
        assert torch.equal(a, b)

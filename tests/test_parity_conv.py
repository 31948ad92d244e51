"""GPU parity of the short convolution (causal depthwise Conv1d + SiLU) against the fp64
oracle: dense and packed rows, halos, dilation, activation off, ragged channel blocks."""
import numpy as np
import pytest
import torch

from chunked_gated_delta_05_gb300 import causal_conv1d_bwd, causal_conv1d_fwd
from oracle import conv
from tests._util import assert_output

pytestmark = pytest.mark.gpu


def make(B, T, C, W, seed, halo_rows=0, N=None):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn(B, T, C, generator=g).to(torch.bfloat16)
    w = (torch.randn(C, W, generator=g) * 0.5).float()
    b = (torch.randn(C, generator=g) * 0.1).float()
    dy = torch.randn(B, T, C, generator=g).to(torch.bfloat16)
    halo = torch.randn(N or B, halo_rows, C, generator=g).to(torch.bfloat16) if halo_rows else None
    return x, w, b, dy, halo


def f64(t):
    return None if t is None else t.double().numpy()


@pytest.mark.parametrize("B,T,C,W,dil,act,packed,halo", [
    (1, 300, 256, 4, 1, True, None, False),
    (2, 77, 1032, 4, 1, True, None, True),
    (1, 200, 64, 3, 2, False, [0, 1, 70, 71, 200], False),
    (1, 333, 136, 8, 1, True, [0, 100, 333], True),
    (3, 65, 8, 1, 1, True, None, False),
    # unit dilation and W <= 4 take the one-pass backward: packed documents shorter than the
    # window, documents starting inside a warp's run, halos, every W
    (1, 300, 256, 3, 1, True, [0, 1, 2, 5, 70, 135, 300], True),
    (1, 260, 128, 2, 1, False, [0, 64, 65, 200, 260], True),
    (1, 200, 520, 4, 1, True, [0, 1, 3, 97, 128, 129, 200], True),
    (2, 130, 64, 4, 1, False, None, False),
    # the halo length (W-1) d selects the kernels: up to 64 rows the shared-memory tiled ones,
    # beyond that the per-row ones
    (1, 200, 264, 6, 3, True, [0, 50, 200], False),
    (1, 400, 256, 8, 5, True, None, False),
    (1, 300, 64, 5, 20, False, None, False),
])
def test_conv_parity(B, T, C, W, dil, act, packed, halo):
    N = B if packed is None else len(packed) - 1
    HW = (W - 1) * dil
    x, w, b, dy, h = make(B, T, C, W, seed=T + C + W, halo_rows=HW if halo and HW else 0, N=N)
    dev = "cuda"
    kw = dict(dilation=dil, activation=act, cu_seqlens=packed)
    y = causal_conv1d_fwd(x.to(dev), w.to(dev), b.to(dev), halo=None if h is None else h.to(dev), **kw)
    dx, dw, db, dh = causal_conv1d_bwd(x.to(dev), w.to(dev), b.to(dev), dy.to(dev),
                                       halo=None if h is None else h.to(dev), **kw)
    torch.cuda.synchronize()
    ref_y = conv.causal_conv1d(f64(x), f64(w), f64(b), halo=f64(h), **kw)
    ref = conv.causal_conv1d_bwd(f64(x), f64(w), f64(b), f64(dy), halo=f64(h), **kw)
    assert_output("y", y.float().cpu().numpy(), ref_y, bf16_rounding=True)
    assert_output("dx", dx.float().cpu().numpy(), ref["dx"], bf16_rounding=True)
    assert_output("dweight", dw.cpu().numpy(), ref["dweight"])
    assert_output("dbias", db.cpu().numpy(), ref["dbias"])
    if h is not None:
        assert_output("dhalo", dh.cpu().numpy(), ref["dhalo"])


def test_conv_parity_bench_shape():
    """The short convolution at the benchmark's shape (the training workload's mixed q/k/v
    width: 2 x 4096 rows x 6144 channels, W = 4, SiLU), every element against the oracle."""
    B, T, C, W = 2, 4096, 6144, 4
    x, w, b, dy, _ = make(B, T, C, W, seed=11)
    dev = "cuda"
    y = causal_conv1d_fwd(x.to(dev), w.to(dev), b.to(dev))
    dx, dw, db, _ = causal_conv1d_bwd(x.to(dev), w.to(dev), b.to(dev), dy.to(dev))
    torch.cuda.synchronize()
    assert_output("y", y.float().cpu().numpy(), conv.causal_conv1d(f64(x), f64(w), f64(b)), bf16_rounding=True)
    ref = conv.causal_conv1d_bwd(f64(x), f64(w), f64(b), f64(dy))
    assert_output("dx", dx.float().cpu().numpy(), ref["dx"], bf16_rounding=True)
    assert_output("dweight", dw.cpu().numpy(), ref["dweight"])
    assert_output("dbias", db.cpu().numpy(), ref["dbias"])

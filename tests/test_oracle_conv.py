"""Pins for the short-convolution oracle (no GPU): library convolutions, the halo and
packed-document readings, and finite differences for the adjoint."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import conv


def problem(B=1, T=37, C=8, W=4, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, T, C)), rng.standard_normal((C, W)) * 0.5, rng.standard_normal(C) * 0.1)


def test_single_channel_matches_numpy_convolve():
    x, w, _ = problem(C=1)
    y = conv.causal_conv1d(x, w, None, activation=False)
    ref = np.convolve(x[0, :, 0], w[0, ::-1])[: x.shape[1]]
    np.testing.assert_allclose(y[0, :, 0], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dilation", [1, 2, 3])
def test_matches_torch_depthwise_conv1d_with_causal_padding(dilation):
    # the eager module: groups = C, zero padding (W-1) d, first T outputs, then SiLU
    x, w, b = problem(B=2, T=29, C=8, W=4, seed=dilation)
    W = w.shape[1]
    xt = torch.tensor(x).transpose(1, 2)
    out = F.conv1d(xt, torch.tensor(w)[:, None, :], torch.tensor(b), padding=(W - 1) * dilation,
                   dilation=dilation, groups=x.shape[2])[:, :, : x.shape[1]]
    ref = F.silu(out).transpose(1, 2).numpy()
    y = conv.causal_conv1d(x, w, b, dilation=dilation)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


def test_halo_equals_prepended_tokens():
    x, w, b = problem(T=20, seed=4)
    HW = 3
    rng = np.random.default_rng(5)
    halo = rng.standard_normal((1, HW, x.shape[2]))
    y = conv.causal_conv1d(x, w, b, halo=halo)
    full = conv.causal_conv1d(np.concatenate([halo, x], axis=1), w, b)
    np.testing.assert_allclose(y, full[:, HW:], rtol=0, atol=1e-12)


def test_packed_documents_are_independent():
    x, w, b = problem(T=31, seed=6)
    cu = [0, 5, 6, 20, 31]
    y = conv.causal_conv1d(x, w, b, cu_seqlens=cu)
    for s, e in zip(cu[:-1], cu[1:]):
        np.testing.assert_allclose(y[:, s:e], conv.causal_conv1d(x[:, s:e], w, b), rtol=0, atol=1e-12)


@pytest.mark.parametrize("activation,dilation,packed,halo", [(True, 1, False, False), (False, 2, True, False),
                                                            (True, 1, True, True), (True, 3, False, True)])
def test_backward_matches_finite_differences(activation, dilation, packed, halo):
    x, w, b = problem(T=13, C=8, W=3, seed=7)
    rng = np.random.default_rng(8)
    cu = [0, 4, 13] if packed else None
    N = 2 if packed else 1
    HW = (w.shape[1] - 1) * dilation
    h = rng.standard_normal((N, HW, x.shape[2])) if halo else None
    dy = rng.standard_normal(x.shape)
    kw = dict(dilation=dilation, activation=activation, cu_seqlens=cu)
    g = conv.causal_conv1d_bwd(x, w, b, dy, halo=h, **kw)
    params = dict(x=x, weight=w, bias=b)
    if halo:
        params["halo"] = h
    names = dict(x="dx", weight="dweight", bias="dbias", halo="dhalo")
    eps = 1e-6
    for name, p in params.items():
        d = rng.standard_normal(p.shape)
        def loss(pp):
            args = dict(params)
            args[name] = pp
            return (conv.causal_conv1d(args["x"], args["weight"], args["bias"], halo=args.get("halo"), **kw) * dy).sum()
        fd = (loss(p + eps * d) - loss(p - eps * d)) / (2 * eps)
        an = (g[names[name]] * d).sum()
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, fd, an)

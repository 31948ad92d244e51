"""Shared test helpers: oracle calls on torch inputs and the tolerance checks."""
import numpy as np
import torch

import oracle

# Tolerances of the method's acceptance bar: bf16 outputs (o, dq, dk, dv, the convolution's y
# and dx) max-abs <= 2e-2 and rel-L2 <= 5e-3, the max-abs bound absolute; fp32 states (final
# state, dh0) rel-L2 <= 1e-3. The gate and beta gradients (dg, dgk, dbeta, and the gate
# activation's parameter gradients) and the convolution's fp32 parameter gradients are sums over
# many tokens with no stated bound of their own: they are judged like bf16 outputs, with the
# max-abs bound scaled by max(1, |ref|_inf).
OUT_MAX_ABS = 2e-2
OUT_REL_L2 = 5e-3
STATE_REL_L2 = 1e-3
SCALED_MAX_ABS = ("dg", "dgk", "dbeta", "da_log", "ddt_bias", "dweight", "dbias", "dhalo")


def f64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def rel_l2(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def assert_output(name, x, ref, scaled=None, bf16_rounding=False):
    """rel-L2 <= 5e-3 and max-abs <= 2e-2; the max-abs bound is scaled by max(1, |ref|_inf)
    only for the gradients named in SCALED_MAX_ABS (``scaled`` overrides the choice). With
    ``bf16_rounding`` each element may also differ by the rounding of its reference value to
    bf16 (2^-8 |ref|): for bf16 outputs whose values exceed 2e-2 / 2^-8 = 5.12 (the short
    convolution's), where one correct rounding alone is larger than the absolute bound."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(x).all(), f"{name}: non-finite values"
    r = rel_l2(x, ref)
    if scaled is None:
        scaled = name.split()[0] in SCALED_MAX_ABS
    bound = OUT_MAX_ABS * (max(1.0, float(np.abs(ref).max()) if ref.size else 1.0) if scaled else 1.0)
    err = np.abs(x - ref)
    if bf16_rounding:
        err = err - 2.0 ** -8 * np.abs(ref)
    m = float(err.max()) if x.size else 0.0
    assert r <= OUT_REL_L2 and m <= bound, f"{name}: rel-L2 {r:.3e} (<= {OUT_REL_L2}), max-abs {m:.3e} (<= {bound:.3e})"
    return r, m


def assert_state(name, x, ref):
    x = np.asarray(x, np.float64)
    assert np.isfinite(x).all(), f"{name}: non-finite values"
    r = rel_l2(x, ref)
    assert r <= STATE_REL_L2, f"{name}: rel-L2 {r:.3e} (<= {STATE_REL_L2})"
    return r


def oracle_fwd(d, *, per_channel=False, use_qk_l2norm=True, use_beta_sigmoid=False, scale=None,
               output_final_state=True):
    return oracle.gdr_fwd(f64(d["q"]), f64(d["k"]), f64(d["v"]), f64(d["g"]), f64(d["beta"]),
                          scale=scale, initial_state=f64(d["h0"]), output_final_state=output_final_state,
                          use_qk_l2norm=use_qk_l2norm, use_beta_sigmoid=use_beta_sigmoid,
                          cu_seqlens=d["cu_seqlens"])


def oracle_bwd(d, *, use_qk_l2norm=True, use_beta_sigmoid=False, scale=None):
    return oracle.gdr_bwd(f64(d["q"]), f64(d["k"]), f64(d["v"]), f64(d["g"]), f64(d["beta"]),
                          f64(d["dO"]), dht=f64(d["dht"]), scale=scale, initial_state=f64(d["h0"]),
                          use_qk_l2norm=use_qk_l2norm, use_beta_sigmoid=use_beta_sigmoid,
                          cu_seqlens=d["cu_seqlens"])


def to_cuda(d):
    out = {}
    for key, val in d.items():
        out[key] = val.cuda() if isinstance(val, torch.Tensor) else val
    return out

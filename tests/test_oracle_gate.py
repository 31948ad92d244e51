"""Pins of the KDA safe-gate oracle (no GPU): the reading g = lower_bound * sigmoid(exp(A_log)
(x + dt_bias)) is tied to its limits and closed forms, its range, and its gradients to finite
differences, alone and composed with the recurrence. These pin the reading (the pages give
the gate's interface, range and gradients, not its formula)."""
import numpy as np
import pytest

import oracle
from oracle import gate


def _params(H, K, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(H) * 0.5, rng.standard_normal((H, K)) * 0.5


def test_limits_and_closed_forms():
    lb = -5.0
    A_log = np.array([0.0, np.log(2.0)])
    dt = np.zeros((2, 3))
    x = np.zeros((1, 4, 2, 3))
    x[0, 0] = 60.0      # saturates at the lower bound
    x[0, 1] = -60.0     # saturates at 0 (no decay)
    x[0, 2] = 0.0       # sigmoid(0) = 1/2
    x[0, 3] = 1.0       # lb sigmoid(exp(A_log))
    g = gate.kda_safe_gate(x, A_log, dt, lb)
    np.testing.assert_allclose(g[0, 0], lb, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g[0, 1], 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g[0, 2], lb / 2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(g[0, 3, 0], -5.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)
    np.testing.assert_allclose(g[0, 3, 1], -5.0 / (1.0 + np.exp(-2.0)), rtol=1e-15)
    # dt_bias shifts the logit: x + dt = 0 gives lb / 2 again
    dt2 = np.full((2, 3), 0.7)
    g2 = gate.kda_safe_gate(np.full((1, 1, 2, 3), -0.7), A_log, dt2, -2.0)
    np.testing.assert_allclose(g2, -1.0, rtol=0, atol=1e-15)


def test_range_is_open_interval_and_monotone():
    H, K = 3, 16
    A_log, dt = _params(H, K, 1)
    x = np.random.default_rng(2).standard_normal((2, 50, H, K)) * 3
    for lb in (-5.0, -1.0, -0.1):
        g = gate.kda_safe_gate(x, A_log, dt, lb)
        assert (g > lb).all() and (g < 0).all()
    # larger logits decay more (g decreases as x increases)
    xs = np.sort(x, axis=1)
    g = gate.kda_safe_gate(xs, A_log, dt, -3.0)
    assert (np.diff(g, axis=1) <= 0).all()


def test_gate_gradients_match_finite_differences():
    H, K = 2, 5
    A_log, dt = _params(H, K, 3)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 3, H, K))
    w = rng.standard_normal(x.shape)
    lb = -4.0
    f = lambda x_, a_, d_: float((w * gate.kda_safe_gate(x_, a_, d_, lb)).sum())
    dx, dA, ddt = gate.kda_safe_gate_bwd(w, x, A_log, dt, lb)
    eps = 1e-6
    for idx in np.ndindex(x.shape):
        e = np.zeros_like(x)
        e[idx] = eps
        fd = (f(x + e, A_log, dt) - f(x - e, A_log, dt)) / (2 * eps)
        assert abs(fd - dx[idx]) <= 1e-8 * max(1.0, abs(fd))
    for h in range(H):
        e = np.zeros(H)
        e[h] = eps
        fd = (f(x, A_log + e, dt) - f(x, A_log - e, dt)) / (2 * eps)
        assert abs(fd - dA[h]) <= 1e-8 * max(1.0, abs(fd))
    for idx in np.ndindex(dt.shape):
        e = np.zeros_like(dt)
        e[idx] = eps
        fd = (f(x, A_log, dt + e) - f(x, A_log, dt - e)) / (2 * eps)
        assert abs(fd - ddt[idx]) <= 1e-8 * max(1.0, abs(fd))


@pytest.mark.parametrize("T", [5, 70])
def test_gate_composed_with_recurrence_matches_finite_differences(T):
    """KDA with the in-kernel gate: the oracle's backward (recurrence adjoint, then the gate's
    chain rule) against central differences of the whole forward in the gate logits and the
    gate parameters."""
    H, K, V = 1, 4, 4
    rng = np.random.default_rng(5 + T)
    q, k, v = (rng.standard_normal((1, T, H, K)) for _ in range(3))
    beta = 1 / (1 + np.exp(-rng.standard_normal((1, T, H))))
    x = rng.standard_normal((1, T, H, K))
    A_log, dt = _params(H, K, 6)
    lb = -5.0
    dO = rng.standard_normal((1, T, H, V))
    dht = rng.standard_normal((1, H, K, V))

    def loss(x_, a_, d_):
        o, hT = oracle.gdr_fwd(q, k, v, gate.kda_safe_gate(x_, a_, d_, lb), beta, use_qk_l2norm=True)
        return float((dO * o).sum() + (dht * hT).sum())

    g = gate.kda_safe_gate(x, A_log, dt, lb)
    ref = oracle.gdr_bwd(q, k, v, g, beta, dO, dht=dht, use_qk_l2norm=True)
    dx, dA, ddt = gate.kda_safe_gate_bwd(ref["dg"], x, A_log, dt, lb)
    eps = 1e-6
    rng2 = np.random.default_rng(7)
    for _ in range(3):
        dirx = rng2.standard_normal(x.shape)
        fd = (loss(x + eps * dirx, A_log, dt) - loss(x - eps * dirx, A_log, dt)) / (2 * eps)
        assert abs(fd - (dx * dirx).sum()) <= 1e-6 * max(1.0, abs(fd))
    e = np.array([eps])
    fd = (loss(x, A_log + e, dt) - loss(x, A_log - e, dt)) / (2 * eps)
    assert abs(fd - dA[0]) <= 1e-6 * max(1.0, abs(fd))
    dird = rng2.standard_normal(dt.shape)
    fd = (loss(x, A_log, dt + eps * dird) - loss(x, A_log, dt - eps * dird)) / (2 * eps)
    assert abs(fd - (ddt * dird).sum()) <= 1e-6 * max(1.0, abs(fd))

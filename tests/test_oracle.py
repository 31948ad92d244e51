"""Pins for the CPU oracle (no GPU). Each test ties the oracle to something other than
itself: hand-worked values, closed forms, special cases, an independent chunked
implementation of the pages' algorithm, invariants, and finite differences."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng_global = np.random.default_rng(1234)


def rand_problem(B, T, H, K, V, *, per_channel=False, seed=0, gmin=None):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    gshape = (B, T, H, K) if per_channel else (B, T, H)
    g = -np.log1p(np.exp(rng.standard_normal(gshape)))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, T, H))))
    return q, k, v, g, beta


def l2(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + 1e-6)


# ---------------------------------------------------------------- hand-worked values

@pytest.mark.parametrize("fname,per_channel", [("hand_k2_t2.json", False), ("hand_kda_k2_t2.json", True)])
def test_hand_worked(fname, per_channel):
    d = json.load(open(os.path.join(GOLDEN, fname)))
    q = np.array(d["q"])[None, :, None, :]
    k = np.array(d["k"])[None, :, None, :]
    v = np.array(d["v"])[None, :, None, :]
    g = np.array(d["g"])[None, :, None] if not per_channel else np.array(d["g"])[None, :, None, :]
    beta = np.array(d["beta"])[None, :, None]
    o, hT = oracle.gdr_fwd(q, k, v, g, beta, scale=1.0, output_final_state=True)
    np.testing.assert_allclose(o[0, :, 0], np.array(d["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(hT[0, 0], np.array(d["final_state"]), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("l2norm", [False, True])
def test_single_token_closed_form(l2norm):
    q, k, v, g, beta = rand_problem(1, 1, 3, 8, 6, seed=1)
    o, hT = oracle.gdr_fwd(q, k, v, g, beta, scale=0.3, use_qk_l2norm=l2norm)
    qh, kh = (l2(q), l2(k)) if l2norm else (q, k)
    for h in range(3):
        b = beta[0, 0, h]
        exp_S = b * np.outer(kh[0, 0, h], v[0, 0, h])
        exp_o = 0.3 * b * (qh[0, 0, h] @ kh[0, 0, h]) * v[0, 0, h]
        np.testing.assert_allclose(hT[0, h], exp_S, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(o[0, 0, h], exp_o, rtol=1e-13, atol=1e-14)


def test_l2norm_eps_inside_sqrt():
    # A tiny key makes the eps visible: kh = k / sqrt(|k|^2 + 1e-6).
    q = np.ones((1, 1, 1, 4))
    k = np.full((1, 1, 1, 4), 1e-4)
    v = np.ones((1, 1, 1, 4))
    g = np.zeros((1, 1, 1))
    beta = np.ones((1, 1, 1))
    _, hT = oracle.gdr_fwd(q, k, v, g, beta, scale=1.0, use_qk_l2norm=True)
    kh = 1e-4 / np.sqrt(4e-8 + 1e-6)
    np.testing.assert_allclose(hT[0, 0], np.full((4, 4), kh), rtol=1e-14)


@pytest.mark.parametrize("per_channel", [False, True])
def test_beta_zero_is_pure_decay(per_channel):
    B, T, H, K, V = 1, 9, 2, 5, 4
    q, k, v, g, beta = rand_problem(B, T, H, K, V, per_channel=per_channel, seed=2)
    beta[:] = 0.0
    S0 = np.random.default_rng(3).standard_normal((1, H, K, V))
    o, hT = oracle.gdr_fwd(q, k, v, g, beta, scale=0.5, initial_state=S0)
    G = np.cumsum(g, axis=1)
    for h in range(H):
        for t in range(T):
            dec = np.exp(G[0, t, h])
            St = (dec[:, None] * S0[0, h]) if per_channel else dec * S0[0, h]
            np.testing.assert_allclose(o[0, t, h], 0.5 * St.T @ q[0, t, h], rtol=1e-12, atol=1e-13)
        decT = np.exp(G[0, -1, h])
        ST = (decT[:, None] * S0[0, h]) if per_channel else decT * S0[0, h]
        np.testing.assert_allclose(hT[0, h], ST, rtol=1e-12, atol=1e-14)


def test_beta_zero_gate_zero_keeps_state():
    q, k, v, g, beta = rand_problem(1, 7, 1, 4, 3, seed=4)
    beta[:] = 0.0
    g[:] = 0.0
    S0 = np.random.default_rng(5).standard_normal((1, 1, 4, 3))
    _, hT = oracle.gdr_fwd(q, k, v, g, beta, initial_state=S0)
    np.testing.assert_array_equal(hT, S0)


def test_orthonormal_keys_exact_retrieval():
    # g=0, beta=1, orthonormal keys: S_T = (I - sum k k^T) S0 + sum k v^T, and S_T^T k_j = v_j.
    K, V, T = 8, 5, 6
    rng = np.random.default_rng(6)
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm[:, :T].T[None, :, None, :].copy()
    q = rng.standard_normal((1, T, 1, K))
    v = rng.standard_normal((1, T, 1, V))
    g = np.zeros((1, T, 1))
    beta = np.ones((1, T, 1))
    S0 = rng.standard_normal((1, 1, K, V))
    _, hT = oracle.gdr_fwd(q, k, v, g, beta, initial_state=S0)
    Kt = k[0, :, 0]
    exp_S = (np.eye(K) - Kt.T @ Kt) @ S0[0, 0] + Kt.T @ v[0, :, 0]
    np.testing.assert_allclose(hT[0, 0], exp_S, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Kt @ hT[0, 0], v[0, :, 0], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("per_channel", [False, True])
def test_gate_minus_infinity_resets_state(per_channel):
    B, T, H, K, V = 1, 12, 1, 6, 5
    q, k, v, g, beta = rand_problem(B, T, H, K, V, per_channel=per_channel, seed=7)
    t_reset = 5
    g[0, t_reset] = -1e4       # exp underflows to exactly 0 in fp64
    o1, h1 = oracle.gdr_fwd(q, k, v, g, beta)
    k2, v2 = k.copy(), v.copy()
    k2[0, :t_reset] += 1.0
    v2[0, :t_reset] -= 2.0
    S0 = np.ones((1, H, K, V))
    o2, h2 = oracle.gdr_fwd(q, k2, v2, g, beta, initial_state=S0)
    np.testing.assert_array_equal(o1[0, t_reset:], o2[0, t_reset:])
    np.testing.assert_array_equal(h1, h2)
    assert not np.allclose(o1[0, :t_reset], o2[0, :t_reset])


def test_per_channel_uniform_gate_equals_scalar_gate():
    B, T, H, K, V = 2, 20, 2, 6, 5
    q, k, v, g, beta = rand_problem(B, T, H, K, V, seed=8)
    gk = np.repeat(g[..., None], K, axis=-1)
    S0 = np.random.default_rng(9).standard_normal((B, H, K, V))
    o1, h1 = oracle.gdr_fwd(q, k, v, g, beta, initial_state=S0, use_qk_l2norm=True)
    o2, h2 = oracle.gdr_fwd(q, k, v, gk, beta, initial_state=S0, use_qk_l2norm=True)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h1, h2, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("per_channel", [False, True])
def test_varlen_is_concatenation_of_independent_runs(per_channel):
    lens = [5, 64, 1, 70, 3]
    T = sum(lens)
    H, K, V = 2, 6, 4
    q, k, v, g, beta = rand_problem(1, T, H, K, V, per_channel=per_channel, seed=10)
    cu = np.cumsum([0] + lens)
    S0 = np.random.default_rng(11).standard_normal((len(lens), H, K, V))
    o, hT = oracle.gdr_fwd(q, k, v, g, beta, initial_state=S0, cu_seqlens=cu, use_qk_l2norm=True)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        on, hn = oracle.gdr_fwd(q[:, s:e], k[:, s:e], v[:, s:e], g[:, s:e], beta[:, s:e],
                                initial_state=S0[n:n + 1], use_qk_l2norm=True)
        np.testing.assert_array_equal(o[:, s:e], on)
        np.testing.assert_array_equal(hT[n:n + 1], hn)


def test_linear_in_values_and_initial_state():
    B, T, H, K, V = 1, 30, 2, 5, 4
    q, k, v1, g, beta = rand_problem(B, T, H, K, V, seed=12)
    rng = np.random.default_rng(13)
    v2 = rng.standard_normal(v1.shape)
    S1 = rng.standard_normal((B, H, K, V))
    S2 = rng.standard_normal((B, H, K, V))
    a, b = 0.7, -1.3
    oa, ha = oracle.gdr_fwd(q, k, v1, g, beta, initial_state=S1)
    ob, hb = oracle.gdr_fwd(q, k, v2, g, beta, initial_state=S2)
    oc, hc = oracle.gdr_fwd(q, k, a * v1 + b * v2, g, beta, initial_state=a * S1 + b * S2)
    np.testing.assert_allclose(oc, a * oa + b * ob, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hc, a * ha + b * hb, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("T,l2norm,h0,C", [(64, True, False, 64), (200, True, True, 64),
                                          (131, False, True, 64), (70, True, True, 16),
                                          (37, True, True, 1)])
def test_recurrence_equals_chunked_form(T, l2norm, h0, C):
    B, H, K, V = 2, 2, 16, 8
    q, k, v, g, beta = rand_problem(B, T, H, K, V, seed=14 + T)
    S0 = np.random.default_rng(15).standard_normal((B, H, K, V)) * 0.1 if h0 else None
    o1, h1 = oracle.gdr_fwd(q, k, v, g, beta, initial_state=S0, use_qk_l2norm=l2norm)
    o2, h2 = chunked.chunk_gated_delta_rule(q, k, v, g, beta, initial_state=S0,
                                            output_final_state=True, use_qk_l2norm=l2norm,
                                            chunk_size=C)
    assert np.linalg.norm(o1 - o2) / np.linalg.norm(o1) < 1e-10
    assert np.linalg.norm(h1 - h2) / np.linalg.norm(h1) < 1e-10


def test_chunk_sizes_agree():
    B, T, H, K, V = 1, 96, 1, 8, 8
    q, k, v, g, beta = rand_problem(B, T, H, K, V, seed=16)
    outs = [chunked.chunk_gated_delta_rule(q, k, v, g, beta, output_final_state=True,
                                           use_qk_l2norm=True, chunk_size=C) for C in (1, 16, 64)]
    for o, h in outs[1:]:
        np.testing.assert_allclose(o, outs[0][0], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(h, outs[0][1], rtol=1e-10, atol=1e-12)


def test_substitution_loop_inverts_unit_lower_triangle():
    q, k, v, g, beta = rand_problem(1, 128, 2, 16, 8, seed=17)
    _, _, mid = chunked.chunk_gated_delta_rule(q, k, v, g, beta, use_qk_l2norm=True,
                                               return_intermediates=True)
    L, A = mid["L"], mid["A"]
    I = np.eye(64)
    err = np.abs((I + L) @ A - I).max()
    assert err < 1e-10


def test_affine_chunk_maps_compose():
    # Each chunk maps its entry state affinely: S_out = M S_in + S_c with
    # M = exp(G_last) I - (k * exp(G_last - G))^T w and S_c = (k * exp(G_last - G))^T u.
    B, T, H, K, V = 1, 192, 1, 8, 6
    q, k, v, g, beta = rand_problem(B, T, H, K, V, seed=18)
    S0 = np.random.default_rng(19).standard_normal((B, H, K, V))
    _, hT, mid = chunked.chunk_gated_delta_rule(q, k, v, g, beta, initial_state=S0,
                                                output_final_state=True, use_qk_l2norm=True,
                                                return_intermediates=True)
    kh = l2(k)[0, :, 0].reshape(3, 64, K)
    S = S0[0, 0]
    for c in range(3):
        G = mid["G"][0, 0, c]
        kd = kh[c] * np.exp(G[-1] - G)[:, None]
        M = np.exp(G[-1]) * np.eye(K) - kd.T @ mid["w"][0, 0, c]
        Sc = kd.T @ mid["u"][0, 0, c]
        S = M @ S + Sc
    np.testing.assert_allclose(S, hT[0, 0], rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- gradients

def _loss(params, dO, dht, kw):
    o, hT = oracle.gdr_fwd(params["q"], params["k"], params["v"], params["g"], params["beta"],
                           initial_state=params.get("h0"), **kw)
    val = (o * dO).sum()
    if dht is not None:
        val += (hT * dht).sum()
    return val


CASES = [
    dict(per_channel=False, l2=True, sig=False, h0=True, dht=True, lens=None, T=5, K=4),
    dict(per_channel=False, l2=False, sig=True, h0=False, dht=False, lens=None, T=70, K=4),
    dict(per_channel=True, l2=True, sig=True, h0=True, dht=True, lens=None, T=70, K=4),
    dict(per_channel=True, l2=False, sig=False, h0=False, dht=True, lens=[3, 2], T=5, K=8),
    dict(per_channel=False, l2=True, sig=False, h0=True, dht=False, lens=[40, 30], T=70, K=8),
]


@pytest.mark.parametrize("case", CASES)
def test_backward_matches_finite_differences(case):
    T, K, V, H = case["T"], case["K"], case["K"], 1
    q, k, v, g, beta = rand_problem(1, T, H, K, V, per_channel=case["per_channel"], seed=20 + T)
    rng = np.random.default_rng(21)
    if case["sig"]:
        beta = rng.standard_normal(beta.shape)
    N = 1 if case["lens"] is None else len(case["lens"])
    cu = None if case["lens"] is None else np.cumsum([0] + case["lens"])
    params = dict(q=q, k=k, v=v, g=g, beta=beta)
    if case["h0"]:
        params["h0"] = rng.standard_normal((N, H, K, V)) * 0.5
    dO = rng.standard_normal((1, T, H, V))
    dht = rng.standard_normal((N, H, K, V)) if case["dht"] else None
    kw = dict(scale=0.4, use_qk_l2norm=case["l2"], use_beta_sigmoid=case["sig"], cu_seqlens=cu,
              output_final_state=True)
    grads = oracle.gdr_bwd(q, k, v, g, beta, dO, dht=dht, scale=0.4, initial_state=params.get("h0"),
                           use_qk_l2norm=case["l2"], use_beta_sigmoid=case["sig"], cu_seqlens=cu)
    name_map = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    eps = 1e-6
    for name in params:
        direction = rng.standard_normal(params[name].shape)
        plus = {n: (p + eps * direction if n == name else p) for n, p in params.items()}
        minus = {n: (p - eps * direction if n == name else p) for n, p in params.items()}
        fd = (_loss(plus, dO, dht, kw) - _loss(minus, dO, dht, kw)) / (2 * eps)
        an = (grads[name_map[name]] * direction).sum()
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, fd, an)


def test_backward_elementwise_small():
    # Elementwise central differences on a 3-token problem (every gradient entry).
    T, K, V = 3, 3, 2
    q, k, v, g, beta = rand_problem(1, T, 1, K, V, per_channel=True, seed=22)
    rng = np.random.default_rng(23)
    h0 = rng.standard_normal((1, 1, K, V))
    dO = rng.standard_normal((1, T, 1, V))
    dht = rng.standard_normal((1, 1, K, V))
    kw = dict(scale=0.7, use_qk_l2norm=True, use_beta_sigmoid=True, output_final_state=True)
    beta = rng.standard_normal(beta.shape)
    params = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)
    grads = oracle.gdr_bwd(q, k, v, g, beta, dO, dht=dht, scale=0.7, initial_state=h0,
                           use_qk_l2norm=True, use_beta_sigmoid=True)
    name_map = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    eps = 1e-6
    for name, p in params.items():
        fd = np.zeros_like(p)
        for idx in np.ndindex(p.shape):
            pp = {n: x.copy() for n, x in params.items()}
            pm = {n: x.copy() for n, x in params.items()}
            pp[name][idx] += eps
            pm[name][idx] -= eps
            fd[idx] = (_loss(pp, dO, dht, kw) - _loss(pm, dO, dht, kw)) / (2 * eps)
        np.testing.assert_allclose(grads[name_map[name]], fd, rtol=1e-6, atol=1e-8)


# ---------------------------------------------------------------- grouped q/k heads

def test_grouped_heads_forward_matches_single_head_runs():
    # value head h reads q/k head h // G (repeat_interleave order): each output head equals
    # an independent single-head run on the matching slices
    B, T, Hk, G, K, V = 1, 70, 2, 3, 4, 4
    H = Hk * G
    rng = np.random.default_rng(31)
    q = rng.standard_normal((B, T, Hk, K))
    k = rng.standard_normal((B, T, Hk, K))
    v = rng.standard_normal((B, T, H, V))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, H))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, T, H))))
    h0 = rng.standard_normal((B, H, K, V)) * 0.3
    o, hT = oracle.gdr_fwd(q, k, v, g, beta, scale=0.5, initial_state=h0, use_qk_l2norm=True)
    for h in range(H):
        hk = h // G
        o1, hT1 = oracle.gdr_fwd(q[:, :, hk:hk + 1], k[:, :, hk:hk + 1], v[:, :, h:h + 1], g[:, :, h:h + 1],
                                 beta[:, :, h:h + 1], scale=0.5, initial_state=h0[:, h:h + 1], use_qk_l2norm=True)
        np.testing.assert_allclose(o[:, :, h:h + 1], o1, rtol=0, atol=1e-12)
        np.testing.assert_allclose(hT[:, h:h + 1], hT1, rtol=0, atol=1e-12)


def test_grouped_heads_backward_matches_finite_differences():
    B, T, Hk, G, K, V = 1, 9, 2, 2, 4, 4
    H = Hk * G
    rng = np.random.default_rng(32)
    q = rng.standard_normal((B, T, Hk, K))
    k = rng.standard_normal((B, T, Hk, K))
    v = rng.standard_normal((B, T, H, V))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, H))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, T, H))))
    dO = rng.standard_normal((B, T, H, V))
    kw = dict(scale=0.6, use_qk_l2norm=True)
    grads = oracle.gdr_bwd(q, k, v, g, beta, dO, **kw)
    assert grads["dq"].shape == q.shape and grads["dk"].shape == k.shape
    eps = 1e-6
    for name, x in (("q", q), ("k", k)):
        direction = rng.standard_normal(x.shape)
        def loss(xx):
            args = dict(q=q, k=k)
            args[name] = xx
            o, _ = oracle.gdr_fwd(args["q"], args["k"], v, g, beta, output_final_state=False, **kw)
            return (o * dO).sum()
        fd = (loss(x + eps * direction) - loss(x - eps * direction)) / (2 * eps)
        an = (grads["d" + name] * direction).sum()
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, fd, an)

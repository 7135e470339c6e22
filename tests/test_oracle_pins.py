"""Pins of the fp64 oracle against facts fixed outside it.

Each test checks the oracle against something it does not share code or
formula with:

* zero projector  -> causal softmax attention from a library routine
  (torch scaled_dot_product_attention, fp64, CPU), as the write-ups state
  ("Parallax: Parameterized Local Linear Attention for Language Modeling",
  "Significance and claims": W_R = 0 recovers the Transformer);
* per-query projector (Sigma_kk + lambda I)^-1 -> the intercept of an
  independently solved ridge weighted-least-squares local-linear fit
  (exact Local Linear Attention, "Problem statement" / "Core mechanism");
* constant values -> the output equals that value for any projector
  (the local weights are affine: they sum to one);
* keys that vary only inside a subspace orthogonal to the projector's range
  -> softmax attention (pins which side of P acts on the query offset);
* linearity of the output in P;
* central finite differences of the forward for every gradient.
"""
import numpy as np
import pytest
import torch

import plx_synth


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _sdpa(q, k, v):
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True).numpy()


def _softmax_weights(q, k):
    """Causal softmax weights [T, T] for one head via torch.softmax (library)."""
    T, d = q.shape
    s = torch.from_numpy(q @ k.T / np.sqrt(d))
    mask = torch.ones(T, T, dtype=torch.bool).tril()
    s = s.masked_fill(~mask, float("-inf"))
    return torch.softmax(s, dim=-1).numpy(), torch.logsumexp(s, dim=-1).numpy()


@pytest.mark.parametrize("T,d", [(1, 4), (2, 4), (7, 8), (33, 8), (33, 64), (70, 16)])
def test_zero_projector_is_softmax_attention(oracle_mod, T, d):
    rng = np.random.default_rng(T * 100 + d)
    B, H = 2, 3
    q, k, v = (_rand(rng, B, H, T, d) for _ in range(3))
    P = np.zeros((H, d, d))
    out, lse, mu_k = oracle_mod.forward(q, k, v, P, nthreads=2)
    np.testing.assert_allclose(out, _sdpa(q, k, v), rtol=0, atol=1e-12)
    # mu_k is softmax attention with the keys as values
    np.testing.assert_allclose(mu_k, _sdpa(q, k, k), rtol=0, atol=1e-12)
    for b in range(B):
        for h in range(H):
            _, L = _softmax_weights(q[b, h], k[b, h])
            np.testing.assert_allclose(lse[b, h], L, rtol=0, atol=1e-12)


def _wls_intercept(p, K, V, q, lam):
    """Intercept a of min_{a,B} sum_i p_i |v_i - a - B (k_i - q)|^2 + lam |B|_F^2."""
    n, d = K.shape
    X = np.concatenate([np.ones((n, 1)), K - q[None, :]], axis=1)
    W = p[:, None]
    A = X.T @ (W * X)
    A[1:, 1:] += lam * np.eye(d)
    theta = np.linalg.solve(A, X.T @ (W * V))
    return theta[0]


@pytest.mark.parametrize("T,d,lam", [(5, 2, 0.1), (16, 4, 0.1), (16, 8, 0.1), (12, 8, 1.0)])
def test_exact_lla_intercept(oracle_mod, T, d, lam):
    rng = np.random.default_rng(7 + T + d)
    B, H = 1, 2
    q, k, v = (_rand(rng, B, H, T, d) for _ in range(3))
    Pq = np.zeros((B, H, T, d, d))
    expect = np.zeros((B, H, T, d))
    for b in range(B):
        for h in range(H):
            W, _ = _softmax_weights(q[b, h], k[b, h])
            for t in range(T):
                p = W[t, :t + 1]
                K, V = k[b, h, :t + 1], v[b, h, :t + 1]
                mk = p @ K
                C = (K - mk).T @ (p[:, None] * (K - mk))
                Pq[b, h, t] = np.linalg.inv(C + lam * np.eye(d))
                expect[b, h, t] = _wls_intercept(p, K, V, q[b, h, t], lam)
    out, _, _ = oracle_mod.forward(q, k, v, Pq, nthreads=2)
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-10)
    # the check is not vacuous: the correction is far from zero here
    assert np.abs(out - _sdpa(q, k, v)).max() > 1e-2


@pytest.mark.parametrize("T,d", [(1, 4), (9, 4), (40, 16)])
def test_constant_values_give_that_value(oracle_mod, T, d):
    rng = np.random.default_rng(11 * T + d)
    B, H = 2, 2
    q, k = _rand(rng, B, H, T, d), _rand(rng, B, H, T, d)
    c = _rand(rng, B, H, 1, d)
    v = np.broadcast_to(c, (B, H, T, d)).copy()
    P = _rand(rng, H, d, d)
    out, _, _ = oracle_mod.forward(q, k, v, P, nthreads=2)
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-11)
    # the first query sees one key only: o_0 = v_0 for any values
    v2 = _rand(rng, B, H, T, d)
    out2, lse2, mu2 = oracle_mod.forward(q, k, v2, P, nthreads=2)
    np.testing.assert_allclose(out2[:, :, 0], v2[:, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(mu2[:, :, 0], k[:, :, 0], rtol=0, atol=1e-12)
    s0 = np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]) / np.sqrt(d)
    np.testing.assert_allclose(lse2[:, :, 0], s0, rtol=0, atol=1e-12)


def test_probe_orientation_subspace(oracle_mod):
    """Keys vary only in span(S); range(P) is orthogonal to span(S) -> softmax.

    The transposed projector has a generic range, so it must NOT reduce.
    """
    rng = np.random.default_rng(3)
    B, H, T, d, r = 1, 2, 24, 8, 3
    Qb, _ = np.linalg.qr(rng.standard_normal((d, d)))
    S, N = Qb[:, :r], Qb[:, r:]
    k = np.empty((B, H, T, d))
    for h in range(H):
        k0 = rng.standard_normal(d)
        k[0, h] = k0[None, :] + rng.standard_normal((T, r)) @ S.T
    q, v = _rand(rng, B, H, T, d), _rand(rng, B, H, T, d)
    P = np.stack([N @ rng.standard_normal((d - r, d)) for _ in range(H)])
    out, _, _ = oracle_mod.forward(q, k, v, P, nthreads=2)
    ref = _sdpa(q, k, v)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    out_t, _, _ = oracle_mod.forward(q, k, v, np.ascontiguousarray(P.transpose(0, 2, 1)), nthreads=2)
    assert np.abs(out_t - ref).max() > 1e-3


def test_linear_in_projector(oracle_mod):
    rng = np.random.default_rng(5)
    B, H, T, d = 2, 2, 30, 8
    q, k, v = (_rand(rng, B, H, T, d) for _ in range(3))
    P = _rand(rng, H, d, d) * 0.3
    o0, l0, m0 = oracle_mod.forward(q, k, v, np.zeros_like(P), nthreads=2)
    o1, l1, m1 = oracle_mod.forward(q, k, v, P, nthreads=2)
    for alpha in (2.5, -0.7):
        oa, la, ma = oracle_mod.forward(q, k, v, alpha * P, nthreads=2)
        np.testing.assert_allclose(oa, o0 + alpha * (o1 - o0), rtol=0, atol=1e-11)
        np.testing.assert_array_equal(la, l0)   # softmax branch does not see P
        np.testing.assert_array_equal(ma, m0)


@pytest.mark.parametrize("T,d", [(1, 3), (5, 3), (8, 4)])
def test_backward_matches_finite_differences(oracle_mod, T, d):
    rng = np.random.default_rng(100 + T * d)
    B, H = 2, 2
    q, k, v = (_rand(rng, B, H, T, d) for _ in range(3))
    P = _rand(rng, H, d, d) * 0.5
    do = _rand(rng, B, H, T, d)
    dq, dk, dv, dP = oracle_mod.backward(q, k, v, P, do, nthreads=2)

    def loss(q_, k_, v_, P_):
        o, _, _ = oracle_mod.forward(q_, k_, v_, P_, nthreads=1)
        return float(np.sum(o * do))

    h = 1e-6
    args = [q, k, v, P]
    grads = [dq, dk, dv, dP]
    for ai, (x, g) in enumerate(zip(args, grads)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            ap = list(args); ap[ai] = xp
            am = list(args); am[ai] = xm
            fd[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        scale = max(1.0, np.abs(fd).max())
        np.testing.assert_allclose(g, fd, rtol=0, atol=2e-8 * scale,
                                   err_msg=f"gradient {['dq', 'dk', 'dv', 'dP'][ai]}")


def test_rows_and_head_subsets_agree_with_full(oracle_mod):
    rng = np.random.default_rng(9)
    B, H, T, d = 2, 3, 19, 8
    q, k, v, do = (_rand(rng, B, H, T, d) for _ in range(4))
    P = _rand(rng, H, d, d) * 0.2
    out, lse, mu = oracle_mod.forward(q, k, v, P, nthreads=3)
    rows = [(1, 2, 18), (0, 0, 0), (1, 0, 7)]
    o_r, l_r, m_r = oracle_mod.forward_rows(q, k, v, P, rows, nthreads=2)
    for j, (b, h, t) in enumerate(rows):
        np.testing.assert_array_equal(o_r[j], out[b, h, t])
        np.testing.assert_array_equal(l_r[j], lse[b, h, t])
        np.testing.assert_array_equal(m_r[j], mu[b, h, t])
    # the given-probe form at selected rows is its full form at those rows
    rho = _rand(rng, B, H, T, d) * 0.3
    po, pl = oracle_mod.forward_probe(q, k, v, rho, nthreads=3)
    po_r, pl_r = oracle_mod.forward_probe_rows(q, k, v, rho, rows, nthreads=2)
    for j, (b, h, t) in enumerate(rows):
        np.testing.assert_array_equal(po_r[j], po[b, h, t])
        np.testing.assert_array_equal(pl_r[j], pl[b, h, t])
    dq, dk, dv, dP = oracle_mod.backward(q, k, v, P, do, nthreads=3)
    sub = [(0, 1), (1, 1)]
    dq2, dk2, dv2, dP2 = oracle_mod.backward(q, k, v, P, do, heads=sub, nthreads=2)
    for b, h in sub:
        np.testing.assert_array_equal(dq2[b, h], dq[b, h])
        np.testing.assert_array_equal(dk2[b, h], dk[b, h])
        np.testing.assert_array_equal(dv2[b, h], dv[b, h])
    np.testing.assert_allclose(dP2[1], dP[1], rtol=0, atol=1e-12)
    assert not dP2[0].any() and not dP2[2].any()


def test_synth_recipe_is_deterministic_and_rounded():
    a = plx_synth.generate(1, 2, 16, 8, "bf16", seed=4, backward=True, norm_mult=True)
    b = plx_synth.generate(1, 2, 16, 8, "bf16", seed=4, backward=True, norm_mult=True)
    for key in ("q", "k", "v", "P", "dout"):
        np.testing.assert_array_equal(a[key], b[key])
    # bf16 round trip is exact
    w = plx_synth.widen(a["q"])
    np.testing.assert_array_equal(plx_synth.to_bf16_bits(w), a["q"])
    # RNE on a tie: 1 + 2^-8 lies halfway between two bf16 values -> even (1.0)
    assert plx_synth.to_bf16_bits(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert plx_synth.to_bf16_bits(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82
    c = plx_synth.generate(1, 2, 8, 4, "fp32", seed=0, key_cov=True)
    assert c["P"].dtype == np.float32 and c["q"].dtype == np.float32


# ---------------------------------------------------------------- given probe
# The one-pass form o = o^SA - Sigma_KV rho with a probe supplied as input
# ("Parallax: Parameterized Local Linear Attention for Language Modeling",
# "Core mechanism": the probe comes from a learned projection of the layer
# input instead of a per-query solve).


@pytest.mark.parametrize("T,d", [(1, 4), (7, 8), (33, 16)])
def test_probe_zero_is_softmax_attention(oracle_mod, T, d):
    rng = np.random.default_rng(300 + T + d)
    B, H = 2, 2
    q, k, v = (_rand(rng, B, H, T, d) for _ in range(3))
    out, lse = oracle_mod.forward_probe(q, k, v, np.zeros((B, H, T, d)), nthreads=2)
    np.testing.assert_allclose(out, _sdpa(q, k, v), rtol=0, atol=1e-12)
    for b in range(B):
        for h in range(H):
            _, L = _softmax_weights(q[b, h], k[b, h])
            np.testing.assert_allclose(lse[b, h], L, rtol=0, atol=1e-12)


@pytest.mark.parametrize("T,d", [(5, 4), (24, 8)])
def test_probe_from_the_projector_is_the_two_pass_layer(oracle_mod, T, d):
    # rho_t = -P_h (q_t - mu_k,t) turns the given-probe form into the layer the
    # library's two-pass path computes (the sign reading R6: o^SA - Sigma rho
    # against mu_v + Sigma u with rho = -u)
    rng = np.random.default_rng(17 + T * d)
    B, H = 2, 2
    q, k, v = (_rand(rng, B, H, T, d) for _ in range(3))
    P = 0.3 * _rand(rng, H, d, d)
    out2, lse2, mu_k = oracle_mod.forward(q, k, v, P, nthreads=2)
    rho = -np.einsum("had,bhtd->bhta", P, q - mu_k)
    out1, lse1 = oracle_mod.forward_probe(q, k, v, rho, nthreads=2)
    np.testing.assert_allclose(out1, out2, rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse1, lse2, rtol=0, atol=1e-12)
    assert np.abs(out1 - _sdpa(q, k, v)).max() > 1e-2  # not vacuous


@pytest.mark.parametrize("T,d,lam", [(6, 2, 0.1), (16, 4, 0.1)])
def test_probe_exact_lla_intercept(oracle_mod, T, d, lam):
    # rho_t = -(Sigma_kk,t + lambda I)^-1 (q_t - mu_k,t) is the exact-LLA probe:
    # the output is the intercept of an independently solved ridge WLS fit
    rng = np.random.default_rng(29 + T + d)
    B, H = 1, 2
    q, k, v = (_rand(rng, B, H, T, d) for _ in range(3))
    rho = np.zeros((B, H, T, d))
    expect = np.zeros((B, H, T, d))
    for b in range(B):
        for h in range(H):
            W, _ = _softmax_weights(q[b, h], k[b, h])
            for t in range(T):
                p = W[t, :t + 1]
                K, V = k[b, h, :t + 1], v[b, h, :t + 1]
                mk = p @ K
                C = (K - mk).T @ (p[:, None] * (K - mk))
                rho[b, h, t] = -np.linalg.solve(C + lam * np.eye(d), q[b, h, t] - mk)
                expect[b, h, t] = _wls_intercept(p, K, V, q[b, h, t], lam)
    out, _ = oracle_mod.forward_probe(q, k, v, rho, nthreads=2)
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-10)


def test_probe_constant_values_and_linearity(oracle_mod):
    rng = np.random.default_rng(5)
    B, H, T, d = 2, 2, 20, 8
    q, k = _rand(rng, B, H, T, d), _rand(rng, B, H, T, d)
    rho = _rand(rng, B, H, T, d)
    c = _rand(rng, B, H, 1, d)
    vc = np.broadcast_to(c, (B, H, T, d)).copy()
    out, _ = oracle_mod.forward_probe(q, k, vc, rho, nthreads=2)
    np.testing.assert_allclose(out, vc, rtol=0, atol=1e-11)  # the covariance of constant values is 0
    v = _rand(rng, B, H, T, d)
    o0, _ = oracle_mod.forward_probe(q, k, v, 0 * rho, nthreads=2)
    o1, _ = oracle_mod.forward_probe(q, k, v, rho, nthreads=2)
    o3, _ = oracle_mod.forward_probe(q, k, v, 2.5 * rho, nthreads=2)
    np.testing.assert_allclose(o3 - o0, 2.5 * (o1 - o0), rtol=0, atol=1e-10)

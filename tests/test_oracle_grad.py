"""Pins of the oracle's bidirectional gradient (CPU only): central finite
differences of the forward oracle in fp64, for every feature map, on every
element of tiny Q, K, V; and the identity that makes the query norm's
gradient vanish (phi(Q) . dphi(Q) = 0 row by row)."""

import numpy as np
import pytest

import oracle as orc


def _loss(Q, K, V, Om, s, dO, features, causal=False):
    fwd = orc.favor_causal if causal else orc.favor_bidirectional
    return float(np.sum(dO * fwd(Q, K, V, Om, s, features)))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("features", ["prf", "relu", "elu1"])
def test_gradient_matches_central_differences(features, causal):
    rng = np.random.default_rng({"prf": 7, "relu": 8, "elu1": 6}[features] + 10 * causal)
    # enough features that no normaliser is zero (under ReLU a causal row
    # with one key can have phi(q).phi(k) = 0)
    L, d, m = 5, 3, 16
    Q, K, V, dO = (rng.standard_normal((L, d)) for _ in range(4))
    Om = rng.standard_normal((m, d))
    if causal:
        K[0] = Q[0]          # phi(q0).phi(k0) = |phi(q0)|^2 > 0 for either map
    s = 0.8
    fwd = orc.favor_causal if causal else orc.favor_bidirectional
    assert np.all(np.isfinite(fwd(Q, K, V, Om, s, features)))
    grad = orc.favor_causal_grad if causal else orc.favor_bidirectional_grad
    dQ, dK, dV = grad(Q, K, V, Om, s, dO, features)
    h = 1e-6
    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        for idx in np.ndindex(X.shape):
            old = X[idx]
            X[idx] = old + h
            up = _loss(Q, K, V, Om, s, dO, features, causal)
            X[idx] = old - h
            dn = _loss(Q, K, V, Om, s, dO, features, causal)
            X[idx] = old
            num = (up - dn) / (2 * h)
            assert abs(num - G[idx]) < 1e-6 * max(1.0, abs(num)), (features, idx, num, G[idx])


def test_batched_gradient_equals_per_head():
    rng = np.random.default_rng(9)
    Q, K, V, dO = (rng.standard_normal((2, 3, 7, 4)) for _ in range(4))
    Om = rng.standard_normal((8, 4))
    g = orc.favor_bidirectional_grad(Q, K, V, Om, 0.7, dO)
    for b in range(2):
        for h in range(3):
            gh = orc.favor_bidirectional_grad(Q[b, h], K[b, h], V[b, h], Om, 0.7, dO[b, h])
            for full, one in zip(g, gh):
                assert np.allclose(full[b, h], one, rtol=1e-13, atol=1e-13)


def test_query_features_get_no_radial_gradient():
    # per-query constants cancel in the output, so sum_i phi_i dphi_i = 0 per
    # row; equivalently the gradient of a query along itself is the
    # projection part only
    rng = np.random.default_rng(10)
    Q, K, V, dO = (rng.standard_normal((6, 4)) for _ in range(4))
    Om = rng.standard_normal((5, 4))
    s = 0.9
    pq = orc.prf_features(s * Q, Om)
    pk = orc.prf_features(s * K, Om)
    S, z = pk.T @ V, pk.sum(0)
    N, D = pq @ S, pq @ z
    O = N / D[:, None]
    dpq = (dO / D[:, None]) @ S.T + (-np.sum(dO * O, 1) / D)[:, None] * z[None, :]
    assert np.max(np.abs(np.sum(pq * dpq, axis=1))) < 1e-12 * np.max(np.abs(pq * dpq))


def test_causal_gradient_of_the_last_row_only_equals_bidirectional():
    # with dO zero except the last row, the causal and bidirectional losses
    # coincide (the last causal row sees every token)
    rng = np.random.default_rng(11)
    Q, K, V = (rng.standard_normal((9, 4)) for _ in range(3))
    dO = np.zeros((9, 4))
    dO[-1] = rng.standard_normal(4)
    Om = rng.standard_normal((7, 4))
    a = orc.favor_causal_grad(Q, K, V, Om, 0.6, dO)
    b = orc.favor_bidirectional_grad(Q, K, V, Om, 0.6, dO)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-12, atol=1e-12)

"""Pins for the oracle's attention (CPU only).

Exact identities the pages fix: the quadratic and the linear order give the
same estimator; the unidirectional form is the lower-triangular part
(diagonal included) computed by a prefix sum; closed-form special cases.
"""

import numpy as np
import pytest

import oracle as orc


def _qkv(B, H, L, d, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((B, H, L, d)) * scale for _ in range(3))


def test_linear_order_equals_quadratic_order():
    Q, K, V = _qkv(2, 3, 97, 16, seed=1)
    Om = orc.build_omega(0, 48, 16)
    s = 16 ** -0.25
    a = orc.favor_bidirectional(Q, K, V, Om, s)
    b = orc.favor_bidirectional_quadratic(Q, K, V, Om, s)
    assert orc.rowwise_rel_err(a, b) < 1e-12


def test_causal_prefix_sum_equals_lower_triangular_form():
    Q, K, V = _qkv(2, 2, 131, 8, seed=2)
    Om = orc.build_omega(1, 24, 8)
    s = 8 ** -0.25
    a = orc.favor_causal(Q, K, V, Om, s)
    b = orc.favor_causal_quadratic(Q, K, V, Om, s)
    assert orc.rowwise_rel_err(a, b) < 1e-12


def test_causal_row_depends_only_on_past():
    Q, K, V = _qkv(1, 1, 64, 8, seed=3)
    Om = orc.build_omega(2, 16, 8)
    s = 8 ** -0.25
    base = orc.favor_causal(Q, K, V, Om, s)
    t = 40
    Q2, K2, V2 = Q.copy(), K.copy(), V.copy()
    rng = np.random.default_rng(4)
    Q2[..., t + 1:, :] = rng.standard_normal(Q2[..., t + 1:, :].shape)
    K2[..., t + 1:, :] = rng.standard_normal(K2[..., t + 1:, :].shape)
    V2[..., t + 1:, :] = rng.standard_normal(V2[..., t + 1:, :].shape)
    pert = orc.favor_causal(Q2, K2, V2, Om, s)
    assert np.array_equal(base[..., : t + 1, :], pert[..., : t + 1, :])
    assert not np.allclose(base[..., t + 1:, :], pert[..., t + 1:, :])


def test_causal_last_row_equals_bidirectional_last_row_and_first_row_is_v0():
    Q, K, V = _qkv(1, 2, 50, 8, seed=5)
    Om = orc.build_omega(3, 32, 8)
    s = 8 ** -0.25
    c = orc.favor_causal(Q, K, V, Om, s)
    b = orc.favor_bidirectional(Q, K, V, Om, s)
    assert np.allclose(c[..., -1, :], b[..., -1, :], rtol=1e-12, atol=1e-13)
    assert np.allclose(c[..., 0, :], V[..., 0, :], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_keys_give_mean_of_values(causal):
    Q, _, V = _qkv(1, 2, 33, 8, seed=6)
    K = np.zeros_like(Q)
    Om = orc.build_omega(4, 16, 8)
    s = 8 ** -0.25
    if causal:
        out = orc.favor_causal(Q, K, V, Om, s)
        want = np.cumsum(V, axis=-2) / np.arange(1, 34)[:, None]
    else:
        out = orc.favor_bidirectional(Q, K, V, Om, s)
        want = np.broadcast_to(V.mean(axis=-2, keepdims=True), V.shape)
    assert np.allclose(out, want, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_reproduced(causal):
    Q, K, _ = _qkv(1, 1, 40, 8, seed=7)
    V = np.full_like(Q, 2.5)
    Om = orc.build_omega(5, 16, 8)
    fn = orc.favor_causal if causal else orc.favor_bidirectional
    out = fn(Q, K, V, Om, 8 ** -0.25)
    assert np.allclose(out, 2.5, rtol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_single_token_returns_value(causal):
    Q, K, V = _qkv(2, 2, 1, 8, seed=8)
    Om = orc.build_omega(6, 16, 8)
    fn = orc.favor_causal if causal else orc.favor_bidirectional
    out = fn(Q, K, V, Om, 8 ** -0.25)
    assert np.allclose(out, V, rtol=1e-13)


def test_query_side_constants_cancel():
    # [su] Simple Derivation: scaling q~ by any positive per-query constant
    # leaves the result unchanged, so dropping ||q||^2/2 changes nothing.
    Q, K, V = _qkv(1, 1, 30, 8, seed=9)
    Om = orc.build_omega(7, 16, 8)
    s = 8 ** -0.25
    pq = orc.prf_features(s * Q, Om)
    pk = orc.prf_features(s * K, Om)
    lam = np.exp(np.random.default_rng(1).standard_normal((1, 1, 30, 1)))
    out1 = (pq @ (np.swapaxes(pk, -1, -2) @ V)) / (pq @ pk.sum(-2)[..., None])
    pq2 = pq * lam
    out2 = (pq2 @ (np.swapaxes(pk, -1, -2) @ V)) / (pq2 @ pk.sum(-2)[..., None])
    assert np.allclose(out1, out2, rtol=1e-12)
    assert np.allclose(out1, orc.favor_bidirectional(Q, K, V, Om, s), rtol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_rows_match_full_output(causal):
    Q, K, V = _qkv(1, 3, 70, 8, seed=10)
    Om = orc.build_omega(8, 16, 8)
    s = 8 ** -0.25
    full = (orc.favor_causal if causal else orc.favor_bidirectional)(Q, K, V, Om, s)[0]
    picks = [(0, 0), (1, 69), (2, 33), (0, 12), (1, 1)]
    rows = orc.favor_rows(Q[0], K[0], V[0], Om, s, picks, causal)
    want = np.stack([full[h, t] for h, t in picks])
    assert np.allclose(rows, want, rtol=1e-12, atol=1e-13)


def test_softmax_reference_matches_direct_formula():
    Q, K, V = _qkv(1, 1, 20, 4, seed=11)
    s = 4 ** -0.25
    S = np.exp((s * Q[0, 0]) @ (s * K[0, 0]).T)
    want = (S / S.sum(-1, keepdims=True)) @ V[0, 0]
    assert np.allclose(orc.softmax_attention(Q, K, V, s)[0, 0], want, rtol=1e-12)
    Sc = S * np.tril(np.ones((20, 20)))
    wantc = (Sc / Sc.sum(-1, keepdims=True)) @ V[0, 0]
    assert np.allclose(orc.softmax_attention(Q, K, V, s, causal=True)[0, 0], wantc, rtol=1e-12)


def test_rowwise_rel_err_definition():
    ref = np.array([[1.0, -2.0], [0.0, 0.5]])
    got = np.array([[1.1, -2.0], [0.0, 0.5]])
    assert orc.rowwise_rel_err(got, ref) == pytest.approx(0.05)

"""Planted mistakes in copies of the oracle's steps must fail the pins.

Each case builds a wrong variant of one oracle step on the CPU (a dropped
term, a flipped sign, a missing factor, a shifted index) and checks that the
pin written for that step rejects it, so the pins can catch such slips.
"""

import math

import numpy as np

import oracle as orc


def _pair(seed=0, d=8, scale=0.35):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(d) * scale, rng.standard_normal(d) * scale


def _mean_estimate(feat, x, y, d, m=8, n=20000, seed=1):
    rng = np.random.default_rng(seed)
    Om = rng.standard_normal((n * m, d))
    fx = feat(x[None], Om)[0] * math.sqrt(n * m) / math.sqrt(m)
    fy = feat(y[None], Om)[0] * math.sqrt(n * m) / math.sqrt(m)
    est = (fx * fy).reshape(n, m).sum(axis=1)
    return est.mean(), est.std(ddof=1) / math.sqrt(n)


def _unbiased(feat):
    x, y = _pair()
    mean, se = _mean_estimate(feat, x, y, 8)
    return abs(mean - float(orc.softmax_kernel(x, y))) < 5 * se


def test_correct_feature_map_passes_unbiasedness():
    assert _unbiased(orc.prf_features)


def test_dropped_norm_term_fails_unbiasedness():
    def bad(X, Om):
        return np.exp(X @ Om.T) / math.sqrt(Om.shape[0])
    assert not _unbiased(bad)


def test_flipped_norm_sign_fails_unbiasedness():
    def bad(X, Om):
        return np.exp(X @ Om.T + 0.5 * np.sum(X * X, -1, keepdims=True)) / math.sqrt(Om.shape[0])
    assert not _unbiased(bad)


def test_missing_sqrt_m_fails_estimator_scale():
    x, y = _pair(2)
    Om = orc.build_omega(0, 4096, 8)
    good = np.sum(orc.prf_features(x[None], Om) * orc.prf_features(y[None], Om))
    bad = good * Om.shape[0]          # features without 1/sqrt(m)
    sm = float(orc.softmax_kernel(x, y))
    assert abs(good - sm) < 0.05 * sm and abs(bad - sm) > 10 * sm


def test_transposed_orf_block_fails_length_pin():
    Om, parts = orc.build_omega(5, 16, 16, return_parts=True)
    lengths = parts[0][2]
    bad = Om.T.copy()
    assert np.allclose(np.linalg.norm(Om, axis=1), lengths, rtol=1e-12)
    assert not np.allclose(np.linalg.norm(bad, axis=1), lengths, rtol=1e-6)


def test_exclusive_diagonal_fails_first_row_pin():
    rng = np.random.default_rng(3)
    Q, K, V = (rng.standard_normal((1, 1, 12, 4)) for _ in range(3))
    Om = orc.build_omega(1, 8, 4)
    s = 4 ** -0.25
    pq = orc.prf_features(s * Q, Om)
    pk = orc.prf_features(s * K, Om)
    A = (pq @ np.swapaxes(pk, -1, -2)) * np.tril(np.ones((12, 12)), k=-1)   # s < t only
    with np.errstate(invalid="ignore", divide="ignore"):
        bad = (A @ V) / A.sum(-1, keepdims=True)
    good = orc.favor_causal(Q, K, V, Om, s)
    assert np.allclose(good[..., 0, :], V[..., 0, :])
    assert not np.allclose(bad[..., 0, :], V[..., 0, :], equal_nan=False)


def test_missing_normaliser_fails_constant_value_pin():
    rng = np.random.default_rng(4)
    Q, K = (rng.standard_normal((1, 1, 20, 4)) for _ in range(2))
    V = np.full((1, 1, 20, 4), 3.0)
    Om = orc.build_omega(2, 8, 4)
    s = 4 ** -0.25
    pq = orc.prf_features(s * Q, Om)
    pk = orc.prf_features(s * K, Om)
    bad = pq @ (np.swapaxes(pk, -1, -2) @ V)
    assert np.allclose(orc.favor_bidirectional(Q, K, V, Om, s), 3.0)
    assert not np.allclose(bad, 3.0, rtol=1e-3)


def test_query_side_norm_kept_on_keys_only_matters():
    # dropping ||k||^2/2 (allowed only on the query side) changes the result
    rng = np.random.default_rng(6)
    Q, K, V = (rng.standard_normal((1, 1, 30, 4)) for _ in range(3))
    Om = orc.build_omega(3, 16, 4)
    s = 4 ** -0.25
    pq = orc.prf_features(s * Q, Om)
    pk_bad = np.exp((s * K) @ Om.T)
    bad = (pq @ (np.swapaxes(pk_bad, -1, -2) @ V)) / (pq @ pk_bad.sum(-2)[..., None])
    good = orc.favor_bidirectional(Q, K, V, Om, s)
    assert orc.rowwise_rel_err(bad, good) > 1e-3

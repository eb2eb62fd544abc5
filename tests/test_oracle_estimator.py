"""Pins for the oracle's feature maps against the pages' theory (CPU only).

Lemma 2 gives the exact MSE of the positive-random-feature estimator for iid
Gaussian projections; Theorem 1 says it is unbiased; Theorem 2 says
orthogonal projections give a strictly smaller MSE; the pages also state that
positive features beat sin/cos features where the kernel value is small, and
that the approximation converges as m grows.  A dropped ||x||^2/2 term, a
wrong sign, a transposed Omega or a missing 1/sqrt(m) fails at least one test.
"""

import math

import numpy as np
import pytest

import oracle as orc


def _pair(d, norm_sum_sq, rng, cos_xy=0.3):
    """x, y in R^d with ||x + y||^2 = norm_sum_sq."""
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    v = rng.standard_normal(d)
    v -= u * (u @ v)
    v /= np.linalg.norm(v)
    a = math.sqrt(norm_sum_sq) / 2.0
    x = a * u + 0.3 * v
    y = a * u - 0.3 * v
    assert abs(np.sum((x + y) ** 2) - norm_sum_sq) < 1e-12
    return x, y


def _iid_single_feature_terms(x, y, n, d, rng):
    """n independent one-feature estimates exp(w.x-|x|^2/2) exp(w.y-|y|^2/2)."""
    Om = rng.standard_normal((n, d))
    fx = orc.prf_features(x[None, :], Om)[0] * math.sqrt(n)
    fy = orc.prf_features(y[None, :], Om)[0] * math.sqrt(n)
    return fx * fy


@pytest.mark.parametrize("d", [4, 16])
@pytest.mark.parametrize("s2", [0.25, 0.5, 1.0])
@pytest.mark.parametrize("m", [1, 4, 16])
def test_lemma2_mse_closed_form(d, s2, m):
    rng = np.random.default_rng(1000 * d + int(100 * s2) + m)
    x, y = _pair(d, s2, rng)
    n_draws = 200_000
    terms = _iid_single_feature_terms(x, y, n_draws * m, d, rng).reshape(n_draws, m)
    est = terms.mean(axis=1)
    sm = float(orc.softmax_kernel(x, y))
    sq = (est - sm) ** 2
    mse = sq.mean()
    se = sq.std(ddof=1) / math.sqrt(n_draws)
    want = orc.lemma2_mse(x, y, m)
    assert abs(mse - want) < 5 * se + 1e-15, (mse, want, se)


def test_lemma2_zero_variance_when_x_is_minus_y():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(8) * 0.7
    y = -x
    for seed in range(5):
        Om = orc.build_omega(seed, 16, 8, orthogonal=(seed % 2 == 0))
        est = orc.prf_estimator(x[None, :], y[None, :], Om)[0]
        assert est == pytest.approx(math.exp(-np.sum(x * x)), rel=1e-13)
    assert orc.lemma2_mse(x, y, 4) == 0.0


@pytest.mark.parametrize("orthogonal", [False, True])
def test_theorem1_unbiased(orthogonal):
    d, m = 8, 8
    rng = np.random.default_rng(17)
    x = rng.standard_normal(d) * 0.35
    y = rng.standard_normal(d) * 0.35
    sm = float(orc.softmax_kernel(x, y))
    n = 3000 if orthogonal else 20000
    ests = np.array([orc.prf_estimator(x[None, :], y[None, :],
                                       orc.build_omega(s, m, d, orthogonal=orthogonal))[0]
                     for s in range(n)]) if orthogonal else None
    if not orthogonal:
        terms = _iid_single_feature_terms(x, y, n * m, d, rng).reshape(n, m)
        ests = terms.mean(axis=1)
    se = ests.std(ddof=1) / math.sqrt(n)
    assert abs(ests.mean() - sm) < 5 * se


@pytest.mark.parametrize("scale", [0.15, 0.2])
def test_theorem2_orthogonal_beats_iid(scale):
    # one full orthogonal block (m = d), where the variance reduction is largest
    d = m = 16
    rng = np.random.default_rng(16)
    x = rng.standard_normal(d) * scale
    y = rng.standard_normal(d) * scale
    sm = float(orc.softmax_kernel(x, y))
    n = 8000
    orf = np.array([orc.prf_estimator(x[None, :], y[None, :], orc.build_omega(s, m, d))[0]
                    for s in range(n)])
    mse_orf = np.mean((orf - sm) ** 2)
    mse_iid = orc.lemma2_mse(x, y, m)
    se = np.std((orf - sm) ** 2, ddof=1) / math.sqrt(n)
    assert abs(np.mean(orf) - sm) < 5 * np.std(orf) / math.sqrt(n)      # still unbiased
    assert mse_orf + 4 * se < mse_iid, (mse_orf, mse_iid, se)


def test_theorem2_blocks_beat_iid_attention_error():
    # the pages' setting: L = 4096, d = 16, sweep m (blocks of d when m > d);
    # inputs with |x|^2 ~ 0.36 so the squared error is not heavy-tailed
    d, L, n_seeds = 16, 4096, 150
    rng = np.random.default_rng(3)
    Q = rng.standard_normal((256, d)) * 0.15
    K = rng.standard_normal((L, d)) * 0.15
    A = np.exp(Q @ K.T)
    for m in (16, 32, 64):
        err = {True: [], False: []}
        for seed in range(n_seeds):
            for orth in (True, False):
                Om = orc.build_omega(100 + seed, m, d, orthogonal=orth)
                approx = orc.prf_features(Q, Om) @ orc.prf_features(K, Om).T
                err[orth].append(np.mean((approx - A) ** 2))
        eo, ei = np.array(err[True]), np.array(err[False])
        se = math.sqrt(eo.var(ddof=1) / n_seeds + ei.var(ddof=1) / n_seeds)
        assert ei.mean() - eo.mean() > 2 * se, (m, eo.mean(), ei.mean(), se)


def test_positive_beats_trigonometric_for_small_kernel_values():
    d, m = 8, 16
    rng = np.random.default_rng(9)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    x = 1.2 * u
    y = -1.1 * u + 0.1 * rng.standard_normal(d)   # x.y < 0: small SM(x, y)
    sm = float(orc.softmax_kernel(x, y))
    assert sm < 0.5
    n = 20000
    Om = rng.standard_normal((n * m, d))
    # PRF
    fx = orc.prf_features(x[None], Om)[0] * math.sqrt(n * m)
    fy = orc.prf_features(y[None], Om)[0] * math.sqrt(n * m)
    prf = (fx * fy).reshape(n, m).mean(axis=1)
    # trig: features [sin, cos], each scaled 1/sqrt(m_total)
    tx = orc.trig_features(x[None], Om)[0] * math.sqrt(n * m)
    ty = orc.trig_features(y[None], Om)[0] * math.sqrt(n * m)
    trig = (tx * ty).reshape(2, n, m).sum(axis=0).mean(axis=1)
    assert abs(trig.mean() - sm) < 5 * trig.std() / math.sqrt(n)   # trig is unbiased too
    mse_prf = np.mean((prf - sm) ** 2)
    mse_trig = np.mean((trig - sm) ** 2)
    assert mse_prf < mse_trig / 5, (mse_prf, mse_trig)
    assert np.all(prf > 0) and np.any(trig < 0)


def test_estimator_matches_kernel_with_many_features():
    # m -> infinity: exp(x^T y) recovered
    d = 8
    rng = np.random.default_rng(21)
    x = rng.standard_normal(d) * 0.4
    y = rng.standard_normal(d) * 0.4
    Om = orc.build_omega(4, 8 * 4096, d)
    est = orc.prf_estimator(x[None], y[None], Om)[0]
    sm = float(orc.softmax_kernel(x, y))
    sd = math.sqrt(orc.lemma2_mse(x, y, 8 * 4096))
    assert abs(est - sm) < 6 * sd


def test_attention_converges_to_softmax_as_m_grows():
    # uniform convergence in m (independent of L).  Inputs with |s q|^2 ~ 1:
    # at larger norms the per-feature variance exp(|q+k|^2) keeps the error
    # pre-asymptotic for any m here (the pages' stated limitation).
    d, L = 16, 256
    rng = np.random.default_rng(12)
    s = d ** -0.25
    Q = rng.standard_normal((L, d)) * 0.5
    K = rng.standard_normal((L, d)) * 0.5
    V = rng.standard_normal((L, d))
    exact = orc.softmax_attention(Q, K, V, s)
    ms = [16, 64, 256, 1024, 4096]
    errs = []
    for m in ms:
        e = [np.sqrt(np.mean((orc.favor_bidirectional(Q, K, V, orc.build_omega(sd, m, d), s) - exact) ** 2))
             for sd in range(8)]
        errs.append(np.mean(e))
    assert all(errs[i + 1] < errs[i] for i in range(len(errs) - 1)), errs
    slope = np.polyfit(np.log(ms), np.log(errs), 1)[0]
    assert -0.8 < slope < -0.25, (slope, errs)

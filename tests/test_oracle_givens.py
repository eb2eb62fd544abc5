"""Pins of the oracle's Givens ORF builder (CPU only): the rotation count's
closed form, the rotation draws against the published SplitMix64 stream
(distinct pair, uniform pairs and angles), a d = 2 block against the
composition of plane rotations, the order of the product against rotating a
vector step by step, exact orthogonality with determinant +1, and the small
bias of the softmax-kernel estimator (the pages: Givens ORFs are slightly
biased, the bias tending to zero as d grows)."""

import math

import numpy as np
import pytest

import oracle as orc


def test_rotation_count_closed_form():
    # 3 d ceil(log2 d)
    assert orc.givens_rotation_count(2) == 6
    assert orc.givens_rotation_count(3) == 18
    assert orc.givens_rotation_count(64) == 3 * 64 * 6
    assert orc.givens_rotation_count(65) == 3 * 65 * 7
    assert orc.givens_rotation_count(128) == 3 * 128 * 7
    with pytest.raises(ValueError):
        orc.givens_rotation_count(1)


def test_draws_are_distinct_uniform_pairs_and_angles():
    d = 6
    pairs = {}
    angles = []
    for b in range(700):
        for i, j, th in orc.givens_rotations(11, b, d):
            assert 0 <= i < d and 0 <= j < d and i != j
            assert 0.0 < th < 2 * math.pi
            pairs[(i, j)] = pairs.get((i, j), 0) + 1
            angles.append(th)
    n = sum(pairs.values())
    assert len(pairs) == d * (d - 1)
    # every ordered pair near n / 30 (1260 draws each: binomial sd ~ 2.8 % of
    # the mean, the bound ~ 5 sd)
    for c in pairs.values():
        assert abs(c / (n / (d * (d - 1))) - 1.0) < 0.15
    # angle quartiles of a uniform (0, 2 pi)
    q = np.quantile(angles, [0.25, 0.5, 0.75]) / (2 * math.pi)
    assert np.allclose(q, [0.25, 0.5, 0.75], atol=0.02)


def test_draws_read_the_splitmix_words_in_order():
    # the top 23 bits of word 2c + 1 give the angle of rotation c of block 0;
    # the first word's top bits choose i (floor(hi32 * d / 2^32))
    d = 8
    rot = orc.givens_rotations(21, 0, d)
    w = orc.splitmix64_stream(21, np.arange(2 * len(rot)))
    for c, (i, j, th) in enumerate(rot):
        k = int(w[2 * c + 1]) >> 41
        assert th == pytest.approx(2 * math.pi * (k + 0.5) / 2 ** 23, rel=1e-15)
        assert i == (int(w[2 * c]) >> 32) * d >> 32
    # block 1 starts right after block 0's words
    rot1 = orc.givens_rotations(21, 1, d)
    w1 = orc.splitmix64_stream(21, [2 * len(rot) + 1])
    assert rot1[0][2] == pytest.approx(2 * math.pi * ((int(w1[0]) >> 41) + 0.5) / 2 ** 23, rel=1e-15)


def test_d2_block_is_the_rotation_by_the_signed_angle_sum():
    # in the plane, the rotation on (0, 1) by theta turns by +theta and the one
    # on (1, 0) by -theta; rotations of the plane compose by adding angles
    for seed in (0, 5, 9):
        phi = sum(th if i == 0 else -th for i, j, th in orc.givens_rotations(seed, 0, 2))
        want = math.sqrt(2) * np.array([[math.cos(phi), -math.sin(phi)], [math.sin(phi), math.cos(phi)]])
        assert np.allclose(orc.build_omega_givens(seed, 2, 2), want, rtol=0, atol=1e-14)


def test_product_order_matches_rotating_a_vector_step_by_step():
    d = 16
    Om = orc.build_omega_givens(8, d, d)
    x = np.random.default_rng(1).standard_normal(d)
    y = x.copy()
    for i, j, th in orc.givens_rotations(8, 0, d):
        c, s = math.cos(th), math.sin(th)
        y[i], y[j] = c * y[i] - s * y[j], s * y[i] + c * y[j]
    assert np.allclose(Om @ x / math.sqrt(d), y, rtol=0, atol=1e-13)


@pytest.mark.parametrize("m,d", [(64, 64), (256, 64), (100, 32), (200, 48), (128, 128)])
def test_blocks_are_rotations_with_rows_of_length_sqrt_d(m, d):
    Om = orc.build_omega_givens(3, m, d)
    assert Om.shape == (m, d)
    for b in range(0, m, d):
        blk = Om[b:b + d]
        assert np.allclose(blk @ blk.T, d * np.eye(blk.shape[0]), rtol=0, atol=1e-9)
        if blk.shape[0] == d:
            assert np.linalg.det(blk / math.sqrt(d)) == pytest.approx(1.0, abs=1e-9)
    if m >= 2 * d:
        assert not np.allclose(Om[:d], Om[d:2 * d])
    assert not np.allclose(orc.build_omega_givens(4, m, d), Om)


def test_rows_are_spread_like_the_sphere():
    # rows uniform on the sphere of radius sqrt(d) have E[w_k^4] = 3d / (d + 2)
    # (d^2 E[u_k^4], u uniform on the unit sphere); rows near coordinate axes
    # (too few rotations) give up to d
    d = 64
    m4 = [float((orc.build_omega_givens(seed, d, d) ** 4).mean()) for seed in range(40)]
    assert np.mean(m4) == pytest.approx(3 * d / (d + 2), rel=0.03)


def _sphere_expectation(z: float, d: int) -> float:
    # E[exp(w.z)] for w uniform on the sphere of radius sqrt(d), |z| = z:
    # Gamma(d/2) (2 / a)^(d/2 - 1) I_(d/2 - 1)(a), a = sqrt(d) z
    special = pytest.importorskip("scipy.special")
    gammaln, ive = special.gammaln, special.ive
    a = math.sqrt(d) * z
    nu = d / 2 - 1
    return math.exp(gammaln(d / 2) + nu * math.log(2 / a) + math.log(ive(nu, a)) + a)


def test_estimator_mean_matches_the_sphere_closed_form():
    # the softmax-kernel estimate exp(-|x|^2/2 - |y|^2/2) mean_i exp(w_i.(x + y))
    # with rows of length sqrt(d) has mean exp(x.y) E_sphere / exp(|x+y|^2 / 2):
    # a small negative bias (-1.7 % here) that the Gaussian rows do not have
    rng = np.random.default_rng(0)
    d = 64
    x = rng.standard_normal(d) * 0.15
    y = rng.standard_normal(d) * 0.15
    exact = math.exp(float(x @ y))
    z = float(np.linalg.norm(x + y))
    want = _sphere_expectation(z, d) / math.exp(z * z / 2) - 1.0
    est = np.array([float(orc.prf_estimator(x, y, orc.build_omega_givens(seed, 256, d))) for seed in range(150)])
    se = est.std() / exact / math.sqrt(len(est))
    assert abs(est.mean() / exact - 1.0 - want) < 4 * se
    assert -0.05 < want < 0

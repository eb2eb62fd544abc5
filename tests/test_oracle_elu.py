"""Pins of the oracle's 1 + elu feature map (CPU only).

"From Performer to Linear Attention" (Su) prints the linear-attention choice
phi(x) = 1 + elu(x) (1 + x for x >= 0, e^x below) and the "Performer" digest
names it as Linear Attention's map; the oracle applies it in the feature-map
slot, to s Omega x.  Fixed here independently of the oracle's code: an
explicit loop, a hand-derived example with Omega = I (plain linear
attention), continuity of the map and its slope at 0, positivity (the
normaliser never vanishes), and the identities every linear attention
satisfies.
"""

import math

import numpy as np
import pytest

import oracle as orc


def test_elu1_features_match_an_explicit_loop():
    rng = np.random.default_rng(21)
    X = rng.standard_normal((4, 5))
    Om = rng.standard_normal((6, 5))
    got = orc.elu1_features(X, Om)
    for t in range(4):
        for i in range(6):
            a = 0.0
            for j in range(5):
                a += Om[i, j] * X[t, j]
            want = (1.0 + a if a >= 0 else math.exp(a)) / math.sqrt(6)
            assert got[t, i] == pytest.approx(want, rel=1e-14, abs=1e-15)


def test_hand_derived_linear_attention_example():
    # Omega = I (m = d = 2), s = 1: phi(x) = (1 + elu(x1), 1 + elu(x2)) / sqrt(2)
    # q = (0, -ln 2) -> (1, 1/2); keys (1, 0) -> (2, 1) and (-ln 4, 2) -> (1/4, 3);
    # scores (common factor 1/2 dropped) 2 + 1/2 = 5/2 and 1/4 + 3/2 = 7/4;
    # values (1, 0), (0, 4):
    #   bidirectional: (5/2 (1, 0) + 7/4 (0, 4)) / (17/4) = (10/17, 28/17)
    #   causal rows: (1, 0); (10/17, 28/17)
    Om = np.eye(2)
    Q = np.array([[0.0, -math.log(2.0)]] * 2)
    K = np.array([[1.0, 0.0], [-math.log(4.0), 2.0]])
    V = np.array([[1.0, 0.0], [0.0, 4.0]])
    bi = orc.favor_bidirectional(Q, K, V, Om, 1.0, "elu1")
    assert np.allclose(bi, [[10 / 17, 28 / 17]] * 2, rtol=0, atol=1e-14)
    ca = orc.favor_causal(Q, K, V, Om, 1.0, "elu1")
    assert np.allclose(ca, [[1.0, 0.0], [10 / 17, 28 / 17]], rtol=0, atol=1e-14)


def test_map_and_slope_are_continuous_at_zero():
    Om = np.eye(1)
    for eps in (1e-7, 1e-9):
        lo = orc.elu1_features(np.array([[-eps]]), Om)[0, 0]
        hi = orc.elu1_features(np.array([[eps]]), Om)[0, 0]
        mid = orc.elu1_features(np.array([[0.0]]), Om)[0, 0]
        assert mid == 1.0
        assert abs(hi - lo) == pytest.approx(2 * eps, rel=1e-6)   # slope 1 on both sides
    # below 0 the map is e^x, above it 1 + x
    assert orc.elu1_features(np.array([[-3.0]]), Om)[0, 0] == pytest.approx(math.exp(-3.0), rel=1e-15)
    assert orc.elu1_features(np.array([[2.5]]), Om)[0, 0] == pytest.approx(3.5, rel=1e-15)


def test_features_are_positive_so_no_normaliser_vanishes():
    rng = np.random.default_rng(22)
    X = 30.0 * rng.standard_normal((200, 8))
    Om = rng.standard_normal((16, 8))
    assert np.all(orc.elu1_features(X, Om) > 0)
    Q, K, V = (rng.standard_normal((40, 8)) for _ in range(3))
    assert np.all(np.isfinite(orc.favor_causal(Q, K, V, Om, 2.0, "elu1")))


@pytest.mark.parametrize("causal", [False, True])
def test_orderings_agree(causal):
    rng = np.random.default_rng(23)
    Q, K, V = (rng.standard_normal((2, 3, 40, 16)) for _ in range(3))
    Om = rng.standard_normal((48, 16))
    s = 16 ** -0.25
    if causal:
        a = orc.favor_causal(Q, K, V, Om, s, "elu1")
        b = orc.favor_causal_quadratic(Q, K, V, Om, s, "elu1")
    else:
        a = orc.favor_bidirectional(Q, K, V, Om, s, "elu1")
        b = orc.favor_bidirectional_quadratic(Q, K, V, Om, s, "elu1")
    assert np.max(np.abs(a - b)) < 1e-12 * np.max(np.abs(b))


def test_causality_constant_values_and_scale_dependence():
    rng = np.random.default_rng(24)
    Q, K, V = (rng.standard_normal((30, 8)) for _ in range(3))
    Om = rng.standard_normal((64, 8))
    base = orc.favor_causal(Q, K, V, Om, 1.0, "elu1")
    K2, V2 = K.copy(), V.copy()
    K2[20:] += 3.0
    V2[20:] -= 7.0
    assert np.array_equal(base[:20], orc.favor_causal(Q, K2, V2, Om, 1.0, "elu1")[:20])
    c = np.full_like(V, -1.5)
    assert np.allclose(orc.favor_bidirectional(Q, K, c, Om, 1.0, "elu1"), -1.5, rtol=0, atol=1e-13)
    # unlike relu, 1 + elu is not homogeneous: the temperature matters
    a = orc.favor_bidirectional(Q, K, V, Om, 0.3, "elu1")
    b = orc.favor_bidirectional(Q, K, V, Om, 3.0, "elu1")
    assert np.max(np.abs(a - b)) > 1e-3

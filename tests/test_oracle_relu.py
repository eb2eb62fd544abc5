"""Pins of the oracle's Performer-ReLU feature map (CPU only).

The pages name the variant ("Rethinking Attention with Performers" summary,
§2 generalized kernelizable attention: other kernels by changing the
feature-map function; §3 applications and §D.2: Performer-ReLU) and print no
formula; the reading is phi(x) = m^-1/2 ReLU(Omega x).  What fixes the
oracle here, independently of its own code: an explicit loop, a hand-derived
example, positive homogeneity (the temperature cancels), and the identities
every linear attention satisfies.
"""

import math

import numpy as np
import pytest

import oracle as orc


def test_relu_features_match_an_explicit_loop():
    rng = np.random.default_rng(1)
    X = rng.standard_normal((3, 5))
    Om = rng.standard_normal((7, 5))
    got = orc.relu_features(X, Om)
    for t in range(3):
        for i in range(7):
            acc = 0.0
            for j in range(5):
                acc += Om[i, j] * X[t, j]
            want = (acc if acc > 0 else 0.0) / math.sqrt(7)
            assert got[t, i] == pytest.approx(want, rel=1e-14, abs=1e-15)


def test_hand_derived_example():
    # Omega = I (m = d = 2), s = 1: phi(x) = (max(x1, 0), max(x2, 0)) / sqrt(2).
    # q = (1, 2); keys (1, 0), (0, 1), (-1, 1) -> features (1, 0), (0, 1),
    # (0, 1) (the -1 is clamped); scores q.phi(k) (common factor 1/2 dropped)
    # 1, 2, 2.  Values (1, 0), (0, 1), (5, 5):
    #   bidirectional row: (1 (1,0) + 2 (0,1) + 2 (5,5)) / 5 = (2.2, 2.4)
    #   causal rows 0, 1, 2: (1, 0); ((1,0) + 2 (0,1)) / 3 = (1/3, 2/3); (2.2, 2.4)
    Om = np.eye(2)
    Q = np.array([[1.0, 2.0]] * 3)
    K = np.array([[1.0, 0.0], [0.0, 1.0], [-1.0, 1.0]])
    V = np.array([[1.0, 0.0], [0.0, 1.0], [5.0, 5.0]])
    bi = orc.favor_bidirectional(Q, K, V, Om, 1.0, "relu")
    assert np.allclose(bi, [[2.2, 2.4]] * 3, rtol=0, atol=1e-14)
    ca = orc.favor_causal(Q, K, V, Om, 1.0, "relu")
    assert np.allclose(ca, [[1.0, 0.0], [1 / 3, 2 / 3], [2.2, 2.4]], rtol=0, atol=1e-14)


def test_temperature_cancels():
    # ReLU is positively homogeneous: phi(c x) = c phi(x) for c > 0, so the
    # numerator and the normaliser scale alike
    rng = np.random.default_rng(2)
    Q, K, V = (rng.standard_normal((2, 24, 8)) for _ in range(3))
    Om = rng.standard_normal((32, 8))
    for causal in (False, True):
        fn = orc.favor_causal if causal else orc.favor_bidirectional
        a = fn(Q, K, V, Om, 0.3, "relu")
        b = fn(Q, K, V, Om, 3.0, "relu")
        assert np.max(np.abs(a - b)) < 1e-12 * np.max(np.abs(a))


@pytest.mark.parametrize("causal", [False, True])
def test_orderings_agree(causal):
    rng = np.random.default_rng(3)
    Q, K, V = (rng.standard_normal((2, 3, 40, 16)) for _ in range(3))
    Om = rng.standard_normal((48, 16))
    s = 16 ** -0.25
    if causal:
        a = orc.favor_causal(Q, K, V, Om, s, "relu")
        b = orc.favor_causal_quadratic(Q, K, V, Om, s, "relu")
    else:
        a = orc.favor_bidirectional(Q, K, V, Om, s, "relu")
        b = orc.favor_bidirectional_quadratic(Q, K, V, Om, s, "relu")
    assert np.max(np.abs(a - b)) < 1e-12 * np.max(np.abs(b))
    picks = [(h, t) for h in (0, 5) for t in (0, 17, 39)]
    rows = orc.favor_rows(Q.reshape(6, 40, 16), K.reshape(6, 40, 16), V.reshape(6, 40, 16), Om, s, picks, causal,
                          "relu")
    ref = np.stack([b.reshape(6, 40, 16)[h, t] for h, t in picks])
    assert np.max(np.abs(rows - ref)) < 1e-12 * np.max(np.abs(ref))


def test_causality_and_constant_values():
    rng = np.random.default_rng(4)
    Q, K, V = (rng.standard_normal((30, 8)) for _ in range(3))
    Om = rng.standard_normal((64, 8))
    base = orc.favor_causal(Q, K, V, Om, 1.0, "relu")
    K2, V2 = K.copy(), V.copy()
    K2[20:] += 3.0
    V2[20:] -= 7.0
    moved = orc.favor_causal(Q, K2, V2, Om, 1.0, "relu")
    assert np.array_equal(base[:20], moved[:20])
    c = np.full_like(V, 2.5)
    assert np.allclose(orc.favor_bidirectional(Q, K, c, Om, 1.0, "relu"), 2.5, rtol=0, atol=1e-13)


def test_features_are_nonnegative_and_zero_on_the_negative_side():
    rng = np.random.default_rng(5)
    X = rng.standard_normal((50, 6))
    Om = rng.standard_normal((20, 6))
    f = orc.relu_features(X, Om)
    proj = X @ Om.T
    assert np.all(f >= 0)
    assert np.all((f == 0) == (proj <= 0))

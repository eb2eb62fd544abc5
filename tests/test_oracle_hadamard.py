"""Pins of the oracle's Hadamard ORF builder (CPU only): the Walsh-Hadamard
matrix against its closed forms and defining identities, the signs against
the published SplitMix64 stream, exact orthogonality and row lengths of the
blocks, a hand-built d = 2 block, and the small bias of the softmax-kernel
estimator (the pages: "small bias tending to zero as d increases")."""

import math

import numpy as np
import pytest

import oracle as orc


def test_walsh_hadamard_closed_forms():
    assert np.allclose(orc.walsh_hadamard(2), np.array([[1, 1], [1, -1]]) / math.sqrt(2), rtol=0, atol=1e-15)
    H4 = np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]]) / 2.0
    assert np.allclose(orc.walsh_hadamard(4), H4, rtol=0, atol=1e-15)
    for d in (8, 16, 64, 128):
        H = orc.walsh_hadamard(d)
        assert np.allclose(H @ H.T, np.eye(d), rtol=0, atol=1e-12)
        # entry (i, j) = (-1)^popcount(i & j) / sqrt(d)
        i, j = np.meshgrid(np.arange(d), np.arange(d), indexing="ij")
        pc = np.vectorize(lambda x: bin(int(x)).count("1"))(i & j)
        assert np.allclose(H, (-1.0) ** pc / math.sqrt(d), rtol=0, atol=1e-15)
    with pytest.raises(ValueError):
        orc.walsh_hadamard(6)


def test_signs_follow_the_splitmix_stream():
    w = orc.splitmix64_stream(99, np.arange(40))
    want = np.where(w >= np.uint64(1 << 63), -1.0, 1.0)
    assert np.array_equal(orc.rademacher_signs(99, np.arange(40)), want)


def test_hand_built_d2_block():
    s = [orc.rademacher_signs(5, np.arange(2) + 2 * p) for p in range(3)]
    H = np.array([[1.0, 1.0], [1.0, -1.0]]) / math.sqrt(2)
    want = math.sqrt(2) * (H @ np.diag(s[0])) @ (H @ np.diag(s[1])) @ (H @ np.diag(s[2]))
    assert np.allclose(orc.build_omega_hadamard(5, 2, 2), want, rtol=0, atol=1e-15)


@pytest.mark.parametrize("m,d", [(64, 64), (256, 64), (100, 32), (512, 128)])
def test_blocks_are_orthogonal_with_rows_of_length_sqrt_d(m, d):
    Om = orc.build_omega_hadamard(3, m, d)
    assert Om.shape == (m, d)
    for b in range(0, m, d):
        blk = Om[b:b + d]
        assert np.allclose(blk @ blk.T, d * np.eye(blk.shape[0]), rtol=0, atol=1e-9)
    # independent blocks differ
    if m >= 2 * d:
        assert not np.allclose(Om[:d], Om[d:2 * d])


def test_estimator_bias_is_small():
    # mean over seeds of the PRF estimate of exp(x.y) with Hadamard Omega
    rng = np.random.default_rng(0)
    d = 64
    x = rng.standard_normal(d) * 0.15
    y = rng.standard_normal(d) * 0.15
    exact = math.exp(float(x @ y))
    est = [float(orc.prf_estimator(x, y, orc.build_omega_hadamard(seed, 64, d))) for seed in range(300)]
    assert abs(np.mean(est) / exact - 1.0) < 0.02

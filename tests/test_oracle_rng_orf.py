"""Pins for the oracle's random numbers and its Omega builder (CPU only).

Each test checks the oracle against something other than itself: published
generator outputs, a library QR, exact identities of the construction, or the
distributions the pages require (Gaussian marginals, orthogonal blocks).
"""

import math
import os

import numpy as np
import pytest
from scipy import stats

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_ints(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [int(x) for x in f.read().split("\n") if x.strip() and not x.startswith("#")]


def test_splitmix64_matches_published_outputs():
    want = _read_ints("splitmix64_seed1234567.txt")
    got = [int(x) for x in orc.splitmix64_stream(1234567, np.arange(5))]
    assert got == want


def test_splitmix64_counter_form_is_the_sequential_generator():
    # word i of a stream equals word 0 of the stream started i increments later
    seed = 0xDEADBEEF
    gam = orc.SPLITMIX_GAMMA
    for i in (0, 1, 7, 1000):
        later = (seed + i * gam) & 0xFFFFFFFFFFFFFFFF
        assert int(orc.splitmix64_stream(seed, [i])[0]) == int(orc.splitmix64_stream(later, [0])[0])


def test_box_muller_normals_are_standard_normal():
    z = orc.counter_normals(7, np.arange(200_000))
    assert abs(z.mean()) < 5 / math.sqrt(z.size)
    assert abs(z.var() - 1.0) < 5 * math.sqrt(2.0 / z.size)
    assert stats.kstest(z, "norm").pvalue > 1e-3


def test_box_muller_field_extraction():
    # word with k1 = 2**22 (u1 = (2**22 + .5) / 2**23) and k2 = 0 (u2 = .5 / 2**23)
    w = np.array([(1 << 63)], dtype=np.uint64)
    u1 = (2 ** 22 + 0.5) / 2 ** 23
    u2 = 0.5 / 2 ** 23
    want = math.sqrt(-2 * math.log(u1)) * math.cos(2 * math.pi * u2)
    assert orc.normals_from_words(w)[0] == pytest.approx(want, rel=1e-15)
    # k2 field taken from bits 18..40; bits below 18 are ignored
    w2 = np.array([(5 << 18) | 0x3FFFF], dtype=np.uint64)
    u1 = 0.5 / 2 ** 23
    u2 = 5.5 / 2 ** 23
    want2 = math.sqrt(-2 * math.log(u1)) * math.cos(2 * math.pi * u2)
    assert orc.normals_from_words(w2)[0] == pytest.approx(want2, rel=1e-15)
    # every u is exactly representable in fp32
    words = orc.splitmix64_stream(3, np.arange(1000))
    k = (words >> np.uint64(41)).astype(np.float64)
    u = (k + 0.5) / 2 ** 23
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)


@pytest.mark.parametrize("d", [4, 16, 64])
def test_gram_schmidt_equals_sign_fixed_library_qr(d):
    rng = np.random.default_rng(d)
    G = rng.standard_normal((d, d))
    Qgs = orc.gram_schmidt_rows(G)
    # rows of G = R^T Q^T with G^T = Q R; Gram–Schmidt gives diag(R) > 0
    q, r = np.linalg.qr(G.T)
    sgn = np.sign(np.diag(r))
    want = (q * sgn).T
    assert np.max(np.abs(Qgs - want)) < 1e-10


@pytest.mark.parametrize("m,d", [(64, 64), (256, 64), (128, 128), (96, 32), (8, 4), (5, 4)])
def test_orf_blocks_orthogonal_and_lengths_chi(m, d):
    Om, parts = orc.build_omega(3, m, d, orthogonal=True, return_parts=True)
    assert Om.shape == (m, d)
    nb = -(-m // d)
    for b in range(nb):
        rows = Om[b * d: min((b + 1) * d, m)]
        G, Qb, lengths = parts[b]
        n = rows.shape[0]
        # row r of the block has length = norm of its independent chi vector
        assert np.allclose(np.linalg.norm(rows, axis=1), lengths[:n], rtol=1e-12)
        # rows of one block are mutually orthogonal
        gram = rows @ rows.T
        off = gram - np.diag(np.diag(gram))
        assert np.max(np.abs(off)) < 1e-9 * np.max(np.diag(gram))
        # directions are the Gram–Schmidt directions of the Gaussian block
        assert np.allclose(rows / lengths[:n, None], Qb[:n], atol=1e-12)


def test_orf_uses_documented_counters():
    d, seed = 4, 11
    Om, parts = orc.build_omega(seed, 8, d, orthogonal=True, return_parts=True)
    for b in range(2):
        G, _, lengths = parts[b]
        for r in range(d):
            for c in range(d):
                idx = orc.orf_index_layout(b, r, c, d, 0)
                assert G[r, c] == orc.counter_normals(seed, [idx])[0]
        chi = np.array([[orc.counter_normals(seed, [orc.orf_index_layout(b, r, c, d, 1)])[0]
                         for c in range(d)] for r in range(d)])
        assert np.allclose(lengths, np.linalg.norm(chi, axis=1), rtol=1e-15)


def test_iid_omega_counters():
    d, m, seed = 8, 5, 2
    Om = orc.build_omega(seed, m, d, orthogonal=False)
    for i in range(m):
        for c in range(d):
            assert Om[i, c] == orc.counter_normals(seed, [(i * d + c) * 2])[0]


def test_orf_marginals_are_gaussian():
    # Orthogonalisation keeps each row N(0, I_d) (pages: marginals preserved).
    d = 16
    rows = np.concatenate([orc.build_omega(s, d, d) for s in range(400)], axis=0)
    # entries of a row ~ N(0, 1)
    assert stats.kstest(rows[:, 0], "norm").pvalue > 1e-3
    assert stats.kstest(rows[::d].ravel(), "norm").pvalue > 1e-3
    # row lengths ~ chi_d
    lens = np.linalg.norm(rows, axis=1)
    assert stats.kstest(lens, stats.chi(d).cdf).pvalue > 1e-3


def test_golden_orf_small():
    # regression pin written by tests/golden/make_golden.py (oracle only)
    path = os.path.join(GOLDEN, "omega_seed0_m8_d4.txt")
    want = np.loadtxt(path)
    got = orc.build_omega(0, 8, 4, orthogonal=True)
    assert np.allclose(got, want, rtol=0, atol=1e-15)

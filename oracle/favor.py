"""fp64 NumPy oracle for FAVOR+ (positive orthogonal random features).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module; it shares no code with the CUDA library and imports nothing from it.

Sources (web pages on "Rethinking Attention with Performers"):
  [digest]  "Performer — Rethinking Attention with Performers" (Korean blog
            digest): §Methods (FAVOR+), §Theoretical bounds, §Key equations
            (핵심 수식), §Method / key components (핵심 구성요소), flowchart.
  [su]      "From Performer to Linear Attention" (Su Jianlin): §Simple
            Derivation (the scale-invariance argument).
  [summary] "Rethinking Attention with Performers" (arXiv:2009.14794v4
            section summary): §2 FAVOR+ mechanism, §3 theoretical results,
            §A.2 unidirectional attention, §B.3 complexity.

Readings where the pages are silent (each also listed in the design notes):
  * A temperature ``scale`` multiplies q and k before the feature map
    (x' = scale * x).  The pages write softmax(QK^T) with no temperature;
    scale = d**-0.25 gives the usual exp(q.k / sqrt(d)).
  * No stabiliser and no epsilon: in fp64 every exponent here is far inside
    the exp range, so the estimator is evaluated literally.
  * The random numbers: a counter-based SplitMix64 (Steele, Lea & Flood,
    "Fast splittable pseudorandom number generators", OOPSLA 2014) turned into
    normals by the Box–Muller transform (cosine branch).  The pages fix no RNG.
  * ORF rows: Gram–Schmidt on the rows of independent d x d Gaussian blocks,
    each row then given the length of an independent N(0, I_d) vector (a chi_d
    sample) so that every row keeps the N(0, I_d) marginal; the first m rows of
    the stacked blocks form Omega.

Parity pins for every function live in ``tests/test_oracle_*.py``.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "SPLITMIX_GAMMA",
    "splitmix64_stream",
    "normals_from_words",
    "counter_normals",
    "gram_schmidt_rows",
    "build_omega",
    "orf_index_layout",
    "walsh_hadamard",
    "rademacher_signs",
    "build_omega_hadamard",
    "givens_rotation_count",
    "givens_rotations",
    "build_omega_givens",
    "prf_features",
    "relu_features",
    "elu1_features",
    "FEATURES",
    "trig_features",
    "softmax_kernel",
    "prf_estimator",
    "lemma2_mse",
    "favor_bidirectional",
    "favor_bidirectional_quadratic",
    "favor_causal",
    "favor_causal_quadratic",
    "favor_rows",
    "favor_bidirectional_grad",
    "favor_causal_grad",
    "softmax_attention",
    "rowwise_rel_err",
]

# --------------------------------------------------------------------------
# Random numbers (not on the pages; published generator definitions)
# --------------------------------------------------------------------------

SPLITMIX_GAMMA = 0x9E3779B97F4A7C15
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (variant 13 of Stafford's mixer)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_stream(seed: int, counters) -> np.ndarray:
    """Word number ``i`` of the SplitMix64 sequence started at ``seed``.

    The sequential generator adds the golden-ratio increment to its state and
    then mixes; word i is therefore mix(seed + (i + 1) * gamma) mod 2**64,
    which makes the generator counter-based.
    """
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (c + np.uint64(1)) * np.uint64(SPLITMIX_GAMMA)
        return _mix64(state)


def normals_from_words(words: np.ndarray) -> np.ndarray:
    """One standard normal per 64-bit word by the Box–Muller transform.

    Two 23-bit fields of the word (bits 41..63 and 18..40) give
    u1, u2 = (k + 1/2) / 2**23 in (0, 1) -- (2k + 1) / 2**24 has at most 24
    significant bits, so the same u is exact in fp32 -- and
    z = sqrt(-2 ln u1) cos(2 pi u2).
    """
    w = np.asarray(words, dtype=np.uint64)
    k1 = (w >> np.uint64(41)).astype(np.float64)
    k2 = ((w >> np.uint64(18)) & np.uint64(0x7FFFFF)).astype(np.float64)
    u1 = (k1 + 0.5) / 8388608.0
    u2 = (k2 + 0.5) / 8388608.0
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def counter_normals(seed: int, counters) -> np.ndarray:
    return normals_from_words(splitmix64_stream(seed, counters))


def orf_index_layout(block: int, row: int, col: int, d: int, kind: int) -> int:
    """Counter of one normal used by :func:`build_omega`.

    kind 0 = entry (row, col) of Gaussian block ``block``; kind 1 = component
    ``col`` of the chi_d length vector of that block's row ``row``.
    """
    return ((block * d + row) * d + col) * 2 + kind


# --------------------------------------------------------------------------
# Omega (the projection): ORF and iid  —  [digest] §Methods (ORF bullet),
# [digest] Zettelkasten "orthogonality strictly reduces variance" (block-wise
# orthogonalisation when m > d), [summary] §A.2 (marginals preserved).
# --------------------------------------------------------------------------


def gram_schmidt_rows(G: np.ndarray) -> np.ndarray:
    """Orthonormalise the rows of ``G`` in order by Gram–Schmidt (fp64).

    Row i loses its components along the already orthonormal rows 0..i-1 (one
    at a time, the modified form), then is divided by its length.
    """
    G = np.asarray(G, dtype=np.float64)
    n = G.shape[0]
    Qm = np.zeros_like(G)
    for i in range(n):
        v = G[i].copy()
        for j in range(i):
            v -= np.dot(Qm[j], v) * Qm[j]
        Qm[i] = v / np.linalg.norm(v)
    return Qm


def build_omega(seed: int, m: int, d: int, orthogonal: bool = True,
                return_parts: bool = False):
    """Projection matrix Omega, shape [m, d], row i = omega_i.

    orthogonal=True: ceil(m/d) independent d x d Gaussian blocks, rows of each
    orthonormalised by Gram–Schmidt, row r of block b rescaled to the length
    of the independent Gaussian vector (kind 1 counters); the first m rows of
    the stacked blocks are kept.  orthogonal=False: iid N(0, 1) entries
    (counter of entry (i, c) = (i*d + c)*2).
    """
    if orthogonal:
        nb = -(-m // d)
        rows = []
        parts = []
        r = np.arange(d)[:, None]
        c = np.arange(d)[None, :]
        for b in range(nb):
            g_idx = ((b * d + r) * d + c) * 2
            G = counter_normals(seed, g_idx)
            chi = counter_normals(seed, g_idx + 1)
            lengths = np.sqrt(np.sum(chi * chi, axis=1))
            Qb = gram_schmidt_rows(G)
            rows.append(Qb * lengths[:, None])
            parts.append((G, Qb, lengths))
        Omega = np.concatenate(rows, axis=0)[:m]
        return (Omega, parts) if return_parts else Omega
    i = np.arange(m)[:, None]
    c = np.arange(d)[None, :]
    Omega = counter_normals(seed, (i * d + c) * 2)
    return (Omega, None) if return_parts else Omega


def walsh_hadamard(d: int) -> np.ndarray:
    """The normalised d x d Walsh-Hadamard matrix (Sylvester's doubling,
    H_1 = [1], H_2k = [[H_k, H_k], [H_k, -H_k]], divided by sqrt(d));
    d must be a power of two."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H / math.sqrt(d)


def rademacher_signs(seed: int, counters) -> np.ndarray:
    """+1 or -1 from the top bit of SplitMix64 word ``counters`` (1 -> -1)."""
    w = splitmix64_stream(seed, counters)
    return np.where((w >> np.uint64(63)) == np.uint64(1), -1.0, 1.0)


def build_omega_hadamard(seed: int, m: int, d: int) -> np.ndarray:
    """Hadamard ORF projection, [m, d].

    [summary] §A.2 (FAVOR+ bullet) and §B.3 name Hadamard ORFs (O(m) space,
    a small bias that tends to zero as d grows) without printing a
    construction; the reading: block b = sqrt(d) (H D_1)(H D_2)(H D_3) with H
    the normalised Walsh-Hadamard matrix and D_p = diag(+-1), sign i of
    product p of block b from SplitMix64 word (b*3 + p)*d + i (its top bit).
    Each block is exactly orthogonal with rows of length sqrt(d) (not a chi_d
    draw: hence the bias).  The first m rows of the stacked blocks are kept.
    """
    H = walsh_hadamard(d)
    blocks = []
    for b in range(-(-m // d)):
        M = np.eye(d)
        for p in range(3):
            D = rademacher_signs(seed, (b * 3 + p) * d + np.arange(d))
            M = M @ (H * D[None, :])          # (H D_p): column i of H times sign i
        blocks.append(math.sqrt(d) * M)
    return np.concatenate(blocks, axis=0)[:m]


def givens_rotation_count(d: int) -> int:
    """Rotations per d x d Givens block: 3 d ceil(log2 d).  Over ceil(m/d)
    blocks that is the O(m log d) numbers the pages give for Givens ORFs; the
    factor 3 is the smallest for which the rows' fourth moment reaches that
    of rows uniform on the sphere of radius sqrt(d) (at d = 64: 5.4 with
    factor 1, 3.03 with 2, 2.91 with 3, against 3d / (d + 2) = 2.91)."""
    if d < 2:
        raise ValueError("a Givens rotation needs d >= 2")
    return 3 * d * (d - 1).bit_length()


def givens_rotations(seed: int, block: int, d: int):
    """(i, j, theta) of each rotation of ``block``, in the order applied.

    Rotation r of block b reads SplitMix64 words 2c and 2c + 1, c = b*K + r
    (K rotations per block).  From the first word w0: i = floor(hi32(w0) d /
    2^32) and j' = floor(lo32(w0) (d - 1) / 2^32), j = j' + [j' >= i] (a
    uniform ordered pair, i != j).  From the second word w1: theta =
    2 pi (k + 1/2) / 2^23 with k its top 23 bits (uniform on (0, 2 pi)).
    """
    K = givens_rotation_count(d)
    c = (np.uint64(block) * np.uint64(K) + np.arange(K, dtype=np.uint64)) * np.uint64(2)
    w0 = splitmix64_stream(seed, c)
    w1 = splitmix64_stream(seed, c + np.uint64(1))
    hi = (w0 >> np.uint64(32)).astype(np.float64)
    lo = (w0 & np.uint64(0xFFFFFFFF)).astype(np.float64)
    i = np.floor(hi * d / 4294967296.0).astype(np.int64)
    jp = np.floor(lo * (d - 1) / 4294967296.0).astype(np.int64)
    j = jp + (jp >= i)
    k = (w1 >> np.uint64(41)).astype(np.float64)
    theta = 2.0 * math.pi * (k + 0.5) / 8388608.0
    return list(zip(i.tolist(), j.tolist(), theta.tolist()))


def build_omega_givens(seed: int, m: int, d: int) -> np.ndarray:
    """Givens ORF projection, [m, d].

    [summary] §A.2 (FAVOR+ bullet) and §B.3 name Givens ORFs (small bias
    tending to zero with d; O(m log d) space) without a construction; the
    reading: block b = sqrt(d) G_K ... G_2 G_1 with G_r the rotation by
    theta_r in the plane of coordinates (i_r, j_r) -- (G x)_i = cos x_i -
    sin x_j, (G x)_j = sin x_i + cos x_j -- drawn by ``givens_rotations``.
    Each block is exactly orthogonal with rows of length sqrt(d) (as the
    Hadamard reading; hence the bias).  The first m stacked rows are kept.
    """
    blocks = []
    for b in range(-(-m // d)):
        M = np.eye(d)
        for i, j, th in givens_rotations(seed, b, d):
            G = np.eye(d)
            G[i, i] = math.cos(th)
            G[i, j] = -math.sin(th)
            G[j, i] = math.sin(th)
            G[j, j] = math.cos(th)
            M = G @ M
        blocks.append(math.sqrt(d) * M)
    return np.concatenate(blocks, axis=0)[:m]


# --------------------------------------------------------------------------
# Feature maps and the softmax-kernel estimator — [digest] §Key equations,
# [digest] §Methods (softmax-kernel decomposition, PRF), [su] §Simple
# Derivation (the m-dimensional vectors q~, k~).
# --------------------------------------------------------------------------


def softmax_kernel(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """SM(x, y) = exp(x^T y) over the last axis."""
    return np.exp(np.sum(np.asarray(x, np.float64) * np.asarray(y, np.float64), axis=-1))


def prf_features(X: np.ndarray, Omega: np.ndarray) -> np.ndarray:
    """Positive random features phi(x) = m^{-1/2} exp(Omega x - ||x||^2 / 2).

    X [..., L, d] (already multiplied by the temperature), Omega [m, d].
    Returns [..., L, m].
    """
    X = np.asarray(X, dtype=np.float64)
    Om = np.asarray(Omega, dtype=np.float64)
    m = Om.shape[0]
    proj = X @ Om.T
    half_sq = 0.5 * np.sum(X * X, axis=-1, keepdims=True)
    return np.exp(proj - half_sq) / math.sqrt(m)


def relu_features(X: np.ndarray, Omega: np.ndarray) -> np.ndarray:
    """Performer-ReLU features phi(x) = m^{-1/2} ReLU(Omega x), elementwise.

    [summary] §2, "Generalized kernelizable attention": FAVOR+ covers other
    kernels by changing the feature-map function applied to the random
    projections; [summary] §3 applications and §D.2 name the Performer-ReLU
    variant.  The pages print no formula: the plainest reading is
    f(w_i^T x) with f = ReLU, the same projection Omega and no ||x||^2 term
    (it belongs to the softmax kernel only).  X [..., L, d] (already times the
    temperature), Omega [m, d]; returns [..., L, m].
    """
    X = np.asarray(X, dtype=np.float64)
    Om = np.asarray(Omega, dtype=np.float64)
    return np.maximum(X @ Om.T, 0.0) / math.sqrt(Om.shape[0])


def elu1_features(X: np.ndarray, Omega: np.ndarray) -> np.ndarray:
    """Linear-attention features phi(x) = m^{-1/2} (1 + elu(Omega x)).

    [su] (the linear-attention choice it compares against): phi(x) = 1 +
    elu(x), i.e. 1 + x for x >= 0 and exp(x) for x < 0, the first-order
    Taylor form of exp near 0; [digest] §Related work names it as the feature
    map of Linear Attention (Katharopoulos 2020).  Read as the same
    feature-map slot as Performer-ReLU, f(w_i^T x) with f = 1 + elu: with
    Omega = I_d (m = d) it is that linear attention itself.  X [..., L, d]
    (already times the temperature), Omega [m, d]; returns [..., L, m].
    """
    X = np.asarray(X, dtype=np.float64)
    Om = np.asarray(Omega, dtype=np.float64)
    a = X @ Om.T
    return np.where(a >= 0.0, 1.0 + a, np.exp(np.minimum(a, 0.0))) / math.sqrt(Om.shape[0])


FEATURES = {"prf": prf_features, "relu": relu_features, "elu1": elu1_features}


def trig_features(X: np.ndarray, Omega: np.ndarray) -> np.ndarray:
    """Trigonometric (sin/cos) random features for the softmax kernel.

    SM(x, y) = exp(||x||^2/2) exp(||y||^2/2) exp(-||x-y||^2/2) and the last
    factor is E[cos(omega^T (x - y))]; so phi(x) = m^{-1/2} exp(||x||^2/2)
    [sin(Omega x), cos(Omega x)] gives an unbiased estimator that can take
    negative values ([digest] §Methods "why positive"; [summary] §2).
    """
    X = np.asarray(X, dtype=np.float64)
    Om = np.asarray(Omega, dtype=np.float64)
    m = Om.shape[0]
    proj = X @ Om.T
    amp = np.exp(0.5 * np.sum(X * X, axis=-1, keepdims=True)) / math.sqrt(m)
    return np.concatenate([amp * np.sin(proj), amp * np.cos(proj)], axis=-1)


def prf_estimator(x: np.ndarray, y: np.ndarray, Omega: np.ndarray) -> np.ndarray:
    """SM^_m^PRF(x, y) = (1/m) sum_i exp(w_i.x - |x|^2/2) exp(w_i.y - |y|^2/2)."""
    return np.sum(prf_features(x, Omega) * prf_features(y, Omega), axis=-1)


def lemma2_mse(x: np.ndarray, y: np.ndarray, m: int) -> float:
    """Lemma 2: MSE = (1/m) exp(|x+y|^2) SM(x,y)^2 (1 - exp(-|x+y|^2))."""
    s2 = float(np.sum((np.asarray(x) + np.asarray(y)) ** 2))
    sm = float(softmax_kernel(x, y))
    return math.exp(s2) * sm * sm * (1.0 - math.exp(-s2)) / m


# --------------------------------------------------------------------------
# Attention — [digest] §Key equations (Attn^ = D^-1 phi(Q)(phi(K)^T V),
# D = diag(phi(Q) phi(K)^T 1_L)), [digest] flowchart, [digest] §Methods
# (causal prefix sum G_t), [summary] §2 (lower-triangular part), §A.2.
# --------------------------------------------------------------------------


def _features_qk(Q, K, Omega, scale, features="prf"):
    q = scale * np.asarray(Q, dtype=np.float64)
    k = scale * np.asarray(K, dtype=np.float64)
    fn = FEATURES[features]
    return fn(q, Omega), fn(k, Omega)


def favor_bidirectional(Q, K, V, Omega, scale: float, features: str = "prf") -> np.ndarray:
    """Bidirectional FAVOR+: D^{-1} phi(Q) (phi(K)^T V), linear order.

    Q, K, V [..., L, d]; returns [..., L, d] in fp64.  ``features`` is "prf"
    (positive random features, the softmax kernel) or "relu".
    """
    pq, pk = _features_qk(Q, K, Omega, scale, features)
    V = np.asarray(V, dtype=np.float64)
    kv = np.swapaxes(pk, -1, -2) @ V              # [..., m, d]  phi(K)^T V
    z = np.sum(pk, axis=-2)                       # [..., m]     phi(K)^T 1_L
    num = pq @ kv                                 # [..., L, d]
    den = np.einsum("...lm,...m->...l", pq, z)    # [..., L]     diag of D
    return num / den[..., None]


def favor_bidirectional_quadratic(Q, K, V, Omega, scale: float, features: str = "prf") -> np.ndarray:
    """Same estimator in quadratic order: row-normalise phi(Q) phi(K)^T, times V."""
    pq, pk = _features_qk(Q, K, Omega, scale, features)
    A = pq @ np.swapaxes(pk, -1, -2)              # [..., L, L]
    A = A / np.sum(A, axis=-1, keepdims=True)
    return A @ np.asarray(V, dtype=np.float64)


def favor_causal(Q, K, V, Omega, scale: float, features: str = "prf") -> np.ndarray:
    """Unidirectional FAVOR+ by the prefix sum of the pages.

    G_t = sum_{s<=t} phi(k_s) v_s^T and z_t = sum_{s<=t} phi(k_s) are carried
    forward one token at a time; out_t = phi(q_t)^T G_t / phi(q_t)^T z_t.
    """
    pq, pk = _features_qk(Q, K, Omega, scale, features)
    V = np.asarray(V, dtype=np.float64)
    lead = V.shape[:-2]
    L, d = V.shape[-2:]
    m = pk.shape[-1]
    G = np.zeros(lead + (m, d))
    z = np.zeros(lead + (m,))
    out = np.empty(lead + (L, d))
    for t in range(L):
        G += pk[..., t, :, None] * V[..., t, None, :]
        z += pk[..., t, :]
        num = np.einsum("...m,...md->...d", pq[..., t, :], G)
        den = np.einsum("...m,...m->...", pq[..., t, :], z)
        out[..., t, :] = num / den[..., None]
    return out


def favor_causal_quadratic(Q, K, V, Omega, scale: float, features: str = "prf") -> np.ndarray:
    """Unidirectional FAVOR+ as the lower-triangular part (diagonal included)
    of phi(Q) phi(K)^T, row-normalised, times V."""
    pq, pk = _features_qk(Q, K, Omega, scale, features)
    A = pq @ np.swapaxes(pk, -1, -2)
    L = A.shape[-1]
    A = A * np.tril(np.ones((L, L)))
    A = A / np.sum(A, axis=-1, keepdims=True)
    return A @ np.asarray(V, dtype=np.float64)


def favor_rows(Q, K, V, Omega, scale: float, bh_rows, causal: bool, features: str = "prf") -> np.ndarray:
    """Selected output rows of the estimator, for large inputs.

    Q, K, V [BH, L, d]; ``bh_rows`` is a list of (head index, t).  Row t of
    head h is sum_{s in S} (phi(q_t).phi(k_s)) v_s / sum_{s in S} phi(q_t).phi(k_s)
    with S = all tokens (bidirectional) or s <= t (causal).  phi(K)^T V over S
    is evaluated as one matrix product per head and range.
    """
    bh_rows = list(bh_rows)
    out = np.empty((len(bh_rows), np.asarray(V).shape[-1]))
    by_head: dict[int, list[tuple[int, int]]] = {}
    for n, (h, t) in enumerate(bh_rows):
        by_head.setdefault(int(h), []).append((int(t), n))
    for h, items in by_head.items():
        k = scale * np.asarray(K[h], dtype=np.float64)
        v = np.asarray(V[h], dtype=np.float64)
        fn = FEATURES[features]
        pk = fn(k, Omega)
        if not causal:
            kv = pk.T @ v
            z = pk.sum(axis=0)
        for t, n in items:
            q = scale * np.asarray(Q[h][t], dtype=np.float64)
            pq = fn(q[None, :], Omega)[0]
            if causal:
                kv = pk[: t + 1].T @ v[: t + 1]
                z = pk[: t + 1].sum(axis=0)
            out[n] = (pq @ kv) / (pq @ z)
    return out


def _map_slope(features: str, a: np.ndarray) -> np.ndarray:
    """f'(a) of the projected feature maps f(a) (relu, 1 + elu)."""
    if features == "relu":
        return (a > 0).astype(np.float64)
    return np.where(a >= 0.0, 1.0, np.exp(np.minimum(a, 0.0)))


def favor_bidirectional_grad(Q, K, V, Omega, scale: float, dO, features: str = "prf"):
    """Gradients (dQ, dK, dV) of sum(dO * favor_bidirectional(Q, K, V)).

    The chain rule through the forward of [digest] §Key equations, step by
    step (Q, K, V [..., L, d], dO like the output; fp64):
      N = phi(Q) S,  S = phi(K)^T V,  D = phi(Q) z,  z = phi(K)^T 1,  O = N / D
      dN = dO / D,   dD = -sum_j(dO O) / D
      dphi(Q) = dN S^T + dD z^T
      dS = phi(Q)^T dN,  dz = phi(Q)^T dD
      dphi(K) = V dS^T + 1 dz^T,  dV = phi(K) dS
    and through the feature map x' = scale x, phi = f(Omega x' ...):
      prf:  d phi_i / d x' = phi_i (w_i - x')
      relu: d phi_i / d x' = m^-1/2 w_i [w_i . x' > 0]
      elu1: d phi_i / d x' = m^-1/2 w_i (1 if w_i . x' >= 0 else exp(w_i . x'))
    then dx = scale dx'.
    """
    Q, K, V, dO = (np.asarray(a, dtype=np.float64) for a in (Q, K, V, dO))
    Om = np.asarray(Omega, dtype=np.float64)
    qs, ks = scale * Q, scale * K
    fn = FEATURES[features]
    pq, pk = fn(qs, Om), fn(ks, Om)
    S = np.swapaxes(pk, -1, -2) @ V                  # [..., m, d]
    z = np.sum(pk, axis=-2)                          # [..., m]
    N = pq @ S                                       # [..., L, d]
    D = np.einsum("...lm,...m->...l", pq, z)         # [..., L]
    O = N / D[..., None]
    dN = dO / D[..., None]
    dD = -np.sum(dO * O, axis=-1) / D
    dpq = dN @ np.swapaxes(S, -1, -2) + dD[..., None] * z[..., None, :]
    dS = np.swapaxes(pq, -1, -2) @ dN
    dz = np.einsum("...lm,...l->...m", pq, dD)
    dpk = V @ np.swapaxes(dS, -1, -2) + dz[..., None, :]
    dV = pk @ dS

    def through_features(x, phi, dphi):
        if features == "prf":
            # sum_i dphi_i phi_i (w_i - x)
            g = dphi * phi
            return g @ Om - x * np.sum(g, axis=-1, keepdims=True)
        return ((dphi * _map_slope(features, x @ Om.T)) @ Om) / math.sqrt(Om.shape[0])

    dQ = scale * through_features(qs, pq, dpq)
    dK = scale * through_features(ks, pk, dpk)
    return dQ, dK, dV


def favor_causal_grad(Q, K, V, Omega, scale: float, dO, features: str = "prf"):
    """Gradients (dQ, dK, dV) of sum(dO * favor_causal(Q, K, V)).

    The chain rule through the prefix-sum forward ([digest] §Methods causal
    bullet), written on the lower-triangular form it equals
    (A = tril(phi(Q) phi(K)^T), diagonal included):
      N = A V,  D = A 1,  O = N / D;  dN = dO / D,  dD = -sum_j(dO O) / D
      dA = tril(dN V^T + dD 1^T)
      dphi(Q) = dA phi(K),  dphi(K) = dA^T phi(Q),  dV = A^T dN
    then through the feature map as in favor_bidirectional_grad.
    """
    Q, K, V, dO = (np.asarray(a, dtype=np.float64) for a in (Q, K, V, dO))
    Om = np.asarray(Omega, dtype=np.float64)
    qs, ks = scale * Q, scale * K
    fn = FEATURES[features]
    pq, pk = fn(qs, Om), fn(ks, Om)
    L = Q.shape[-2]
    mask = np.tril(np.ones((L, L)))
    A = (pq @ np.swapaxes(pk, -1, -2)) * mask
    N = A @ V
    D = np.sum(A, axis=-1)
    O = N / D[..., None]
    dN = dO / D[..., None]
    dD = -np.sum(dO * O, axis=-1) / D
    dA = (dN @ np.swapaxes(V, -1, -2) + dD[..., None]) * mask
    dpq = dA @ pk
    dpk = np.swapaxes(dA, -1, -2) @ pq
    dV = np.swapaxes(A, -1, -2) @ dN

    def through_features(x, phi, dphi):
        if features == "prf":
            g = dphi * phi
            return g @ Om - x * np.sum(g, axis=-1, keepdims=True)
        return ((dphi * _map_slope(features, x @ Om.T)) @ Om) / math.sqrt(Om.shape[0])

    return scale * through_features(qs, pq, dpq), scale * through_features(ks, pk, dpk), dV


def softmax_attention(Q, K, V, scale: float, causal: bool = False) -> np.ndarray:
    """Exact softmax((scale Q)(scale K)^T) V, the quantity FAVOR+ estimates."""
    q = scale * np.asarray(Q, dtype=np.float64)
    k = scale * np.asarray(K, dtype=np.float64)
    S = q @ np.swapaxes(k, -1, -2)
    if causal:
        L = S.shape[-1]
        S = np.where(np.tril(np.ones((L, L), dtype=bool)), S, -np.inf)
    S = S - np.max(S, axis=-1, keepdims=True)
    P = np.exp(S)
    P = P / np.sum(P, axis=-1, keepdims=True)
    return P @ np.asarray(V, dtype=np.float64)


def rowwise_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of max_j |got - ref| / max_j |ref| (normwise per row)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.max(np.abs(got - ref), axis=-1)
    den = np.max(np.abs(ref), axis=-1)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(num / den))

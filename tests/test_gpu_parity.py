"""GPU parity: the CUDA library against the fp64 oracle, element by element.

Inputs come from ``workloads`` (seeded), the projection Omega is the one the
library built (copied back), and the oracle evaluates the literal FAVOR+
estimator in fp64.  Error metric: max over rows of max_j |gpu - oracle| /
max_j |oracle|; bars 1e-4 (fp32 storage) and 2e-2 (bf16 storage).
"""

import math

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from helpers import TOL, sample_rows, to_np

pytestmark = pytest.mark.gpu


def _run(favor, causal, Q, K, V, om, scale, status=None):
    B, H, L, d = Q.shape
    ws = favor.new_workspace(causal, B, H, L, d, om.shape[0], Q.dtype)
    fn = favor.fwd_causal if causal else favor.fwd_bidir
    return fn(Q, K, V, om, scale, ws, dev_status=status)


def _status(device="cuda"):
    return torch.zeros(1, dtype=torch.int32, device=device)


# ---------------------------------------------------------------------------
# a0: the projection
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed,m,d", [(0, 64, 64), (1, 256, 64), (7, 128, 128), (3, 512, 128), (5, 96, 32),
                                      (9, 5, 4), (11, 200, 100),
                                      # odd panel counts (helper pairing, barrier counts), a ragged
                                      # last part, and blocks with fewer rows than drawing CTAs
                                      (13, 30, 13), (17, 120, 40), (19, 150, 72), (23, 3, 1), (29, 5, 2)])
def test_orf_matches_oracle(cuda_lib, seed, m, d):
    om = to_np(cuda_lib.new_omega(seed, m, d))
    want, parts = orc.build_omega(seed, m, d, return_parts=True)
    for b, (G, _, lengths) in enumerate(parts):
        rows = slice(b * d, min((b + 1) * d, m))
        got, ref = om[rows], want[rows]
        # fp32 Box–Muller (a few ulp) and fp32 Gram–Schmidt: the error of a QR
        # factor grows with the condition number of the Gaussian block.
        kappa = np.linalg.cond(G)
        tol = 64 * kappa * 2.0 ** -23 * max(1.0, float(np.max(np.abs(ref))))
        assert np.max(np.abs(got - ref)) < tol, (b, np.max(np.abs(got - ref)), tol, kappa)
        # exact structure: lengths and orthogonality
        assert np.allclose(np.linalg.norm(got, axis=1), lengths[: got.shape[0]], rtol=2e-6)
        dirs = got / np.linalg.norm(got, axis=1, keepdims=True)
        assert np.max(np.abs(dirs @ dirs.T - np.eye(dirs.shape[0]))) < 2e-6


@pytest.mark.parametrize("seed,m,d", [(0, 64, 64), (1, 256, 64), (2, 512, 128), (3, 100, 32), (4, 3, 2)])
def test_hadamard_omega_matches_oracle(cuda_lib, seed, m, d):
    om = torch.empty((m, d), dtype=torch.float32, device="cuda")
    cuda_lib.build_orf(seed, om, orthogonal="hadamard")
    got, want = to_np(om), orc.build_omega_hadamard(seed, m, d)
    assert np.max(np.abs(got - want)) < 1e-5 * np.max(np.abs(want))
    for b in range(0, m, d):
        blk = got[b:b + d]
        assert np.max(np.abs(blk @ blk.T - d * np.eye(blk.shape[0]))) < 1e-4 * d


def test_hadamard_omega_in_attention(cuda_lib):
    # a Hadamard projection runs through the same kernels as any other Omega
    w = wl.Workload("had", "bidir", "bf16", 1, 2, 500, 64, 256, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=6))
    om = torch.empty((w.m, w.d), dtype=torch.float32, device="cuda")
    cuda_lib.build_orf(6, om, orthogonal="hadamard")
    O = _run(cuda_lib, False, Q, K, V, om, w.qk_scale)
    ref = orc.favor_bidirectional(to_np(Q), to_np(K), to_np(V), to_np(om), w.qk_scale)
    assert orc.rowwise_rel_err(to_np(O), ref) < TOL[torch.bfloat16]


@pytest.mark.parametrize("seed,m,d", [(0, 64, 64), (7, 256, 64), (3, 100, 32), (9, 200, 48), (2, 256, 128),
                                     (5, 6, 2), (1, 50, 3)])
def test_givens_omega_matches_oracle(cuda_lib, seed, m, d):
    om = torch.empty((m, d), dtype=torch.float32, device="cuda")
    cuda_lib.build_orf(seed, om, orthogonal="givens")
    got, want = to_np(om), orc.build_omega_givens(seed, m, d)
    # fp32 rotations, 3 d ceil(log2 d) of them: rounding grows like their square root
    assert np.max(np.abs(got - want)) < 1e-4 * np.max(np.abs(want))
    for b in range(0, m, d):
        blk = got[b:b + d]
        assert np.max(np.abs(blk @ blk.T - d * np.eye(blk.shape[0]))) < 1e-4 * d


def test_givens_omega_in_attention(cuda_lib):
    w = wl.Workload("giv", "causal", "bf16", 1, 2, 500, 64, 256, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=8))
    om = torch.empty((w.m, w.d), dtype=torch.float32, device="cuda")
    cuda_lib.build_orf(8, om, orthogonal="givens")
    O = _run(cuda_lib, True, Q, K, V, om, w.qk_scale)
    ref = orc.favor_causal(to_np(Q), to_np(K), to_np(V), to_np(om), w.qk_scale)
    assert orc.rowwise_rel_err(to_np(O), ref) < TOL[torch.bfloat16]


def test_iid_omega_matches_oracle(cuda_lib):
    om = to_np(cuda_lib.new_omega(4, 300, 70, orthogonal=False))
    want = orc.build_omega(4, 300, 70, orthogonal=False)
    assert np.max(np.abs(om - want)) < 1e-5 * np.max(np.abs(want))


def test_orf_deterministic_and_seed_dependent(cuda_lib):
    a = cuda_lib.new_omega(123, 256, 64)
    b = cuda_lib.new_omega(123, 256, 64)
    c = cuda_lib.new_omega(124, 256, 64)
    assert torch.equal(a, b)
    assert not torch.allclose(a, c)


# ---------------------------------------------------------------------------
# a1..a5: attention, small shapes (whole output) incl. ragged tails
# ---------------------------------------------------------------------------

SMALL = [
    # (B, H, L, d, m)
    (1, 1, 1, 64, 64), (1, 2, 2, 64, 64), (2, 1, 17, 64, 128), (1, 1, 128, 64, 128), (1, 2, 129, 64, 256),
    (2, 2, 300, 64, 256), (1, 1, 257, 128, 128), (1, 2, 513, 128, 256), (1, 1, 200, 128, 512),
    (1, 1, 64, 32, 48), (1, 1, 77, 100, 200), (3, 1, 1000, 64, 256),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,H,L,d,m", SMALL)
def test_small_shapes_match_oracle(cuda_lib, causal, dtype, B, H, L, d, m):
    w = wl.Workload("small", "causal" if causal else "bidir", "f32" if dtype == torch.float32 else "bf16",
                    B, H, L, d, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=L + d + m))
    om = cuda_lib.new_omega(L + m, m, d)
    st = _status()
    O = _run(cuda_lib, causal, Q, K, V, om, w.qk_scale, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    fn = orc.favor_causal if causal else orc.favor_bidirectional
    if causal and L > 600:
        fn = orc.favor_causal_quadratic
    ref = fn(to_np(Q), to_np(K), to_np(V), to_np(om), w.qk_scale)
    err = orc.rowwise_rel_err(to_np(O), ref)
    assert err < TOL[dtype], err


# ---------------------------------------------------------------------------
# the workloads at full size: sampled rows against the oracle
# ---------------------------------------------------------------------------

FULL = list(wl.WORKLOADS) + [n for n in wl.SWEEP
                             if ("L16384" in n) or ("L65536" in n and "m512" in n) or n.startswith("sweep-bidir")]


@pytest.mark.parametrize("name", FULL)
def test_workload_full_size_sampled_rows(cuda_lib, name):
    w = wl.get(name)
    causal = w.mode == "causal"
    Q, K, V = (t.cuda() for t in wl.make_qkv(w))
    om = cuda_lib.new_omega(wl.omega_seed_for_call(w, 0), w.m, w.d)
    st = _status()
    O = _run(cuda_lib, causal, Q, K, V, om, w.qk_scale, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.isfinite(O.float()).all()
    BH = w.B * w.H
    picks = sample_rows(BH, w.L, 12 if w.L <= 16384 else 8, seed=1)
    heads = sorted({h for h, _ in picks})
    q3 = Q.view(BH, w.L, w.d)
    k3 = K.view(BH, w.L, w.d)
    v3 = V.view(BH, w.L, w.d)
    o3 = O.view(BH, w.L, w.d)
    omn = to_np(om)
    ref_rows, got_rows = [], []
    for h in heads:
        hp = [(0, t) for hh, t in picks if hh == h]
        ref_rows.append(orc.favor_rows(to_np(q3[h:h + 1]), to_np(k3[h:h + 1]), to_np(v3[h:h + 1]), omn,
                                       w.qk_scale, hp, causal))
        got_rows.append(np.stack([to_np(o3[h, t]) for _, t in hp]))
    err = orc.rowwise_rel_err(np.concatenate(got_rows), np.concatenate(ref_rows))
    assert err < TOL[w.torch_dtype], (name, err)


@pytest.mark.parametrize("name", ["causal-bf16-B4H8L8192-d64-m256", "causal-bf16-B2H8L12288-d64-m256"])
def test_causal_full_size_chunk_boundaries(cuda_lib, name):
    # every 128-token chunk boundary of one head (rows 128k - 1 and 128k),
    # so every superchunk boundary and the last tile of every superchunk
    # are checked at the full workload size, whatever the split
    w = wl.get(name)
    Q, K, V = (t.cuda() for t in wl.make_qkv(w))
    om = cuda_lib.new_omega(wl.omega_seed_for_call(w, 0), w.m, w.d)
    st = _status()
    O = _run(cuda_lib, True, Q, K, V, om, w.qk_scale, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    BH = w.B * w.H
    h = BH // 2 + 1
    rows = sorted({0, w.L - 1} | {t for k in range(1, w.L // 128) for t in (128 * k - 1, 128 * k)})
    q3, k3, v3, o3 = (X.view(BH, w.L, w.d)[h:h + 1] for X in (Q, K, V, O))
    ref = orc.favor_rows(to_np(q3), to_np(k3), to_np(v3), to_np(om), w.qk_scale, [(0, t) for t in rows], True)
    got = to_np(o3[0])[rows]
    assert orc.rowwise_rel_err(got, ref) < TOL[torch.bfloat16], name


@pytest.mark.parametrize("m", [128, 256])
def test_causal_multichunk_walk(cuda_lib, m):
    # B*H = 128 heads of 512 tokens: one superchunk per head walks 4 chunks
    # of 128 (G carried across chunks); sampled rows of sampled heads
    w = wl.Workload("walk", "causal", "bf16", 8, 16, 512, 64, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=m))
    om = cuda_lib.new_omega(m, m, w.d)
    st = _status()
    O = _run(cuda_lib, True, Q, K, V, om, w.qk_scale, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    BH = w.B * w.H
    picks = [(h, t) for h in (0, 37, 127) for t in (0, 127, 128, 300, 511)]
    q3, k3, v3, o3 = (X.view(BH, w.L, w.d) for X in (Q, K, V, O))
    ref = orc.favor_rows(to_np(q3), to_np(k3), to_np(v3), to_np(om), w.qk_scale, picks, True)
    got = np.stack([to_np(o3[h, t]) for h, t in picks])
    assert orc.rowwise_rel_err(got, ref) < TOL[torch.bfloat16]


@pytest.mark.parametrize("L", [640, 768, 4096])
@pytest.mark.parametrize("m", [128, 256])
def test_causal_initial_states_summed_either_way(cuda_lib, L, m):
    # one head split into superchunks of one chunk each on a 152-SM GPU: at
    # L = 640 the last of 5 superchunks starts from the sum of 4 earlier
    # partials (the scan kernel adds them), at 768 from 5 (the prefix kernel
    # does) and at 4096 from 31; whole output against the oracle
    w = wl.Workload("init", "causal", "bf16", 1, 1, L, 64, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=L + m))
    om = cuda_lib.new_omega(L, m, w.d)
    st = _status()
    O = _run(cuda_lib, True, Q, K, V, om, w.qk_scale, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    fn = orc.favor_causal if L <= 800 else orc.favor_causal_quadratic
    ref = fn(to_np(Q), to_np(K), to_np(V), to_np(om), w.qk_scale)
    assert orc.rowwise_rel_err(to_np(O), ref) < TOL[torch.bfloat16]


def test_redrawn_omega_per_call(cuda_lib):
    # the 12288-token pixel workload draws a fresh Omega (seed base + i) each call
    w = wl.get("causal-bf16-B2H8L12288-d64-m256").with_(B=1, H=2, L=1024)
    Q, K, V = (t.cuda() for t in wl.make_qkv(w))
    outs = []
    for i in range(2):
        om = cuda_lib.new_omega(wl.omega_seed_for_call(w, i), w.m, w.d)
        O = _run(cuda_lib, True, Q, K, V, om, w.qk_scale)
        ref = orc.favor_causal_quadratic(to_np(Q), to_np(K), to_np(V), to_np(om), w.qk_scale)
        assert orc.rowwise_rel_err(to_np(O), ref) < TOL[torch.bfloat16]
        outs.append(O)
    assert not torch.equal(outs[0], outs[1])


# ---------------------------------------------------------------------------
# properties
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_causal_rows_do_not_see_the_future(cuda_lib, dtype):
    w = wl.Workload("p", "causal", "f32" if dtype == torch.float32 else "bf16", 1, 2, 700, 64, 256, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=3))
    om = cuda_lib.new_omega(2, w.m, w.d)
    base = _run(cuda_lib, True, Q, K, V, om, w.qk_scale).clone()
    t = 333
    g = torch.Generator(device="cuda").manual_seed(9)
    for X in (Q, K, V):
        X[:, :, t + 1:] = torch.randn(X[:, :, t + 1:].shape, generator=g, device="cuda").to(dtype)
    pert = _run(cuda_lib, True, Q, K, V, om, w.qk_scale)
    assert torch.equal(base[:, :, : t + 1], pert[:, :, : t + 1])
    assert not torch.equal(base[:, :, t + 1:], pert[:, :, t + 1:])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_bitwise_deterministic(cuda_lib, causal, dtype):
    w = wl.Workload("p", "bidir", "f32" if dtype == torch.float32 else "bf16", 2, 4, 4096, 64, 256, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=5))
    om = cuda_lib.new_omega(6, w.m, w.d)
    a = _run(cuda_lib, causal, Q, K, V, om, w.qk_scale).clone()
    b = _run(cuda_lib, causal, Q, K, V, om, w.qk_scale)
    assert torch.equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_zero_keys_give_mean_of_values(cuda_lib, causal, dtype):
    B, H, L, d, m = 1, 2, 513, 64, 128
    g = torch.Generator(device="cuda").manual_seed(1)
    Q = torch.randn((B, H, L, d), generator=g, device="cuda").to(dtype)
    V = torch.randn((B, H, L, d), generator=g, device="cuda").to(dtype)
    K = torch.zeros_like(Q)
    om = cuda_lib.new_omega(3, m, d)
    O = to_np(_run(cuda_lib, causal, Q, K, V, om, d ** -0.25))
    v = to_np(V)
    want = (np.cumsum(v, axis=-2) / np.arange(1, L + 1)[:, None]) if causal else \
        np.broadcast_to(v.mean(axis=-2, keepdims=True), v.shape)
    assert orc.rowwise_rel_err(O, want) < TOL[dtype]


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_reproduced(cuda_lib, causal):
    B, H, L, d, m = 1, 1, 300, 64, 256
    g = torch.Generator(device="cuda").manual_seed(2)
    Q = torch.randn((B, H, L, d), generator=g, device="cuda").to(torch.bfloat16)
    K = torch.randn((B, H, L, d), generator=g, device="cuda").to(torch.bfloat16)
    V = torch.full((B, H, L, d), 1.5, device="cuda", dtype=torch.bfloat16)
    om = cuda_lib.new_omega(4, m, d)
    O = _run(cuda_lib, causal, Q, K, V, om, d ** -0.25).float()
    assert torch.allclose(O, torch.full_like(O, 1.5), rtol=1e-2)


def test_stage_calls_equal_full_call(cuda_lib):
    w = wl.Workload("p", "bidir", "bf16", 1, 4, 2000, 64, 256, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=8))
    om = cuda_lib.new_omega(8, w.m, w.d)
    for causal in (False, True):
        ws = cuda_lib.new_workspace(causal, 1, 4, 2000, 64, 256, torch.bfloat16)
        full = (cuda_lib.fwd_causal if causal else cuda_lib.fwd_bidir)(Q, K, V, om, w.qk_scale, ws).clone()
        if causal:
            cuda_lib.causal_state(K, V, om, w.qk_scale, ws)
            staged = cuda_lib.causal_output(Q, K, V, om, w.qk_scale, ws)
        else:
            cuda_lib.bidir_state(K, V, om, w.qk_scale, ws)
            staged = cuda_lib.bidir_output(Q, om, w.qk_scale, ws)
        assert torch.equal(full, staged)


@pytest.mark.parametrize("dtype,q_mult,k_mult,m", [
    (torch.float32, 8.0, 3.0, 256), (torch.bfloat16, 8.0, 3.0, 256), (torch.bfloat16, 8.0, 3.0, 128),
    (torch.bfloat16, 1.0, 4.0, 256), (torch.bfloat16, 1.0, 4.0, 128)])
def test_large_norm_inputs_stay_finite(cuda_lib, dtype, q_mult, k_mult, m):
    # queries 8x the unit scale: s w.q reaches ~60 and differs from the
    # Cauchy-Schwarz bound s |q| max|w| by ~160, so a query reference taken
    # from that bound would underflow every feature; the per-row maximum
    # keeps the largest feature at 1.  Keys 3x or 4x the unit scale: their
    # largest features fall to ~e^-40 under the data-free key reference.
    # m = 128 (one feature block) and m = 256 (two) take different routes
    # to the row maximum in the causal kernel.
    w = wl.Workload("p", "bidir", "f32" if dtype == torch.float32 else "bf16", 1, 2, 1024, 64, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=10))
    Q = (Q.float() * q_mult).to(dtype)
    K = (K.float() * k_mult).to(dtype)
    om = cuda_lib.new_omega(10, w.m, w.d)
    for causal in (False, True):
        st = _status()
        O = _run(cuda_lib, causal, Q, K, V, om, w.qk_scale, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        fn = orc.favor_causal_quadratic if causal else orc.favor_bidirectional
        ref = fn(to_np(Q), to_np(K), to_np(V), to_np(om), w.qk_scale)
        assert np.all(np.isfinite(ref))
        assert orc.rowwise_rel_err(to_np(O), ref) < TOL[dtype], causal


def test_dev_status_flags_nonfinite_normaliser(cuda_lib):
    B, H, L, d, m = 1, 1, 64, 64, 64
    Q = torch.zeros((B, H, L, d), device="cuda")
    Q[0, 0, 5, 0] = float("nan")
    K = torch.zeros_like(Q)
    V = torch.ones_like(Q)
    om = cuda_lib.new_omega(1, m, d)
    st = _status()
    _run(cuda_lib, False, Q, K, V, om, 1.0, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5

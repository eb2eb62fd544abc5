"""GPU parity of the bidirectional backward (favor_bwd_bidir) against the
fp64 oracle gradient (itself pinned by finite differences).

Metric: per head, max |gpu - oracle| over the head's gradient entries
divided by the head's largest oracle entry (a gradient row can be near zero,
so a row-wise ratio would measure cancellation, not the kernels).  Bars: the
fp32 arithmetic of the kernels over sums of at most L m terms gives ~1e-6 for
fp32 storage (bar 1e-4); bf16 storage rounds every stored gradient to 2^-9
relative (bar 2e-2, as for the forward).
"""

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from helpers import TOL, to_np

pytestmark = pytest.mark.gpu


def _per_head_err(got, ref):
    g = got.reshape(-1, got.shape[-2] * got.shape[-1])
    r = ref.reshape(-1, ref.shape[-2] * ref.shape[-1])
    return float(np.max(np.max(np.abs(g - r), axis=1) / np.max(np.abs(r), axis=1)))


@pytest.mark.parametrize("features", ["prf", "relu", "elu1"])
@pytest.mark.parametrize("dtype,B,H,L,d,m", [(torch.float32, 2, 2, 200, 64, 128),
                                             (torch.float32, 1, 3, 65, 32, 100),
                                             (torch.bfloat16, 2, 4, 1000, 64, 256),
                                             (torch.bfloat16, 1, 2, 300, 128, 512)])
def test_backward_matches_oracle(cuda_lib, features, dtype, B, H, L, d, m):
    w = wl.Workload("bwd", "bidir", "f32" if dtype == torch.float32 else "bf16", B, H, L, d, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=L + m))
    gen = torch.Generator(device="cpu")
    gen.manual_seed(L * m)
    dO = torch.randn((B, H, L, d), generator=gen).to(dtype).cuda()
    om = cuda_lib.new_omega(m + 2, m, d)
    s = d ** -0.25
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dQ, dK, dV = cuda_lib.bwd_bidir(Q, K, V, dO, om, s, feature_map=features, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rQ, rK, rV = orc.favor_bidirectional_grad(to_np(Q), to_np(K), to_np(V), to_np(om), s, to_np(dO), features)
    errs = {n: _per_head_err(to_np(g), r) for n, g, r in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV))}
    assert max(errs.values()) < TOL[dtype], errs


def test_backward_is_deterministic(cuda_lib):
    B, H, L, d, m = 1, 2, 300, 64, 128
    w = wl.Workload("bwd", "bidir", "f32", B, H, L, d, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=1))
    dO = torch.ones_like(Q)
    om = cuda_lib.new_omega(1, m, d)
    a = cuda_lib.bwd_bidir(Q, K, V, dO, om, 0.4)
    b = cuda_lib.bwd_bidir(Q, K, V, dO, om, 0.4)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("features", ["prf", "relu", "elu1"])
@pytest.mark.parametrize("dtype,B,H,L,d,m", [(torch.float32, 2, 2, 75, 64, 128),
                                             (torch.float32, 1, 2, 33, 32, 100),
                                             (torch.bfloat16, 2, 3, 300, 64, 256),
                                             (torch.bfloat16, 1, 2, 50, 128, 512),
                                             # 304 heads: chunks of several tiles (64 and 80
                                             # tokens on 152 SMs) with a ragged last chunk
                                             (torch.float32, 16, 19, 200, 32, 64),
                                             (torch.bfloat16, 8, 38, 264, 64, 128)])
def test_causal_backward_matches_oracle(cuda_lib, features, dtype, B, H, L, d, m):
    w = wl.Workload("cbwd", "causal", "f32" if dtype == torch.float32 else "bf16", B, H, L, d, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=3 * L + m))
    if features == "relu":
        # the first row's only key is itself: phi(q0).phi(k0) = |phi(q0)|^2 > 0
        K[:, :, 0] = Q[:, :, 0]
    gen = torch.Generator(device="cpu")
    gen.manual_seed(L + 2 * m)
    dO = torch.randn((B, H, L, d), generator=gen).to(dtype).cuda()
    om = cuda_lib.new_omega(m + 5, m, d)
    s = d ** -0.25
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dQ, dK, dV = cuda_lib.bwd_causal(Q, K, V, dO, om, s, feature_map=features, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rQ, rK, rV = orc.favor_causal_grad(to_np(Q), to_np(K), to_np(V), to_np(om), s, to_np(dO), features)
    errs = {n: _per_head_err(to_np(g), r) for n, g, r in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV))}
    assert max(errs.values()) < TOL[dtype], errs


def test_causal_backward_last_row_equals_bidirectional(cuda_lib):
    # dO zero except the last row: the two losses coincide
    B, H, L, d, m = 1, 2, 70, 64, 128
    w = wl.Workload("cbwd", "causal", "f32", B, H, L, d, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=4))
    dO = torch.zeros_like(Q)
    dO[:, :, -1] = torch.randn((B, H, d), generator=torch.Generator().manual_seed(4)).cuda()
    om = cuda_lib.new_omega(4, m, d)
    a = cuda_lib.bwd_causal(Q, K, V, dO, om, 0.4)
    b = cuda_lib.bwd_bidir(Q, K, V, dO, om, 0.4)
    for x, y in zip(a, b):
        assert _per_head_err(to_np(x), to_np(y)) < 1e-4


# ---------------------------------------------------------------------------
# bf16, d = 64, m in {128, 256}: the tensor-core kernels (tc_bwd.cu)
# ---------------------------------------------------------------------------
def _bwd_case(cuda_lib, B, H, L, m, features, seed, q_scale=1.0, k_scale=1.0):
    w = wl.Workload("tcbwd", "bidir", "bf16", B, H, L, 64, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=seed))
    Q = (Q.float() * q_scale).to(torch.bfloat16)
    K = (K.float() * k_scale).to(torch.bfloat16)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 1)
    dO = torch.randn((B, H, L, 64), generator=gen).to(torch.bfloat16).cuda()
    om = cuda_lib.new_omega(seed + 2, m, 64)
    return Q, K, V, dO, om


@pytest.mark.parametrize("features", ["prf", "relu", "elu1"])
@pytest.mark.parametrize("B,H,L,m", [(1, 2, 128, 256),     # one tile
                                     (1, 3, 777, 128),     # ragged last tile
                                     (3, 5, 2500, 128),    # several CTAs per head
                                     (2, 3, 3000, 256),
                                     (5, 10, 500, 256),    # CTAs that cross from one head into the next
                                     (1, 1, 20000, 128)])  # one head over every CTA of the grid
def test_tc_backward_matches_oracle(cuda_lib, features, B, H, L, m):
    Q, K, V, dO, om = _bwd_case(cuda_lib, B, H, L, m, features, seed=L + m)
    s = 64 ** -0.25
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dQ, dK, dV = cuda_lib.bwd_bidir(Q, K, V, dO, om, s, feature_map=features, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rQ, rK, rV = orc.favor_bidirectional_grad(to_np(Q), to_np(K), to_np(V), to_np(om), s, to_np(dO), features)
    errs = {n: _per_head_err(to_np(g), r) for n, g, r in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV))}
    assert max(errs.values()) < TOL[torch.bfloat16], errs


def test_tc_backward_full_size_sampled_heads(cuda_lib):
    # the 4096-token, 64-head workload, every head computed; two heads checked
    B, H, L, m = 8, 8, 4096, 256
    Q, K, V, dO, om = _bwd_case(cuda_lib, B, H, L, m, "prf", seed=11)
    s = 64 ** -0.25
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dQ, dK, dV = cuda_lib.bwd_bidir(Q, K, V, dO, om, s, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b, h in ((0, 0), (7, 5)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        rQ, rK, rV = orc.favor_bidirectional_grad(to_np(Q[sl]), to_np(K[sl]), to_np(V[sl]), to_np(om), s,
                                                  to_np(dO[sl]), "prf")
        errs = {n: _per_head_err(to_np(g[sl]), r) for n, g, r in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV))}
        assert max(errs.values()) < TOL[torch.bfloat16], (b, h, errs)


@pytest.mark.parametrize("q_scale,k_scale", [(8.0, 1.0), (4.0, 2.0)])
def test_tc_backward_large_norm_inputs(cuda_lib, q_scale, k_scale):
    # the query reference is the row's own largest exponent, so phi(q) never
    # underflows as a whole however large q is
    B, H, L, m = 1, 2, 600, 256
    Q, K, V, dO, om = _bwd_case(cuda_lib, B, H, L, m, "prf", seed=5, q_scale=q_scale, k_scale=k_scale)
    s = 64 ** -0.25
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dQ, dK, dV = cuda_lib.bwd_bidir(Q, K, V, dO, om, s, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rQ, rK, rV = orc.favor_bidirectional_grad(to_np(Q), to_np(K), to_np(V), to_np(om), s, to_np(dO), "prf")
    errs = {n: _per_head_err(to_np(g), r) for n, g, r in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV))}
    assert max(errs.values()) < TOL[torch.bfloat16], errs


def test_tc_backward_is_deterministic(cuda_lib):
    Q, K, V, dO, om = _bwd_case(cuda_lib, 2, 4, 2000, 256, "prf", seed=7)
    a = cuda_lib.bwd_bidir(Q, K, V, dO, om, 0.35)
    b = cuda_lib.bwd_bidir(Q, K, V, dO, om, 0.35)
    for x, y in zip(a, b):
        assert torch.equal(x, y)

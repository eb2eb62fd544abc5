"""GPU parity of incremental causal decoding (one token per call, the prefix
state carried in an fp32 array) against the fp64 oracle.

Row t of the causal estimator (the oracle's lower-triangular quadratic form)
must come out of the t-th decode step, from a zero state or from the state
that favor_decode_prefill builds for a prompt; bars as for the full passes
(row-wise normwise 1e-4 fp32, 2e-2 bf16).
"""

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from helpers import TOL, to_np

pytestmark = pytest.mark.gpu


def _inputs(B, H, L, d, dtype, seed):
    w = wl.Workload("dec", "causal", "f32" if dtype == torch.float32 else "bf16", B, H, L, d, 64, "normal")
    return [t.cuda() for t in wl.make_qkv(w, seed=seed)]


def _decode_all(favor, Q, K, V, om, s, state, t0=0, status=None):
    outs = []
    for t in range(t0, Q.shape[2]):
        outs.append(favor.decode_step(Q[:, :, t].contiguous(), K[:, :, t].contiguous(), V[:, :, t].contiguous(), om,
                                      s, state, dev_status=status))
    return torch.stack(outs, dim=2)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d,m", [(64, 256), (64, 128), (32, 100), (128, 512), (16, 8)])
def test_decode_steps_match_causal_rows(cuda_lib, dtype, d, m):
    B, H, L = 2, 3, 37
    Q, K, V = _inputs(B, H, L, d, dtype, seed=d + m)
    om = cuda_lib.new_omega(m + 1, m, d)
    s = d ** -0.25
    state = cuda_lib.new_decode_state(B, H, m, d)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _decode_all(cuda_lib, Q, K, V, om, s, state, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.favor_causal_quadratic(to_np(Q), to_np(K), to_np(V), to_np(om), s)
    assert orc.rowwise_rel_err(to_np(got), ref) < TOL[dtype]
    # the first step is v_0 itself (one token attends only to itself)
    assert np.max(np.abs(to_np(got)[:, :, 0] - to_np(V)[:, :, 0])) <= 1e-6 + TOL[dtype] * np.max(np.abs(to_np(V)))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("q_scale", [4.0, 8.0])
def test_decode_large_norm_queries(cuda_lib, dtype, q_scale):
    # the query reference is the query's own largest exponent, so phi(q)
    # never underflows as a whole however large q is
    B, H, L, d, m = 2, 2, 20, 64, 256
    Q, K, V = _inputs(B, H, L, d, dtype, seed=7)
    Q = (Q.float() * q_scale).to(dtype)
    om = cuda_lib.new_omega(9, m, d)
    s = d ** -0.25
    state = cuda_lib.new_decode_state(B, H, m, d)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _decode_all(cuda_lib, Q, K, V, om, s, state, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.isfinite(got.float()).all()
    ref = orc.favor_causal_quadratic(to_np(Q), to_np(K), to_np(V), to_np(om), s)
    assert orc.rowwise_rel_err(to_np(got), ref) < TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,H,d,m", [(40, 16, 64, 256), (37, 7, 48, 96), (5, 3, 64, 256), (40, 16, 64, 100)])
def test_decode_many_heads(cuda_lib, dtype, B, H, d, m):
    # more heads than SMs (several heads per CTA, both shared-memory buffers
    # reused), fewer heads than SMs, and a feature count off the
    # double-buffered form's multiple of 4
    L = 5
    Q, K, V = _inputs(B, H, L, d, dtype, seed=B * H + m)
    om = cuda_lib.new_omega(m + 2, m, d)
    s = d ** -0.25
    state = cuda_lib.new_decode_state(B, H, m, d)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _decode_all(cuda_lib, Q, K, V, om, s, state, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.favor_causal_quadratic(to_np(Q), to_np(K), to_np(V), to_np(om), s)
    assert orc.rowwise_rel_err(to_np(got), ref) < TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_continues_a_prefilled_prompt(cuda_lib, dtype):
    B, H, L0, L, d, m = 2, 4, 300, 308, 64, 256
    Q, K, V = _inputs(B, H, L, d, dtype, seed=5)
    om = cuda_lib.new_omega(3, m, d)
    s = d ** -0.25
    state = cuda_lib.new_decode_state(B, H, m, d)
    cuda_lib.decode_prefill(K[:, :, :L0].contiguous(), V[:, :, :L0].contiguous(), om, s, state)
    got = _decode_all(cuda_lib, Q, K, V, om, s, state, t0=L0)
    picks = [(bh, t) for bh in range(B * H) for t in range(L0, L)]
    ref = orc.favor_rows(to_np(Q).reshape(B * H, L, d), to_np(K).reshape(B * H, L, d),
                         to_np(V).reshape(B * H, L, d), to_np(om), s, picks, True)
    assert orc.rowwise_rel_err(to_np(got).reshape(B * H * (L - L0), d), ref) < TOL[dtype]


def test_prefill_equals_token_by_token_state(cuda_lib):
    B, H, L, d, m = 1, 2, 50, 64, 128
    Q, K, V = _inputs(B, H, L, d, torch.float32, seed=8)
    om = cuda_lib.new_omega(8, m, d)
    s = d ** -0.25
    stepped = cuda_lib.new_decode_state(B, H, m, d)
    _decode_all(cuda_lib, Q, K, V, om, s, stepped)
    pre = cuda_lib.decode_prefill(K, V, om, s, cuda_lib.new_decode_state(B, H, m, d))
    a, b = to_np(stepped), to_np(pre)
    # same features and the same reference; only the summation order differs
    assert np.max(np.abs(a - b)) <= 1e-5 * np.max(np.abs(b))


def test_decode_flags_a_nonfinite_normaliser(cuda_lib):
    B, H, d, m = 1, 1, 64, 64
    q = torch.zeros((B, H, d), device="cuda")
    q[0, 0, 3] = float("nan")
    k = torch.zeros_like(q)
    v = torch.ones_like(q)
    om = cuda_lib.new_omega(1, m, d)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.decode_step(q, k, v, om, 1.0, cuda_lib.new_decode_state(B, H, m, d), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5

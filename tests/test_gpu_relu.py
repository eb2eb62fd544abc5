"""GPU parity of the Performer-ReLU feature map (favor_fwd_*_fm with
FAVOR_FM_RELU) against the fp64 oracle's relu features, on the tensor-core
(bf16) and CUDA-core (fp32) paths; bars as for the softmax features."""

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from helpers import TOL, to_np

pytestmark = pytest.mark.gpu


def _qkv(B, H, L, d, dtype, seed):
    w = wl.Workload("relu", "bidir", "f32" if dtype == torch.float32 else "bf16", B, H, L, d, 64, "normal")
    return [t.cuda() for t in wl.make_qkv(w, seed=seed)]


def _run(favor, causal, Q, K, V, om, s, status=None):
    B, H, L, d = Q.shape
    ws = favor.new_workspace(causal, B, H, L, d, om.shape[0], Q.dtype)
    fn = favor.fwd_causal if causal else favor.fwd_bidir
    return fn(Q, K, V, om, s, ws, dev_status=status, feature_map="relu")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,d,m,L", [(torch.bfloat16, 64, 256, 1000), (torch.bfloat16, 64, 128, 300),
                                         (torch.float32, 64, 64, 300), (torch.float32, 32, 100, 129)])
def test_relu_matches_oracle(cuda_lib, causal, dtype, d, m, L):
    B, H = 2, 3
    Q, K, V = _qkv(B, H, L, d, dtype, seed=m + L)
    om = cuda_lib.new_omega(m + 7, m, d)
    s = d ** -0.25
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    O = _run(cuda_lib, causal, Q, K, V, om, s, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    fn = orc.favor_causal_quadratic if causal else orc.favor_bidirectional
    ref = fn(to_np(Q), to_np(K), to_np(V), to_np(om), s, "relu")
    assert orc.rowwise_rel_err(to_np(O), ref) < TOL[dtype]


def test_relu_long_causal_sampled_rows(cuda_lib):
    # several superchunks per head: the scan's initial states come from the
    # superchunk partials, as for the softmax features
    B, H, L, d, m = 2, 8, 8192, 64, 256
    Q, K, V = _qkv(B, H, L, d, torch.bfloat16, seed=77)
    om = cuda_lib.new_omega(77, m, d)
    s = d ** -0.25
    O = _run(cuda_lib, True, Q, K, V, om, s)
    picks = [(h, t) for h in (0, 9, 15) for t in (0, 1, 4095, 4096, 6000, 8191)]
    q3, k3, v3, o3 = (X.view(B * H, L, d) for X in (Q, K, V, O))
    ref = orc.favor_rows(to_np(q3), to_np(k3), to_np(v3), to_np(om), s, picks, True, "relu")
    got = np.stack([to_np(o3[h, t]) for h, t in picks])
    assert orc.rowwise_rel_err(got, ref) < TOL[torch.bfloat16]


def test_relu_differs_from_softmax_features(cuda_lib):
    B, H, L, d, m = 1, 2, 256, 64, 128
    Q, K, V = _qkv(B, H, L, d, torch.float32, seed=3)
    om = cuda_lib.new_omega(3, m, d)
    ws = cuda_lib.new_workspace(False, B, H, L, d, m, Q.dtype)
    a = cuda_lib.fwd_bidir(Q, K, V, om, 0.35, ws)
    b = cuda_lib.fwd_bidir(Q, K, V, om, 0.35, ws, feature_map="relu")
    assert not torch.allclose(a, b)

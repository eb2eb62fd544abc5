"""GPU parity of the 1 + elu feature map (favor_fwd_*_fm with FAVOR_FM_ELU1)
against the fp64 oracle's elu1 features, on the tensor-core kernels (bf16,
d = 64 and 128) and the CUDA-core kernels (fp32, other shapes); bars as for
the softmax features.  Omega = I gives plain linear attention."""

import pytest
import torch

import oracle as orc
import workloads as wl
from helpers import TOL, to_np

pytestmark = pytest.mark.gpu


def _qkv(B, H, L, d, dtype, seed):
    w = wl.Workload("elu", "bidir", "f32" if dtype == torch.float32 else "bf16", B, H, L, d, 64, "normal")
    return [t.cuda() for t in wl.make_qkv(w, seed=seed)]


def _run(favor, causal, Q, K, V, om, s, status=None):
    B, H, L, d = Q.shape
    ws = favor.new_workspace(causal, B, H, L, d, om.shape[0], Q.dtype, feature_map="elu1")
    fn = favor.fwd_causal if causal else favor.fwd_bidir
    return fn(Q, K, V, om, s, ws, dev_status=status, feature_map="elu1")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,d,m,L", [(torch.bfloat16, 64, 256, 1000), (torch.bfloat16, 64, 128, 300),
                                         (torch.bfloat16, 64, 256, 4100), (torch.bfloat16, 128, 512, 700),
                                         (torch.bfloat16, 128, 128, 129),
                                         (torch.float32, 64, 64, 300), (torch.float32, 32, 100, 129)])
def test_elu1_matches_oracle(cuda_lib, causal, dtype, d, m, L):
    B, H = 2, 3
    Q, K, V = _qkv(B, H, L, d, dtype, seed=m + L + 1)
    om = cuda_lib.new_omega(m + 9, m, d)
    s = d ** -0.25
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    O = _run(cuda_lib, causal, Q, K, V, om, s, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    fn = orc.favor_causal_quadratic if causal else orc.favor_bidirectional
    ref = fn(to_np(Q), to_np(K), to_np(V), to_np(om), s, "elu1")
    assert orc.rowwise_rel_err(to_np(O), ref) < TOL[dtype]


@pytest.mark.parametrize("causal", [False, True])
def test_identity_projection_is_linear_attention(cuda_lib, causal):
    B, H, L, d = 1, 4, 257, 64
    Q, K, V = _qkv(B, H, L, d, torch.float32, seed=31)
    om = torch.eye(d, dtype=torch.float32, device="cuda")
    O = _run(cuda_lib, causal, Q, K, V, om, 1.0)
    fn = orc.favor_causal_quadratic if causal else orc.favor_bidirectional
    ref = fn(to_np(Q), to_np(K), to_np(V), to_np(om), 1.0, "elu1")
    assert orc.rowwise_rel_err(to_np(O), ref) < TOL[torch.float32]


@pytest.mark.parametrize("causal", [False, True])
def test_elu1_takes_the_plain_calls_workspace(cuda_lib, causal):
    # every feature map takes the plain call's path: the same workspace size,
    # and a call with the plain workspace runs
    B, H, L, d, m = 2, 4, 1000, 64, 256
    assert cuda_lib.workspace_bytes(causal, B, H, L, d, m, torch.bfloat16, feature_map="elu1") == \
        cuda_lib.workspace_bytes(causal, B, H, L, d, m, torch.bfloat16)
    Q, K, V = _qkv(B, H, L, d, torch.bfloat16, seed=3)
    om = cuda_lib.new_omega(3, m, d)
    ws = cuda_lib.new_workspace(causal, B, H, L, d, m, torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn = cuda_lib.fwd_causal if causal else cuda_lib.fwd_bidir
    O = fn(Q, K, V, om, d ** -0.25, ws, dev_status=st, feature_map="elu1")
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = (orc.favor_causal_quadratic if causal else orc.favor_bidirectional)(
        to_np(Q), to_np(K), to_np(V), to_np(om), d ** -0.25, "elu1")
    assert orc.rowwise_rel_err(to_np(O), ref) < TOL[torch.bfloat16]

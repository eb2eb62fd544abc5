"""The allocation-free bidirectional entry point, favor_fwd_bidir_static.

Some callers cannot allocate device memory where they run the attention:
code inside a host framework that owns all device memory and forbids
allocation on its request path, or latency-critical code that must not enter
the allocator (cudaMalloc can synchronise the device).  For them the library
runs favor_fwd_bidir with its scratch in one fixed device array instead of a
caller workspace.  These tests call that entry point through the C ABI and
compare it with favor_fwd_bidir, twice in a row (the array keeps the previous
call's contents, which must not leak into the next result).

The file sorts last so that a run stopping at the first failure has already
run every other test; it also passes when run alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from helpers import TOL, to_np

pytestmark = pytest.mark.gpu

CASES = [
    # (dtype, B, H, L, d, m): tensor-core path and CUDA-core path
    (torch.bfloat16, 2, 4, 1000, 64, 256),
    (torch.float32, 1, 2, 513, 64, 64),
]


def _static_call(lib, Q, K, V, O, om, scale, status):
    B, H, L, d = Q.shape
    dt = 1 if Q.dtype == torch.bfloat16 else 0
    return lib.favor_fwd_bidir_static(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), B, H, L, d,
                                      om.data_ptr(), om.shape[0], dt, ctypes.c_float(scale), status.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype,B,H,L,d,m", CASES)
def test_static_scratch_matches_workspace_entry(cuda_lib, dtype, B, H, L, d, m):
    lib = cuda_lib.load()
    w = wl.Workload("static", "bidir", "bf16" if dtype == torch.bfloat16 else "f32", B, H, L, d, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=L + m))
    om = cuda_lib.new_omega(L, m, d)
    ws = cuda_lib.new_workspace(False, B, H, L, d, m, dtype)
    ref = cuda_lib.fwd_bidir(Q, K, V, om, w.qk_scale, ws).clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for call in range(2):
        # a different second input set: stale scratch from call 0 must not matter
        if call == 1:
            Q2, K2, V2 = (t.cuda() for t in wl.make_qkv(w, seed=L + m + 1))
            ref = cuda_lib.fwd_bidir(Q2, K2, V2, om, w.qk_scale, ws).clone()
            Q, K, V = Q2, K2, V2
        O = torch.full_like(Q, float("nan"))
        code = _static_call(lib, Q, K, V, O, om, w.qk_scale, status)
        torch.cuda.synchronize()
        assert code == 0, cuda_lib.status_string(code)
        assert int(status.item()) == 0
        assert orc.rowwise_rel_err(to_np(O), to_np(ref)) < TOL[dtype]
        outs.append(O)
    # and both agree with the fp64 oracle on the last inputs
    exact = orc.favor_bidirectional(to_np(Q), to_np(K), to_np(V), to_np(om), w.qk_scale)
    assert orc.rowwise_rel_err(to_np(outs[1]), exact) < TOL[dtype]


def test_static_scratch_rejects_oversized_shapes(cuda_lib):
    lib = cuda_lib.load()
    limit = lib.favor_static_scratch_bytes()
    assert limit == 16 << 20
    B, H, L, d, m = 64, 64, 4096, 64, 256          # needs far more than the fixed array
    assert lib.favor_workspace_bytes(0, B, H, L, d, m, 1) > limit
    small = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    om = torch.zeros((m, d), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = lib.favor_fwd_bidir_static(small.data_ptr(), small.data_ptr(), small.data_ptr(), None, B, H, L, d,
                                      om.data_ptr(), m, 1, ctypes.c_float(0.35), status.data_ptr(), None)
    assert code == 2                                # FAVOR_ERR_UNSUPPORTED, nothing launched
    assert np.all(to_np(small) == 0)


def test_static_scratch_at_its_limit(cuda_lib):
    # the largest head count whose scratch fits the fixed array (the array's
    # tail in use) runs and matches favor_fwd_bidir; one head more is rejected
    lib = cuda_lib.load()
    limit = lib.favor_static_scratch_bytes()
    B, L, d, m = 1, 300, 64, 256
    need = {H: lib.favor_workspace_bytes(0, B, H, L, d, m, 1) for H in range(1, 4097)}
    fits = [H for H, n in need.items() if 0 < n <= limit]
    H = max(fits)
    assert need[H] > 0.9 * limit, (H, need[H], limit)
    assert need[H + 1] > limit
    w = wl.Workload("static", "bidir", "bf16", B, H, L, d, m, "normal")
    Q, K, V = (t.cuda() for t in wl.make_qkv(w, seed=21))
    om = cuda_lib.new_omega(21, m, d)
    ws = cuda_lib.new_workspace(False, B, H, L, d, m, torch.bfloat16)
    ref = cuda_lib.fwd_bidir(Q, K, V, om, w.qk_scale, ws).clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    O = torch.full_like(Q, float("nan"))
    code = _static_call(lib, Q, K, V, O, om, w.qk_scale, status)
    torch.cuda.synchronize()
    assert code == 0, cuda_lib.status_string(code)
    assert int(status.item()) == 0
    assert orc.rowwise_rel_err(to_np(O), to_np(ref)) < TOL[torch.bfloat16]
    # one head more: rejected before anything is launched, O untouched
    w2 = w.with_(H=H + 1)
    Q2, K2, V2 = (t.cuda() for t in wl.make_qkv(w2, seed=22))
    O2 = torch.zeros_like(Q2)
    code = _static_call(lib, Q2, K2, V2, O2, om, w.qk_scale, status)
    torch.cuda.synchronize()
    assert code == 2
    assert torch.count_nonzero(O2).item() == 0

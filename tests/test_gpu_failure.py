"""Failure handling of the bounded device waits, on the GPU without a fault.

A wait on an mbarrier that nothing completes must give up after the wait
limit (1 s), store FAVOR_ERR_TIMEOUT in the device status and raise the
CTA's abort flag, so that a second wait started later returns at once; the
context stays usable for the next call."""

import pytest
import torch

import oracle as orc
import workloads as wl
from helpers import TOL, to_np

pytestmark = pytest.mark.gpu

FAVOR_ERR_TIMEOUT = 4


def test_a_wait_that_runs_out_reports_and_aborts_the_other(cuda_lib):
    status, returned, t = cuda_lib.selftest_wait_timeout()
    assert status == FAVOR_ERR_TIMEOUT
    assert returned == [2, 2]                       # both waits gave up
    first = (t[1] - t[0]) / 1e9
    second_after_first = (t[2] - t[1]) / 1e9
    assert 0.9 < first < 3.0                         # the 1 s limit
    # warp 1 began 0.5 s in: alone it would give up near 1.5 s; with the
    # abort flag it returns right after warp 0
    assert abs(second_after_first) < 0.2


def test_context_stays_usable_after_a_timeout(cuda_lib):
    cuda_lib.selftest_wait_timeout()
    w = wl.Workload("after", "causal", "bf16", 1, 2, 300, 64, 256, "normal")
    Q, K, V = (x.cuda() for x in wl.make_qkv(w, seed=12))
    om = cuda_lib.new_omega(12, w.m, w.d)
    ws = cuda_lib.new_workspace(True, 1, 2, 300, 64, 256, torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    O = cuda_lib.fwd_causal(Q, K, V, om, w.qk_scale, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = orc.favor_causal_quadratic(to_np(Q), to_np(K), to_np(V), to_np(om), w.qk_scale)
    assert orc.rowwise_rel_err(to_np(O), ref) < TOL[torch.bfloat16]

"""The seeded input recipes (CPU only): determinism, dtype and layout, the
token-indexed structure of the sequence workloads, the LayerNorm of the
sweep, the Omega seed schedule, and the N(0, 1) draws' moments."""

import pytest
import torch

import workloads as wl


def test_same_seed_same_inputs_and_seeds_differ():
    w = wl.get("bidir-bf16-B8H8L4096-d64-m256")
    a = wl.make_qkv(w, seed=3, B=1, H=2, L=64)
    b = wl.make_qkv(w, seed=3, B=1, H=2, L=64)
    c = wl.make_qkv(w, seed=4, B=1, H=2, L=64)
    for x, y, z in zip(a, b, c):
        assert torch.equal(x, y)
        assert not torch.equal(x, z)
        assert x.dtype == torch.bfloat16 and x.shape == (1, 2, 64, 64) and x.is_contiguous()
    # Q, K and V are independent draws
    assert not torch.equal(a[0], a[1]) and not torch.equal(a[1], a[2])


def test_fp32_workload_stays_fp32():
    q, k, v = wl.make_qkv(wl.get("bidir-f32-B1H1L512-d64-m64"))
    assert q.dtype == torch.float32 and q.shape == (1, 1, 512, 64)


def test_normal_draws_have_unit_moments():
    q, _, _ = wl.make_qkv(wl.get("bidir-f32-B1H1L512-d64-m64"), seed=9)
    assert abs(float(q.mean())) < 0.02
    assert abs(float(q.var()) - 1.0) < 0.03


@pytest.mark.parametrize("name,vocab", [("causal-bf16-B4H8L8192-d64-m256", 36),
                                        ("causal-bf16-B2H8L12288-d64-m256", 256)])
def test_token_workloads_pick_rows_of_a_table(name, vocab):
    w = wl.get(name)
    B, H, L = 2, 3, 600
    for x in wl.make_qkv(w, seed=5, B=B, H=H, L=L):
        for b in range(B):
            for h in range(H):
                rows = torch.unique(x[b, h].float(), dim=0)
                assert rows.shape[0] <= vocab          # at most one distinct row per token value
        # the same token picks the same row in every head's slice of the table
        assert x.shape == (B, H, L, w.d)
    q, k, _ = wl.make_qkv(w, seed=5, B=B, H=H, L=L)
    # positions holding equal query rows hold equal key rows (one token sequence)
    qb, kb = q[0, 0].float(), k[0, 0].float()
    same = (qb[:, None, :] == qb[None, :, :]).all(-1)
    same_k = (kb[:, None, :] == kb[None, :, :]).all(-1)
    assert torch.equal(same, same_k)


def test_sweep_layer_norms_queries_and_keys_only():
    w = wl.get("sweep-bidir-bf16-B1H16L16384-d128-m256")
    q, k, v = wl.make_qkv(w, seed=2, B=1, H=2, L=256)
    for x in (q, k):
        xf = x.float()
        assert float(xf.mean(-1).abs().max()) < 0.02         # bf16 rounding of a zero-mean row
        assert float((xf.var(-1, unbiased=False) - 1.0).abs().max()) < 0.03
    vf = v.float()
    assert float((vf.var(-1, unbiased=False) - 1.0).abs().max()) > 0.05   # V is not normalised


def test_omega_seed_schedule():
    fixed = wl.get("causal-bf16-B4H8L8192-d64-m256")
    redraw = wl.get("causal-bf16-B2H8L12288-d64-m256")
    assert [wl.omega_seed_for_call(fixed, i) for i in range(3)] == [fixed.omega_seed] * 3
    assert [wl.omega_seed_for_call(redraw, i) for i in range(3)] == [redraw.omega_seed + i for i in range(3)]


def test_workload_registry():
    assert len(wl.WORKLOADS) == 4
    assert len(wl.SWEEP) == 18
    for name, w in {**wl.WORKLOADS, **wl.SWEEP}.items():
        assert wl.get(name) is w
        assert w.qk_scale == pytest.approx(w.d ** -0.25)

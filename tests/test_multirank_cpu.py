"""The replicas' host logic on two CPU ranks (gloo, world size 2).

The path shards by (batch, head) with no exchange: each rank runs its own
inputs, and the bench reports every rank's tokens over the slowest rank's
time.  What crosses ranks is checked here without a GPU: the barrier, the
maximum over ranks, distinct per-rank inputs and the whole-job value.
"""

import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_multirank", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _load_bench()
        import workloads as wl
        ranks = bench.Ranks(world, torch.device("cpu"))
        ranks.barrier()
        # per-rank times 2.0 and 5.0 ms: every rank sees the slower one
        slowest = ranks.max_over_ranks(2.0 + 3.0 * rank)
        w = wl.Workload("mr", "bidir", "f32", 1, 2, 48, 16, 32, "normal")
        q, k, v = wl.make_qkv(w, seed=bench.rank_input_seed(rank, 0))
        sums = [torch.zeros(3, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sums, torch.tensor([float(t.double().sum()) for t in (q, k, v)], dtype=torch.float64))
        value = bench.whole_job_value(world, w.B * w.L, 10, slowest)
        ranks.barrier()
        torch.save({"slowest": slowest, "sums": torch.stack(sums), "value": value},
                   os.path.join(out_dir, f"rank{rank}.pt"))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [torch.load(tmp_path / f"rank{r}.pt") for r in range(world)]
    for r in res:
        assert r["slowest"] == 5.0
        # 2 ranks x 48 tokens x 10 steps over 5 ms
        assert r["value"] == pytest.approx(2 * 48 * 10 / 5e-3, rel=1e-12)
    # both ranks gathered the same table, and their inputs differ
    assert torch.equal(res[0]["sums"], res[1]["sums"])
    assert not torch.equal(res[0]["sums"][0], res[0]["sums"][1])


def test_single_rank_needs_no_process_group():
    bench = _load_bench()
    ranks = bench.Ranks(1, torch.device("cpu"))
    ranks.barrier()
    assert ranks.max_over_ranks(7.5) == 7.5
    assert bench.whole_job_value(1, 32768, 4, 2.0) == pytest.approx(32768 * 4 / 2e-3)
    assert bench.rank_input_seed(0, 3) != bench.rank_input_seed(1, 3)

"""bench.py's host-side accounting (CPU only).

The roofline line divides algorithmic work by measured time, so the per-stage
byte and flop counts are checked against the per-head-token figures they come
from (read Q, K, V and write O: 4 d e bytes; two projections 4 m d flops plus
state and output 4 m (d + 1) flops), and the committed profile summaries are
checked to parse into the traffic field.
"""

import importlib.util
import os
import re

import pytest

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", ["bidir-bf16-B8H8L4096-d64-m256", "bidir-f32-B1H1L512-d64-m64",
                                  "causal-bf16-B4H8L8192-d64-m256"])
def test_algorithmic_work_matches_per_token_figures(bench, name):
    w = wl.get(name)
    e = 4 if w.dtype == "f32" else 2
    ht = w.B * w.H * w.L
    per_tok_flops = 4 * w.m * w.d + 4 * w.m * (w.d + 1)
    # the causal scan does the whole per-token work; the bidirectional pass
    # splits it between the state and the output kernels
    b, f = bench.algorithmic(w, "causal_output")
    assert b == ht * 4 * w.d * e and f == ht * per_tok_flops
    bs, fs = bench.algorithmic(w, "bidir_state")
    bo, fo = bench.algorithmic(w, "bidir_output")
    assert fs + fo == ht * per_tok_flops
    assert bs == ht * 2 * w.d * e + w.B * w.H * w.m * (w.d + 1) * 4
    assert bo == ht * 2 * w.d * e + w.B * w.H * w.m * (w.d + 1) * 4


def test_headline_workload_figures(bench):
    # B8 H8 L4096 d64 m256 bf16: 134.2 MB and 34.6 GF per causal launch
    w = wl.get(bench.DEFAULT_WORKLOAD)
    b, f = bench.algorithmic(w, "causal_output")
    assert b == 134217728
    assert f == 34628173824


def test_committed_profile_parses(bench):
    pdir = os.path.join(ROOT, "profiles")
    files = [f for f in os.listdir(pdir) if f.endswith(".md")]
    assert files, "profiles/ holds no summary"
    found = False
    for f in files:
        text = open(os.path.join(pdir, f)).read()
        assert "ncu" in text and "--clock-control none" in text      # the command that made it
        if re.search(r"^traffic_bytes_per_launch:", text, re.M):
            found = True
            stage = re.search(r"^stage:\s*(\S+)", text, re.M).group(1)
            workload = re.search(r"^workload:\s*(\S+)", text, re.M).group(1)
            src = re.search(r"^source_hash:\s*(\S+)", text, re.M).group(1)
            value = bench.profiled_traffic(stage, workload)
            if src == bench.kernel_source_hash():
                assert value is not None and value > 0
            else:
                assert value is None          # stale counters are never reported
    assert found


def test_source_hash_is_stable(bench):
    assert bench.kernel_source_hash() == bench.kernel_source_hash()
    assert re.fullmatch(r"[0-9a-f]{16}", bench.kernel_source_hash())

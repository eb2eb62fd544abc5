"""Throughput of the FAVOR+ forward hot path on GB300.

One step = the whole hot path over one batch of synthetic input:
  build Omega (ORF) -> bidirectional FAVOR+ (state + output) -> causal
  FAVOR+ (superchunk states + scan/output), on the same Q, K, V.
Metric: tokens per second, a token being one (batch, position) with all H
heads, processed by both the bidirectional and the causal forward pass.

Default workload: bidir/causal bf16, B=8 H=8 L=4096 d=64 m=256 (the Regular
Transformer attention shape, 8 heads of 64).  ``--workload`` selects another
(see ``workloads``).  Prints ONE JSON line (rank 0).

Timed region: K replays of a CUDA graph holding one step, input sets rotated
so that the bytes touched between two uses of a set exceed L2; CUDA events on
the launching stream; barrier + synchronize on both sides; max over ranks.
Per-kernel durations (roofline) come from an event-instrumented pass of the
same steps.  ``--impl reference`` times the fp64 CPU oracle instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as wl  # noqa: E402

DEFAULT_WORKLOAD = "bidir-bf16-B8H8L4096-d64-m256"
L2_BYTES = 129 * 1024 * 1024
STAGES = ("build_orf", "bidir_state", "bidir_output", "causal_state", "causal_output")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--decode-steps", type=int, default=200)
    ap.add_argument("--relu-steps", type=int, default=100)
    ap.add_argument("--elu-steps", type=int, default=100)
    ap.add_argument("--bwd-steps", type=int, default=10)
    ap.add_argument("--config-steps", type=int, default=20,
                    help="calls timed per configuration line (0: no per-configuration lines)")
    ap.add_argument("--config-cpu-s", type=float, default=1.5,
                    help="seconds of oracle time per configuration line's cpu_baseline (0: none)")
    ap.add_argument("--call", default=None, metavar="WORKLOAD",
                    help="only run WORKLOAD's full forward call --calls times and print its mean time "
                         "(a small driver for profilers)")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--call-mode", default=None, choices=["bidir", "causal"],
                    help="with --call: run this pass instead of the workload's own")
    ap.add_argument("--call-backward", action="store_true",
                    help="with --call: run the pass's backward (dQ, dK, dV for a seeded dO) instead")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


class Ranks:
    """Host-side coordination of the replicas: a barrier around each timed
    region and the maximum of a per-rank time.  The path shards by (batch,
    head) with no exchange, so nothing else crosses ranks."""

    def __init__(self, world: int, device):
        self.world = world
        self.device = device

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(self, x: float) -> float:
        if self.world > 1:
            import torch.distributed as dist
            t = torch.tensor([x], dtype=torch.float64, device=self.device)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            return float(t.item())
        return x


def rank_input_seed(rank: int, i: int) -> int:
    """Seed of input set i on a rank: every rank processes its own units."""
    return 1000 * rank + i


def whole_job_value(world: int, tokens_per_step: int, steps: int, elapsed_ms_max: float) -> float:
    """Tokens per second of the whole job: every rank's tokens over the
    slowest rank's time (weak scaling: the per-rank workload is fixed)."""
    return world * tokens_per_step * steps / (elapsed_ms_max / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def workload_for(name: str):
    w = wl.get(name)
    return w


# ---------------------------------------------------------------------------
# algorithmic work per launch (per head-token figures times B*H*L)
# ---------------------------------------------------------------------------

def algorithmic(w, stage: str):
    """(bytes, flops) that the stage must move / compute for one launch."""
    e = 4 if w.dtype == "f32" else 2
    ht = w.B * w.H * w.L
    md, md1 = w.m * w.d, w.m * (w.d + 1)
    state_bytes = w.B * w.H * w.m * (w.d + 1) * 4
    if stage == "bidir_state":
        return ht * 2 * w.d * e + state_bytes, ht * (2 * md + 2 * md1)
    if stage == "bidir_output":
        return ht * 2 * w.d * e + state_bytes, ht * (2 * md + 2 * md1)
    if stage == "causal_state":
        return ht * 2 * w.d * e, ht * (2 * md + 2 * md1)
    if stage == "causal_output":
        return ht * 4 * w.d * e, ht * (4 * md + 4 * md1)
    if stage == "build_orf":
        return w.m * w.d * 4, 0
    raise KeyError(stage)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="favor_clocks_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# traffic from the committed ncu summary (null when the kernel source changed)
# ---------------------------------------------------------------------------

# The sources the tensor-core kernels (the profiled stages) are built from:
# a committed profile's counters stay valid while their code (comments and
# layout aside) does not change.
KERNEL_SOURCES = ("linear_softmax_attention_gb300/csrc/tc.cu", "linear_softmax_attention_gb300/csrc/tc_fs.cu",
                  "linear_softmax_attention_gb300/csrc/tc_bwd.cu",
                  "linear_softmax_attention_gb300/csrc/tc_util.cuh", "linear_softmax_attention_gb300/csrc/tc_ptx.cuh",
                  "linear_softmax_attention_gb300/csrc/common.cuh", "linear_softmax_attention_gb300/csrc/prep.cu",
                  "linear_softmax_attention_gb300/csrc/orf.cu", "linear_softmax_attention_gb300/csrc/decode.cu",
                  "include/favor.h")
_C_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def source_code_text(text: str) -> str:
    """C/C++ source without comments, whitespace runs collapsed (no comment
    marker sits inside a string literal in these files)."""
    return " ".join(_C_COMMENT.sub(" ", text).split())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as fh:
            h.update(source_code_text(fh.read()).encode())
            h.update(b"\0")
    return h.hexdigest()[:16]


def profiled_traffic(stage: str, workload: str):
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    src = kernel_source_hash()
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md"):
            continue
        text = open(os.path.join(pdir, f)).read()
        m_stage = re.search(r"^stage:\s*(\S+)", text, re.M)
        m_wl = re.search(r"^workload:\s*(\S+)", text, re.M)
        m_src = re.search(r"^source_hash:\s*(\S+)", text, re.M)
        m_tr = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        if m_stage and m_wl and m_src and m_tr and m_stage.group(1) == stage and m_wl.group(1) == workload:
            return float(m_tr.group(1)) if m_src.group(1) == src else None
    return None


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, rank, world, local_rank):
    import linear_softmax_attention_gb300 as favor

    favor.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = workload_for(args.workload)
    dt = w.torch_dtype
    B, H, L, d, m = w.B, w.H, w.L, w.d, w.m
    bytes_per_set = 3 * B * H * L * d * (4 if w.dtype == "f32" else 2)
    n_sets = max(2, -(-2 * L2_BYTES // bytes_per_set) + 1)
    n_sets = min(n_sets, 8)
    sets = []
    for i in range(n_sets):
        q, k, v = wl.make_qkv(w, seed=rank_input_seed(rank, i), device=dev)
        sets.append((q, k, v))
    O_b = torch.empty_like(sets[0][0])
    O_c = torch.empty_like(sets[0][0])
    # Omega is double-buffered: each step builds the next step's Omega on a
    # second stream while its own attention kernels (which leave SMs free)
    # run on the current one; every step builds one Omega and uses one
    omegas = [torch.empty((m, d), dtype=torch.float32, device=dev) for _ in range(2)]
    omega = omegas[0]
    side = torch.cuda.Stream(device=dev)
    # the causal pass runs on its own stream beside the bidirectional one:
    # the passes are independent and each kernel leaves SMs idle (grids of
    # whole heads' tiles), so their kernels overlap
    second = torch.cuda.Stream(device=dev)
    ev_fork = torch.cuda.Event()
    ev_join = torch.cuda.Event()
    ev_join2 = torch.cuda.Event()
    ws_b = favor.new_workspace(False, B, H, L, d, m, dt, device=dev)
    ws_c = favor.new_workspace(True, B, H, L, d, m, dt, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    s = w.qk_scale
    stream = torch.cuda.Stream(device=dev)

    def step(i, seed_call):
        q, k, v = sets[i % n_sets]
        cur, nxt = omegas[i % 2], omegas[(i + 1) % 2]
        ev_fork.record(stream)
        side.wait_event(ev_fork)
        second.wait_event(ev_fork)
        favor.build_orf(seed_call, nxt, stream=side)
        favor.causal_state(k, v, cur, s, ws_c, dev_status=status, stream=second)
        favor.causal_output(q, k, v, cur, s, ws_c, O=O_c, dev_status=status, stream=second)
        favor.bidir_state(k, v, cur, s, ws_b, dev_status=status, stream=stream)
        favor.bidir_output(q, cur, s, ws_b, O=O_b, dev_status=status, stream=stream)
        ev_join.record(side)
        stream.wait_event(ev_join)
        ev_join2.record(second)
        stream.wait_event(ev_join2)

    # the input sets and workspaces were made on the current stream; every
    # step runs on `stream`
    torch.cuda.synchronize(dev)
    favor.build_orf(wl.omega_seed_for_call(w, 0), omegas[0], stream=stream)

    # kernels of this library per step: tensor-core path = ORF, prep + state,
    # output, prep + state, causal scan; CUDA-core path = ORF, prep + partial
    # states + merge, output, prep + partial states, causal scan
    launches_per_step = 7 if favor.path_name(False, d, m, dt) != "simt" else 8

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i, wl.omega_seed_for_call(w, i + 1))
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up: "
                           f"{favor.status_string(int(status.item()))}")

    # graphs: one per input set (and per Omega seed when Omega is redrawn) for
    # the whole step, and one per stage for the per-kernel durations
    n_graphs = n_sets if not w.redraw_omega else max(n_sets, 4)
    n_graphs += n_graphs % 2          # graphs alternate the two Omega buffers
    stage_fns = (
        lambda i, q, k, v: favor.build_orf(wl.omega_seed_for_call(w, i), omega, stream=stream),
        lambda i, q, k, v: favor.bidir_state(k, v, omega, s, ws_b, dev_status=status, stream=stream),
        lambda i, q, k, v: favor.bidir_output(q, omega, s, ws_b, O=O_b, dev_status=status, stream=stream),
        lambda i, q, k, v: favor.causal_state(k, v, omega, s, ws_c, dev_status=status, stream=stream),
        lambda i, q, k, v: favor.causal_output(q, k, v, omega, s, ws_c, O=O_c, dev_status=status, stream=stream),
    )
    graphs, stage_graphs = [], []
    with torch.cuda.stream(stream):
        for i in range(n_graphs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(i, wl.omega_seed_for_call(w, i + 1))
            graphs.append(g)
            per = []
            for fn in stage_fns:
                gs = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gs, stream=stream):
                    fn(i, *sets[i % n_sets])
                per.append(gs)
            stage_graphs.append(per)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            graphs[i % n_graphs].replay()
            for gs in stage_graphs[i % n_graphs]:
                gs.replay()
    torch.cuda.synchronize(dev)

    ranks = Ranks(world, dev)
    barrier, max_over_ranks = ranks.barrier, ranks.max_over_ranks

    # timed region 1: K replays of the whole-step graph (the headline value)
    barrier()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    t_wall0 = time.perf_counter()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(args.steps):
            graphs[i % n_graphs].replay()
        end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    barrier()

    # timed region 2: the same K steps as per-stage graphs, an event on the
    # launching stream after each stage: per-kernel average launch durations
    n_ev = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)] for _ in range(n_ev)]
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(n_ev):
            e = evs[i]
            e[0].record(stream)
            for j, gs in enumerate(stage_graphs[i % n_graphs]):
                gs.replay()
                e[j + 1].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier()
    stage_ms = {st: max_over_ranks(statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n_ev)))
                for j, st in enumerate(STAGES)}
    elapsed_ms = max_over_ranks(start.elapsed_time(end))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the timed region")

    ms_per_step = elapsed_ms / args.steps
    tokens_per_step = B * L
    value = whole_job_value(world, tokens_per_step, args.steps, elapsed_ms)

    # e2e through the public calls (favor_build_orf, favor_fwd_bidir,
    # favor_fwd_causal) with pinned host buffers: every step copies its Q, K,
    # V host -> device and both outputs device -> host inside the timed
    # region.  Three streams pipeline the steps: the copies in of step i+1
    # and out of step i-1 run while step i computes (inputs and outputs
    # double-buffered on the device).
    e2e = None
    if args.e2e_steps > 0:
        hq, hk, hv = (t.cpu().pin_memory() for t in sets[0])
        dev_in = [tuple(torch.empty_like(t) for t in sets[0]) for _ in range(2)]
        dev_out = [(torch.empty_like(O_b), torch.empty_like(O_c)) for _ in range(2)]
        host_out = [tuple(torch.empty(O_b.shape, dtype=O_b.dtype, pin_memory=True) for _ in range(2))
                    for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        d2h = O_b.numel() * O_b.element_size() * 2
        s_in = [torch.cuda.Stream(device=dev) for _ in range(3)]   # one per input tensor
        s_out = torch.cuda.Stream(device=dev)
        ev_in = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        om_e2e = torch.empty((m, d), dtype=torch.float32, device=dev)
        ev_om, ev_c2 = torch.cuda.Event(), torch.cuda.Event()

        def e2e_step(i):
            b_ = i % 2
            dq, dk, dv = dev_in[b_]
            ob, oc = dev_out[b_]
            hob, hoc = host_out[b_]
            for j, (dst, src) in enumerate(((dq, hq), (dk, hk), (dv, hv))):
                with torch.cuda.stream(s_in[j]):
                    if i >= 2:
                        s_in[j].wait_event(ev_comp[b_])     # step i-2 has read these inputs
                    dst.copy_(src, non_blocking=True)
                    ev_in[b_][j].record(s_in[j])
                stream.wait_event(ev_in[b_][j])
            if i >= 2:
                stream.wait_event(ev_out[b_])               # step i-2's outputs have left
            favor.build_orf(wl.omega_seed_for_call(w, i), om_e2e, stream=stream)
            ev_om.record(stream)
            second.wait_event(ev_om)
            favor.fwd_causal(dq, dk, dv, om_e2e, s, ws_c, O=oc, dev_status=status, stream=second)
            favor.fwd_bidir(dq, dk, dv, om_e2e, s, ws_b, O=ob, dev_status=status, stream=stream)
            ev_c2.record(second)
            stream.wait_event(ev_c2)
            ev_comp[b_].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b_])
                hob.copy_(ob, non_blocking=True)
                hoc.copy_(oc, non_blocking=True)
                ev_out[b_].record(s_out)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for st_ in s_in:
            st_.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(args.e2e_steps):
            e2e_step(i)
        stream.wait_event(ev_out[(args.e2e_steps - 1) % 2])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} after the end-to-end steps")
        e2e = {"value": world * tokens_per_step / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "pipeline": "H2D of step i+1 (one stream per input) and D2H of step i-1 overlap step i"}

    hbm, tc_burst, tc_sus, peak_kind = load_peaks()
    decode = measure_decode(favor, args.decode_steps, stream, status, hbm, dev) if args.decode_steps > 0 else None
    bwd = None
    if args.bwd_steps > 0:
        bwd = measure_backward(favor, args.bwd_steps, sets, omegas[0], s, stream, status, dev, tokens_per_step, hbm)
    relu = None
    if args.relu_steps > 0:
        relu = measure_feature_map(favor, "relu", args.relu_steps, sets, omegas[0], s, ws_b, ws_c, O_b, O_c, stream,
                                   status, dev, tokens_per_step)
    elu1 = None
    if args.elu_steps > 0:
        elu1 = measure_feature_map(favor, "elu1", args.elu_steps, sets, omegas[0], s, ws_b, ws_c, O_b, O_c, stream,
                                   status, dev, tokens_per_step)
    configs = measure_configs(favor, args, dev, stream, status, hbm, tc_burst) if args.config_steps > 0 else None
    # dominant kernel: largest share of the step
    # the stage times come from sub-millisecond graph replays of one kernel
    # each: the burst tensor peak applies (the sustained one is for a kernel
    # timed inside a seconds-long loop)
    dom = max((st for st in STAGES if st != "build_orf"), key=lambda st: stage_ms[st])
    nbytes, nflops = algorithmic(w, dom)
    t_dom = stage_ms[dom] / 1e3
    t_hbm = nbytes / (hbm * 1e9)
    t_tc = nflops / (tc_burst * 1e12)
    if t_tc > t_hbm:
        roof = {"bound": "tensor", "achieved": nflops / t_dom / 1e12, "peak": tc_burst, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": nbytes / t_dom / 1e9, "peak": hbm, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profiled_traffic(dom, w.name)
    roof["kernel"] = dom
    roof["peak_source"] = f"{peak_kind} ({'burst bf16' if roof['bound'] == 'tensor' else 'HBM copy'})"
    roof["algorithmic_bytes_per_launch"] = nbytes
    roof["algorithmic_flops_per_launch"] = nflops
    stages_out = {}
    for st in STAGES:
        b_, f_ = algorithmic(w, st)
        t_ = stage_ms[st] / 1e3
        stages_out[st] = {"ms": stage_ms[st], "GB/s": b_ / t_ / 1e9, "TFLOP/s": f_ / t_ / 1e12,
                          "hbm_frac": b_ / t_ / 1e9 / hbm,
                          "roofline_frac": max(b_ / (hbm * 1e9), f_ / (tc_burst * 1e12)) / t_}
    bidir_ms = stage_ms["bidir_state"] + stage_ms["bidir_output"]
    causal_ms = stage_ms["causal_state"] + stage_ms["causal_output"]

    line = {
        "metric": "FAVOR+ fwd tokens/sec (bidir & causal) on 1 GB300; % of roofline",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; workloads module)",
        "config": {"workload": w.name, "B": B, "H": H, "L": L, "d": d, "m": m, "qk_scale": s,
                   "step": "build Omega + bidirectional + causal forward", "tokens_per_step": tokens_per_step,
                   "path": favor.path_name(False, d, m, dt), "l2": f"{n_sets} rotating input sets "
                   f"({n_sets * bytes_per_set / 2**20:.0f} MiB > L2)", "timing": "CUDA graph replay per step; per-kernel times from per-stage graphs with events between stages",
                   "omega": "each step builds the next step's Omega on a side stream (double-buffered) while its attention kernels run",
                   "streams": "the bidirectional and the causal pass on two streams (independent passes; their kernels overlap)",
                   "parallelism": f"replicas x{world}"},
        "modes": {"head_tokens_per_s": value * H,
                  "bidir_tokens_per_s": tokens_per_step / (bidir_ms / 1e3),
                  "causal_tokens_per_s": tokens_per_step / (causal_ms / 1e3),
                  "build_orf_ms": stage_ms["build_orf"],
                  "build_orf_hadamard_ms": time_build(favor, "hadamard", m, d, stream, dev),
                  "build_orf_givens_ms": time_build(favor, "givens", m, d, stream, dev)},
        "stages": stages_out,
        "roofline": roof,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "wall_s_timed": t_wall,
        "e2e": e2e,
        "decode": decode,
        "relu": relu,
        "elu1": elu1,
        "backward": bwd,
        "configs": configs,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=12.0)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


# ---------------------------------------------------------------------------
# one line per configuration: the full public call on each workload
# ---------------------------------------------------------------------------

CONFIGS = [
    # (configuration number, workload names)
    (1, ["bidir-f32-B1H1L512-d64-m64"]),
    (2, ["bidir-bf16-B8H8L4096-d64-m256"]),
    (3, ["causal-bf16-B4H8L8192-d64-m256"]),
    (4, ["causal-bf16-B2H8L12288-d64-m256"]),
    (5, list(wl.SWEEP)),
]


def alu_peak_tflops(dev) -> float:
    """fp32 FMA peak of the CUDA cores: SMs x 128 lanes x 2 flop x max SM clock."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
    except (OSError, KeyError, ValueError):
        mhz = 2070.0
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def call_roofline(w, ms: float, hbm: float, tc_burst: float, alu: float):
    """Roofline of one full forward call (state + output): algorithmic bytes
    4 d e and flops 4 m d + 4 m (d + 1) per head-token.  bf16 runs against the
    burst tensor peak and the HBM copy rate; fp32 storage runs on the CUDA
    cores, so against their FMA peak."""
    e = 4 if w.dtype == "f32" else 2
    ht = w.B * w.H * w.L
    nbytes = ht * 4 * w.d * e
    nflops = ht * (4 * w.m * w.d + 4 * w.m * (w.d + 1))
    t = ms / 1e3
    peak_f, unit_f, bound_f = (alu, "TFLOP/s", "alu") if w.dtype == "f32" else (tc_burst, "TFLOP/s", "tensor")
    if nflops / (peak_f * 1e12) > nbytes / (hbm * 1e9):
        r = {"bound": bound_f, "achieved": nflops / t / 1e12, "peak": peak_f, "unit": unit_f}
    else:
        r = {"bound": "hbm", "achieved": nbytes / t / 1e9, "peak": hbm, "unit": "GB/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["algorithmic_bytes_per_call"] = nbytes
    r["algorithmic_flops_per_call"] = nflops
    return r


def oracle_mode_rate(w, budget_s: float):
    """Head-tokens per second of the fp64 oracle on one head of a token
    prefix of the workload, in the workload's own mode, sized to take about
    ``budget_s`` (the oracle is linear in L in both modes)."""
    import numpy as np

    import oracle as orc
    causal = w.mode == "causal"
    f64 = (lambda t: t.float().numpy().astype(np.float64))
    om = orc.build_omega(wl.omega_seed_for_call(w, 0), w.m, w.d)

    def run(L):
        q, k, v = wl.make_qkv(w, seed=0, B=1, H=1, L=L)
        t0 = time.perf_counter()
        (orc.favor_causal if causal else orc.favor_bidirectional)(f64(q), f64(k), f64(v), om, w.qk_scale)
        return time.perf_counter() - t0

    L0 = min(w.L, 256)
    t0 = run(L0)
    Ls = int(min(w.L, max(L0, L0 * budget_s / max(t0, 1e-6))))
    t = run(Ls) if Ls != L0 else t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return Ls / t, Ls, cores


def measure_configs(favor, args, dev, stream, status, hbm, tc_burst):
    """Every configuration through the public full call (favor_fwd_bidir or
    favor_fwd_causal; for the redrawn-Omega workload favor_build_orf with the
    call's seed first, on the same stream).  Each call is timed alone with
    CUDA events on its stream, after a write of 2 x L2 that flushes the
    cache; value = B L tokens per mean call time."""
    alu = alu_peak_tflops(dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    out = {}
    cpu_done = set()
    for number, names in CONFIGS:
        for name in names:
            w = wl.get(name)
            causal = w.mode == "causal"
            q, k, v = wl.make_qkv(w, seed=0, device=dev)
            O = torch.empty_like(q)
            om = favor.new_omega(wl.omega_seed_for_call(w, 0), w.m, w.d, device=dev)
            ws = favor.new_workspace(causal, w.B, w.H, w.L, w.d, w.m, w.torch_dtype, device=dev)
            fn = favor.fwd_causal if causal else favor.fwd_bidir
            # inputs, Omega and workspace were made on the current stream; the
            # calls below run on `stream`
            torch.cuda.synchronize(dev)

            def call(i, build, part="both"):
                if build:
                    favor.build_orf(wl.omega_seed_for_call(w, i), om, stream=stream)
                if part == "both":
                    fn(q, k, v, om, w.qk_scale, ws, O=O, dev_status=status, stream=stream)
                elif part == "state":
                    (favor.causal_state if causal else favor.bidir_state)(k, v, om, w.qk_scale, ws,
                                                                         dev_status=status, stream=stream)
                elif causal:
                    favor.causal_output(q, k, v, om, w.qk_scale, ws, O=O, dev_status=status, stream=stream)
                else:
                    favor.bidir_output(q, om, w.qk_scale, ws, O=O, dev_status=status, stream=stream)

            def timed(build, part="both"):
                with torch.cuda.stream(stream):
                    for i in range(3):
                        call(i, build, part)
                torch.cuda.synchronize(dev)
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(args.config_steps)]
                with torch.cuda.stream(stream):
                    for i, (e0, e1) in enumerate(evs):
                        flush.fill_(i & 0xFF)
                        e0.record(stream)
                        call(i + 3, build, part)
                        e1.record(stream)
                torch.cuda.synchronize(dev)
                if int(status.item()) != 0:
                    raise RuntimeError(f"device status {int(status.item())} on {name}")
                return statistics.mean(a.elapsed_time(b) for a, b in evs)

            ms = timed(w.redraw_omega)
            line = {"config": number, "mode": w.mode, "dtype": w.dtype, "B": w.B, "H": w.H, "L": w.L, "d": w.d,
                    "m": w.m, "path": favor.path_name(causal, w.d, w.m, w.torch_dtype),
                    "value": w.B * w.L / (ms / 1e3), "unit": "tokens/s",
                    "head_tokens_per_s": w.B * w.H * w.L / (ms / 1e3), "ms_per_call": ms,
                    "calls": args.config_steps, "roofline": call_roofline(w, ms, hbm, tc_burst, alu),
                    "stage_ms": {"state": timed(False, "state"), "output": timed(False, "output")}}
            if w.redraw_omega:
                ms_c = timed(False)
                line["call"] = "favor_build_orf (seed of the call) + favor_fwd_causal, one stream"
                line["omega_cached"] = {"ms_per_call": ms_c, "value": w.B * w.L / (ms_c / 1e3)}
                line["build_share"] = (ms - ms_c) / ms
            # the oracle on a bounded sample: every named workload, and the
            # longest sequence of each (mode, m) of the sweep
            key = (w.mode, w.m) if number == 5 else name
            if args.config_cpu_s > 0 and key not in cpu_done and (number != 5 or w.L == 65536):
                cpu_done.add(key)
                rate, Ls, cores = oracle_mode_rate(w, args.config_cpu_s)
                line["cpu_baseline"] = {"value": rate / w.H, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                        "sample": f"one head of the first {Ls} tokens, {w.mode}, fp64 NumPy; "
                                                  f"tokens = head-tokens / H"}
            out[name] = line
            del q, k, v, O, ws
    del flush
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# CPU oracle: the reported baseline and the reference arm
# ---------------------------------------------------------------------------

def oracle_sample_step(w, heads: int, seed: int, L: int | None = None):
    """One bounded oracle step: Omega + bidirectional + causal on `heads` heads
    of the workload (optionally its first L tokens)."""
    import numpy as np

    import oracle as orc
    q, k, v = wl.make_qkv(w, seed=seed, B=1, H=heads, L=L)
    f64 = (lambda t: t.float().numpy().astype(np.float64))
    Q, K, V = f64(q), f64(k), f64(v)
    om = orc.build_omega(wl.omega_seed_for_call(w, seed), w.m, w.d)
    orc.favor_bidirectional(Q, K, V, om, w.qk_scale)
    orc.favor_causal(Q, K, V, om, w.qk_scale)


def cpu_baseline(w, budget_s: float):
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    heads = 1
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle_sample_step(w, heads, seed=n)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt_s = time.perf_counter() - t0
    # a step covers B*L tokens x H heads; the sample covers `heads` heads of L tokens
    tokens = n * w.L * heads / w.H
    return {"value": tokens / dt_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} x (Omega build + bidirectional + causal) on {heads} head(s) of L={w.L}, "
                      f"d={w.d}, m={w.m} in fp64 NumPy; tokens = head-tokens / H"}


def run_reference(args, rank, world):
    """The fp64 CPU oracle as the reference arm: exactly K timed steps, each
    on one head of a token prefix sized so that the run stays within minutes."""
    if rank != 0:
        return
    w = workload_for(args.workload)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    t0 = time.perf_counter()
    oracle_sample_step(w, 1, seed=0)
    t_full = time.perf_counter() - t0
    budget = 90.0
    Ls = w.L if args.steps * t_full <= budget else max(64, int(w.L * budget / (args.steps * t_full)))
    for i in range(max(0, min(args.warmup, 3) - 1)):
        oracle_sample_step(w, 1, seed=1 + i, L=Ls)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_sample_step(w, 1, seed=100 + i, L=Ls)
    dt_s = time.perf_counter() - t0
    tokens_per_step = Ls / w.H
    value = tokens_per_step * args.steps / dt_s
    sample = f"one head of {Ls} tokens per step (Omega build + bidirectional + causal, fp64 NumPy); " \
             f"tokens = head-tokens / H"
    line = {
        "impl": "reference",
        "metric": "FAVOR+ fwd tokens/sec (bidir & causal) on 1 GB300; % of roofline",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt_s / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; workloads module)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d, "m": w.m,
                   "step": "build Omega + bidirectional + causal forward"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def time_build(favor, kind, m, d, stream, dev, reps=20):
    """Mean duration of favor_build_orf of the given kind (CUDA events)."""
    om = torch.empty((m, d), dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        favor.build_orf(0, om, orthogonal=kind, stream=stream)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(reps):
            favor.build_orf(i, om, orthogonal=kind, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps


def measure_backward(favor, n_steps, sets, omega, s, stream, status, dev, tokens_per_step, hbm):
    """favor_bwd_bidir and favor_bwd_causal on the step's workload (the
    bidirectional pass on the tensor-core kernels, the causal pass on the
    CUDA-core ones): dQ, dK, dV for a seeded dO, inputs rotating over the
    sets, one CUDA graph per set.
    Algorithmic bytes: read Q, K, V, dO and write dQ, dK, dV (7 d e per
    head-token)."""
    q0 = sets[0][0]
    B, H, L, d = q0.shape
    gen = torch.Generator(device="cpu")
    gen.manual_seed(5)
    dO = torch.randn(q0.shape, generator=gen).to(q0.dtype).to(dev)
    ws = torch.empty(favor.bwd_workspace_bytes(B, H, L, d, omega.shape[0], q0.dtype), dtype=torch.uint8, device=dev)
    dQ, dK, dV = torch.empty_like(q0), torch.empty_like(q0), torch.empty_like(q0)
    torch.cuda.synchronize(dev)      # dO was made on the current stream
    out = {}
    for causal in (False, True):
        graphs = []
        for q, k, v in sets:
            with torch.cuda.stream(stream):
                favor.bwd_bidir(q, k, v, dO, omega, s, ws, dQ=dQ, dK=dK, dV=dV, dev_status=status, stream=stream,
                                causal=causal)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                favor.bwd_bidir(q, k, v, dO, omega, s, ws, dQ=dQ, dK=dK, dV=dV, dev_status=status, stream=stream,
                                causal=causal)
            graphs.append(g)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            graphs[0].replay()
            e0.record(stream)
            for i in range(n_steps):
                graphs[i % len(graphs)].replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} after the backward steps")
        ms = e0.elapsed_time(e1) / n_steps
        nbytes = 7 * q0.numel() * q0.element_size()
        out["causal" if causal else "bidir"] = {
            "value": tokens_per_step / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "steps": n_steps,
            "hbm_frac": nbytes / (ms / 1e3) / 1e9 / hbm}
    out["step"] = "backward (dQ, dK, dV) of each pass: bidirectional on tcgen05, causal on CUDA cores"
    return out


def measure_feature_map(favor, fm, n_steps, sets, omega, s, ws_b, ws_c, O_b, O_c, stream, status, dev,
                        tokens_per_step):
    """The bidirectional and causal forward passes of the step with another
    feature map (Performer-ReLU, 1 + elu): same workload, Omega built once,
    inputs rotating over the sets (above L2), one CUDA graph per input set."""
    graphs = []
    for q, k, v in sets:
        with torch.cuda.stream(stream):
            for _ in range(2):
                favor.fwd_bidir(q, k, v, omega, s, ws_b, O=O_b, dev_status=status, stream=stream, feature_map=fm)
                favor.fwd_causal(q, k, v, omega, s, ws_c, O=O_c, dev_status=status, stream=stream, feature_map=fm)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            favor.fwd_bidir(q, k, v, omega, s, ws_b, O=O_b, dev_status=status, stream=stream, feature_map=fm)
            favor.fwd_causal(q, k, v, omega, s, ws_c, O=O_c, dev_status=status, stream=stream, feature_map=fm)
        graphs.append(g)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for g in graphs:
            g.replay()
        e0.record(stream)
        for i in range(n_steps):
            graphs[i % len(graphs)].replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the {fm} steps")
    ms = e0.elapsed_time(e1) / n_steps
    return {"feature_map": fm, "value": tokens_per_step / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "steps": n_steps, "step": "bidirectional + causal forward (Omega built once)"}


DECODE_B, DECODE_H, DECODE_D, DECODE_M = 256, 8, 64, 256


def measure_decode(favor, n_steps, stream, status, hbm, dev):
    """Incremental causal decoding (favor_decode_step): one token for each of
    B sequences x H heads per step, d64 m256 bf16.  The fp32 state
    [B, H, d + 1, m] is 136 MB, above the 129 MB L2, so every step reads and
    writes it from HBM; algorithmic bytes per step = state read + write +
    q, k, v, o.  Steps are replayed from a CUDA graph of 10 launches."""
    B, H, d, m = DECODE_B, DECODE_H, DECODE_D, DECODE_M
    gen = torch.Generator(device="cpu")
    gen.manual_seed(11)
    q, k, v = (torch.randn((B, H, d), generator=gen).to(torch.bfloat16).to(dev) for _ in range(3))
    om = favor.new_omega(11, m, d)
    state = favor.new_decode_state(B, H, m, d)
    o = torch.empty_like(q)
    s = d ** -0.25
    per_graph = 10
    torch.cuda.synchronize(dev)      # inputs, Omega and state were made on the current stream
    with torch.cuda.stream(stream):
        for _ in range(3):
            favor.decode_step(q, k, v, om, s, state, o=o, dev_status=status, stream=stream)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(per_graph):
            favor.decode_step(q, k, v, om, s, state, o=o, dev_status=status, stream=stream)
    reps = max(1, n_steps // per_graph)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after the decode steps")
    ms = e0.elapsed_time(e1) / (reps * per_graph)
    state_bytes = B * H * m * (d + 1) * 4
    nbytes = 2 * state_bytes + 4 * B * H * d * 2
    achieved = nbytes / (ms / 1e3) / 1e9
    return {"workload": f"decode-bf16-B{B}H{H}-d{d}-m{m}", "value": B / (ms / 1e3), "unit": "tokens/s",
            "ms_per_step": ms, "steps": reps * per_graph, "state_bytes": state_bytes,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "algorithmic_bytes_per_launch": nbytes}}


def run_call_only(args):
    """One workload's public full call (favor_fwd_bidir or favor_fwd_causal,
    or with --call-backward favor_bwd_*), --calls times on the current
    stream, Omega built once."""
    import linear_softmax_attention_gb300 as favor

    favor.load()
    dev = torch.device("cuda", 0)
    w = workload_for(args.call)
    causal = (args.call_mode or w.mode) == "causal"
    q, k, v = wl.make_qkv(w, seed=0, device=dev)
    om = favor.new_omega(wl.omega_seed_for_call(w, 0), w.m, w.d, device=dev)
    ws = favor.new_workspace(causal, w.B, w.H, w.L, w.d, w.m, w.torch_dtype, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    fn = favor.fwd_causal if causal else favor.fwd_bidir
    O = torch.empty_like(q)
    if args.call_backward:
        gen = torch.Generator(device="cpu")
        gen.manual_seed(5)
        dO = torch.randn(q.shape, generator=gen).to(q.dtype).to(dev)
        ws = torch.empty(favor.bwd_workspace_bytes(w.B, w.H, w.L, w.d, w.m, w.torch_dtype), dtype=torch.uint8,
                         device=dev)
        grads = (torch.empty_like(q), torch.empty_like(q), torch.empty_like(q))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record()
    for _ in range(args.calls):
        if args.call_backward:
            favor.bwd_bidir(q, k, v, dO, om, w.qk_scale, ws, dQ=grads[0], dK=grads[1], dV=grads[2],
                            dev_status=status, causal=causal)
        else:
            fn(q, k, v, om, w.qk_scale, ws, O=O, dev_status=status)
    e1.record()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} on {w.name}")
    print(json.dumps({"call": w.name, "mode": "causal" if causal else "bidir", "backward": args.call_backward,
                      "calls": args.calls,
                      "ms_per_call": e0.elapsed_time(e1) / args.calls,
                      "path": favor.path_name(causal, w.d, w.m, w.torch_dtype)}))


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.call is not None:
        run_call_only(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()

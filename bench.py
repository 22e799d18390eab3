#!/usr/bin/env python3
"""Benchmark of the topology-aware expert-routing plan on GB300.

One step = the whole hot path on one batch of synthetic routing ids already
resident in HBM: topo_hist -> topo_plan -> topo_reroute_layout (rerouting and
dispatch layout in one pass over the pairs).  The workload is the stress configuration (T = 1,048,576
tokens x k = 10 over E = 512 experts, R = 128 ranks in 16 nodes of 8, 64
replica slots per rank, 4 microbatches planned per call): 41.9 M
(token, slot) pairs per step, 168 MB of ids -- larger than the 129 MB L2, so
no flush is needed between steps.

Printed (one JSON line, rank 0): pairs/s for the device-resident step
(`value`), the same through host buffers with the copies inside the timed
region (`e2e`), the dominant call's roofline against the measured HBM
bandwidth, the oracle timed on a bounded sample of the same workload on the
host cores (`cpu_baseline`), plus the planner latency on the T = 16384,
E = 64, R = 32 workload and the co-occurrence kernel's HBM fraction on the
L = 8, T = 262144, E = 128 workload as secondary figures.

--impl reference times the CPU oracle (the only reference this method has)
on bounded samples of the same workload.
Multi-GPU (torchrun): each rank plans its own independent replica of the
workload (weak scaling, no data-path collective); time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

# algorithmic HBM bytes per (token, slot) pair: hist reads the id; the fused
# reroute+layout reads the id and writes dst_inst and sorted_pairs
BYTES_PER_PAIR = {"hist": 4, "reroute_layout": 12}
KERNELS_PER_CALL = {"hist": 2, "plan": 4, "reroute_layout": 5, "cooccur": 2, "dedup": 4, "gate": 2, "shuffle": 2, "place": 1}
CALLS = ("hist", "plan", "reroute_layout")
# kernel sources of each call (with the shared header): recorded DRAM traffic
# counts only while these are unchanged
CALL_SOURCE = {"hist": ("k_hist.cu",), "plan": ("k_plan.cu",),
               "reroute_layout": ("k_prep.cu", "k_route.cu"), "cooccur": ("k_cooccur_mma.cu",)}
CALL_KERNEL = {"hist": "k_hist_tiles", "reroute_layout": "k_route_tiles", "cooccur": "k_cooccur"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--skip-secondary", action="store_true", help="only the main line's fields")
    ap.add_argument("--skip-cpu", action="store_true", help="no oracle baseline")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--only", choices=("plan_latency", "cooccur", "pack", "dedup", "gate", "shuffle", "place",
                                       "configs", "solver", "chain"),
                    help="run one secondary measurement alone and print it (for profiling); chain: the "
                         "hot path hist -> plan -> reroute_layout twice, untimed (an ncu target)")
    ap.add_argument("--microbatches", type=int, default=0,
                    help="--only gate / chain: microbatches of the workload to use (0 = all; 1 for ncu captures)")
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="--impl reference: seconds the oracle steps should take in total")
    return ap.parse_args()


# ----------------------------------------------------------------------- utils

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def source_sha(call: str) -> str:
    h = hashlib.sha256()
    for name in CALL_SOURCE[call] + ("common.cuh",):
        with open(os.path.join(ROOT, "moe_expert_routing_ids_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(call: str, units: int):
    """DRAM bytes per launch of the call's main kernel from the committed ncu
    summary, scaled to `units` pairs (or ids), or None if absent or stale."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f).get(call)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_sha") != source_sha(call):
        return None
    return rec["dram_bytes"] * units / rec["units"]


def host_info() -> dict:
    """The host the oracle baseline ran on: logical CPUs and CPU model."""
    import platform
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                if key.strip().lower() in ("model name", "cpu model", "hardware"):
                    model = val.strip()
                    break
    except OSError:
        pass
    if not model:                                  # Arm kernels list no model name; lscpu does
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            model = next((l.split(":", 1)[1].strip() for l in out.splitlines()
                          if l.lower().startswith("model name")), "")
        except (OSError, subprocess.SubprocessError):
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.processor() or platform.machine()}


def max_over_ranks(x: float, device="cpu") -> float:
    """The largest x over the ranks of the default process group (x itself
    without one): the job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [int(r[1]) for r in rows]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": int(statistics.median(sm)), "sm_max_mhz": int(rows[0][2]),
                "reasons": reasons, "samples": len(rows)}


class GraphEvents:
    """CUDA events recorded as graph nodes (cudaEventRecordExternal), so a
    captured step keeps per-call timestamps on every replay."""

    def __init__(self, n):
        import ctypes
        import ctypes.util
        names = ["libcudart.so.13", "libcudart.so", ctypes.util.find_library("cudart") or ""]
        for n_ in names:
            try:
                self.rt = ctypes.CDLL(n_)
                break
            except OSError:
                continue
        else:
            raise RuntimeError("libcudart not found")
        self.ct = ctypes
        self.ev = []
        for _ in range(n):
            h = ctypes.c_void_p()
            if self.rt.cudaEventCreate(ctypes.byref(h)) != 0:
                raise RuntimeError("cudaEventCreate failed")
            self.ev.append(h)

    def record(self, i, stream):
        rc = self.rt.cudaEventRecordWithFlags(self.ev[i], self.ct.c_void_p(stream.cuda_stream), 1)
        if rc != 0:
            raise RuntimeError(f"cudaEventRecordWithFlags failed: {rc}")

    def elapsed(self, i, j):
        ms = self.ct.c_float()
        if self.rt.cudaEventElapsedTime(self.ct.byref(ms), self.ev[i], self.ev[j]) != 0:
            raise RuntimeError("cudaEventElapsedTime failed")
        return ms.value

    def close(self):
        for h in self.ev:
            self.rt.cudaEventDestroy(h)


def cpu_sample_chain(w, ids_layer):
    """Oracle chain on one microbatch of ids [1, T', k] (T' may be a slice of
    the workload's T, a multiple of R): (seconds, pairs)."""
    import oracle
    cfg = dict(w.plan_cfg, T=int(ids_layer.shape[1]))
    t0 = time.perf_counter()
    h = oracle.hist(ids_layer, w.R, w.E)
    p = oracle.plan(cfg, h)
    d = oracle.reroute(cfg, ids_layer, p)
    oracle.layout(cfg, d)
    return time.perf_counter() - t0, int(ids_layer.size)


def reference_slice_tokens(w, rate: float, steps: int, warmup: int, budget_s: float) -> int:
    """Tokens per oracle step so that warm-up + steps take about budget_s at
    `rate` pairs/s: a multiple of R, between R and T."""
    per_step = budget_s / max(1, steps + warmup)
    t = int(per_step * rate / w.k) // w.R * w.R
    return max(w.R, min(w.T, t))


# ------------------------------------------------------------------ reference

def run_reference(args, rank):
    """CPU oracle arm, rank 0 only: exactly `steps` timed steps, each the
    oracle chain (hist, plan, reroute, layout) on one token slice of a stress
    microbatch; the slice is sized from a calibration run so the whole arm
    takes about --ref-budget-s seconds, and consecutive steps take
    consecutive slices.  Metric and unit as ours."""
    if rank != 0:
        return
    import oracle
    from moe_expert_routing_ids_gb300 import workloads as W
    oracle.build()
    w = W.STRESS
    ids = w.ids(n_layers=1)
    cal_t = max(w.R, (w.T // 64) // w.R * w.R)
    cal_s, cal_n = cpu_sample_chain(w, ids[:, :cal_t])
    t_s = reference_slice_tokens(w, cal_n / max(cal_s, 1e-9), args.steps, args.warmup,
                                 args.ref_budget_s)
    n_slices = max(1, w.T // t_s)

    def step(i):
        o = (i % n_slices) * t_s
        return cpu_sample_chain(w, ids[:, o:o + t_s])

    for i in range(args.warmup):
        step(i)
    secs, pairs = 0.0, 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        s, n = step(args.warmup + i)
        secs += s
        pairs += n
    wall = time.perf_counter() - t0
    value = pairs / secs
    sample = (f"per step {t_s} of the {w.T} tokens of one stress microbatch ({t_s * w.k} pairs), "
              f"oracle hist+plan+reroute+layout single-threaded; {args.steps} steps, {secs:.1f} s")
    line = {"impl": "reference", "metric": "routed (token,slot) pairs/sec", "value": value,
            "unit": "pairs/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * wall / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "E": w.E, "k": w.k, "R": w.R,
                       "ranks_per_node": w.ranks_per_node, "n_slot": w.n_slot,
                       "microbatches": w.n_layers, "tokens_per_step": t_s,
                       "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": "pairs/s", "cores": 1, "kind": "oracle", "host": host_info(),
                             "sample": sample},
            "e2e": {"value": value, "unit": "pairs/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------ ours

STEPS_PER_GRAPH = 20


def capture_steps(P, d_ids, n_steps, stream, gev):
    """One CUDA graph of n_steps whole steps, with an event node before every
    call and after the last one (len(CALLS) * n_steps + 1 events)."""
    import torch
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for k in range(n_steps):
            base = k * len(CALLS)
            gev.record(base, stream)
            P.hist(d_ids)
            gev.record(base + 1, stream)
            P.make_plan()
            gev.record(base + 2, stream)
            P.reroute_layout(d_ids)
        gev.record(n_steps * len(CALLS), stream)
    return graph


def capture_plain(P, d_ids, n_steps, stream):
    """One CUDA graph of n_steps whole steps, nothing between the calls."""
    import torch
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(n_steps):
            P.hist(d_ids)
            P.make_plan()
            P.reroute_layout(d_ids)
    return graph


CALL_REPLAYS = 5      # replays of the event-instrumented graph for the per-call times


def time_chain(P, d_ids, steps, stream):
    """Times exactly `steps` steps, replayed from CUDA graphs of up to 20 steps
    with nothing between the calls (an event node between calls breaks the
    programmatic launch chain and costs about 4% of the step); returns total
    ms (events around all replays).  Then, for the per-call times, replays the
    same steps captured with an event node before every call CALL_REPLAYS
    times and returns each call's mean."""
    import torch
    n_in = min(STEPS_PER_GRAPH, steps)
    full, rem = divmod(steps, n_in)
    g_main = capture_plain(P, d_ids, n_in, stream)
    g_rem = capture_plain(P, d_ids, rem, stream) if rem else None
    gev = GraphEvents(n_in * len(CALLS) + 1)
    g_ev = capture_steps(P, d_ids, n_in, stream, gev)
    for g in (g_main, g_rem, g_ev):                 # settle
        if g is not None:
            g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(full):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        t1.record(stream)
    t1.synchronize()
    total = t0.elapsed_time(t1)
    per_call = {c: [] for c in CALLS}
    for _ in range(CALL_REPLAYS):
        with torch.cuda.stream(stream):
            g_ev.replay()
        torch.cuda.synchronize()
        for k in range(n_in):
            for i, c in enumerate(CALLS):
                per_call[c].append(gev.elapsed(k * len(CALLS) + i, k * len(CALLS) + i + 1))
    gev.close()
    del g_main, g_rem, g_ev
    return total, steps, {c: statistics.mean(v) for c, v in per_call.items()}


def secondary_plan_latency(dev, stream):
    """topo_plan latency per layer on the T=16384, E=64, R=32 workload: 200
    calls captured in one CUDA graph, after 20 warm-up calls (TopoEP §6.3
    protocol), mean per call."""
    import torch
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Planner
    w = W.PLAN_LATENCY
    P = Planner(w.plan_cfg, w.n_layers, dev, stream=stream)
    ids = torch.as_tensor(w.ids(), device=dev)
    with torch.cuda.stream(stream):
        P.hist(ids)
        for _ in range(20):
            P.make_plan()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(200):
            P.make_plan()
    graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        graph.replay()
        b.record(stream)
    b.synchronize()
    us = a.elapsed_time(b) * 1e3 / 200 / w.n_layers
    return {"workload": w.name, "us_per_layer": round(us, 2), "reps": 200, "warmup": 20,
            "target_us": 40, "timing": "200 calls in one CUDA graph"}


def bf16_peak():
    """Measured dense bf16 tensor throughput (TFLOP/s, burst) and its kind."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def secondary_cooccur(dev, stream, hbm_peak):
    """topo_cooccur on the L = 8, T = 262144, E = 128, k = 8 workload, L2
    flushed before each call, median of 10 after 3 warm-up replays: the
    tensor-core path (count tiles in e4m3, tcgen05.mma into float32 tensor
    memory) against its dense-contraction FLOPs and the fp8 peak (the
    measured bf16 peak x 2, the nominal fp8 : bf16 ratio), and the same call
    on the shared-atomic kernels beside it."""
    import torch
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Cooccur
    w = W.COOCCUR
    ids = torch.as_tensor(w.ids(), device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for tc in (True, False):
        C = Cooccur(w.n_layers, w.T, w.E, w.k, dev, tensor_cores=tc)
        gev = GraphEvents(2)
        with torch.cuda.stream(stream):
            C.run(ids, stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            flush.fill_(1)                          # evict the ids from L2 (64 MiB < L2)
            gev.record(0, stream)
            C.run(ids, stream)
            gev.record(1, stream)
        times = []
        for _ in range(13):
            graph.replay()
            torch.cuda.synchronize()
            times.append(gev.elapsed(0, 1))
        gev.close()
        if C.error() != 0:
            raise RuntimeError("device error in the co-occurrence measurement")
        out[tc] = statistics.median(times[3:])
        del graph, C
    ms = out[True]
    nbytes = w.n_layers * w.T * w.k * 4 + (2 * w.n_layers - 1) * w.E * w.E * 8
    gbs = nbytes / (ms * 1e-3) / 1e9
    # dense contraction the tensor cores run: M = 128 experts, N = 256 (co and
    # tr together) for layers with a successor, 128 for the last, K = T
    flops = sum(2 * 128 * (256 if l + 1 < w.n_layers else 128) * w.T for l in range(w.n_layers))
    bf16, kind = bf16_peak()
    tflops = flops / (ms * 1e-3) / 1e12
    return {"workload": w.name, "ms": round(ms, 4), "path": "tensor cores (tcgen05, e4m3 counts, fp32 accumulate)",
            "algorithmic_bytes": nbytes, "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
            "tensor_roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": 2 * bf16,
                                "unit": "TFLOP/s", "frac": round(tflops / (2 * bf16), 4),
                                "peak_kind": f"{kind} bf16 x 2 (fp8)", "flops": flops},
            "atomics_ms": round(out[False], 4),
            "l2": "flushed (256 MB write) before each call",
            "traffic": profiled_traffic("cooccur", w.n_layers * w.T * w.k)}


L2_BYTES = 129 << 20


def plan_quality(w, stats, lstats, hist):
    """Plan-quality and locality figures of one call over all its layers, the
    numbers the pages judge a plan by: rank-load imbalance max/mean (TopoEP §6
    Fig. 10, Fig. 13b), the share of token-expert assignments that cross
    nodes and the share served by replicas (Fig. 16), and the intra- and
    inter-node dispatch bytes (§2.3 Fig. 3).  stats / lstats: the plan and
    layout statistics [L, 8]; hist: Omega [L, R, E], used only for the static
    placement's inter-node share (every pair on its expert's main rank)."""
    L = stats.shape[0]
    pairs = w.T * w.k * L
    mean = stats[:, 7] / w.R
    e_r = w.E // w.R
    dom_src = np.arange(w.R) // w.ranks_per_node
    dom_main = (np.arange(w.E) // e_r) // w.ranks_per_node
    cross = dom_src[:, None] != dom_main[None, :]
    static_inter = int(sum(int(hist[l][cross].sum()) for l in range(L)))
    return {
        "L_max": stats[:, 0].tolist(), "L_max_static": stats[:, 1].tolist(),
        "imbalance_max_over_mean": [round(float(a / m), 4) if m else None for a, m in zip(stats[:, 0], mean)],
        "imbalance_static": [round(float(a / m), 4) if m else None for a, m in zip(stats[:, 1], mean)],
        "replicas": int(stats[:, 2].sum()), "replicas_inter_node_stage": int(stats[:, 3].sum()),
        "refine_commits": int(stats[:, 4].sum()),
        "inter_node_pairs_frac": round(float(lstats[:, 2].sum()) / max(pairs, 1), 5),
        "inter_node_pairs_frac_static": round(static_inter / max(pairs, 1), 5),
        "replica_served_pairs_frac": round(float(lstats[:, 6].sum()) / max(pairs, 1), 5),
        "pairs_local_intra_inter": [int(lstats[:, i].sum()) for i in (0, 1, 2)],
        "bytes_local_intra_inter": [int(lstats[:, i].sum()) for i in (3, 4, 5)],
        "T_token": int(stats[:, 5].sum()), "T_replica": int(stats[:, 6].sum())}


def oracle_chain_stats(w, ids):
    """The oracle's plan and layout statistics and Omega for the same ids."""
    import oracle
    cfg = w.plan_cfg
    h = oracle.hist(ids, w.R, w.E)
    p = oracle.plan(cfg, h)
    d = oracle.reroute(cfg, ids, p)
    _, _, _, st = oracle.layout(cfg, d)
    return np.asarray(p["stats"]).reshape(-1, 8), np.asarray(st).reshape(-1, 8), h


def config_lines(dev, stream, hbm_peak, check_oracle=True):
    """Every plan workload (the T=4096 E=8, T=16384 E=64, four-layer and stress
    configurations): the whole chain hist -> plan -> reroute_layout timed as
    200 steps after 20 warm-up steps (TopoEP §6.3 protocol) in CUDA graphs with
    event nodes between the calls; pairs/s, per-layer plan latency, %HBM
    where the ids exceed L2 (else the replayed steps are L2-resident and only
    latency is reported); and the plan-quality figures, checked equal to the
    oracle's on the same ids."""
    import torch
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Planner
    out = {}
    for w in W.PLAN_WORKLOADS:
        ids = w.ids()
        d_ids = torch.as_tensor(ids, device=dev)
        P = Planner(w.plan_cfg, w.n_layers, dev, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(20):
                P.run(d_ids)
        if P.error() != 0:
            raise RuntimeError(f"device error on {w.name}")
        total, n, per_call = time_chain(P, d_ids, 200, stream)
        if P.error() != 0:
            raise RuntimeError(f"device error on {w.name}")
        ms = total / n
        pairs = int(ids.size)
        b = P.numpy()
        entry = {"pairs": pairs, "layers": w.n_layers, "ms_per_step": round(ms, 5),
                 "pairs_per_s": round(pairs / (ms * 1e-3), 1),
                 "us_per_call": {c: round(per_call[c] * 1e3, 2) for c in CALLS},
                 "plan_us_per_layer": round(per_call["plan"] * 1e3 / w.n_layers, 2),
                 "ids_bytes": int(ids.nbytes)}
        if ids.nbytes > L2_BYTES:
            entry["hbm_frac"] = {c: round(BYTES_PER_PAIR[c] * pairs / (per_call[c] * 1e-3) / 1e9 / hbm_peak, 4)
                                 for c in BYTES_PER_PAIR}
        else:
            entry["hbm_frac"] = None
            entry["l2"] = "ids fit in L2: latency only"
        entry["quality"] = plan_quality(w, b["stats"], b["layout_stats"], b["hist"])
        if check_oracle:
            ost, olst, oh = oracle_chain_stats(w, ids)
            entry["quality_equals_oracle"] = bool(np.array_equal(ost, b["stats"]) and
                                                  np.array_equal(olst, b["layout_stats"]) and
                                                  np.array_equal(oh, b["hist"]))
        out[w.name] = entry
        del P, d_ids
    return out


def solver_sweep(dev, stream):
    """topo_plan latency shaped like TopoEP §6.3 Fig. 11: (a) E = 640, Top-8,
    EP 8..128; (b) EP 32 over a 16x range of expert counts.  Each point: one
    hist, 20 warm-up plan calls, then 200 calls in one CUDA graph, mean per
    call; the oracle's plan of the same Omega timed beside it (one call,
    single-threaded), and the plan's imbalance."""
    import torch
    import oracle
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Planner
    res = {}
    for label, pts in (("rank_scaling_e640", W.SOLVER_RANKS), ("expert_scaling_r32", W.SOLVER_EXPERTS)):
        rows = []
        for w in pts:
            ids = w.ids()
            P = Planner(w.plan_cfg, 1, dev, stream=stream)
            d_ids = torch.as_tensor(ids, device=dev)
            with torch.cuda.stream(stream):
                P.hist(d_ids)
                for _ in range(20):
                    P.make_plan()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(200):
                    P.make_plan()
            graph.replay()
            torch.cuda.synchronize()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                graph.replay()
                z.record(stream)
            z.synchronize()
            us = a.elapsed_time(z) * 1e3 / 200
            if P.error() != 0:
                raise RuntimeError(f"device error on {w.name}")
            st = P.buf.stats.cpu().numpy()[0]
            h = oracle.hist(ids, w.R, w.E)
            t0 = time.perf_counter()
            ost = oracle.plan(w.plan_cfg, h)["stats"].reshape(-1)
            o_us = (time.perf_counter() - t0) * 1e6
            rows.append({"E": w.E, "R": w.R, "T": w.T, "us": round(us, 2), "oracle_us": round(o_us, 1),
                         "imbalance": round(float(st[0] / (st[7] / w.R)), 4),
                         "imbalance_static": round(float(st[1] / (st[7] / w.R)), 4),
                         "replicas": int(st[2]), "refine_commits": int(st[4]),
                         "stats_equal_oracle": bool(np.array_equal(st, ost))})
            del graph, P, d_ids
        res[label] = rows
    res["setup"] = ("Top-8, n_slot 2, 4096 tokens per rank, 8 ranks per node, Zipf(1.2), hidden 2048, "
                    "intermediate 768; 200 calls after 20 warm-ups, mean")
    return res


SHUFFLE_RANKS = 16           # EP16 over the co-occurrence workload's 128 experts
PLACE_RANKS = 8              # EP8, the scale at which the pages report deduplication savings


def secondary_place(dev, stream):
    """topo_place_experts on the co-occurrence workload's 8 layers (E = 128)
    at EP8: one call for all layers timed with CUDA events (median of 5 after
    2 warm-up calls), then, for its first layer, the rows the deduplicated
    dispatch layout sends with the contiguous and with the correlated map
    (plan with no replica slots, so every pair goes to its expert's main
    rank)."""
    import torch
    import moe_expert_routing_ids_gb300 as topo
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Cooccur, Planner
    w = W.COOCCUR
    L, T, E, k, R = w.n_layers, w.T, w.E, w.k, PLACE_RANKS
    ids_np = w.ids()
    ids = torch.as_tensor(ids_np, device=dev)
    C = Cooccur(L, T, E, k, dev, transitions=False)
    with torch.cuda.stream(stream):
        C.run(ids, stream)
    mr = torch.empty((L, E), dtype=torch.int32, device=dev)
    st = torch.empty((L, topo.TOPO_PLACE_STATS), dtype=torch.int64, device=dev)
    s = stream.cuda_stream
    times = []
    for i in range(7):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            topo.topo_place_experts(L, E, R, 0, C.co, mr, st, s)
            b.record(stream)
        b.synchronize()
        if i >= 2:
            times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    stn = st.cpu().numpy()
    # the swap phase: uniform random co-selection counts (no planted groups),
    # where the greedy map leaves gainful swaps; stats checked against the oracle
    import oracle
    co_r = W.random_cooccur(31, L, E)
    d_co = torch.as_tensor(co_r, device=dev)
    mr2 = torch.empty_like(mr)
    st2 = torch.empty_like(st)
    t_sw = []
    for i in range(7):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            topo.topo_place_experts(L, E, R, 0, d_co, mr2, st2, s)
            b.record(stream)
        b.synchronize()
        if i >= 2:
            t_sw.append(a.elapsed_time(b))
    st_r = st2.cpu().numpy()
    mr_o, st_o = oracle.place(co_r, R)
    swaps = {"workload": f"uniform random counts, {L} layers, E = {E}, EP{R}",
             "ms": round(statistics.median(t_sw), 4), "swaps": int(st_r[:, 3].sum()),
             "within_weight_greedy": int(st_r[:, 1].sum()), "within_weight_final": int(st_r[:, 2].sum()),
             "equals_oracle": bool(np.array_equal(st_r, st_o) and np.array_equal(mr2.cpu().numpy(), mr_o))}
    res = {"workload": f"{w.name} as EP{R}", "ms": round(ms, 4), "layers_in_parallel": L,
           "swap_phase": swaps,
           "within_weight_contiguous": int(stn[:, 0].sum()), "within_weight_greedy": int(stn[:, 1].sum()),
           "within_weight_final": int(stn[:, 2].sum()), "swaps": int(stn[:, 3].sum()),
           "timing": "CUDA events around one call for all layers, median of 5 after 2 warm-up calls",
           "gpu_launches_per_call": KERNELS_PER_CALL["place"]}
    # deduplication at EP8 on layer 0, contiguous against correlated placement
    saved = {}
    for name, m in (("contiguous", None), ("correlated", mr[0].contiguous())):
        cfg = dict(T=T, E=E, k=k, R=R, ranks_per_node=R, n_slot=0, tok_bytes=2048, expert_bytes=1 << 20,
                   c_intra=1, c_inter=4, max_refine_iters=0, main_rank=m)
        P = Planner(cfg, 1, dev, stream=stream)
        with torch.cuda.stream(stream):
            P.run(ids[:1])
        c = topo.make_cfg(**{**cfg, "main_rank": P.main_rank})
        nb = topo.topo_workspace_bytes(c, 1, topo.TOPO_CALL_DEDUP)
        ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
        o = [torch.empty((1, R + 1), dtype=torch.int32, device=dev),
             torch.empty((1, T * k), dtype=torch.int32, device=dev),
             torch.empty((1, T * k), dtype=torch.int64, device=dev),
             torch.empty((1, T, 1), dtype=torch.int64, device=dev),
             torch.empty((1, R, R), dtype=torch.int64, device=dev),
             torch.empty((1, topo.TOPO_DEDUP_STATS), dtype=torch.int64, device=dev)]
        with torch.cuda.stream(stream):
            topo.topo_dedup_layout(c, 1, P.buf.dst_inst, *o, ws, nb, s)
        torch.cuda.synchronize()
        if P.error() != 0 or topo.topo_read_error(ws) != 0:
            raise RuntimeError("device error in the placement measurement")
        dst = o[5].cpu().numpy()[0]
        saved[name] = round(1 - dst[0] / dst[1], 4)
    res["dedup_rows_saved_layer0"] = saved
    return res



def secondary_shuffle(dev, stream, hbm_peak):
    """topo_shuffle_targets over the co-occurrence workload (8 layers of
    262144 tokens, E = 128, k = 8) as EP16, with its own GPU transition
    counts; L2 flushed (256 MB write) before each call; CUDA events inside one
    captured graph per call, median of 10 after 3 warm-up replays.  Also the
    prediction statistics of the four-layer workload, whose layers are
    correlated."""
    import torch
    import moe_expert_routing_ids_gb300 as topo
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Cooccur
    res = {}
    for w, timed in ((W.COOCCUR, True), (W.FOUR_LAYER, False)):
        R = SHUFFLE_RANKS if timed else w.R
        L, T, E, k = w.n_layers, w.T, w.E, w.k
        C = Cooccur(L, T, E, k, dev)
        ids = torch.as_tensor(w.ids(), device=dev)
        with torch.cuda.stream(stream):
            C.run(ids, stream)
        nb = topo.topo_shuffle_workspace_bytes(L, E, R)
        ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
        target = torch.empty((L - 1, T), dtype=torch.int32, device=dev)
        stats = torch.empty((L - 1, topo.TOPO_SHUFFLE_STATS), dtype=torch.int64, device=dev)
        s = stream.cuda_stream

        def call():
            topo.topo_shuffle_targets(L, T, E, k, R, ids, C.tr, None, None, target, stats, ws, nb, s)
        with torch.cuda.stream(stream):
            call()
        torch.cuda.synchronize()
        if topo.topo_read_error(ws) != 0 or C.error() != 0:
            raise RuntimeError("device error in the shuffle measurement")
        st = stats.cpu().numpy().sum(axis=0)
        entry = {"workload": f"{w.name} as EP{R}", "next_pairs_on_target": int(st[0]),
                 "next_pairs_on_source": int(st[1]), "tokens_moved": int(st[2]),
                 "next_pairs": int(st[3]),
                 "locality_target": round(st[0] / max(st[3], 1), 4),
                 "locality_source": round(st[1] / max(st[3], 1), 4)}
        if timed:
            flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
            gev = GraphEvents(2)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                flush.fill_(1)
                gev.record(0, stream)
                call()
                gev.record(1, stream)
            times = []
            for _ in range(13):
                graph.replay()
                torch.cuda.synchronize()
                times.append(gev.elapsed(0, 1))
            gev.close()
            ms = statistics.median(times[3:])
            # algorithmic: every layer's ids read once (a layer is the next
            # layer of one prediction and the current layer of the following
            # one, but its bytes need to leave HBM only once), the
            # transitions, the targets written
            nbytes = L * T * k * 4 + (L - 1) * E * E * 8 + (L - 1) * T * 4
            gbs = nbytes / (ms * 1e-3) / 1e9
            entry.update({"ms": round(ms, 4), "algorithmic_bytes": nbytes, "achieved_gbs": round(gbs, 1),
                          "frac": round(gbs / hbm_peak, 4), "l2": "flushed (256 MB write) before each call",
                          "gpu_launches_per_call": KERNELS_PER_CALL["shuffle"]})
            res["timed"] = entry
        else:
            res["correlated_layers"] = entry
    return res


PACK_WORKLOAD_H = 7168       # hidden size of the four-layer workload (bf16 rows)


def secondary_pack(dev, stream, hbm_peak):
    """topo_permute and topo_combine on the first layer of the T=65536, E=256,
    k=8, R=64 workload with H = 7168 bf16 rows: x 0.94 GB, send buffer 7.5 GB
    (both far above L2).  Layout from the library's own chain; each call timed
    with CUDA events, median of 5 after 2 warm-up calls."""
    import torch
    import moe_expert_routing_ids_gb300 as topo
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Planner
    w = W.FOUR_LAYER
    T, k, H = w.T, w.k, PACK_WORKLOAD_H
    P = Planner(w.plan_cfg, 1, dev, stream=stream)
    ids = torch.as_tensor(w.ids(n_layers=1), device=dev)
    with torch.cuda.stream(stream):
        P.run(ids)
    cfg = topo.make_cfg(**w.plan_cfg)
    ws_bytes = topo.topo_workspace_bytes(cfg, 1, topo.TOPO_CALL_PACK)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    g = torch.Generator(device=dev).manual_seed(5)
    x = (torch.randn((1, T, H), generator=g, device=dev) * 4).to(torch.bfloat16).view(torch.int16)
    y = torch.empty((1, T * k, H), dtype=torch.int16, device=dev)
    out = torch.empty((1, T, H), dtype=torch.int16, device=dev)
    gw = torch.rand((1, T, k), generator=g, device=dev)
    sp = P.buf.sorted_pairs

    def timed(fn):
        times = []
        for i in range(7):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                fn()
                b.record(stream)
            b.synchronize()
            if i >= 2:
                times.append(a.elapsed_time(b))
        return statistics.median(times)

    s = stream.cuda_stream
    ms_p = timed(lambda: topo.topo_permute(cfg, 1, H, x, sp, y, ws, ws_bytes, s))
    ms_c = timed(lambda: topo.topo_combine(cfg, 1, H, y, sp, gw, out, ws, ws_bytes, s))
    torch.cuda.synchronize()
    if topo.topo_read_error(ws) != 0 or P.error() != 0:
        raise RuntimeError("device error in the pack measurement")
    row = H * 2
    # algorithmic: permute reads each token row once and writes it k times;
    # combine reads the k rows and the k weights and writes one row; both also
    # read the layout and build its inverse (12 B per pair)
    b_p = T * row + T * k * row + 12 * T * k
    b_c = T * k * row + T * row + 4 * T * k + 12 * T * k
    res = {}
    for name, ms, nb in (("permute", ms_p, b_p), ("combine", ms_c, b_c)):
        gbs = nb / (ms * 1e-3) / 1e9
        res[name] = {"ms": round(ms, 4), "algorithmic_bytes": nb, "achieved_gbs": round(gbs, 1),
                     "frac": round(gbs / hbm_peak, 4)}
    res.update({"workload": f"{w.name} (first layer), H={H} bf16", "timing":
                "CUDA events around one call, median of 5 after 2 warm-up calls"})
    del y, x, out
    return res


def secondary_gate(dev, stream, hbm_peak, microbatches=0):
    """topo_gate_hist on the T = 1048576, E = 512, k = 10, R = 128 workload, all
    4 microbatches: router logits = standard Gumbel noise, bias = log of the
    workload's Zipf(1.4) expert probabilities (random logits with a fixed
    expert-specific bias), float32 (8.6 GB) and bf16 (4.3 GB), both far above
    L2.  No score output.  Each call timed with CUDA events, median of 5 after
    2 warm-up calls."""
    import torch
    import moe_expert_routing_ids_gb300 as topo
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Planner
    w = W.STRESS
    L, T, E, k = w.n_layers, w.T, w.E, w.k
    if microbatches:
        L = min(L, microbatches)
    P = Planner(w.plan_cfg, L, dev, stream=stream)
    g = torch.Generator(device=dev).manual_seed(17)
    x = torch.empty((L, T, E), dtype=torch.float32, device=dev)
    x.uniform_(generator=g).clamp_(min=1e-12).log_().neg_().log_().neg_()
    p = 1.0 / torch.arange(1, E + 1, dtype=torch.float64, device=dev) ** w.zipf_s
    perm = torch.randperm(E, generator=g, device=dev)
    bias = torch.log(p / p.sum())[perm].float()
    ids = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    res = {"workload": f"{w.name}, {L} microbatches", "timing":
           "CUDA events around one call, median of 5 after 2 warm-up calls"}
    for name in ("f32", "bf16"):
        if name == "f32":
            logits = x
        else:
            logits = x.to(torch.bfloat16)
            del x                                   # only the bf16 copy stays referenced
        times = []
        for i in range(7):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                P.gate_hist(logits, ids, bias)
                b.record(stream)
            b.synchronize()
            if i >= 2:
                times.append(a.elapsed_time(b))
        if P.error() != 0:
            raise RuntimeError("device error in the gating measurement")
        ms = statistics.median(times)
        # algorithmic: read the logits once, write the ids
        nb = L * T * E * logits.element_size() + L * T * k * 4
        gbs = nb / (ms * 1e-3) / 1e9
        res[name] = {"ms": round(ms, 4), "tokens_per_s": round(L * T / (ms * 1e-3), 1),
                     "algorithmic_bytes": nb, "achieved_gbs": round(gbs, 1),
                     "frac": round(gbs / hbm_peak, 4)}
        del logits
    res["gpu_launches_per_call"] = KERNELS_PER_CALL["gate"]
    return res


def secondary_dedup(P, w, dev, stream, hbm_peak):
    """topo_dedup_layout on the destinations of the timed workload (all its
    microbatches; dst_inst 168 MB > 129 MB L2).  The call timed with CUDA
    events, median of 5 after 2 warm-up calls."""
    import torch
    import moe_expert_routing_ids_gb300 as topo
    L, T, k, R = w.n_layers, w.T, w.k, w.R
    RW = (R + 63) // 64
    cfg = topo.make_cfg(**w.plan_cfg)
    ws_bytes = topo.topo_workspace_bytes(cfg, L, topo.TOPO_CALL_DEDUP)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    o = dict(seg=torch.empty((L, R + 1), dtype=torch.int32, device=dev),
             row_token=torch.empty((L, T * k), dtype=torch.int32, device=dev),
             row_slots=torch.empty((L, T * k), dtype=torch.int64, device=dev),
             tok_dst=torch.empty((L, T, RW), dtype=torch.int64, device=dev),
             send=torch.empty((L, R, R), dtype=torch.int64, device=dev),
             stats=torch.empty((L, topo.TOPO_DEDUP_STATS), dtype=torch.int64, device=dev))
    s = stream.cuda_stream
    times = []
    for i in range(7):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            topo.topo_dedup_layout(cfg, L, P.buf.dst_inst, o["seg"], o["row_token"], o["row_slots"],
                                   o["tok_dst"], o["send"], o["stats"], ws, ws_bytes, s)
            b.record(stream)
        b.synchronize()
        if i >= 2:
            times.append(a.elapsed_time(b))
    torch.cuda.synchronize()
    if topo.topo_read_error(ws) != 0:
        raise RuntimeError("device error in the deduplicated layout measurement")
    ms = statistics.median(times)
    st = o["stats"].cpu().numpy()
    rows, pairs = int(st[:, 0].sum()), int(st[:, 1].sum())
    # algorithmic: read the destinations once, write the token bitmaps and one
    # (token, slot mask) row of 12 B per row
    nb = 4 * pairs + 8 * L * T * RW + 12 * rows
    gbs = nb / (ms * 1e-3) / 1e9
    return {"workload": f"{w.name}, all {L} microbatches", "ms": round(ms, 4),
            "rows": rows, "pairs": pairs, "rows_remote": int(st[:, 2].sum()),
            "pairs_remote": int(st[:, 3].sum()), "pairs_per_s": round(pairs / (ms * 1e-3), 1),
            "algorithmic_bytes": nb, "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
            "timing": "CUDA events around one call, median of 5 after 2 warm-up calls",
            "gpu_launches_per_call": KERNELS_PER_CALL["dedup"]}


def run_only(name, microbatches=0):
    """One secondary measurement on cuda:0, printed as its own JSON line."""
    import torch
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    hbm, _ = peaks()
    if name == "plan_latency":
        res = secondary_plan_latency(dev, stream)
    elif name == "cooccur":
        res = secondary_cooccur(dev, stream, hbm)
    elif name == "pack":
        res = secondary_pack(dev, stream, hbm)
    elif name == "gate":
        res = secondary_gate(dev, stream, hbm, microbatches)
    elif name == "shuffle":
        res = secondary_shuffle(dev, stream, hbm)
    elif name == "place":
        res = secondary_place(dev, stream)
    elif name == "configs":
        res = {"configs": config_lines(dev, stream, hbm)}
    elif name == "solver":
        res = solver_sweep(dev, stream)
    elif name == "chain":
        w = W.STRESS
        L = min(w.n_layers, microbatches) if microbatches else w.n_layers
        ids = torch.as_tensor(w.ids()[:L], device=dev).contiguous()
        P = Planner(w.plan_cfg, L, dev, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(2):
                P.run(ids)
        torch.cuda.synchronize(dev)
        if P.error() != 0:
            raise RuntimeError("device error in the plan chain")
        res = {"workload": f"{w.name}, {L} microbatch(es)", "pairs": int(ids.numel()), "runs": 2}
    else:
        w = W.STRESS
        P = Planner(w.plan_cfg, w.n_layers, dev, stream=stream)
        with torch.cuda.stream(stream):
            P.run(torch.as_tensor(w.ids(), device=dev))
        torch.cuda.synchronize(dev)
        if P.error() != 0:
            raise RuntimeError("device error in the plan chain")
        res = secondary_dedup(P, w, dev, stream, hbm)
    print(json.dumps({"measurement": name, **res}), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Planner

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    w = W.STRESS
    ids = w.ids(replica=rank)
    pairs = int(ids.size)
    d_ids = torch.as_tensor(ids, device=dev)
    P = Planner(w.plan_cfg, w.n_layers, dev, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            P.run(d_ids)
    torch.cuda.synchronize(dev)
    err = P.error()
    if err != 0:
        raise RuntimeError(f"device error word {err}")

    clocks = Clocks(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    total_ms, steps_run, per_call = time_chain(P, d_ids, args.steps, stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    if P.error() != 0:
        raise RuntimeError("device error after the timed region")
    total_ms = max_over_ranks(total_ms, dev)
    if rank != 0:
        return
    ms_step = total_ms / steps_run
    value = pairs * world / (ms_step * 1e-3)
    hbm, peak_kind = peaks()
    # dominant HBM call
    scan = {c: per_call[c] for c in BYTES_PER_PAIR}
    dom = max(scan, key=scan.get)
    achieved = BYTES_PER_PAIR[dom] * pairs / (per_call[dom] * 1e-3) / 1e9
    traffic = profiled_traffic(dom, pairs)
    calls = {c: {"ms": round(per_call[c], 4),
                 **({"achieved_gbs": round(BYTES_PER_PAIR[c] * pairs / (per_call[c] * 1e-3) / 1e9, 1)}
                    if c in BYTES_PER_PAIR else {})} for c in CALLS}
    calls["plan"]["us_per_microbatch"] = round(per_call["plan"] * 1e3 / w.n_layers, 2)
    line = {"metric": "routed (token,slot) pairs/sec", "value": value, "unit": "pairs/s",
            "n_gpus": world, "steps": steps_run, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "E": w.E, "k": w.k, "R": w.R,
                       "ranks_per_node": w.ranks_per_node, "n_slot": w.n_slot,
                       "microbatches": w.n_layers, "pairs_per_step": pairs,
                       "parallelism": f"replicas x{world}",
                       "l2": "ids 168 MB > 129 MB L2 per step, no flush"},
            "gpu_launches": steps_run * sum(KERNELS_PER_CALL[c] for c in CALLS),
            "timing": f"exactly {steps_run} steps replayed from CUDA graphs of "
                      f"{min(STEPS_PER_GRAPH, args.steps)} steps with nothing between the calls, CUDA "
                      "events around all replays; per-call times (and the roofline) from the same steps "
                      f"captured with an event node before every call, replayed {CALL_REPLAYS} times after "
                      "them (those nodes break the programmatic launch chain: about 4% slower)",
            "calls": calls,
            "roofline": {"bound": "hbm", "kernel": f"{dom} call ({CALL_KERNEL[dom]} + its index kernels)",
                         "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4), "peak_kind": peak_kind,
                         "algorithmic_bytes_per_pair": BYTES_PER_PAIR[dom],
                         "traffic": traffic}}
    if clk:
        line["clocks"] = clk
    if not args.skip_e2e:
        n_e2e = max(3, min(args.steps, 20))
        line["e2e"] = e2e(P, w, ids, dev, stream, n_e2e)
        line["e2e_full_outputs"] = e2e(P, w, ids, dev, stream, n_e2e, _outputs,
                                       "every plan and layout output (dst_inst, sorted_pairs, tables)")
    if not args.skip_secondary:
        line["configs"] = config_lines(dev, stream, hbm)
        line["solver_latency"] = solver_sweep(dev, stream)
        line["plan_latency"] = secondary_plan_latency(dev, stream)
        line["cooccur"] = secondary_cooccur(dev, stream, hbm)
        line["pack"] = secondary_pack(dev, stream, hbm)
        line["dedup"] = secondary_dedup(P, w, dev, stream, hbm)
        line["gate"] = secondary_gate(dev, stream, hbm)
        line["shuffle"] = secondary_shuffle(dev, stream, hbm)
        line["place"] = secondary_place(dev, stream)
    if not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline(w, ids)
    print(json.dumps(line), flush=True)


def _outputs(Q):
    b = Q.buf
    return [b.dst_inst, b.sorted_pairs, b.seg_off, b.send_counts, b.layout_stats, b.slot_expert,
            b.rank_load, b.stats]


def _result(Q):
    """The step's result read back by the host: the plan and layout statistics
    and the rank loads (the plan and layout themselves stay on the device for
    the dispatch that consumes them)."""
    b = Q.buf
    return [b.stats, b.layout_stats, b.rank_load]


def e2e(P, w, ids, dev, stream, steps, outputs=_result, what="the plan and layout statistics"):
    """Same metric through host buffers.  Every step copies its ids in from
    pinned host memory, runs the three calls, and copies `outputs` back to
    pinned host memory.  Steps are pipelined over two slots
    (two planners, two device input buffers): step i's input copy and step
    i-1's output copy overlap step i's compute, on their own streams.  Timed
    from before the first input copy to after the last output copy."""
    import torch
    from moe_expert_routing_ids_gb300.planner import Planner
    Ps = [P, Planner(w.plan_cfg, w.n_layers, dev, stream=stream)]
    h_ids = torch.from_numpy(ids).pin_memory()
    h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outputs(Q)] for Q in Ps]
    d_ids = [torch.empty(ids.shape, dtype=torch.int32, device=dev) for _ in Ps]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done = [torch.cuda.Event() for _ in Ps]
    run_done = [torch.cuda.Event() for _ in Ps]
    out_done = [torch.cuda.Event() for _ in Ps]

    def step(i):
        k = i % 2
        Q = Ps[k]
        s_in.wait_event(run_done[k])               # slot k's ids no longer read
        with torch.cuda.stream(s_in):
            d_ids[k].copy_(h_ids, non_blocking=True)
        in_done[k].record(s_in)
        stream.wait_event(in_done[k])
        stream.wait_event(out_done[k])             # slot k's outputs copied out
        with torch.cuda.stream(stream):
            Q.run(d_ids[k])
        run_done[k].record(stream)
        s_out.wait_event(run_done[k])
        with torch.cuda.stream(s_out):
            for h, d in zip(h_out[k], outputs(Q)):
                h.copy_(d, non_blocking=True)
        out_done[k].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize(dev)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(steps):
        step(i)
    z.record(s_out)
    z.synchronize()
    ms = a.elapsed_time(z) / steps
    for Q in Ps:
        if Q.error() != 0:
            raise RuntimeError("device error in the end-to-end run")
    return {"value": ids.size / (ms * 1e-3), "unit": "pairs/s", "ms_per_step": ms,
            "h2d_bytes_per_step": int(ids.nbytes),
            "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in outputs(P))),
            "read_back": what, "steps": steps,
            "pipeline": "2 slots; input copy, compute, output copy on 3 streams"}


def cpu_baseline(w, ids):
    import oracle
    oracle.build()
    secs, pairs, n = 0.0, 0, 0
    while secs < 10.0 and n < w.n_layers * 3:
        s, p = cpu_sample_chain(w, ids[n % w.n_layers][None])
        secs += s
        pairs += p
        n += 1
    return {"value": pairs / secs, "unit": "pairs/s", "cores": 1, "kind": "oracle", "host": host_info(),
            "sample": f"{n} microbatch(es) of the workload, {pairs} pairs, oracle chain "
                      f"hist+plan+reroute+layout single-threaded, {secs:.1f} s"}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank)
        else:
            import __graft_entry__
            __graft_entry__.build()
            if args.only:
                if rank == 0:
                    run_only(args.only, args.microbatches)
            else:
                run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

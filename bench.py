#!/usr/bin/env python
"""Benchmark of the Q4_K MoE FFN decode path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload: one Qwen3-30B-A3B-shaped MoE layer (hidden 2048, 128
experts, top-8, intermediate 768, Q4_K experts resident in HBM), 1024
independent tokens decoded one at a time (bs=1).  One step = the 1024
sequential single-token forwards (router GEMV, softmax/top-k, gate/up
dequant-GEMV + SwiGLU, down dequant-GEMV + weighted combine), replayed as one
CUDA graph.  The layer's 339.7 MB of experts exceed the 129 MB L2, so no
flush is inserted between steps.

Printed: one JSON line with value = tokens/s over all ranks, the dominant
kernel's HBM roofline (its CUDA-event time on its own stream), the whole
chain's achieved bandwidth, nvidia-smi clocks sampled during the timed
region, an end-to-end figure with host<->device copies in the timed
region, the CPU oracle's throughput on a bounded sample, and (unless
--no-extras) the 48-layer stack, the 4-token deduplicated workload, the
headline workload as a pre-normed block, the 4096-token grouped prefill
with its tensor-core roofline, the headline decode and the prefill with
NVFP4 experts, the headline decode in the int8-activation mode, and the
headline decode and the prefill with Q5_K experts.

--impl reference times the CPU oracle (the reference implementation of the
method) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode tok/s at bs=1 (Qwen3-30B-A3B shape, Q4_K); HBM GB/s vs peak"
FALLBACK_HBM_GBS = 6800.0


# DRAM bytes per launch of the dominant kernel from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only while the
# kernel's sources are the ones that were profiled (sha256 over the files).
PROFILED_TRAFFIC = {
    "k_expert_cluster": {
        "bytes": 21299456,
        "capture": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum "
                   "-k regex:k_expert_cluster -s 20 -c 3 on bench.py --tokens 64 --steps 2 --warmup 1 "
                   "--no-extras --no-cpu-baseline (launch 21)",
        "sources": ["quantized_moe_expert_gemv_gb300/csrc/si_expert_cluster.cu",
                    "quantized_moe_expert_gemv_gb300/csrc/si_device.cuh",
                    "quantized_moe_expert_gemv_gb300/csrc/si_internal.h"],
        "sha256": "097bff69832111ab8820282b18f51d29857e4bb15f37c4bb7543e63bb0c0a86f",
    },
}


def profiled_traffic(kernel: str):
    """(bytes per launch, note) from the stored ncu capture, or (None, why not)."""
    import hashlib
    ent = PROFILED_TRAFFIC.get(kernel)
    if ent is None:
        return None, "no ncu capture for this kernel"
    root = os.path.dirname(os.path.abspath(__file__))
    h = hashlib.sha256()
    for f in ent["sources"]:
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != ent["sha256"]:
        return None, "kernel sources changed since the ncu capture"
    return ent["bytes"], "dram__bytes_read.sum + dram__bytes_write.sum: " + ent["capture"]


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the stack, dedup, pre-normed, prefill, NVFP4, int8-activation and Q5_K workloads")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--tokens", type=int, default=0,
                   help="tokens per step of the headline layer (default 1024; small values for ncu)")
    p.add_argument("--prefill-only", action="store_true",
                   help="time only the grouped prefill workload (for profiling its kernels)")
    p.add_argument("--dedup-probe", type=int, default=0, metavar="S",
                   help="run only S steps of the 4-token deduplicated workload as plain launches and print "
                        "each step's distinct experts (for a per-launch DRAM capture of the expert kernel)")
    p.add_argument("--cpu-sample-tokens", type=int, default=0,
                   help="tokens of the CPU oracle sample (default: 16 per host core, at least 64)")
    return p.parse_args()


# ------------------------------------------------------------------ helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s)"


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.file.read())) if len(r) >= 9]
        self.file.close()
        os.unlink(self.file.name)
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        power = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


class Dist:
    def __init__(self, n_gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.device = "cuda" if n_gpus > 0 else "cpu"  # where the reduction tensors live (nccl / gloo)
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl" if n_gpus > 0 else "gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t)
        return float(t.item())


# --------------------------------------------------------- CPU oracle timing
_ORACLE_INPUTS = {}


def oracle_tokens_per_s(n_tokens: int, threads: int):
    """The CPU oracle, unchanged, on n_tokens of the headline layer (one token
    per task, `threads` tasks at a time).  Returns (tok/s, seconds, threads)."""
    import oracle
    from quantized_moe_expert_gemv_gb300 import synth
    wl = synth.WORKLOADS["layer"]
    if "layer" not in _ORACLE_INPUTS:
        _ORACLE_INPUTS["layer"] = synth.make_layer(wl["shape"], seed=wl["seed"])
    layer = _ORACLE_INPUTS["layer"]
    x = synth.make_tokens(wl["shape"], seed=wl["seed"], n_tokens=n_tokens)
    oracle.build()
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda t: oracle.moe_token(layer, x[t]), range(n_tokens)))
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt


def oracle_prefill_tokens_per_s(n_tokens: int, threads: int):
    """The CPU oracle, unchanged, as a grouped prefill of n_tokens tokens of the
    prefill workload's layer: routing of every token, counts / offsets / perm,
    then every expert's pairs through the oracle's expert FFN with one expert
    per task (`threads` tasks at a time), and the weighted combine in slot
    order.  Returns (tok/s, seconds)."""
    import numpy as np
    import oracle
    from quantized_moe_expert_gemv_gb300 import synth
    wl = synth.WORKLOADS["prefill"]
    shape = wl["shape"]
    if "prefill" not in _ORACLE_INPUTS:
        _ORACLE_INPUTS["prefill"] = synth.make_layer(shape, seed=wl["seed"])
    layer = _ORACLE_INPUTS["prefill"]
    x = synth.make_tokens(shape, seed=wl["seed"], n_tokens=n_tokens)
    H, I, k = shape.hidden, shape.intermediate, shape.top_k
    oracle.build()
    t0 = time.perf_counter()
    ids, w, _, _ = oracle.route_tokens(layer.router_w, x, k)
    counts, offsets, perm = oracle.counts_offsets_perm(ids, shape.n_experts)
    x64 = synth.bf16_to_f32(x).astype(np.float64)
    y = np.empty((n_tokens * k, H), dtype=np.float64)

    def one_expert(e):
        for p in perm[offsets[e]:offsets[e + 1]]:
            _, y[p] = oracle.expert_ffn(layer.w_gate[e], layer.w_up[e], layer.w_down[e], x64[p // k], H, I)
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one_expert, [e for e in range(shape.n_experts) if counts[e] > 0]))
    out = np.zeros((n_tokens, H), dtype=np.float64)
    for slot in range(k):
        out += w[:, slot, None] * y[np.arange(n_tokens) * k + slot]
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, dist):
    """--impl reference: the CPU oracle, timed per step on a bounded sample."""
    if dist.rank != 0:
        return
    cores = cpu_cores()
    sample = max(cores, 8)
    steps_t = []
    for i in range(args.warmup + args.steps):
        tps, dt = oracle_tokens_per_s(sample, cores)
        if i >= args.warmup:
            steps_t.append(dt)
    total = sum(steps_t)
    value = sample * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Q4_K experts, bf16 N(0,1) tokens)",
        "config": {"workload": "qwen3-30b-a3b-moe-layer-decode-bs1", "hidden": 2048,
                   "intermediate": 768, "experts": 128, "top_k": 8,
                   "tokens_per_step": sample, "l2_policy": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample} tokens of the headline layer per step, one per thread"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- GPU workloads
def build_layer_graph(binding, plan, L, x_rows, out_rows, scratch, stream, n_tok=1, route=None,
                      events=None):
    """Capture one CUDA graph of len(x_rows) sequential decode calls."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for t in range(len(x_rows)):
                ro = route[t] if route is not None else None
                if events is not None:
                    binding.si_debug_decode_events(plan, L, x_rows[t], n_tok, out_rows[t], ro, scratch,
                                                   events[t], stream=stream)
                else:
                    binding.si_moe_forward_decode(plan, L, x_rows[t], n_tok, out_rows[t], ro, scratch,
                                                  stream=stream)
    return g


def time_graph(g, stream, steps, warmup, dist, sampler=None):
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            g.replay()
        end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    dist.barrier()
    ms = start.elapsed_time(end)
    return dist.max(ms), clocks


def e2e_per_token(binding, device, plan, L, x_pin, scratch, stream, shape, dist, torch, n, warmup):
    """A bs=1 caller without a graph, that needs each token's output on the
    host: per token its 4 KiB x from pinned host memory in, one decode, its
    8 KiB output back to pinned host memory, and a wait for it.  Timed two
    ways by the host wall clock over n tokens: through the library's
    host-buffer entry point (one C call per token: one replay of a graph
    holding the copies and the two kernels, the wait and the status read),
    and with torch's copies around the device entry point (three
    Python-level calls and a stream wait per token)."""
    x_one = torch.empty((shape.hidden,), dtype=torch.int16, device="cuda")
    out_one = torch.empty((shape.hidden,), dtype=torch.float32, device="cuda")
    out_pin = torch.empty((n, shape.hidden), dtype=torch.float32).pin_memory()
    host_scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE_HOST, 1)
    rows = x_pin.shape[0]

    def via_host_entry(t):
        binding.si_moe_forward_decode_host(plan, L, x_pin[t % rows], 1, out_pin[t % n], None, host_scratch,
                                           stream=stream)

    def via_torch_copies(t):
        with torch.cuda.stream(stream):
            x_one.copy_(x_pin[t % rows], non_blocking=True)
            binding.si_moe_forward_decode(plan, L, x_one, 1, out_one, None, scratch, stream=stream)
            out_pin[t % n].copy_(out_one, non_blocking=True)
        stream.synchronize()

    def wall(one):
        for t in range(warmup):
            one(t)
        torch.cuda.synchronize()
        dist.barrier()
        t0 = time.perf_counter()
        for t in range(n):
            one(t)
        return dist.max(time.perf_counter() - t0)

    w_host = wall(via_host_entry)
    w_torch = wall(via_torch_copies)
    st = binding.si_moe_read_status(plan, scratch, stream)
    assert st == binding.SI_OK, binding.si_status_string(st)
    return {"value": dist.sum(n / w_host), "unit": "tok/s", "us_per_token": 1e6 * w_host / n, "tokens": n,
            "h2d_bytes_per_token": shape.hidden * 2, "d2h_bytes_per_token": shape.hidden * 4,
            "timing": "host wall clock; per token one si_moe_forward_decode_host call (one replay of its "
                      "captured graph: copy in, two kernels, copy out; stream wait, status read)",
            "torch_copies": {"value": dist.sum(n / w_torch), "unit": "tok/s", "us_per_token": 1e6 * w_torch / n,
                             "timing": "per token torch copy in, si_moe_forward_decode, torch copy out, "
                                       "stream wait"}}


def bench_layer(args, dist, binding, device, synth, torch, hbm_peak):
    wl = synth.WORKLOADS["layer"]
    shape, seed, T = wl["shape"], wl["seed"], (args.tokens or wl["n_tokens"])
    layer = synth.make_layer(shape, seed=seed)
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape), torch.cuda.current_device())
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    x_host = synth.make_tokens(shape, seed=seed, n_tokens=T)
    x = device.tokens_to_device(x_host)
    out = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
    L = dl.struct()
    stream = torch.cuda.Stream()
    g = build_layer_graph(binding, plan, L, [x[t] for t in range(T)], [out[t] for t in range(T)],
                          scratch, stream)
    sampler = ClockSampler(torch.cuda.current_device())
    ms, clocks = time_graph(g, stream, args.steps, args.warmup, dist, sampler)
    st = binding.si_moe_read_status(plan, scratch, stream)
    assert st == binding.SI_OK, binding.si_status_string(st)
    ms_step = ms / args.steps
    total_tokens = dist.sum(T * args.steps)
    value = total_tokens / (ms / 1e3)

    # Per-kernel CUDA-event timing of the same 1024-token step (events around
    # each of the three kernels, recorded on the launch stream inside a graph).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(T)]
    with torch.cuda.stream(stream):
        for row in ev:          # torch creates the CUDA event on its first record
            for e in row:
                e.record(stream)
    torch.cuda.synchronize()
    gi = build_layer_graph(binding, plan, L, [x[t] for t in range(T)], [out[t] for t in range(T)],
                           scratch, stream, events=ev)
    for _ in range(2):
        gi.replay()
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 10))
    sums = [0.0, 0.0, 0.0]
    for _ in range(reps):
        with torch.cuda.stream(stream):
            gi.replay()
        torch.cuda.synchronize()
        for t in range(T):
            for k in range(3):
                sums[k] += ev[t][k].elapsed_time(ev[t][k + 1])
    per_launch_ms = [s / (reps * T) for s in sums]
    nbh, nbi = shape.blocks_per_gate_row, shape.blocks_per_down_row
    gateup_bytes = shape.top_k * 2 * shape.intermediate * nbh * 144
    down_bytes = shape.top_k * shape.hidden * nbi * 144
    router_bytes = shape.n_experts * shape.hidden * 4 + shape.hidden * 2
    expert_bytes = gateup_bytes + down_bytes
    path = binding.si_debug_decode_fused(plan, 1)
    plan_info = binding.si_debug_plan_info(plan)
    fused = path >= 1
    # The roofline is taken on the whole per-token chain (router + expert
    # kernel), timed without anything between the kernels: the step time of
    # the timed graph divided by its tokens.  The expert kernel overlaps the
    # router through programmatic dependent launch, so its own duration is at
    # most this and its achieved bandwidth at least the figure below.  Events
    # recorded between the two kernels (kernels_ms_per_token_events) break that
    # overlap and serialise them; they only show how a token's time splits.
    # The column-split router serves plain single tokens of the cluster kernel
    # for E in {64, 128} and H in {1024, 2048}; other shapes take k_router_topk.
    router = ("k_router_one" if path == 2 and shape.n_experts in (64, 128) and shape.hidden in (1024, 2048)
              else "k_router_topk")
    dom_name = ((router + " + " + ("k_expert_cluster" if path == 2 else "k_expert") +
                 " (router GEMV + top-k; fused gate/up dequant-GEMV + SwiGLU + down dequant-GEMV + combine)")
                if fused else router + " + k_gateup_generic + k_down_generic")
    dom_bytes, dom_ms = expert_bytes, ms_step / T
    dom_gbs = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic, traffic_note = profiled_traffic("k_expert_cluster") if path == 2 else \
        (None, "no ncu capture for this kernel")

    # End to end: pinned host tokens in, pinned host outputs back, every step.
    x_pin = torch.from_numpy(x_host.view("int16")).pin_memory()
    out_pin = torch.empty((T, shape.hidden), dtype=torch.float32).pin_memory()
    x16 = x.view(torch.int16)

    def e2e_step():
        with torch.cuda.stream(stream):
            x16.copy_(x_pin, non_blocking=True)
            g.replay()
            out_pin.copy_(out, non_blocking=True)
    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    e1.synchronize()
    e2e_ms = dist.max(e0.elapsed_time(e1))
    e2e_value = total_tokens / (e2e_ms / 1e3)
    try:
        e2e_tok = e2e_per_token(binding, device, plan, L, x_pin, scratch, stream, shape, dist, torch,
                                n=min(T, 512), warmup=max(args.warmup, 16))
    except Exception as exc:  # reported in the line; the headline figures above stand
        e2e_tok = {"error": repr(exc)}

    tok_per_s_rank = T * args.steps / (ms / 1e3)
    chain_gbs = expert_bytes * tok_per_s_rank / 1e9
    result = {
        "value": value, "unit": "tok/s", "ms_per_step": ms_step,
        "config": {"workload": "qwen3-30b-a3b-moe-layer-decode-bs1", "hidden": shape.hidden,
                   "intermediate": shape.intermediate, "experts": shape.n_experts, "top_k": shape.top_k,
                   "weights": "Q4_K (GGUF, 144 B / 256 weights)", "tokens_per_step": T, "seed": seed,
                   "global_batch": 1, "parallelism": f"replicas x{dist.world}",
                   "l2_policy": "inputs larger than L2: 339.7 MB of resident experts per layer vs "
                                "129 MB L2; no flush between steps",
                   "graph": "one CUDA graph per step (1024 sequential decode calls)",
                   "plan": plan_info},
        "roofline": {"bound": "hbm", "kernel": dom_name,
                     "achieved": dom_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": dom_gbs / hbm_peak,
                     "traffic": traffic, "traffic_source": traffic_note,
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "launch_ms": dom_ms,
                     "timing": "ms_per_step / tokens_per_step: CUDA events on the launch stream around the "
                               "timed graph replays, nothing between the kernels (the expert kernel overlaps "
                               "the router by programmatic dependent launch, so its own duration is at most "
                               "this)",
                     "check": {"launch_ms_x_launches": dom_ms * T, "ms_per_step": ms_step,
                               "ok": dom_ms * T <= ms_step * (1 + 1e-9)}},
        "kernels_ms_per_token_events": dict(
            ({"router_topk": per_launch_ms[0], "expert_fused": per_launch_ms[1] + per_launch_ms[2]} if fused else
             {"router_topk": per_launch_ms[0], "gateup": per_launch_ms[1], "down": per_launch_ms[2]}),
            note="events recorded between the kernels inside the graph serialise them (no overlap); "
                 "their sum exceeds the per-token step time"),
        "chain": {"expert_bytes_per_token": expert_bytes, "router_bytes_per_token": router_bytes,
                  "achieved_gbs": chain_gbs, "frac_of_peak": chain_gbs / hbm_peak,
                  "us_per_token": 1e3 * ms_step / T},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": T * shape.hidden * 2,
                "d2h_bytes_per_step": T * shape.hidden * 4},
        "e2e_per_token": e2e_tok,
        "gpu_launches": (2 if fused else 3) * T * args.steps,
    }
    del g, gi
    return result


def bench_stack48(args, dist, binding, device, synth, torch, hbm_peak):
    wl = synth.WORKLOADS["stack48"]
    shape, seed, NL, S = wl["shape"], wl["seed"], wl["n_layers"], wl["n_steps"]
    plan = binding.si_moe_plan(device.desc_for(shape), torch.cuda.current_device())
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    layers = []
    for l in range(NL):
        wg, wu, wd, rw = synth.make_layer_torch(shape, seed, l)
        layers.append((binding.layer_struct(wg, wu, wd, rw), (wg, wu, wd, rw)))
    x = synth.make_tokens_torch(S * NL, shape.hidden, (seed, "stack-x")).view(S, NL, shape.hidden)
    out = torch.empty((S, NL, shape.hidden), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for s in range(S):
                for l in range(NL):
                    binding.si_moe_forward_decode(plan, layers[l][0], x[s, l], 1, out[s, l], None, scratch,
                                                  stream=stream)
    steps = max(1, args.steps // 4)
    ms, clocks = time_graph(g, stream, steps, min(args.warmup, 2), dist, ClockSampler(torch.cuda.current_device()))
    st = binding.si_moe_read_status(plan, scratch, stream)
    assert st == binding.SI_OK
    tok_s = S * steps / (ms / 1e3)
    step_bytes = NL * shape.top_k * shape.expert_bytes
    gbs = step_bytes * tok_s / 1e9
    del g
    return {"workload": "48-layer stack, 256 decode steps (16.3 GB Q4_K resident)",
            "tok_per_s": dist.sum(tok_s), "layer_tok_per_s": dist.sum(tok_s) * NL,
            "us_per_step": 1e6 / tok_s, "expert_bytes_per_step": step_bytes,
            "achieved_gbs": gbs, "frac_of_peak": gbs / hbm_peak, "clocks": clocks,
            "gpu_launches": (2 if binding.si_debug_decode_fused(plan, 1) >= 1 else 3) * NL * S * steps}


def bench_dedup4(args, dist, binding, device, synth, torch, hbm_peak):
    wl = synth.WORKLOADS["dedup4"]
    shape, seed, n, S = wl["shape"], wl["seed"], wl["tokens_per_step"], wl["n_steps"]
    bias = synth.dedup_router_bias(seed, synth.load_dedup_beta())
    layer = synth.make_layer(shape, seed=seed, router_bias=bias)
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape), torch.cuda.current_device())
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, n)
    x = device.tokens_to_device(synth.make_tokens(shape, seed, n * S)).view(S, n, shape.hidden)
    out = torch.empty((S, n, shape.hidden), dtype=torch.float32, device="cuda")
    counts = torch.zeros((S, shape.n_experts), dtype=torch.int32, device="cuda")
    routes = [binding.route_struct(expert_counts=counts[s]) for s in range(S)]
    stream = torch.cuda.Stream()
    g = build_layer_graph(binding, plan, dl.struct(), [x[s] for s in range(S)], [out[s] for s in range(S)],
                          scratch, stream, n_tok=n, route=routes)
    steps = max(1, args.steps // 2)
    ms, clocks = time_graph(g, stream, steps, args.warmup, dist, ClockSampler(torch.cuda.current_device()))
    st = binding.si_moe_read_status(plan, scratch, stream)
    assert st == binding.SI_OK, binding.si_status_string(st)
    U = (counts > 0).sum(dim=1).double()
    u_mean = float(U.mean())
    tok_s = n * S * steps / (ms / 1e3)
    step_s = S * steps / (ms / 1e3)
    bytes_per_step = u_mean * shape.expert_bytes
    gbs = bytes_per_step * step_s / 1e9
    del g
    return {"workload": "4 tokens/step deduplicated decode, 512 steps, biased routing (32 hot experts, 60% mass)",
            "tok_per_s": dist.sum(tok_s), "us_per_step": 1e6 / step_s, "mean_unique_experts": u_mean,
            "expert_bytes_per_step": bytes_per_step,
            "non_dedup_bytes_per_step": n * shape.top_k * shape.expert_bytes,
            "achieved_gbs": gbs, "frac_of_peak": gbs / hbm_peak, "clocks": clocks,
            "gpu_launches": (2 if binding.si_debug_decode_fused(plan, n) >= 1 else 3) * S * steps}


def bench_prenorm(args, dist, binding, device, synth, torch, hbm_peak):
    """The headline decode workload as a pre-normed block with its residual
    (out = x + MoE(x * gamma / rms(x))): 1024 sequential single-token calls."""
    wl = synth.WORKLOADS["layer"]
    shape, seed, T = wl["shape"], wl["seed"], 1024
    layer = synth.make_layer(shape, seed=seed)
    layer.norm_weight = synth.make_norm_weight(shape, seed=seed)
    layer.norm_eps = 1e-6
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape), torch.cuda.current_device())
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    x = device.tokens_to_device(synth.make_tokens(shape, seed + dist.rank, T))
    out = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    g = build_layer_graph(binding, plan, dl.struct(), [x[t] for t in range(T)], [out[t] for t in range(T)],
                          scratch, stream)
    steps = max(1, args.steps // 2)
    ms, clocks = time_graph(g, stream, steps, args.warmup, dist, ClockSampler(torch.cuda.current_device()))
    st = binding.si_moe_read_status(plan, scratch, stream)
    assert st == binding.SI_OK, binding.si_status_string(st)
    tok_s = T * steps / (ms / 1e3)
    expert_bytes = shape.top_k * shape.expert_bytes
    gbs = expert_bytes * tok_s / 1e9
    path = binding.si_debug_decode_fused(plan, 1)
    del g
    return {"workload": "qwen3-30b-a3b-moe-layer-decode-bs1 as a pre-normed block (RMSNorm gain U[0.5,1.5], "
                        "eps 1e-6, residual added)",
            "tok_per_s": dist.sum(tok_s), "us_per_token": 1e6 / tok_s, "expert_bytes_per_token": expert_bytes,
            "achieved_gbs": gbs, "frac_of_peak": gbs / hbm_peak, "clocks": clocks,
            "gpu_launches": {2: 2, 1: 2}.get(path, 3) * T * steps}


def bench_nvfp4(args, dist, binding, device, synth, torch, hbm_peak):
    """The headline decode workload (1024 sequential single-token calls in one
    CUDA graph) with NVFP4 experts: E2M1 codes, E4M3 scales per 16 weights, an
    fp32 tensor scale per expert matrix, 144 bytes per 256 weights."""
    wl = synth.WORKLOADS["layer"]
    shape, seed, T = wl["shape"], wl["seed"], 1024
    layer = synth.make_layer_nvfp4(shape, seed=seed)
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape, wtype=binding.SI_WTYPE_NVFP4), torch.cuda.current_device())
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    x = device.tokens_to_device(synth.make_tokens(shape, seed, T))
    out = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    g = build_layer_graph(binding, plan, dl.struct(), [x[t] for t in range(T)], [out[t] for t in range(T)],
                          scratch, stream)
    steps = max(1, args.steps // 2)
    ms, clocks = time_graph(g, stream, steps, args.warmup, dist, ClockSampler(torch.cuda.current_device()))
    st = binding.si_moe_read_status(plan, scratch, stream)
    assert st == binding.SI_OK, binding.si_status_string(st)
    tok_s = T * steps / (ms / 1e3)
    expert_bytes = shape.top_k * shape.expert_bytes
    gbs = expert_bytes * tok_s / 1e9
    path = binding.si_debug_decode_fused(plan, 1)
    del g
    return {"workload": "qwen3-30b-a3b-moe-layer-decode-bs1 with NVFP4 experts (synthetic codes and scales, "
                        "144 B / 256 weights), 1024 tokens",
            "tok_per_s": dist.sum(tok_s), "us_per_token": 1e6 / tok_s, "expert_bytes_per_token": expert_bytes,
            "achieved_gbs": gbs, "frac_of_peak": gbs / hbm_peak, "clocks": clocks,
            "gpu_launches": {2: 2, 1: 2}.get(path, 3) * T * steps}


def bench_q5k(args, dist, binding, device, synth, torch, hbm_peak):
    """The headline decode workload (1024 sequential single-token calls in one
    CUDA graph) with Q5_K experts (176 bytes per 256 weights)."""
    wl = synth.WORKLOADS["layer"]
    shape, seed, T = wl["shape"], wl["seed"], 1024
    layer = synth.make_layer_q5k(shape, seed=seed)
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape, wtype=binding.SI_WTYPE_Q5_K), torch.cuda.current_device())
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    x = device.tokens_to_device(synth.make_tokens(shape, seed, T))
    out = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    g = build_layer_graph(binding, plan, dl.struct(), [x[t] for t in range(T)], [out[t] for t in range(T)],
                          scratch, stream)
    steps = max(1, args.steps // 2)
    ms, clocks = time_graph(g, stream, steps, args.warmup, dist, ClockSampler(torch.cuda.current_device()))
    st = binding.si_moe_read_status(plan, scratch, stream)
    assert st == binding.SI_OK, binding.si_status_string(st)
    tok_s = T * steps / (ms / 1e3)
    expert_bytes = shape.top_k * 3 * shape.hidden * shape.intermediate // 256 * synth.Q5K_BLOCK_BYTES
    gbs = expert_bytes * tok_s / 1e9
    path = binding.si_debug_decode_fused(plan, 1)
    del g
    return {"workload": "qwen3-30b-a3b-moe-layer-decode-bs1 with Q5_K experts (176 B / 256 weights), 1024 tokens",
            "tok_per_s": dist.sum(tok_s), "us_per_token": 1e6 / tok_s, "expert_bytes_per_token": expert_bytes,
            "achieved_gbs": gbs, "frac_of_peak": gbs / hbm_peak, "clocks": clocks,
            "gpu_launches": {2: 2, 1: 2}.get(path, 3) * T * steps}


def bench_act8(args, dist, binding, device, synth, torch, hbm_peak):
    """The headline decode workload (1024 sequential single-token calls in one
    CUDA graph) in the int8-activation mode (SI_FLAG_ACT_INT8: x and h int8
    per 32 columns, dp4a).  An approximation with its own tolerance, measured
    by tests/test_gpu_act8.py against the exact block; this entry times it."""
    wl = synth.WORKLOADS["layer"]
    shape, seed, T = wl["shape"], wl["seed"], 1024
    layer = synth.make_layer(shape, seed=seed)
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape, flags=binding.SI_FLAG_ACT_INT8), torch.cuda.current_device())
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, 1)
    x = device.tokens_to_device(synth.make_tokens(shape, seed, T))
    out = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    g = build_layer_graph(binding, plan, dl.struct(), [x[t] for t in range(T)], [out[t] for t in range(T)],
                          scratch, stream)
    steps = max(1, args.steps // 2)
    ms, clocks = time_graph(g, stream, steps, args.warmup, dist, ClockSampler(torch.cuda.current_device()))
    st = binding.si_moe_read_status(plan, scratch, stream)
    assert st == binding.SI_OK, binding.si_status_string(st)
    tok_s = T * steps / (ms / 1e3)
    expert_bytes = shape.top_k * shape.expert_bytes
    gbs = expert_bytes * tok_s / 1e9
    path = binding.si_debug_decode_fused(plan, 1)
    del g
    return {"workload": "qwen3-30b-a3b-moe-layer-decode-bs1, int8 activations per 32 columns (approximate mode), "
                        "1024 tokens",
            "dtype": "q4k-w x int8-act (per 32 columns) -> fp32 accumulate",
            "tok_per_s": dist.sum(tok_s), "us_per_token": 1e6 / tok_s, "expert_bytes_per_token": expert_bytes,
            "achieved_gbs": gbs, "frac_of_peak": gbs / hbm_peak, "clocks": clocks,
            "gpu_launches": {2: 2, 1: 2}.get(path, 3) * T * steps}


def tensor_peak():
    """Dense 16-bit tensor-core peak (TFLOP/s): the measured bf16 GEMM figure
    (fp16 has the same dense rate on this part)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured (MEASURED_PEAKS.json bf16_tflops burst / bf16_tflops_sustained)"
    return 1900.0, 1700.0, "fallback (1.9 PFLOP/s burst, 1.7 sustained)"


def bench_prefill(args, dist, binding, device, synth, torch, nvfp4=False, q5k=False):
    """Grouped prefill of 4096 tokens through one layer of the Qwen3-30B-A3B
    shape: routing + two tensor-core GEMMs + combine, per call (Q4_K experts,
    NVFP4 experts with nvfp4=True, Q5_K experts with q5k=True)."""
    wl = synth.WORKLOADS["prefill"]
    shape, seed, T = wl["shape"], wl["seed"], wl["n_tokens"]
    layer = (synth.make_layer_nvfp4(shape, seed=seed) if nvfp4 else
             synth.make_layer_q5k(shape, seed=seed) if q5k else synth.make_layer(shape, seed=seed))
    dl = device.to_device(layer)
    wtype = binding.SI_WTYPE_NVFP4 if nvfp4 else binding.SI_WTYPE_Q5_K if q5k else binding.SI_WTYPE_Q4_K
    plan = binding.si_moe_plan(device.desc_for(shape, max_tokens=T, wtype=wtype), torch.cuda.current_device())
    scratch = device.alloc_scratch(plan, binding.SI_MODE_PREFILL, T)
    x = device.tokens_to_device(synth.make_tokens(shape, seed, T))
    out = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
    L = dl.struct()
    stream = torch.cuda.Stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    with torch.cuda.stream(stream):
        for e in ev:  # torch creates the CUDA event on its first record
            e.record(stream)
        for _ in range(max(3, args.warmup)):
            binding.si_moe_forward_prefill(plan, L, x, T, out, None, scratch, stream=stream)
    stream.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        binding.si_moe_forward_prefill(plan, L, x, T, out, None, scratch, stream=stream)
    stream.synchronize()
    one = time.perf_counter() - t0
    reps = int(min(2000, max(10, 0.6 / max(one, 1e-5))))  # ~0.6 s timed, so the clock sampler sees it
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        binding.si_moe_forward_prefill(plan, L, x, T, out, None, scratch, stream=stream)
    e1.record(stream)
    e1.synchronize()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / reps
    parts = [0.0] * 4
    nev = min(reps, 20)
    for _ in range(nev):
        binding.si_debug_prefill_events(plan, L, x, T, out, None, scratch, events=ev, stream=stream)
        ev[4].synchronize()
        for i in range(4):
            parts[i] += ev[i].elapsed_time(ev[i + 1]) / nev
    assert binding.si_moe_read_status(plan, scratch, stream) == binding.SI_OK
    pairs = T * shape.top_k
    f_gateup = 2.0 * pairs * 2 * shape.intermediate * shape.hidden
    f_down = 2.0 * pairs * shape.hidden * shape.intermediate
    burst, sustained, src = tensor_peak()
    gemm_ms = parts[1] + parts[2]
    tflops = (f_gateup + f_down) / (gemm_ms * 1e-3) / 1e12
    tok_s = T / (ms * 1e-3)
    del scratch
    return {"workload": "grouped prefill, 4096 tokens x top-8 of 128 experts, one Qwen3-30B-A3B layer, seed 4" +
                        (", NVFP4 experts" if nvfp4 else ", Q5_K experts" if q5k else ""),
            "tok_per_s": dist.sum(tok_s), "ms_per_call": ms,
            "kernels_ms": {"routing_counts_perm": parts[0], "gemm_gateup_swiglu": parts[1],
                           "gemm_down_weight": parts[2], "combine": parts[3]},
            "gemm_flop": f_gateup + f_down,
            "roofline": {"bound": "tensor", "kernel": "k_prefill_gemm<0> + k_prefill_gemm<1> (fp16 operands, "
                                                      "fp32 accumulation in tensor memory)",
                         "achieved": tflops, "peak": burst, "unit": "TFLOP/s", "frac": tflops / burst,
                         "frac_of_sustained": tflops / sustained, "peak_source": src,
                         "gateup_tflops": f_gateup / (parts[1] * 1e-3) / 1e12,
                         "down_tflops": f_down / (parts[2] * 1e-3) / 1e12},
            "calls_timed": reps, "clocks": clocks, "gpu_launches": 6 * reps}


def dedup_probe(args, binding, device, synth, torch):
    """S steps of the dedup4 workload, launched one after another on a stream (no
    graph), so that a profiler sees one expert-kernel launch per step; prints the
    distinct experts of every step and the bytes each of them has."""
    wl = synth.WORKLOADS["dedup4"]
    shape, seed, n = wl["shape"], wl["seed"], wl["tokens_per_step"]
    S = args.dedup_probe
    bias = synth.dedup_router_bias(seed, synth.load_dedup_beta())
    layer = synth.make_layer(shape, seed=seed, router_bias=bias)
    dl = device.to_device(layer)
    plan = binding.si_moe_plan(device.desc_for(shape), torch.cuda.current_device())
    scratch = device.alloc_scratch(plan, binding.SI_MODE_DECODE, n)
    x = device.tokens_to_device(synth.make_tokens(shape, seed, n * S)).view(S, n, shape.hidden)
    out = torch.empty((S, n, shape.hidden), dtype=torch.float32, device="cuda")
    counts = torch.zeros((S, shape.n_experts), dtype=torch.int32, device="cuda")
    L = dl.struct()
    for s in range(S):
        binding.si_moe_forward_decode(plan, L, x[s], n, out[s], binding.route_struct(expert_counts=counts[s]),
                                      scratch)
    torch.cuda.synchronize()
    st = binding.si_moe_read_status(plan, scratch)
    assert st == binding.SI_OK, binding.si_status_string(st)
    U = (counts > 0).sum(dim=1).tolist()
    return {"dedup_probe_steps": S, "unique_experts_per_step": U, "bytes_per_expert": shape.expert_bytes,
            "expert_kernel": {3: "k_expert_cluster (distinct-expert units)", 1: "k_expert"}.get(
                binding.si_debug_decode_fused(plan, n), "generic")}


def run_ours(args, dist):
    import torch
    from quantized_moe_expert_gemv_gb300 import binding, build, device, synth
    build.build()
    binding.load_library()
    torch.cuda.set_device(dist.local)
    if args.dedup_probe:
        res = dedup_probe(args, binding, device, synth, torch)
        if dist.rank == 0:
            print(json.dumps(res), flush=True)
        return
    if args.prefill_only:
        res = bench_prefill(args, dist, binding, device, synth, torch)
        if dist.rank == 0:
            print(json.dumps(res), flush=True)
        return
    hbm_peak, peak_src = peaks()
    res = bench_layer(args, dist, binding, device, synth, torch, hbm_peak)
    res["roofline"]["peak_source"] = peak_src
    line = {"metric": METRIC, "value": res["value"], "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "q4k-w x int16-act (per 64 columns) -> fp32 accumulate",
            "data": "synthetic (seeded Q4_K experts, bf16 N(0,1) tokens)"}
    for k in ("config", "roofline", "kernels_ms_per_token_events", "chain", "clocks", "e2e", "e2e_per_token",
              "gpu_launches"):
        line[k] = res[k]
    if not args.no_extras:
        torch.cuda.empty_cache()
        try:
            line["stack48"] = bench_stack48(args, dist, binding, device, synth, torch, hbm_peak)
        except Exception as exc:  # report, do not hide the headline
            line["stack48"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        try:
            line["dedup4"] = bench_dedup4(args, dist, binding, device, synth, torch, hbm_peak)
        except Exception as exc:
            line["dedup4"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        try:
            line["prenorm"] = bench_prenorm(args, dist, binding, device, synth, torch, hbm_peak)
        except Exception as exc:
            line["prenorm"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        try:
            line["prefill"] = bench_prefill(args, dist, binding, device, synth, torch)
        except Exception as exc:
            line["prefill"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        try:
            line["nvfp4"] = bench_nvfp4(args, dist, binding, device, synth, torch, hbm_peak)
            line["nvfp4"]["prefill"] = bench_prefill(args, dist, binding, device, synth, torch, nvfp4=True)
        except Exception as exc:
            line["nvfp4"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        try:
            line["act8"] = bench_act8(args, dist, binding, device, synth, torch, hbm_peak)
        except Exception as exc:
            line["act8"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        try:
            line["q5k"] = bench_q5k(args, dist, binding, device, synth, torch, hbm_peak)
            line["q5k"]["prefill"] = bench_prefill(args, dist, binding, device, synth, torch, q5k=True)
        except Exception as exc:
            line["q5k"] = {"error": repr(exc)}
    # two-sided guard: an achieved fraction of a measured peak above 1.0 means the timed
    # region did not do the work it is credited with
    fracs = {"roofline": line["roofline"].get("frac"), "chain": line.get("chain", {}).get("frac_of_peak")}
    for key in ("stack48", "dedup4", "prenorm", "nvfp4"):
        if isinstance(line.get(key), dict):
            fracs[key] = line[key].get("frac_of_peak")
    if isinstance(line.get("prefill"), dict) and "roofline" in line["prefill"]:
        fracs["prefill"] = line["prefill"]["roofline"].get("frac")
    over = {k: v for k, v in fracs.items() if v is not None and v > 1.0}
    line["guard"] = {"max_frac_ok": not over, "over": over}
    if over:
        print("bench: achieved fraction above 1.0 -- rejected: %s" % over, file=sys.stderr)
    if dist.rank == 0 and not args.no_cpu_baseline:
        cores = cpu_cores()
        # bounded samples: about 20 s of oracle work in all on a 16-core host
        n = args.cpu_sample_tokens or max(256, 160 * cores)
        tps, dt = oracle_tokens_per_s(n, cores)
        tps1, dt1 = oracle_tokens_per_s(64, 1)
        line["cpu_baseline"] = {"value": tps, "unit": "tok/s", "cores": cores, "kind": "oracle",
                                "sample": f"{n} tokens of the headline layer, one per thread, {dt:.1f} s",
                                "single_thread": {"value": tps1, "unit": "tok/s", "cores": 1,
                                                  "sample": f"64 tokens of the headline layer, {dt1:.1f} s"}}
        if isinstance(line.get("prefill"), dict) and "tok_per_s" in line["prefill"]:
            np_ = max(256, 64 * cores)
            ptps, pdt = oracle_prefill_tokens_per_s(np_, cores)
            ptps1, pdt1 = oracle_prefill_tokens_per_s(64, 1)
            line["prefill"]["cpu_baseline"] = {
                "value": ptps, "unit": "tok/s", "cores": cores, "kind": "oracle",
                "sample": f"{np_} tokens of the prefill workload's layer (routing, counts/offsets/perm, "
                          f"one expert per thread, slot-order combine), {pdt:.1f} s",
                "single_thread": {"value": ptps1, "unit": "tok/s", "cores": 1,
                                  "sample": f"64 tokens of the prefill workload's layer, {pdt1:.1f} s"}}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    dist = Dist(args.gpus)
    if args.impl == "reference":
        run_reference(args, dist)
    else:
        run_ours(args, dist)
    if dist.pg:
        dist.pg.destroy_process_group()


if __name__ == "__main__":
    main()

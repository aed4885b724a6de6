#!/usr/bin/env python
"""Benchmark of the DSA indexer path with IndexCache on GB300.

A step of the default workload (stack61) is one forward through a 61-layer
DSA stack with IndexCache freq 4: the 16 F layers each run the whole indexer
path over a mixed batch of 64 decode tokens at 32768 context plus one
4096-token prefill chunk (K quantisation and paged-cache write of the step's
tokens, q quantisation with the weight fold, the FP8 tensor-core scores,
per-row top-k with the logical->physical conversion), and the 45 S layers
reuse the F layer's buffers. The same stack with freq 1 (61 F layers) is
timed beside it. The line's ``workloads`` object carries the single-layer
workloads decode8x128k, prefill4x8k and decode32, each with its own
roofline. Inputs are synthetic (seeded normals), resident in HBM.

Prints one JSON line (rank 0). ``--gpus N`` runs one replica of the workload
per GPU (N ranks under torch.distributed.run, started by this script when it
is not already under it; no collective on the data path). ``--impl
reference`` times the CPU oracle on the host cores instead (a bounded sample
of the same workload per step). ``--dry-run`` exercises the multi-rank
launcher and timing on CPU (gloo), without a GPU.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from dsa_sparse_attention_quant_gb300 import synth  # noqa: E402

METRIC = "indexer score-pairs/s (q·k ×64 heads) + top-k rows/s; % of HBM/FP8 roofline"
L2_BYTES = 129 * 1024 * 1024
HBM_FALLBACK_GBS = 6800.0
# Nominal GB300 figures, reported beside the measured-peak fractions: HBM3e
# at about 8 TB/s, dense FP8 tensor cores at 4.5 PFLOP/s.
NOMINAL_HBM_GBS = 8000.0
NOMINAL_FP8_TFLOPS = 4500.0
FLOP_PER_PAIR = 64 * 128 * 2  # one causal (token, key) pair: 64 heads x 128-dim dot products
DEFAULT_WORKLOAD = "stack61"
DEFAULT_SUB_WORKLOADS = "decode8x128k,prefill4x8k,decode32"

STACK_LAYERS, STACK_FREQ = 61, 4
WORKLOAD_DESC = {
    "decode32": ("decode32: 32 decode requests x 1 query token, context uniform on [4096, 8192] (seed 1), 64 FP8 "
                 "heads x 128, 132 B/slot paged K cache (64-slot pages, permuted block table), top-2048, 1 indexer "
                 "layer"),
    "decode8x128k": ("decode8x128k: 8 decode requests at 131072 context, random block table, top-2048, "
                     "logical->physical conversion included"),
    "prefill4x8k": ("prefill4x8k: 4 causal prefills of 8192 tokens (32768 query tokens), shuffled pages, K quant + "
                    "cache write fused with logits/top-k, top-2048"),
    "prefill512": "prefill512: 1 request, causal prefill of 512 tokens, RoPE inputs, top-128",
    "stack61": ("stack61: 61 DSA layers, IndexCache freq=4 (skip = max(l-1,0)%4 != 0: 16 F layers run the indexer, "
                "45 S layers reuse the persistent top-k buffer); per F layer a mixed batch of 64 decode tokens at "
                "32768 context + one fresh 4096-token prefill chunk, independent per-layer K caches, top-2048; "
                "compared with freq=1 (all 61 layers run the indexer)"),
}


def host_workload(name: str):
    """The workload's seeded host batch (for stack61: one F layer of the stack)."""
    if name == "stack61":
        return synth.stack_layer(0)
    if name in synth.WORKLOADS:
        return synth.WORKLOADS[name]()
    raise SystemExit(f"unknown workload {name}")


LOGITS_SOURCES = ("logits.cu", "common.cuh")
GATHER_SOURCES = ("gather.cu", "common.cuh")


def kernel_source_sha(sources=LOGITS_SOURCES) -> str:
    """First 16 hex digits of the sha256 of the named csrc/ files, in order."""
    import hashlib

    csrc = os.path.join(ROOT, "dsa_sparse_attention_quant_gb300", "csrc")
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary: str, sources=LOGITS_SOURCES):
    """DRAM bytes per launch from an ncu summary in profiles/, or None when the
    summary is missing or was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        line = line.strip().strip("|").strip()
        if line.startswith("source_sha:"):
            fields["sha"] = line.split(":", 1)[1].strip()
        elif line.startswith("dram_bytes_per_launch"):
            fields["bytes"] = line.split("|")[-1].strip()
    if fields.get("sha") != kernel_source_sha(sources) or "bytes" not in fields:
        return None
    return int(fields["bytes"])


# --------------------------------------------------------------------- ranks

class Ranks:
    """This process's place in the run: world size, rank, local rank, device."""

    def __init__(self, world: int, rank: int, local: int, dev):
        self.world, self.rank, self.local, self.dev = world, rank, local, dev


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over the ranks of the process group (x itself on
    one rank). The timed region of a multi-GPU run is the slowest rank's."""
    import torch
    import torch.distributed as dist

    if not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def gather_over_ranks(x: float, device) -> list:
    """x of every rank, in rank order ([x] on one rank)."""
    import torch
    import torch.distributed as dist

    if not dist.is_initialized() or dist.get_world_size() == 1:
        return [float(x)]
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    out = [torch.zeros_like(t) for _ in range(dist.get_world_size())]
    dist.all_gather(out, t)
    return [float(o.item()) for o in out]


def barrier(ranks: Ranks) -> None:
    import torch.distributed as dist

    if ranks.world > 1:
        dist.barrier()


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Throughput of the whole job: every rank processed its own replica of the
    workload (weak scaling), all within the slowest rank's time."""
    return units_per_rank * world / seconds


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def relaunch_cmd(n: int, argv) -> list:
    """The torch.distributed.run command that starts this script on n ranks."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__), *argv]


def init_ranks(args) -> Ranks:
    """Ranks from the torch.distributed.run environment (one GPU per rank)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.dry_run:
        if world > 1:
            import torch.distributed as dist

            dist.init_process_group("gloo")
        return Ranks(world, rank, local, "cpu")
    import torch

    if args.impl == "reference":
        return Ranks(world, rank, local, "cpu")
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return Ranks(world, rank, local, torch.device("cuda", torch.cuda.current_device()))


# --------------------------------------------------------------------- peaks and rooflines

def read_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm": float(p["hbm_gbs"]), "bf16_burst": float(p["bf16_tflops"]),
                "bf16_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "src": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm": HBM_FALLBACK_GBS, "bf16_burst": 1900.0, "bf16_sustained": 1700.0, "src": "fallback"}


def hbm_roofline(kernel: str, nbytes: float, ms: float, peaks: dict, b2b_ms=None, traffic=None) -> dict:
    """Roofline of a bandwidth-bound kernel: algorithmic bytes / event-timed duration."""
    achieved = nbytes / (ms / 1e3) / 1e9
    r = {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
         "frac": achieved / peaks["hbm"], "traffic": traffic, "algorithmic_bytes_per_launch": nbytes,
         "avg_launch_ms": ms,
         "peak_source": f"{peaks['src']} (of measured): MEASURED_PEAKS.json hbm_gbs, copy bandwidth",
         "frac_nominal": achieved / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS}
    if b2b_ms is not None:
        r["back_to_back_ms"] = b2b_ms
        r["frac_back_to_back"] = nbytes / (b2b_ms / 1e3) / 1e9 / peaks["hbm"]
        r["frac_back_to_back_nominal"] = nbytes / (b2b_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS
    return r


def tensor_roofline(kernel: str, flops: float, ms: float, peaks: dict, b2b_ms=None, traffic=None) -> dict:
    """Roofline of the FP8 contraction. Every duration here is a launch timed
    on its own (well under a second), so the denominator is the burst figure:
    FP8 = 2 x the measured bf16 cuBLAS burst rate (the nominal FP8/bf16 ratio
    of 4.5 / 2.25 PFLOP/s). kind::f8f6f4 runs E2M1 operands at the FP8 rate."""
    peak = 2.0 * peaks["bf16_burst"]
    achieved = flops / (ms / 1e3) / 1e12
    r = {"bound": "tensor", "kernel": kernel, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
         "frac": achieved / peak, "traffic": traffic, "algorithmic_flops_per_launch": flops, "avg_launch_ms": ms,
         "peak_source": f"{peaks['src']} (of measured): 2 x MEASURED_PEAKS.json bf16_tflops (burst; the launch is "
                        "timed alone)",
         "frac_nominal": achieved / NOMINAL_FP8_TFLOPS, "nominal_peak": NOMINAL_FP8_TFLOPS,
         "frac_of_sustained": achieved / (2.0 * peaks["bf16_sustained"])}
    if b2b_ms is not None:
        r["back_to_back_ms"] = b2b_ms
        r["frac_back_to_back"] = flops / (b2b_ms / 1e3) / 1e12 / peak
    return r


def decode_score_bytes(pairs: int, tokens: int, slot_bytes: int) -> int:
    """Algorithmic bytes of the decode score kernel: each visible K slot (132 B
    FP8, 68 B FP4) streams from HBM once per pair and each pair's fp32 score is
    written once; q codes (8 KB) and folded weights (256 B) once per token."""
    return pairs * (slot_bytes + 4) + tokens * (64 * 128 + 64 * 4)


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if t0 is not None and not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}




# --------------------------------------------------------------------- our arm

def replica_count(hb, kcache: str, requested: int = 0) -> tuple:
    """Input replicas the steps rotate over (so that their total exceeds twice
    the L2 and every step reads its K cache from HBM), and one replica's bytes."""
    slot_bytes = 68 if kcache == "fp4" else 132
    per_replica = hb.num_blocks * 64 * slot_bytes + hb.num_tokens * (64 * 128 * 2 + 64 * 4 + 128 * 2)
    n_rep = requested or max(1, min(16, math.ceil(2 * L2_BYTES / per_replica)))
    return n_rep, per_replica


def workload_config(name: str, hb, args, world: int) -> dict:
    """The `config` object of a line; the same for both arms of the run."""
    fp4 = args.kcache == "fp4"
    cfg = {
        "workload": WORKLOAD_DESC[name],
        "k_cache": ("FP4: E2M1 codes + ue8m0 fp32 scale per token, 68 B/slot (the reading of use_fp4_cache)"
                    if fp4 else "FP8: E4M3 codes + ue8m0 fp32 scale per token, 132 B/slot"),
        "query_tokens": hb.num_tokens,
        "topk": hb.topk,
        "parallelism": f"one replica per GPU x{world}, no collective on the data path" if world > 1 else "1 GPU",
        "rope": "q and new K rotated (RoPE) in the layer prologue" if args.rope else "inputs arrive rotated",
    }
    if name == "stack61":
        if args.stack_layers != STACK_LAYERS:
            cfg["workload"] += f" [profiling case: the first {args.stack_layers} layers]"
        slot_bytes = 68 if fp4 else 132
        n_f = sum(1 for l in range(args.stack_layers) if max(l - 1, 0) % STACK_FREQ == 0)
        cfg.update({"layers": args.stack_layers, "freq": STACK_FREQ, "f_layers": n_f,
                    "pairs_per_step": n_f * hb.num_pairs(),
                    "l2": f"inputs larger than L2: every F layer reads its own "
                          f"{hb.num_blocks * 64 * slot_bytes / 1e6:.0f} MB K cache"})
    else:
        n_rep, per_replica = replica_count(hb, args.kcache, args.replicas)
        cfg.update({"pairs_per_step": hb.num_pairs(),
                    "l2": f"inputs larger than L2: {n_rep} rotating input replicas, "
                          f"{n_rep * per_replica / 1e6:.0f} MB > 2x 129 MB"})
    return cfg


class Replica:
    """One independent copy of a step's device inputs (K cache, q, w, new K)."""

    def __init__(self, hb, dsa, torch, dev, ctx_k, ctx_slots, kcache="fp8"):
        self.k_cache = dsa.new_k_cache(hb.num_blocks, kcache, device=dev)
        dsa.indexer_k_quant_write(ctx_k, ctx_slots, self.k_cache)
        self.q = torch.from_numpy(hb.q.view(np.int16)).view(torch.bfloat16).to(dev)
        self.w = torch.from_numpy(hb.w).to(dev)
        self.k_new = torch.from_numpy(hb.k_new.view(np.int16)).view(torch.bfloat16).to(dev)


def capture_graph(torch, cap, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        fn()
    return g


def run_layer(args, name: str, ranks: Ranks, with_cpu: bool):
    """One indexer layer (decode32, decode8x128k, prefill4x8k, prefill512):
    returns rank 0's line (None on the other ranks)."""
    import torch

    import dsa_sparse_attention_quant_gb300 as dsa

    dev, world = ranks.dev, ranks.world
    hb = host_workload(name)
    T, k = hb.num_tokens, hb.topk
    pairs = hb.num_pairs()
    batch = dsa.Batch.from_host(hb, dev)
    slots = torch.from_numpy(hb.slot_mapping).to(dev)
    fs, _ = dsa.schedule_build(1, True, 4)

    fp4 = args.kcache == "fp4"
    slot_bytes = 68 if fp4 else 132
    n_rep, per_replica = replica_count(hb, args.kcache, args.replicas)
    ctx_k = torch.from_numpy(hb.ctx_k.view(np.int16)).view(torch.bfloat16).to(dev)
    ctx_slots = torch.from_numpy(hb.ctx_slots).to(dev)
    reps = [Replica(hb, dsa, torch, dev, ctx_k, ctx_slots, args.kcache) for _ in range(n_rep)]
    del ctx_k, ctx_slots

    ws = torch.empty(dsa.layer_stack_workspace_size(batch, k), dtype=torch.uint8, device=dev)
    topk = torch.empty((T, k), dtype=torch.int32, device=dev)
    phys = torch.empty((T, k), dtype=torch.int32, device=dev)
    valid = torch.empty(T, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    layers = [[dict(q=r.q, w=r.w, k_new=r.k_new, k_cache=r.k_cache)] for r in reps]
    # per step: fused prologue (S1 K quant + cache write, S2a q quant + fold, plan),
    # the score kernel(s) (S2b), top-k with the id conversion fused (S3 + S5):
    # the decode rows' select, the prefill rows' per-row top-k
    has_dec = hb.num_decodes > 0
    has_pre = hb.num_reqs > hb.num_decodes
    kernels = ["prologue"] + (["logits<1>"] if has_dec else []) + (["logits<4>"] if has_pre else []) + \
        (["select"] if has_dec else []) + (["topk"] if has_pre else [])
    launches_per_step = len(kernels)  # timeline marks per step
    # decode rows that one CTA stages (up to 32768 scores) take one top-k
    # launch; longer ones a chunk launch and a resolving launch, timed together
    # as "select"
    long_rows = has_dec and (batch.max_seq_len + 3) // 4 * 4 > 32768
    kernel_launches = launches_per_step + (1 if long_rows else 0)

    # --rope: q and the new K rows arrive un-rotated and the layer's prologue
    # applies RoPE (positions + cos/sin table) before quantising them
    positions = torch.from_numpy(hb.positions).to(dev) if args.rope else None
    rope_cs = torch.from_numpy(synth.rope_cos_sin(int(hb.seq_lens.max()) + 1)).to(dev) if args.rope else None

    def step(i, ev=None):
        # S4: the IndexCache runner over this one-layer stack ('F'); one C-ABI call
        if ev is not None:
            dsa.binding.set_launch_events(ev)
        dsa.layer_stack_run(batch, fs, layers[i % n_rep], k, slot_mapping=slots, topk_buf=topk, phys_buf=phys,
                            valid_buf=valid, ws=ws, dev_err=err, positions=positions, rope_cos_sin=rope_cs)
        if ev is not None:
            dsa.binding.set_launch_events(())

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if dsa.check_device_error(err):
        raise SystemExit(f"device error word set: {int(err.item()):#x}")

    # Device-timed region. Each step is one CUDA-graph replay of the calls
    # above (the launch cost of the small kernels would otherwise leave the GPU
    # idle between them); the kernels of a step overlap their set-up with the
    # previous kernel (programmatic dependent launch). Pass 1 times K plain
    # steps: the value. Pass 2 replays the same K steps from graphs that carry a
    # timeline of external event nodes around every kernel, so each launch's
    # device time is measured on its own stream; the event nodes between
    # kernels stop that overlap, so pass 2's kernel times add up to more than
    # pass 1's step.
    stream = torch.cuda.current_stream()
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(launches_per_step + 1)] for _ in range(args.steps)]
    for evs in kev:  # materialise the event handles before capture
        for e in evs:
            e.record(stream)
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    plain = [capture_graph(torch, cap, lambda i=i: step(i)) for i in range(n_rep)]
    timeline = [capture_graph(torch, cap, lambda i=i: step(i, kev[i])) for i in range(args.steps)]
    stream.wait_stream(cap)
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clocks:
        # keep the GPU busy for a short clock window before the timed steps
        t_warm = time.perf_counter()
        i = 0
        while time.perf_counter() - t_warm < args.clock_window:
            plain[i % n_rep].replay()
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        barrier(ranks)
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        t_start.record(stream)
        for i in range(args.steps):
            plain[i % n_rep].replay()
        t_end.record(stream)
        torch.cuda.synchronize()
        wall1 = time.perf_counter()
        barrier(ranks)
        elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), dev)
        for i in range(args.steps):
            timeline[i].replay()
        torch.cuda.synchronize()
        # per launch: elapsed time between the timeline events around it
        per_kernel = np.array([[evs[j].elapsed_time(evs[j + 1]) for j in range(launches_per_step)] for evs in kev])

        # The score kernels alone, K launches back to back on the replicas' q
        # codes, weights and caches: two events around the run give the
        # per-launch time when a launch's set-up overlaps the previous launch's
        # tail (programmatic dependent launch), as it overlaps the prologue
        # inside a step. Reported beside the isolated launches above.
        plan_ws = dsa.indexer_plan(batch)
        qw = [dsa.indexer_q_quant_fold(r.q, r.w) for r in reps]
        b2b_scores = torch.empty((T, (batch.max_seq_len + 3) // 4 * 4), dtype=torch.float32, device=dev)

        def score_launch(i):
            q8_i, _, wf_i = qw[i % n_rep]
            dsa.indexer_logits(batch, q8_i, wf_i, reps[i % n_rep].k_cache, logits=b2b_scores, ws=plan_ws,
                               dev_err=err)

        for i in range(n_rep + 2):
            score_launch(i)
        torch.cuda.synchronize()
        b2b0, b2b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b2b0.record(stream)
        for i in range(args.steps):
            score_launch(i)
        b2b1.record(stream)
        torch.cuda.synchronize()
        b2b_ms = max_over_ranks(b2b0.elapsed_time(b2b1) / args.steps, dev)
        del qw, b2b_scores

        e2e = e2e_layer(args, hb, batch, fs, reps, ws, topk, err, rope_cs, n_rep, ranks, dsa, torch)
    torch.cuda.synchronize()
    if dsa.check_device_error(err):
        raise SystemExit(f"device error word set: {int(err.item()):#x}")
    if ranks.rank != 0:
        return None

    ms_per_step = elapsed_ms / args.steps
    peaks = read_peaks()
    breakdown = {kname: float(per_kernel[:, j].mean() * 1e3) for j, kname in enumerate(kernels)}
    score_cols = [j for j, kname in enumerate(kernels) if kname.startswith("logits")]
    kernel_avg_ms = float(per_kernel[:, score_cols].sum(axis=1).mean())
    traffic = profiled_traffic(f"logits_kernel_{name}{'_fp4' if fp4 else ''}.md")
    mma = "tcgen05 kind::f8f6f4 E2M1 K x E4M3 q" if fp4 else "tcgen05 FP8"
    if not has_pre:
        roofline = hbm_roofline(f"dsa::logits_kernel<1> (decode scores, {mma})",
                                decode_score_bytes(pairs, T, slot_bytes), kernel_avg_ms, peaks, b2b_ms, traffic)
    else:
        roofline = tensor_roofline(f"dsa::logits_kernel (scores, {mma})", pairs * FLOP_PER_PAIR, kernel_avg_ms,
                                   peaks, b2b_ms, traffic)
    roofline["timing"] = ("CUDA events on the launching stream around every launch of the score kernel, in a second "
                          "timed pass over the same K steps (each launch starts cold)")
    roofline["timing_back_to_back"] = ("K launches of the score kernel alone (dsa_indexer_logits on the rotating "
                                       "replicas) between two CUDA events on its stream: each launch's set-up "
                                       "overlaps the previous launch's tail, as it overlaps the prologue in a step")
    line = {
        "metric": METRIC,
        "value": whole_job_rate(pairs, world, ms_per_step / 1e3),
        "unit": "pairs/s",
        "topk_rows_per_s": whole_job_rate(T, world, ms_per_step / 1e3),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp4_e2m1 (K) x fp8_e4m3 (q) -> fp32" if fp4 else "fp8_e4m3 x fp8_e4m3 -> fp32",
        "data": "synthetic (seeded normals, bf16-rounded)",
        "config": workload_config(name, hb, args, world),
        "roofline": roofline,
        "breakdown_us": breakdown,
        "e2e": e2e,
        "gpu_launches": kernel_launches * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed_region": wall1 - wall0,
    }
    if world == 1 and with_cpu and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(hb, args.cpu_seconds, args.kcache)
    return line


def e2e_layer(args, hb, batch, fs, reps, ws, topk, err, rope_cs, n_rep, ranks, dsa, torch) -> dict:
    """End to end through the public API from pinned host memory. Every step
    uploads its inputs (q, w, new K, slots, the batch metadata, positions with
    --rope) packed in one pinned buffer with one copy, runs the layer runner (a
    prepared dsa.LayerStack on views of that upload), and reads the physical
    ids and valid counts back with one copy. Consecutive steps alternate
    between two streams, each with its own workspace and output buffers (and
    their inputs are different replicas): a step's upload overlaps the previous
    step's kernels and its read-back, while its kernels still start only after
    the previous step's kernels (an event), so the device work per step is
    that of the device-timed steps. The host waits for step i's result before
    it enqueues step i + 2."""
    dev = ranks.dev
    T, k = hb.num_tokens, hb.topk
    parts = [("q", hb.q), ("w", hb.w), ("k_new", hb.k_new), ("slots", hb.slot_mapping),
             ("qsl", hb.query_start_loc.astype(np.int32)), ("seq", hb.seq_lens.astype(np.int32)),
             ("bt", hb.block_table.astype(np.int32)), ("req", hb.req_id_per_token.astype(np.int32))]
    if args.rope:
        parts.append(("pos", hb.positions.astype(np.int64)))
    offs, total = {}, 0
    for pname, arr in parts:
        offs[pname] = (total, np.ascontiguousarray(arr))
        total += (arr.nbytes + 255) // 256 * 256
    host_in = torch.empty(max(total, 256), dtype=torch.uint8).pin_memory()
    hv = host_in.numpy()
    for pname, (o, arr) in offs.items():
        hv[o:o + arr.nbytes] = arr.reshape(-1).view(np.uint8)
    out_bytes = (T * k * 4 + 255) // 256 * 256 + T * 4
    host_out = torch.empty(max(out_bytes, 256), dtype=torch.uint8).pin_memory()

    def view(buf, pname, dtype, shape):
        o, arr = offs[pname]
        return buf[o:o + arr.nbytes].view(dtype).view(shape)

    lanes = 2 if n_rep >= 2 else 1
    voff = (T * k * 4 + 255) // 256 * 256
    lane_bufs = []  # per stream: workspace, logical ids, packed device output, pinned host output
    for ln in range(lanes):
        dev_out = torch.empty(max(out_bytes, 256), dtype=torch.uint8, device=dev)
        lane_bufs.append(dict(
            ws=ws if ln == 0 else torch.empty_like(ws), topk=topk if ln == 0 else torch.empty_like(topk),
            dev_out=dev_out, phys=dev_out[:T * k * 4].view(torch.int32).view(T, k),
            valid=dev_out[voff:voff + T * 4].view(torch.int32),
            host_out=host_out if ln == 0 else torch.empty_like(host_out).pin_memory()))
    stacks, dev_in = [[] for _ in range(lanes)], []
    for r in reps:
        d = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
        d.copy_(host_in)
        be = dsa.Batch(view(d, "qsl", torch.int32, (-1,)), view(d, "seq", torch.int32, (-1,)),
                       view(d, "bt", torch.int32, tuple(hb.block_table.shape)), view(d, "req", torch.int32, (-1,)),
                       hb.num_decodes, hb.num_blocks, batch.max_seq_len, batch.num_decode_tokens)
        le = [dict(q=view(d, "q", torch.bfloat16, (T, 64, 128)), w=view(d, "w", torch.float32, (T, 64)),
                   k_new=view(d, "k_new", torch.bfloat16, (T, 128)), k_cache=r.k_cache)]
        for ln, lb in enumerate(lane_bufs):
            stacks[ln].append(dsa.LayerStack(be, fs, le, k, slot_mapping=view(d, "slots", torch.int64, (-1,)),
                                             topk_buf=lb["topk"], phys_buf=lb["phys"], valid_buf=lb["valid"],
                                             ws=lb["ws"], dev_err=err,
                                             positions=view(d, "pos", torch.int64, (-1,)) if args.rope else None,
                                             rope_cos_sin=rope_cs))
        dev_in.append(d)
    h2d, d2h = host_in.numel(), host_out.numel()  # the bytes each step copies
    streams = [torch.cuda.current_stream()] + [torch.cuda.Stream() for _ in range(lanes - 1)]
    kernels_done = [torch.cuda.Event() for _ in range(lanes)]
    started = [False]

    def e2e_step(i):
        ln, j = i % lanes, i % n_rep
        st, lb = streams[ln], lane_bufs[ln]
        with torch.cuda.stream(st):
            dev_in[j].copy_(host_in, non_blocking=True)
            if started[0]:
                st.wait_event(kernels_done[(i - 1) % lanes])  # one step's kernels at a time
            stacks[ln][j].run(st)
            kernels_done[ln].record(st)
            started[0] = True
            lb["host_out"].copy_(lb["dev_out"], non_blocking=True)
        if lanes == 1:
            st.synchronize()
        elif i > 0:
            streams[(i - 1) % lanes].synchronize()  # step i - 1's result is on the host

    for i in range(args.warmup):
        e2e_step(i)
    streams[(args.warmup - 1) % lanes].synchronize()
    torch.cuda.synchronize()
    barrier(ranks)
    e0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    streams[(args.steps - 1) % lanes].synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - e0, dev)
    return {
        "value": whole_job_rate(hb.num_pairs(), ranks.world, e2e_s / args.steps),
        "unit": "pairs/s",
        "h2d_bytes_per_step": h2d,
        "d2h_bytes_per_step": d2h,
        "ms_per_step": e2e_s / args.steps * 1e3,
        "path": "per step: pinned host -> device (one copy), LayerStack.run (one C call), device -> pinned host "
                "(one copy); steps alternate between two streams with their own buffers so that copies overlap "
                "the neighbouring steps' kernels, kernels of consecutive steps ordered by an event; the host waits "
                "for each step's result one step later and for the last at the end",
    }


def compact(line: dict) -> dict:
    """A sub-workload's line without the keys the main line already carries."""
    keep = ("value", "unit", "topk_rows_per_s", "ms_per_step", "dtype", "config", "roofline", "breakdown_us", "e2e",
            "gpu_launches", "clocks", "wall_s_timed_region")
    return {k: line[k] for k in keep if k in line}


# --------------------------------------------------------------------- stack61

def stack_inputs(meta, n_layers, dev, dsa, torch, kcache="fp8"):
    """Per-layer q, w, new K and K cache of the stack, drawn on the device.

    Layer l draws from torch's CUDA generator seeded with 5000 + l (N(0,1),
    rounded to bf16 where the path reads bf16); the metadata (lengths, block
    table, slots) is the host generator's. Drawing 61 caches of 2M tokens on
    the host would take minutes.
    """
    slots_ctx = torch.from_numpy(meta.ctx_slots).to(dev)
    n_ctx, T = int(meta.ctx_slots.shape[0]), meta.num_tokens
    layers = []
    for l in range(n_layers):
        g = torch.Generator(device=dev)
        g.manual_seed(5000 + l)
        cache = dsa.new_k_cache(meta.num_blocks, kcache, device=dev)
        for c0 in range(0, n_ctx, 1 << 20):
            c1 = min(n_ctx, c0 + (1 << 20))
            k = torch.randn((c1 - c0, 128), generator=g, device=dev).to(torch.bfloat16)
            dsa.indexer_k_quant_write(k, slots_ctx[c0:c1], cache)
        q = torch.randn((T, 64, 128), generator=g, device=dev).to(torch.bfloat16)
        w = torch.randn((T, 64), generator=g, device=dev)
        kn = torch.randn((T, 128), generator=g, device=dev).to(torch.bfloat16)
        layers.append(dict(q=q, w=w, k_new=kn, k_cache=cache))
    torch.cuda.synchronize()
    return layers


def stack_host_batch(meta, dev, torch):
    """Layer 0 of the stack as a host batch (the same draws), for the oracle's sample."""
    g = torch.Generator(device=dev)
    g.manual_seed(5000)
    n_ctx, T = int(meta.ctx_slots.shape[0]), meta.num_tokens
    ks = []
    for c0 in range(0, n_ctx, 1 << 20):
        c1 = min(n_ctx, c0 + (1 << 20))
        ks.append(torch.randn((c1 - c0, 128), generator=g, device=dev).to(torch.bfloat16).cpu())
    q = torch.randn((T, 64, 128), generator=g, device=dev).to(torch.bfloat16).cpu()
    w = torch.randn((T, 64), generator=g, device=dev).cpu()
    kn = torch.randn((T, 128), generator=g, device=dev).to(torch.bfloat16).cpu()
    import dataclasses
    u16 = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    return dataclasses.replace(meta, q=u16(q), w=w.numpy(), k_new=u16(kn), ctx_k=u16(torch.cat(ks)))


def run_stack(args, ranks: Ranks, with_cpu: bool):
    """The 61-layer IndexCache stack: one step = one forward through the 61
    layers (the indexer on the F layers, the S layers reuse the buffers).
    Returns rank 0's line (None on the other ranks)."""
    import torch

    import dsa_sparse_attention_quant_gb300 as dsa

    dev, world = ranks.dev, ranks.world
    meta = synth.stack_layer(0, with_data=False)
    T, k = meta.num_tokens, meta.topk
    batch = dsa.Batch.from_host(meta, dev)
    if args.sm_split == "off":
        batch.work = (0, 0)  # no work given: decode and prefill scores one after the other
    slots = torch.from_numpy(meta.slot_mapping).to(dev)
    n_layers = args.stack_layers
    fs4, _ = dsa.schedule_build(n_layers, True, STACK_FREQ)
    fs1, _ = dsa.schedule_build(n_layers, True, 1)
    n_f = fs4.count("F")
    layers = stack_inputs(meta, n_layers, dev, dsa, torch, args.kcache)
    l4 = [layers[l] if fs4[l] == "F" else None for l in range(n_layers)]
    ws = torch.empty(dsa.layer_stack_workspace_size(batch, k), dtype=torch.uint8, device=dev)
    topk = torch.empty((T, k), dtype=torch.int32, device=dev)
    phys = torch.empty((T, k), dtype=torch.int32, device=dev)
    valid = torch.empty(T, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # the batch carries its work (decode keys, prefill pairs) from the host
    # metadata: in the step, each F layer scores the decode rows on this many
    # SMs beside the prefill rows on the rest
    dec_sms = dsa.LayerStack(batch, fs4, l4, k, topk_buf=topk, phys_buf=phys, valid_buf=valid, ws=ws).decode_sms()

    def run(fs, L, ev=None):
        if ev is not None:
            dsa.binding.set_launch_events(ev)
        dsa.layer_stack_run(batch, fs, L, k, slot_mapping=slots, topk_buf=topk, phys_buf=phys, valid_buf=valid,
                            ws=ws, dev_err=err)
        if ev is not None:
            dsa.binding.set_launch_events(())

    for _ in range(args.warmup):
        run(fs4, l4)
        run(fs1, layers)
    torch.cuda.synchronize()
    if dsa.check_device_error(err):
        raise SystemExit(f"device error word set: {int(err.item()):#x}")

    # one F layer alone, with a timeline event after each of its kernels
    kernels = ["prologue", "logits<1>", "logits<4>", "select", "topk"]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(kernels) + 1)] for _ in range(args.steps)]
    stream = torch.cuda.current_stream()
    for evs in kev:
        for e in evs:
            e.record(stream)
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    g4 = capture_graph(torch, cap, lambda: run(fs4, l4))
    g1 = capture_graph(torch, cap, lambda: run(fs1, layers))
    one = [capture_graph(torch, cap, lambda i=i: run("F", [layers[i % n_layers]], kev[i]))
           for i in range(args.steps)]
    stream.wait_stream(cap)
    torch.cuda.synchronize()

    def timed(g, steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(ranks)
        a.record(stream)
        for _ in range(steps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(ranks)
        return max_over_ranks(a.elapsed_time(b) / steps, dev)

    with ClockSampler(torch.cuda.current_device()) as clocks:
        t_warm = time.perf_counter()
        while time.perf_counter() - t_warm < args.clock_window:
            g4.replay()
            torch.cuda.synchronize()
        wall0 = time.perf_counter()
        ms4 = timed(g4, args.steps)
        wall1 = time.perf_counter()
        ms1 = timed(g1, args.steps)
        for g in one:
            g.replay()
        torch.cuda.synchronize()
        per_kernel = np.array([[evs[j].elapsed_time(evs[j + 1]) for j in range(len(kernels))] for evs in kev])

        # end to end: the F layers' q, w and new K and the step's metadata from
        # pinned host memory, the stack, the physical ids back. Consecutive
        # steps alternate between two streams, each with its own device copy
        # of the inputs and metadata and its own outputs: a step's uploads
        # overlap the previous step's kernels, while its kernels start only
        # after the previous step's kernels (an event). The host waits for
        # step i's result before it enqueues step i + 2.
        host = [dict(q=L["q"].cpu().pin_memory(), w=L["w"].cpu().pin_memory(), k_new=L["k_new"].cpu().pin_memory())
                if L is not None else None for L in l4]
        meta_host = {
            "slots": torch.from_numpy(meta.slot_mapping).pin_memory(),
            "qsl": torch.from_numpy(meta.query_start_loc.astype(np.int32)).pin_memory(),
            "seq": torch.from_numpy(meta.seq_lens.astype(np.int32)).pin_memory(),
            "bt": torch.from_numpy(meta.block_table.astype(np.int32)).pin_memory(),
            "req": torch.from_numpy(meta.req_id_per_token.astype(np.int32)).pin_memory(),
        }
        h2d = sum(t.numel() * t.element_size() for h in host if h is not None for t in h.values()) + \
            sum(t.numel() * t.element_size() for t in meta_host.values())
        d2h = T * k * 4 + T * 4
        lanes = []
        for ln in range(2):
            mdev = {n_: t.to(dev) for n_, t in meta_host.items()}
            lb = dsa.Batch(mdev["qsl"], mdev["seq"], mdev["bt"], mdev["req"], meta.num_decodes, meta.num_blocks,
                           batch.max_seq_len, batch.num_decode_tokens)
            lb.work = batch.work
            ll = [dict(q=torch.empty_like(L["q"]), w=torch.empty_like(L["w"]), k_new=torch.empty_like(L["k_new"]),
                       k_cache=L["k_cache"]) if L is not None else None for L in l4]
            o_t, o_p = torch.empty_like(topk), torch.empty_like(phys)
            o_v = torch.empty_like(valid)
            lanes.append(dict(
                meta=mdev, layers=ll, phys=o_p, valid=o_v,
                stack=dsa.LayerStack(lb, fs4, ll, k, slot_mapping=mdev["slots"], topk_buf=o_t, phys_buf=o_p,
                                     valid_buf=o_v, ws=ws if ln == 0 else torch.empty_like(ws), dev_err=err),
                out_phys=torch.empty((T, k), dtype=torch.int32).pin_memory(),
                out_valid=torch.empty(T, dtype=torch.int32).pin_memory(),
                stream=stream if ln == 0 else torch.cuda.Stream(), done=torch.cuda.Event(), ready=torch.cuda.Event()))
        issued = []

        def e2e_step():
            i = len(issued)
            lane = lanes[i % 2]
            st = lane["stream"]
            with torch.cuda.stream(st):
                for L, h in zip(lane["layers"], host):
                    if L is None:
                        continue
                    for pname in ("q", "w", "k_new"):
                        L[pname].copy_(h[pname], non_blocking=True)
                for n_, t in meta_host.items():
                    lane["meta"][n_].copy_(t, non_blocking=True)
                if issued:
                    st.wait_event(lanes[(i - 1) % 2]["done"])  # one step's kernels at a time
                lane["stack"].run(st)
                lane["done"].record(st)
                lane["out_phys"].copy_(lane["phys"], non_blocking=True)
                lane["out_valid"].copy_(lane["valid"], non_blocking=True)
                lane["ready"].record(st)
            issued.append(i)
            if i >= 1:
                lanes[(i - 1) % 2]["ready"].synchronize()  # step i - 1's result is on the host

        def e2e_drain():
            lanes[(len(issued) - 1) % 2]["ready"].synchronize()

        for _ in range(args.warmup):
            e2e_step()
        e2e_drain()
        barrier(ranks)
        e0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        e2e_drain()
        e2e_s = max_over_ranks((time.perf_counter() - e0) / args.steps, dev)
    torch.cuda.synchronize()
    if dsa.check_device_error(err):
        raise SystemExit(f"device error word set: {int(err.item()):#x}")
    if ranks.rank != 0:
        return None

    layer_pairs = meta.num_pairs()
    pairs = n_f * layer_pairs
    n_dec = meta.num_decodes
    dec_pairs = int((meta.positions[:n_dec] + 1).sum())
    pre_pairs = layer_pairs - dec_pairs
    peaks = read_peaks()
    ms = {kname: float(per_kernel[:, j].mean()) for j, kname in enumerate(kernels)}
    slot_bytes = 68 if args.kcache == "fp4" else 132
    mma = "tcgen05 kind::f8f6f4 E2M1 K x E4M3 q" if args.kcache == "fp4" else "tcgen05 FP8"
    fp4_tag = "_fp4" if args.kcache == "fp4" else ""
    phases = {
        "decode_scores": hbm_roofline(f"dsa::logits_kernel<1> (decode scores, {mma})",
                                      decode_score_bytes(dec_pairs, n_dec, slot_bytes), ms["logits<1>"], peaks,
                                      traffic=profiled_traffic(f"logits_kernel_decode_stack61{fp4_tag}.md")),
        "prefill_scores": tensor_roofline(f"dsa::logits_kernel<4> (prefill scores, {mma})",
                                          pre_pairs * FLOP_PER_PAIR, ms["logits<4>"], peaks,
                                          traffic=profiled_traffic(f"logits_kernel_prefill_stack61{fp4_tag}.md")),
        "decode_topk": {"kernel": "dsa::select_kernel", "bound": "latency", "avg_launch_ms": ms["select"],
                        "rows": n_dec, "rows_per_s": n_dec / (ms["select"] / 1e3)},
        "prefill_topk": {"kernel": "dsa::topk_kernel", "bound": "latency", "avg_launch_ms": ms["topk"],
                         "rows": T - n_dec, "rows_per_s": (T - n_dec) / (ms["topk"] / 1e3)},
    }
    dom = "prefill_scores" if ms["logits<4>"] >= ms["logits<1>"] else "decode_scores"
    roofline = dict(phases[dom])
    roofline.update({"phases": phases, "dominant_phase": dom,
                     "timing": "CUDA events on the launching stream around each kernel of one F layer (a one-layer "
                               "stack replayed alone), averaged over K layers; each kernel alone on the whole GPU "
                               "(the launch timeline turns the decode/prefill SM split off)"})
    line = {
        "metric": METRIC,
        "value": whole_job_rate(pairs, world, ms4 / 1e3),
        "unit": "pairs/s",
        "topk_rows_per_s": whole_job_rate(n_f * T, world, ms4 / 1e3),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms4,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp4_e2m1 (K) x fp8_e4m3 (q) -> fp32" if args.kcache == "fp4" else "fp8_e4m3 x fp8_e4m3 -> fp32",
        "data": "synthetic (seeded normals, bf16-rounded; per-layer tensors from torch's seeded CUDA generator)",
        "config": workload_config("stack61", meta, args, world),
        "indexcache": {"freq4_ms_per_step": ms4, "freq1_ms_per_step": ms1, "freq4_speedup_vs_freq1": ms1 / ms4,
                       "f_layer_ms_in_step": ms4 / n_f},
        "sm_split": {"decode_score_sms": dec_sms, "prefill_score_sms": torch.cuda.get_device_properties(dev)
                     .multi_processor_count - dec_sms if dec_sms else None,
                     "note": "in the step each F layer scores its decode rows on decode_score_sms SMs beside its "
                             "prefill rows on the rest (two streams), each segment's top-k after its scores"},
        "roofline": roofline,
        "breakdown_us": {kname: v * 1e3 for kname, v in ms.items()},
        "e2e": {"value": whole_job_rate(pairs, world, e2e_s), "unit": "pairs/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                "path": "per step: the F layers' q, w and new K and the step's metadata copied from pinned host "
                        "memory, the 61-layer stack (one C call), physical ids and valid counts copied back; "
                        "steps alternate between two streams with their own device inputs and outputs (a step's "
                        "uploads overlap the previous step's kernels, its kernels follow them), the host waits for "
                        "each step's result before it enqueues the step after next"},
        "gpu_launches": args.steps * len(kernels) * n_f,
        "clocks": clocks.summary(),
        "wall_s_timed_region": wall1 - wall0,
    }
    if world == 1 and with_cpu and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(stack_host_batch(meta, dev, torch), args.cpu_seconds, args.kcache)
    return line


# --------------------------------------------------------------------- gather

GATHER_DESC = ("gather64x2048: the consumer's read of the selected rows — 64 decode tokens x 2048 physical "
               "slots each, 656-byte rows (an FP8 MLA KV row size) from a 2,097,152-row paged cache "
               "(1.38 GB), ids drawn uniformly (seeded)")


def run_gather(args, ranks: Ranks, with_cpu: bool):
    """Times dsa_gather_rows on its own: value = gathered rows per second."""
    import torch

    import dsa_sparse_attention_quant_gb300 as dsa

    dev, world = ranks.dev, ranks.world
    R, T, k, rb = 64 * 32768, 64, 2048, 656
    g = torch.Generator(device=dev)
    g.manual_seed(6000)
    rows = torch.randint(0, 256, (R, rb), dtype=torch.uint8, device=dev, generator=g)
    n_sets = 4  # rotating id sets
    phys = [torch.randint(0, R, (T, k), dtype=torch.int32, device=dev, generator=g) for _ in range(n_sets)]
    out = torch.empty((T, k, rb), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for i in range(args.warmup):
        dsa.gather_rows(rows, phys[i % n_sets], rb, out=out, dev_err=err)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clocks:
        barrier(ranks)
        a.record()
        for i in range(args.steps):
            dsa.gather_rows(rows, phys[i % n_sets], rb, out=out, dev_err=err)
        b.record()
        torch.cuda.synchronize()
        barrier(ranks)
    if dsa.check_device_error(err):
        raise SystemExit(f"device error word set: {int(err.item()):#x}")
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, dev)
    if ranks.rank != 0:
        return None
    moved = 2 * T * k * rb + T * k * 4
    roofline = hbm_roofline("dsa::gather_rows_kernel", moved, ms, read_peaks(),
                            traffic=profiled_traffic("gather_rows_kernel_gather64x2048.md", GATHER_SOURCES))
    roofline["timing"] = "K launches back to back between two CUDA events on the launching stream"
    return {
        "metric": "gathered KV rows/s (the consumer's read of the selected rows)",
        "value": whole_job_rate(T * k, world, ms / 1e3), "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8", "data": "synthetic",
        "config": {"workload": GATHER_DESC, "l2": "inputs larger than L2 (1.38 GB of rows, 4 rotating id sets)",
                   "parallelism": f"one replica per GPU x{world}" if world > 1 else "1 GPU"},
        "roofline": roofline,
        "gpu_launches": args.steps, "clocks": clocks.summary(),
    }


def run_named(args, name: str, ranks: Ranks, with_cpu: bool):
    if name == "stack61":
        return run_stack(args, ranks, with_cpu)
    if name == "gather64x2048":
        return run_gather(args, ranks, with_cpu)
    return run_layer(args, name, ranks, with_cpu)


# --------------------------------------------------------------------- oracle

def oracle_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    import ctypes

    try:
        return int(ctypes.CDLL("libgomp.so.1").omp_get_max_threads())
    except (OSError, AttributeError):
        return os.cpu_count() or 1


def oracle_state(hb, kcache="fp8"):
    import oracle

    cache = oracle.new_cache(hb.num_blocks, kcache)
    oracle.k_quant_write(hb.ctx_k, hb.ctx_slots, cache)  # the cache state before the step
    return oracle, cache


def oracle_step(ora, hb, cache, rows):
    """The whole path on the oracle for the given query rows."""
    ora.k_quant_write(hb.k_new, hb.slot_mapping, cache)
    ora.schedule(1, True, 4)
    topk = ora.indexer(hb, cache, rows=rows)
    ora.convert(topk, hb.req_id_per_token[rows], hb.block_table)
    return int((hb.positions[rows] + 1).sum())


def cpu_baseline(hb, budget_s: float, kcache: str = "fp8"):
    ora, cache = oracle_state(hb, kcache)
    T = hb.num_tokens
    # size the sample: grow the row count until one pass takes about the budget
    n_rows, dt, p = 1, 0.0, 0
    while True:
        rows = np.arange(n_rows, dtype=np.int64)
        t0 = time.perf_counter()
        p = oracle_step(ora, hb, cache, rows)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 2 or n_rows >= T:
            break
        n_rows = int(min(T, max(2 * n_rows, n_rows * budget_s / max(dt, 1e-3))))
    reps = 1
    if n_rows >= T and dt < budget_s / 4:  # the whole step is quick: time several passes of it
        reps = int(min(1000, max(2, budget_s / 2 / max(dt, 1e-4))))
        t0 = time.perf_counter()
        for _ in range(reps):
            p = oracle_step(ora, hb, cache, rows)
        dt = (time.perf_counter() - t0) / reps
    return {"value": p / dt, "unit": "pairs/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{n_rows} of {T} query rows of the same step ({p} pairs; K write of all {T} new tokens, "
                      f"fp64 scores, full-sort top-k, conversion), {dt:.2f} s per pass, {reps} pass(es), "
                      f"OpenMP over rows"}


def run_reference(args, ranks: Ranks):
    """The oracle on the host cores, on this arm's workload, metric and config:
    each step is a bounded sample of the workload's query rows."""
    if ranks.rank != 0:
        return None
    name = args.workload
    hb = host_workload(name)
    ora, cache = oracle_state(hb, args.kcache)
    T = hb.num_tokens
    t0 = time.perf_counter()
    oracle_step(ora, hb, cache, np.arange(1, dtype=np.int64))
    t_one = max(time.perf_counter() - t0, 1e-4)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    n_rows = int(max(1, min(T, per_step / t_one)))
    rows = np.arange(n_rows, dtype=np.int64)
    for _ in range(args.warmup):
        oracle_step(ora, hb, cache, rows)
    t0 = time.perf_counter()
    p = 0
    for _ in range(args.steps):
        p += oracle_step(ora, hb, cache, rows)
    dt = time.perf_counter() - t0
    value = p / dt
    sample = (f"{n_rows} of {T} query rows per step of one F layer of the stack" if name == "stack61" else
              f"{n_rows} of {T} query rows per step")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "pairs/s",
        "n_gpus": ranks.world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded normals, bf16-rounded)",
        "config": workload_config(name, hb, args, ranks.world),
        "cpu_baseline": {"value": value, "unit": "pairs/s", "cores": oracle_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "pairs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# --------------------------------------------------------------------- dry run

def run_dry(args, ranks: Ranks):
    """The multi-rank launch and timing without a GPU: every rank times its own
    CPU task (rank r sleeps (r + 1) ms per step, so the ranks differ), the
    timed region is bracketed by barriers, and rank 0 reports the slowest
    rank's time and the units of every rank."""
    import os as _os

    def work():
        time.sleep(1e-3 * (ranks.rank + 1))

    for _ in range(args.warmup):
        work()
    barrier(ranks)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        work()
    mine = (time.perf_counter() - t0) / args.steps
    barrier(ranks)
    slowest = max_over_ranks(mine, "cpu")
    per_rank = gather_over_ranks(mine, "cpu")
    rank_ids = gather_over_ranks(float(_os.environ.get("RANK", "0")), "cpu")
    if ranks.rank != 0:
        return None
    units = 1000.0
    return {"metric": "dry run: units/s", "value": whole_job_rate(units, ranks.world, slowest), "unit": "units/s",
            "n_gpus": ranks.world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": slowest * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "none", "data": "none",
            "dry_run": True, "ranks": [int(r) for r in rank_ids], "rank_ms_per_step": [x * 1e3 for x in per_rank],
            "config": {"workload": "dry run", "parallelism": f"one replica per rank x{ranks.world}"}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=["stack61", "decode32", "decode8x128k", "prefill4x8k", "prefill512", "gather64x2048"])
    ap.add_argument("--sub-workloads", default=DEFAULT_SUB_WORKLOADS,
                    help="single-layer workloads measured after stack61 and reported under `workloads` "
                         "('' for none)")
    ap.add_argument("--replicas", type=int, default=0)
    ap.add_argument("--stack-layers", type=int, default=STACK_LAYERS,
                    help="layers of the stack61 workload (fewer only to profile a small case)")
    ap.add_argument("--clock-window", type=float, default=1.0, help="seconds of untimed steps while sampling clocks")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kcache", choices=["fp8", "fp4"], default="fp8",
                    help="indexer K cache: FP8 (132 B/slot) or FP4 E2M1 (68 B/slot)")
    ap.add_argument("--rope", action="store_true",
                    help="q and new K arrive un-rotated; the layer prologue applies RoPE before quantising")
    ap.add_argument("--sm-split", choices=["auto", "off"], default="auto",
                    help="stack61: score each F layer's decode rows on a share of the SMs beside its prefill rows "
                         "(auto, from the step's work) or one after the other on the whole GPU (off)")
    ap.add_argument("--dry-run", action="store_true",
                    help="no GPU: exercise the rank launcher and the slowest-rank timing on CPU (gloo)")
    argv = sys.argv[1:] if argv is None else argv
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference" and "WORLD_SIZE" in os.environ:
        # torch.distributed.run sets one OpenMP thread per rank; rank 0 alone
        # runs the oracle here, on all host cores
        os.environ["OMP_NUM_THREADS"] = str(os.cpu_count() or 1)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: start this script on --gpus ranks
        return subprocess.call(relaunch_cmd(args.gpus, argv))
    ranks = init_ranks(args)
    try:
        if args.dry_run:
            line = run_dry(args, ranks)
        elif args.impl == "reference":
            line = run_reference(args, ranks)
        else:
            line = run_named(args, args.workload, ranks, with_cpu=True)
            subs = [s for s in args.sub_workloads.split(",") if s] if args.workload == "stack61" else []
            if subs:
                res = {}
                for name in subs:
                    sub = run_named(args, name, ranks, with_cpu=False)
                    if sub is not None:
                        res[name] = compact(sub)
                if line is not None:
                    line["workloads"] = res
        if line is not None:
            print(json.dumps(line), flush=True)
    finally:
        import torch.distributed as dist

        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

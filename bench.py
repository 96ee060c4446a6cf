"""Throughput of the Titans/ATLAS memory-layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one forward of the whole memory layer (every chunk of every unit)
over one batch of synthetic inputs that already sit in HBM.  The default
workload is the largest single-GPU one by work, ATLAS with Muon (MLP
128 -> 512 -> 128, B=2, H=16, T=16384, C=64, Omega window 8, five
Newton-Schulz iterations per token and weight matrix); ``--workload NAME``
times any other.  One JSON line goes to stdout on rank 0.

Under torchrun (N > 1) every rank runs its own batch of the same shape on its
own GPU (the (batch, head) units are independent: no collective on the data
path); the timed region is bracketed by barriers and the slowest rank's time
is reported.  ``--impl reference`` times the fp64 CPU oracle on a bounded
sample of the same workload on the host's cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from harness import PROLOGUES, WORKLOADS, make_inputs, make_prologue_inputs  # noqa: E402

METRIC = "memory-layer tokens/s (B*H*T/s) on 1 GB300"
DEFAULT_WORKLOAD = "atlas_muon"

# fp32 FMA peak of the whole GPU for paths bound by plain ALU issue: 152 SMs
# x 128 fp32 lanes x 2 FLOP per FMA x the 2070 MHz maximum SM clock
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


# --------------------------------------------------------------- accounting
def flops_per_chunk(w) -> float:
    """Algorithmic FLOPs of one chunk of one unit: the dual form without
    Newton-Schulz, or the per-token orthogonalisation path with it."""
    C, Kw = w.C, w.C + w.c - 1
    F, dv, h = w.feat_dim, w.d_v, w.hidden
    feat = 0.0
    if w.proj_dim:
        feat = 2.0 * w.poly_dim * w.proj_dim * (C + C)     # keys and queries of the chunk
    surprise = w.ns_iters > 0 and getattr(w, "ns_target", "momentum") == "surprise"
    if getattr(w, "update", "per_token") == "chunkwise":
        # one update per chunk: the forward/backward at W_bar, one summed
        # gradient product per matrix, Newton-Schulz once per matrix, and
        # every token's read-out through the memory
        mats = [(F, dv)] if w.depth == 1 else [(F, h), (h, dv)]
        fwd = 2.0 * Kw * F * dv if w.depth == 1 else 3 * 2.0 * Kw * F * h
        state = sum(2.0 * r * c * C for (r, c) in mats)
        read = C * sum(2.0 * r * c for (r, c) in mats)
        ns = sum(w.ns_iters * (2.0 * min(r, c) ** 2 * max(r, c) * 2 + 2.0 * min(r, c) ** 3) for (r, c) in mats)
        return feat + fwd + state + read + ns
    if w.ns_iters == 0 or surprise:
        extra = 0.0
        if surprise:
            # c x c Newton-Schulz cores per token and matrix, Gram bands of
            # the window factors, banded coefficient mixes in the read-out
            # and the chunk-end state (the rest is the plain dual form)
            mats = [(F, dv)] if w.depth == 1 else [(F, h), (h, dv)]
            band = 2 * w.c - 1
            for (r, c) in mats:
                extra += 2.0 * Kw * band * (r + c)                          # Gram bands
                extra += C * w.ns_iters * 5 * 2.0 * w.c ** 3                # cores
                extra += C * 2.0 * Kw * band + 2 * 2.0 * Kw * band * c      # read-out mix, M_e R
        if w.depth == 1:
            fwd = 2.0 * Kw * F * dv
            read = 2.0 * C * 2 * F * dv + 2.0 * C * Kw * F + 2.0 * C * Kw * dv
            state = 2 * 2.0 * F * dv * Kw
        else:
            fwd = 3 * 2.0 * Kw * F * h
            read = (2.0 * C * 2 * F * h + 2.0 * C * Kw * F + 2.0 * C * Kw * h
                    + 2.0 * C * 2 * h * dv + 2.0 * C * Kw * h + 2.0 * C * Kw * dv)
            state = 2 * 2 * 2.0 * F * h * Kw
        return feat + fwd + read + state + extra
    # Newton-Schulz: per token and matrix, S_t from the window factors, k
    # quintic steps on the short side, decay scan and read-out.
    mats = [(F, dv)] if w.depth == 1 else [(F, h), (h, dv)]
    fwd = 2.0 * Kw * F * dv if w.depth == 1 else 3 * 2.0 * Kw * F * h
    per_tok = 0.0
    for (r, c) in mats:
        m, n = min(r, c), max(r, c)
        per_tok += 2.0 * m * n * Kw                                   # S_t
        per_tok += w.ns_iters * (2.0 * m * m * n * 2 + 2.0 * m ** 3)  # NS
        per_tok += 2.0 * m * n * 2                                    # scan + read-out
    return feat + fwd + C * per_tok


def algorithmic_flops_per_token(w) -> float:
    """Algorithmic FLOPs per token by the hot-path scope table's accounting:
    the work the method must do in the dual form, with no per-token state
    in HBM.

    * Newton-Schulz on the momentum (per token): the quintic steps only,
      sum over matrices of k (2 m^2 n * 2 + 2 m^3) on the short side m,
      plus phi P (2 * monomials * proj per key and per query) when the
      features are projected;
    * depth 2 without it: forward and backward at W_bar (3 * 2 F h), the
      chunk-end state products (W and S, both matrices) and the dual-form
      read-out through W_bar and S_bar (both matrices);
    * depth 1 without it: phi(k) W_bar, the S and W updates, phi(q) W_bar
      and S_bar, and the intra-chunk Gram phi(q) X^T over the window rows.

    The chunk-wise rule and Newton-Schulz on the surprise keep the per-chunk
    counts of flops_per_chunk."""
    surprise = w.ns_iters > 0 and getattr(w, "ns_target", "momentum") == "surprise"
    if getattr(w, "update", "per_token") == "chunkwise" or surprise:
        return flops_per_chunk(w) / w.C
    F, dv, h = w.feat_dim, w.d_v, w.hidden
    mats = [(F, dv)] if w.depth == 1 else [(F, h), (h, dv)]
    feat = 2.0 * 2.0 * w.poly_dim * w.proj_dim if w.proj_dim else 0.0
    if w.ns_iters:
        ns = sum(w.ns_iters * (2.0 * min(r, c) ** 2 * max(r, c) * 2 + 2.0 * min(r, c) ** 3) for r, c in mats)
        return ns + feat
    if w.depth == 2:
        fwd = 3 * 2.0 * F * h
        state = 2 * sum(2.0 * r * c for r, c in mats)
        read = 2 * sum(2.0 * r * c for r, c in mats)
        return fwd + state + read + feat
    Kw = w.C + w.c - 1
    return 2.0 * F * dv + 2 * 2.0 * F * dv + 2 * 2.0 * F * dv + 2.0 * F * Kw + feat


def roofline_bound(w, flops, nbytes, peaks) -> str:
    """'alu' on the fp32 SIMT paths; else 'tensor' when the step's
    arithmetic intensity is above the ridge of the measured bf16 tensor
    peak over the measured HBM bandwidth, 'hbm' below it."""
    if path_dtype(w) == "f32":
        return "alu"
    ridge = peaks.get("bf16_tflops_sustained", 1700.0) * 1e12 / (peaks.get("hbm_gbs", 6800.0) * 1e9)
    return "tensor" if flops / max(nbytes, 1.0) >= ridge else "hbm"


def path_dtype(w) -> str:
    """Arithmetic type of the path a workload runs on: the fused MLP kernel
    multiplies bf16 operands (fp32 accumulation and state); the tensor-core
    Newton-Schulz path and the tensor-core depth-1 (polynomial-feature)
    kernel multiply split bf16 pairs (three products, about fp32 accuracy);
    everything else is fp32."""
    fused = (w.depth == 2 and w.ns_iters == 0 and w.c == 1 and w.p == 1 and w.proj_dim == 0 and w.d_k == 64
             and w.d_v == 64 and w.hidden == 256 and w.C == 64)
    if fused:
        return "bf16"
    if w.ns_iters and getattr(w, "ns_target", "momentum") == "momentum" and w.depth == 2:
        return "bf16x3"
    depth1_tc = (w.depth == 1 and w.ns_iters == 0 and w.update == "per_token"
                 and w.qkv_dtype == "bf16" and w.proj_dim == 0 and w.p in (1, 2) and w.d_k % 8 == 0
                 and w.d_k <= 32 and w.d_v % 8 == 0 and w.d_v <= 64 and w.C <= 64 and w.C + w.c - 1 <= 80
                 and w.feat_dim <= 768)
    if depth1_tc:
        return "bf16x3"
    surprise_tc = (w.depth == 2 and w.ns_iters > 0 and getattr(w, "ns_target", "momentum") == "surprise"
                   and w.feat_dim % 16 == 0 and w.feat_dim <= 128 and w.feat_dim == w.d_v and w.hidden % 64 == 0
                   and w.d_v % 32 == 0 and w.C <= 64 and w.C + w.c - 1 <= 80 and w.c <= 16)
    if surprise_tc:   # the read-out's and the chunk-end state's products on the tensor cores
        return "bf16x3"
    return "f32"


def bytes_per_step(w) -> float:
    es = 2 if w.qkv_dtype == "bf16" else 4
    per_tok = es * (2 * w.d_k + w.d_v) + 4 * 3 + (4 if w.use_gamma else 0) + 4 * w.d_v
    state = sum(r * c for r, c in w.matrix_shapes()) * 4 * 4   # W0, S0 in; W, S out
    return w.tokens * per_tok + w.units * state


# sources of the kernel whose DRAM counters profiles/traffic.json records:
# the record is used only while these files are unchanged
TRAFFIC_SOURCES = {"titans_mlp": ("k_mlp_tc.cu", "tc.cuh", "atlas_common.cuh"),
                   "atlas_muon": ("k_ns_tc.cu", "tc.cuh", "atlas_common.cuh"),
                   "atlas_poly_c4": ("k_dual1_tc.cu", "tc.cuh", "atlas_common.cuh")}


def source_digest(files=None) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "test_learned_neural_gb300", "csrc")
    for fn in sorted(files if files is not None else os.listdir(csrc)):
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of the GPU's clocks and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,pci.bus_id")

    def __init__(self, bus_id=None):
        self.bus_id = (bus_id or "").lower()
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = self.rows
        if self.bus_id:
            mine = [r for r in rows if r[8].lower().endswith(self.bus_id[-7:])]
            rows = mine or rows
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------- CPU oracle
_ORACLE_INPUTS = {}


def _oracle_job(args):
    """Worker: oracle forward of one sample; returns its compute seconds
    (input generation is cached per process and not timed)."""
    name, units, T = args
    import oracle
    w = WORKLOADS[name]
    if name not in _ORACLE_INPUTS:
        _ORACLE_INPUTS[name] = make_inputs(w)
    t0 = time.perf_counter()
    oracle.forward(w, _ORACLE_INPUTS[name], units=units, T=T)
    return time.perf_counter() - t0


# fp64 oracle cost per token and unit on one host core, measured (x86 and
# Arm hosts within a factor of two); sizes the bounded samples below
ORACLE_S_PER_TOKEN = {"atlas_muon": 0.019, "atlas_muon_surprise": 0.019, "atlas_muon_chunkwise": 0.0005,
                      "atlas_long": 0.0034}


def oracle_sample(w, budget_s=None):
    """Bounded sample of the workload for the CPU oracle: (units, tokens)
    from the start of the sequence.  Without a budget: up to 8 units (one
    process each) x 2C tokens on the Newton-Schulz workloads, else x 4096;
    with one, the token count is cut so that one unit's pass takes about
    budget_s seconds (at least 8 tokens)."""
    cores = os.cpu_count() or 1
    units = list(range(min(8, w.units, cores)))
    T = 2 * w.C if w.ns_iters else min(w.T, 4096)
    if budget_s is not None:
        per_tok = ORACLE_S_PER_TOKEN.get(w.name, 0.0006)
        T = max(8, min(T, int(budget_s / per_tok)))
    return units, T


def time_oracle(name, reps=1, budget_s=None):
    """Time the oracle on its sample, one spawned process per unit (one BLAS
    thread each, all in parallel).  A rep takes as long as its slowest unit.
    Returns (tokens/s, cores used, description, per-rep seconds)."""
    import multiprocessing as mp
    w = WORKLOADS[name]
    units, T = oracle_sample(w, budget_s)
    cores = min(len(units), os.cpu_count() or 1)
    env_keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in env_keep:
        os.environ[k] = "1"
    ctx = mp.get_context("spawn")
    times = []
    try:
        with ctx.Pool(cores) as pool:
            pool.map(_oracle_job, [(name, [u], w.C) for u in units])      # inputs + imports, untimed
            for _ in range(reps):
                per_unit = pool.map(_oracle_job, [(name, [u], T) for u in units])
                waves = -(-len(units) // cores)
                times.append(max(per_unit) * waves)
    finally:
        for k, v in env_keep.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    tokens = len(units) * T
    desc = f"{len(units)} units x first {T} tokens of {w.name} (fp64 numpy, one process per unit, {cores} cores)"
    return tokens / statistics.median(times), cores, desc, times


# -------------------------------------------------------------- reference
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    # warm-up: time_oracle runs one untimed pass per worker before the timed
    # reps.  Each step's sample is cut so that all K steps take about a
    # minute of oracle work in total.
    budget = 60.0 / max(args.steps, 1)
    tps, cores, desc, times = time_oracle(args.workload, reps=args.steps, budget_s=budget)
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, harness recipe)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "sample": desc},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- multi-rank
def replica_workload(w, rank: int):
    """Every rank runs its own batch of the same shape (weak scaling): the
    (batch, head) units are independent, so no data crosses ranks."""
    return w.scaled(seed=w.seed + 1000 * rank) if rank else w


def max_over_ranks(x: float, device=None) -> float:
    """Slowest rank's value (the timed region ends when the last rank ends)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, steps: int, slowest_seconds: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world * steps / slowest_seconds


# ------------------------------------------------------------------- ours
def run_ours(args):
    import torch
    import torch.distributed as dist

    import test_learned_neural_gb300 as tln
    from test_learned_neural_gb300.runner import Memory, tensors_from_numpy

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = WORKLOADS[args.workload]
    if args.geometry:
        w = w.scaled(**args.geometry)
    w = replica_workload(w, rank)
    inp = make_inputs(w)
    t = tensors_from_numpy(inp, device=dev)
    mem = Memory(w)
    out = mem.alloc_outputs(w.B, w.H, w.T, dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)   # > L2 (129 MB)
    stream = torch.cuda.current_stream()

    def step():
        mem.forward(t, out=out)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    mem.status()
    launches = tln.atlas_mem_last_launches(mem.h)

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    clocks = ClockSampler(f"{bus:02x}:00" if isinstance(bus, int) else None)
    clocks.start()
    time.sleep(0.3)   # nvidia-smi needs a moment before its first sample
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()                    # evict L2 between timed steps
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    mem.status()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_s = max_over_ranks(sum(step_ms) / 1e3, dev)
    value = job_throughput(w.tokens, world, args.steps, total_s)

    # end to end through the host-buffer entry point (pinned host memory)
    e2e = None
    if not args.no_e2e:
        th = tensors_from_numpy(inp, device="cpu", pin=True)
        oh = mem.alloc_outputs(w.B, w.H, w.T, "cpu")
        for key, val in list(oh.items()):
            oh[key] = [x.pin_memory() for x in val] if isinstance(val, list) else val.pin_memory()
        h2d = sum(x.numel() * x.element_size() for k, x in th.items() if k not in ("W0", "S0") and x is not None)
        h2d += sum(x.numel() * x.element_size() for x in th["W0"] + th["S0"])
        d2h = oh["y"].numel() * 4 + sum(x.numel() * 4 for x in oh["W"] + oh["S"])
        mem.forward(th, out=oh, host=True)
        reps = max(3, min(args.steps, 10))
        # clocks during these steps too: they follow the timed region without
        # a pause, so a GPU that heats up shows it here first
        clocks_e2e = ClockSampler(f"{bus:02x}:00" if isinstance(bus, int) else None)
        clocks_e2e.start()
        time.sleep(0.3)
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(reps):
            mem.forward(th, out=oh, host=True)
        e2e_s = max_over_ranks((time.perf_counter() - t0) / reps, dev)
        e2e = {"value": job_throughput(w.tokens, world, 1, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "clocks": clocks_e2e.stop()}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, src = measured_peaks()
    fl = algorithmic_flops_per_token(w) * w.tokens
    nbytes = bytes_per_step(w)
    step_s = statistics.mean(step_ms) / 1e3
    bound = roofline_bound(w, fl, nbytes, peaks)
    # a step of a second or more runs under the power cap: sustained peak
    sustained = step_s >= 0.1
    if bound == "alu":
        achieved, peak, runit = fl / step_s / 1e12, FP32_ALU_TFLOPS, "TFLOP/s"
        peak_src = "fp32 FMA issue: 152 SMs x 128 lanes x 2 x 2070 MHz (derived)"
    elif bound == "hbm":
        achieved, peak, runit = nbytes / step_s / 1e9, peaks.get("hbm_gbs", 6800.0), "GB/s"
        peak_src = f"hbm_gbs ({src})"
    else:
        key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
        achieved, peak, runit = fl / step_s / 1e12, peaks.get(key, 1700.0 if sustained else 1900.0), "TFLOP/s"
        peak_src = f"{key} ({src})"
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath) and not args.geometry:
        rec = json.load(open(tpath)).get(w.name)
        if rec and rec.get("source_digest") == source_digest(TRAFFIC_SOURCES.get(w.name)):
            traffic = rec.get("dram_bytes_per_step")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": path_dtype(w),
        "data": "synthetic (seeded, harness recipe), inputs resident in HBM",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "depth": w.depth, "d": w.d_v,
                   "hidden": w.hidden, "C": w.C, "c": w.c, "p": w.p, "ns_iters": w.ns_iters,
                   "l2": "flushed between timed steps (256 MB write)", "parallelism": f"replicas x{world}",
                   **({"geometry": "reduced (--geometry), profiling case"} if args.geometry else {})},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": runit,
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                     "kernel": ("atlas::k_mlp_dual_tc (the step's only launch)" if launches == 1
                                else f"whole forward ({launches} launches per step)"),
                     "algorithmic_flops_per_token": algorithmic_flops_per_token(w),
                     "algorithmic_flops_per_step": fl, "algorithmic_bytes_per_step": nbytes},
        "gpu_launches": launches * args.steps,
        "e2e": e2e,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline and world == 1:
        tps, cores, desc, _ = time_oracle(w.name, reps=1)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ------------------------------------------- stage in front of the memory
PROLOGUE_METRIC = "stage tokens/s (B*T/s, x -> q, k, v, gates) on 1 GB300"


def prologue_bytes_per_step(p) -> float:
    """Algorithmic bytes of one call: x and W_in read, taps and biases read,
    q, k, v and the gates written (the fp32 projection in between is the
    implementation's, not the method's)."""
    es = 2 if p.qkv_dtype == "bf16" else 4
    return (p.tokens * p.D * es + p.D * p.N * es + 4 * (p.Nc * p.conv + p.G * p.H)
            + p.tokens * p.H * (es * (2 * p.d_k + p.d_v) + 4 * p.G))


def time_prologue_oracle(p, T=1024):
    """The oracle on the first T tokens of batch row 0 (one process)."""
    import oracle
    inp = make_prologue_inputs(p.scaled(B=1))
    from harness import bf16_from_bits
    dec = (lambda a: bf16_from_bits(a).astype(np.float64)) if p.qkv_dtype == "bf16" else (lambda a: a.astype(np.float64))
    T = min(T, p.T)
    x, W = dec(inp["x"])[0, :T], dec(inp["W_in"])
    t0 = time.perf_counter()
    oracle.prologue_row(p, x, W, inp["conv_w"], inp["gate_b"])
    dt = time.perf_counter() - t0
    return T / dt, 1, f"batch row 0 x first {T} tokens of {p.name} (fp64 numpy, one process)"


def run_prologue(args):
    import torch
    from test_learned_neural_gb300.runner import Prologue, prologue_tensors_from_numpy

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    p = PROLOGUES[args.workload]
    if args.impl == "reference":
        tps, cores, desc = time_prologue_oracle(p)
        print(json.dumps({"impl": "reference", "metric": PROLOGUE_METRIC, "value": tps, "unit": "tokens/s",
                          "n_gpus": args.gpus, "steps": 1, "warmup": 0, "ms_per_step": 1e3 * p.tokens / tps,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic (seeded, harness recipe)", "config": {"workload": p.name},
                          "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                           "sample": desc},
                          "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    torch.cuda.set_device(0)
    inp = make_prologue_inputs(p)
    pro = Prologue(p)
    t = prologue_tensors_from_numpy(inp)
    out = pro.alloc_outputs(p.B, p.T, "cuda")
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 0)):
        pro.forward(t, out=out)
    torch.cuda.synchronize()
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        pro.forward(t, out=out)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_s = sum(step_ms) / 1e3
    peaks, src = measured_peaks()
    byt = prologue_bytes_per_step(p)
    achieved = byt / (statistics.mean(step_ms) / 1e3) / 1e9
    peak = peaks.get("hbm_gbs", 6800.0)
    line = {
        "metric": PROLOGUE_METRIC, "value": p.tokens * args.steps / total_s, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": p.qkv_dtype,
        "data": "synthetic (seeded, harness recipe), inputs resident in HBM",
        "config": {"workload": p.name, "B": p.B, "T": p.T, "D": p.D, "H": p.H, "d_k": p.d_k, "d_v": p.d_v,
                   "conv": p.conv, "l2": "flushed between timed steps (256 MB write)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "peak_source": f"hbm_gbs ({src})",
                     "kernel": "whole stage (k_proj_tc projection GEMM + k_prologue: 2 launches per step)",
                     "algorithmic_bytes_per_step": byt,
                     "algorithmic_flops_per_step": 2.0 * p.tokens * p.D * p.N},
        "gpu_launches": 2 * args.steps,
        "e2e": None,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline:
        tps, cores, desc = time_prologue_oracle(p)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    pro.status()
    pro.close()
    return 0


# measured ms per forward on one GB300, to size the default step count
APPROX_MS = {"atlas_muon": 1040, "atlas_long": 920, "atlas_muon_surprise": 122, "atlas_muon_chunkwise": 82,
             "atlas_poly_c4": 1.7, "atlas_poly_c16": 1.7}


def default_steps(name: str) -> int:
    """About 10 s of timed steps, between 10 and 100."""
    ms = APPROX_MS.get(name, 0.5)
    return int(max(10, min(100, 10000 // ms)))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about 10 s of timed work: 10 on the default workload)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS) + sorted(PROLOGUES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--geometry", default=None, metavar="B,H,T",
                    help="run the workload's method at a smaller batch x heads x length (for profiler captures; "
                         "the JSON line's config names the geometry and is not a headline number)")
    args = ap.parse_args(argv)
    if args.geometry is not None:
        b, h, t = (int(v) for v in args.geometry.split(","))
        args.geometry = {"B": b, "H": h, "T": t}
    if args.steps is None:
        args.steps = default_steps(args.workload)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.workload in PROLOGUES:
        if args.geometry:
            ap.error("--geometry applies to the memory workloads only")
        return run_prologue(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark: allowed-pair TFLOP/s of the block-sparse masked attention forward pass.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--pass fwd|bwd|decode] [--decode-workload NAME]

--pass fwd (default) is the headline described below.  --pass bwd times one spattn_bwd
over the whole batch (10 d pairs flops per step, against the bf16 peak); --pass decode
times one generation step (ring-buffer append + decode, spattn_decode_append) and reports GB/s of cached K/V
read per step against the measured HBM bandwidth; its timed steps are captured once into a
CUDA graph and replayed (each step still appends, decodes at its own position and merges).

One step = one spattn_fwd call over the whole batch (every (batch, head)) of the
workload, inputs already resident in HBM.  Warm-up: at least W steps, and for steps
shorter than 0.2 ms at least 0.2 s of back-to-back steps before the timed region (a kernel
of tens of microseconds would otherwise be timed while the GPU ramps up from the idle of
the host-side legs).  value = 4 d B H pairs_per_head / t_step
(2d flops for q.k and 2d for the weighted values per allowed pair: the glossary's
O(E (d_k + d_v)) cost, "Sparse attention", section "When the cost is linear").
Under torchrun each rank runs its own copy of the workload on its GPU (heads are
independent; there is no collective on the data path), and value sums over ranks.

At N = 1 the default run also times, after the headline, the other forward workloads
(the 128K / 8K pair that shows density-proportional cost, the 16K long-document mask,
the dilated and BigBird masks, and the short 2048- and 512-token configs on the HBM
roofline) on device-drawn seeded inputs, each with its own clock record, under the
line's "secondary" key; --no-secondary skips them.

--impl reference times the fp64 CPU oracle (the reference arm of this method) on a
bounded sample of the same workload, on the host cores: query rows of one head for the
forward, dQ of sampled rows for --pass bwd, sampled (batch, kv head) groups for --pass
decode, each in its pass's metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import spattn_workloads as W  # noqa: E402

METRIC = "allowed-pair TFLOP/s (4·d·pairs/s) & % of B300 bf16 tensor peak, 1 GPU"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "t32k_w4096"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# DRAM bytes (read + write) per launch of the tensor-core forward kernel on the
# 32K / W=4096 workload, from the ncu capture summarised in
# the forward kernel's profile summary (captured with H=8, 250.7 MB, scaled by 32/8 heads),
# valid only for the kernel source with this hash; any other source reports null.
TRAFFIC = {"kernel_sha": "c098de61ca126cd1", "bytes_per_launch": 999.9e6, "workload": "t32k_w4096"}
# The same for the backward's dominant kernel (bwd_dkdv_tc, H=4 capture x 8) and the
# decode kernel (B=8 capture, x 4 for B=32), keyed by their source hashes.
BWD_TRAFFIC = {"kernel_sha": "a4acc78bd1403ef0", "bytes_per_launch": 1358.0e6,
               "workload": "t32k_w4096", "file": "bwd_tc.cu"}
DEC_TRAFFIC = {"kernel_sha": "01872e9be1b20281", "file": "decode.cu",
               "bytes_per_launch": {"decode_b8_w4096": 140.0e6, "decode_b32_w4096": 560.1e6}}


def kernel_sha(name: str = "fwd_tc.cu") -> str:
    p = os.path.join(ROOT, "sparse_masked_attention_plan_b300", "csrc", name)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def mask_desc(p):
    if p["causal"]:
        s = f"causal window={p['window'] or 'none'}"
    else:
        s = f"bidirectional radius={p['radius']}"
    if p["stride"]:
        s += f", stride={p['stride']} offset={p['offset']}"
    if len(p["global_pos"]):
        s += f", {len(p['global_pos'])} global tokens"
    if p.get("dilation", 1) > 1:
        s += f", dilation {p['dilation']}"
    if p.get("rand_block"):
        s += f", {len(p['rand_pairs'])} random blocks of {p['rand_block']}"
    return s


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(backend: str = "nccl"):
    """(world, rank, local_rank) from the torchrun environment; joins the process
    group when world > 1 (NCCL for the GPU arm, gloo for CPU-only use)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


L2_BYTES = 126e6  # B300 L2 cache


class StepTimer:
    """Per-step CUDA events on the launching stream.  When a step's inputs fit in L2
    (in_bytes <= L2), a 2 x L2 buffer is rewritten before every timed step, outside the
    events, so no step starts with its inputs already in L2; larger inputs evict
    themselves.  `l2` says which of the two applies."""

    def __init__(self, torch, dev, stream, steps, in_bytes, what):
        self.torch, self.stream, self.steps = torch, stream, steps
        self.flush = None
        if in_bytes <= L2_BYTES:
            self.flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.int32, device=dev)
            self.l2 = (f"L2 flushed before every timed step ({in_bytes / 1e6:.0f} MB of {what} "
                       f"fit in L2)")
        else:
            self.l2 = f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB of {what})"
        mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        self.t0, self.t1 = mk(), mk()

    def run(self, step):
        for s in range(self.steps):
            if self.flush is not None:
                with self.torch.cuda.stream(self.stream):
                    self.flush.fill_(s)
            self.t0[s].record(self.stream)
            step()
            self.t1[s].record(self.stream)

    def per_step_ms(self):
        return [a.elapsed_time(b) for a, b in zip(self.t0, self.t1)]


# Configurations whose forward is bound by HBM traffic and launch latency rather than the
# tensor cores (arithmetic intensity below the ridge point): the 512- and 2048-token
# shapes.  Their roofline is GB/s of algorithmic bytes against the measured HBM bandwidth.
HBM_BOUND = ("t512_w128_s0", "t512_w128_s64", "t512_full_causal", "t2048_w256_s0",
             "t2048_w256_s64")

SECONDARY = ["t128k_w4096_s1024", "t8k_full_causal", "t16k_r256_s16_g128", "t32k_w512_d2",
             "t4096_bigbird", "t2048_w256_s0", "t2048_w256_s64", "t512_w128_s0"]


def fwd_algo_bytes(B, H, T, d, elem=2):
    """Algorithmic bytes of one forward launch: Q, K, V read and O written (d elements
    each per token per head) plus the fp32 LSE."""
    return B * H * T * (4 * d * elem + 4)


def fwd_roofline(name, cfg, flops, ms, peaks):
    """(bound, achieved, peak, unit) of a forward step taking `ms`."""
    if name in HBM_BOUND:
        gbs = fwd_algo_bytes(cfg["B"], cfg["H"], cfg["T"], cfg["d"]) / (ms / 1e3) / 1e9
        return "hbm", gbs, peaks["hbm_gbs"], "GB/s"
    return "tensor", flops / (ms / 1e3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"


def time_secondary(torch, sp, names, steps, warmup, dev, stream):
    """Time one forward step of each named workload (whole batch, inputs resident, the
    same per-step CUDA events and L2 rule as the headline), each with its own clocks.
    Inputs are seeded N(0,1) bf16 drawn on the device (these lines are throughput only;
    the parity tests use the host-drawn inputs)."""
    peaks, _ = load_peaks()
    out = {}
    for name in names:
        cfg = W.WORKLOADS[name]
        p = W.mask_params(name)
        B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
        g = torch.Generator(device=dev).manual_seed(1)
        with torch.cuda.stream(stream):
            q, k, v = (torch.randn(B, H, T, d, generator=g, device=dev, dtype=torch.float32)
                       .to(torch.bfloat16) for _ in range(3))
            o = torch.empty_like(q)
            lse = torch.empty(B, H, T, dtype=torch.float32, device=dev)
        plan = sp.Plan(T, d, **p, stream=stream)
        info = plan.info()
        flops = 4.0 * d * B * H * info["pairs_per_head"]
        scale = 1.0 / math.sqrt(d)

        def step():
            sp.fwd(plan, q, k, v, scale, out=o, lse=lse, stream=stream)

        warm_up(torch, stream, step, warmup)
        timer = StepTimer(torch, dev, stream, steps, 3 * q.numel() * q.element_size(), "Q/K/V")
        with ClockSampler(dev.index or 0) as clk:
            torch.cuda.synchronize(dev)
            timer.run(step)
            torch.cuda.synchronize(dev)
        plan.check_device(stream)
        ms = statistics.mean(timer.per_step_ms())
        bound, achieved, peak, unit = fwd_roofline(name, cfg, flops, ms, peaks)
        packing = plan.columns().size > 0 or len(p["global_pos"]) > 0
        out[name] = {"B": B, "H": H, "T": T, "d": d, "mask": mask_desc(p),
                     "pairs_per_head": info["pairs_per_head"], "ms_per_step": ms,
                     "tflops": flops / (ms / 1e3) / 1e12,
                     "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak,
                     "step": "k_pack + fwd_tc" if packing else "fwd_tc",
                     "l2": timer.l2, "clocks": clk.summary()}
        plan.close()
        del q, k, v, o, lse
        torch.cuda.empty_cache()
    a, b = out.get("t128k_w4096_s1024"), out.get("t8k_full_causal")
    if a and b:
        pr = (a["pairs_per_head"] * a["B"] * a["H"]) / (b["pairs_per_head"] * b["B"] * b["H"])
        ma, mb = a["clocks"]["sm_mhz"], b["clocks"]["sm_mhz"]
        out["density"] = {
            "pairs_ratio_128k_over_8k": pr,
            "time_ratio": a["ms_per_step"] / b["ms_per_step"],
            "cycles_ratio": (a["ms_per_step"] * ma) / (b["ms_per_step"] * mb) if ma and mb else None,
            "note": "cycles_ratio = (time x median SM MHz) of the 128K step over the 8K step"}
    return out


MIN_WARM_S = 0.2  # warm-up wall time before the timed region of a short step
SHORT_STEP_S = 2e-4  # steps shorter than this get MIN_WARM_S of warm-up


def warm_up(torch, stream, step, steps):
    """Run `steps` untimed steps; while the steps are short (< SHORT_STEP_S each) go on
    until MIN_WARM_S of wall time has passed, so a kernel of tens of microseconds is not
    timed while the GPU is still ramping up from idle (after the host-side legs of the
    run: measured, 30 ms of such steps were not enough, 0.2 s was).  Longer steps stop at
    `steps`: their own warm-up already brings the clocks up, and more of it would only
    heat the chip into its power limit."""
    t0 = time.perf_counter()
    n = 0
    while True:
        step()
        n += 1
        if n % 8 == 0 or n >= steps:
            stream.synchronize()
        if n < steps:
            continue
        el = time.perf_counter() - t0
        if el >= MIN_WARM_S or el / n >= SHORT_STEP_S:
            break
    stream.synchronize()
    return n


def max_over_ranks(x: float, world: int) -> float:
    """The maximum of x over all ranks (x itself when world == 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(total_ms: float, steps: int, flops_per_step_per_rank: float, world: int):
    """(ms_per_step, TFLOP/s) of the whole job: the slowest rank's time, every rank's work."""
    ms = max_over_ranks(total_ms, world) / steps
    return ms, world * flops_per_step_per_rank / (ms / 1e3) / 1e12


# ----------------------------------------------------------------- CPU oracle arm

def oracle_sample_rate(cfg, p, Q, K, V, budget_s: float, seed: int = 0):
    """Time the oracle (as it stands) on seeded sampled query rows of head (0, 0).

    Returns (pairs per second, pairs processed, rows, seconds, threads)."""
    import oracle
    oracle.build()
    T, d = cfg["T"], cfg["d"]
    m = oracle.Mask.from_params(T, p)
    q, k, v = (oracle.bf16_bits(x[0, 0]) for x in (Q, K, V))
    scale = 1.0 / math.sqrt(d)
    # calibrate on growing row counts, then size the sample to the budget
    n, dt = 32, 0.0
    while n < T:
        rows = W.sample_rows(T, n, seed)
        t0 = time.perf_counter()
        oracle.attention(m, q, k, v, scale, rows)
        dt = time.perf_counter() - t0
        if dt > 0.25 * budget_s / 8 or dt > 0.5:
            break
        n *= 4
    n = int(min(T, max(32, n * budget_s / max(dt, 1e-3))))
    rows = W.sample_rows(T, n, seed + 1)
    pairs = sum(len(m.row_set(int(r))) for r in rows)
    t0 = time.perf_counter()
    oracle.attention(m, q, k, v, scale, rows)
    secs = time.perf_counter() - t0
    return pairs / secs, pairs, len(rows), secs, oracle.num_threads()


def run_reference(args, cfg, p):
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return 0
    import torch
    import oracle
    oracle.build()
    B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
    g = torch.Generator().manual_seed(0)
    # one head's inputs are all the oracle sample touches
    Q, K, V = (torch.randn(1, 1, T, d, generator=g).to(torch.bfloat16) for _ in range(3))
    m = oracle.Mask.from_params(T, p)
    q, k, v = (oracle.bf16_bits(x[0, 0]) for x in (Q, K, V))
    scale = 1.0 / math.sqrt(d)
    step_budget = 2.0
    rows = W.sample_rows(T, 32, 11)
    t0 = time.perf_counter()
    oracle.attention(m, q, k, v, scale, rows)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(T, max(32, 32 * step_budget / dt)))
    samples = [W.sample_rows(T, n, 100 + s) for s in range(args.warmup + args.steps)]
    pairs = [sum(len(m.row_set(int(r))) for r in rs) for rs in samples]
    for s in range(args.warmup):
        oracle.attention(m, q, k, v, scale, samples[s])
    t0 = time.perf_counter()
    for s in range(args.warmup, args.warmup + args.steps):
        oracle.attention(m, q, k, v, scale, samples[s])
    secs = time.perf_counter() - t0
    done = sum(pairs[args.warmup:])
    value = 4 * d * done / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "H": H, "T": T, "d": d,
                   "mask": mask_desc(p),
                   "step": f"{n} seeded query rows of one head per step (bounded sample)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{args.steps} steps x {n} rows of head (0,0), "
                                   f"{done} allowed pairs"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_reference_bwd(args, cfg, p):
    """The backward's reference arm: the oracle's dQ of seeded sampled rows of one head
    (each row's dQ needs only its own allowed set), bounded per step.  It is credited
    with the full backward's 10 d flops per pair although it computes only dQ, so the
    arm is if anything overstated."""
    world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import torch
    import oracle
    oracle.build()
    B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
    g = torch.Generator().manual_seed(0)
    Q, K, V, dO = (torch.randn(T, d, generator=g).to(torch.bfloat16) for _ in range(4))
    m = oracle.Mask.from_params(T, p)
    q, k, v, do = (oracle.bf16_bits(x) for x in (Q, K, V, dO))
    scale = 1.0 / math.sqrt(d)
    rows = W.sample_rows(T, 16, 11)
    t0 = time.perf_counter()
    oracle.attention_bwd_dq(m, q, k, v, do, scale, rows)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(T, max(16, 16 * 2.0 / dt)))
    samples = [W.sample_rows(T, n, 100 + s) for s in range(args.warmup + args.steps)]
    pairs = [sum(len(m.row_set(int(r))) for r in rs) for rs in samples]
    for s in range(args.warmup):
        oracle.attention_bwd_dq(m, q, k, v, do, scale, samples[s])
    t0 = time.perf_counter()
    for s in range(args.warmup, args.warmup + args.steps):
        oracle.attention_bwd_dq(m, q, k, v, do, scale, samples[s])
    secs = time.perf_counter() - t0
    done = sum(pairs[args.warmup:])
    value = 10 * d * done / secs / 1e12
    line = {
        "impl": "reference", "metric": BWD_METRIC, "pass": "bwd", "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "H": H, "T": T, "d": d,
                   "mask": mask_desc(p),
                   "step": f"dQ of {n} seeded query rows of one head per step (bounded "
                           f"sample, credited with 10 d flops per pair)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{args.steps} steps x dQ of {n} rows, {done} allowed pairs"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_reference_decode(args):
    """The decode step's reference arm: the oracle's decode of every query head of
    seeded sampled (batch, kv head) groups, bounded per step; the bytes are each
    group's cached K/V rows of the window, counted once for its G heads (as the GPU
    arm counts them)."""
    world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import torch
    import oracle
    oracle.build()
    cfg = W.DECODE_WORKLOADS[args.decode_workload]
    B, Hq, Hkv, cap, w, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["cap"], cfg["window"], cfg["d"]
    G = Hq // Hkv
    g = torch.Generator().manual_seed(0)
    Kc, Vc = (oracle.bf16_bits(torch.randn(cap, d, generator=g).to(torch.bfloat16))
              for _ in range(2))
    qs = [oracle.bf16_bits(torch.randn(d, generator=g).to(torch.bfloat16)) for _ in range(G)]
    pos = W.decode_positions(B, cap, 0)
    scale = 1.0 / math.sqrt(d)
    group_bytes = w * d * 2 * 2

    def groups(n, s):  # n groups: every head of the group at its sequence's position
        for i in range(n):
            t = int(pos[(s * n + i) % B]) + s
            for h in range(G):
                oracle.decode(qs[h], Kc, Vc, t, w, scale)

    t0 = time.perf_counter()
    groups(1, 0)
    dt = max(time.perf_counter() - t0, 1e-4)
    n = int(max(1, min(B * Hkv, 1.0 / dt)))
    for s in range(args.warmup):
        groups(n, s)
    t0 = time.perf_counter()
    for s in range(args.warmup, args.warmup + args.steps):
        groups(n, s)
    secs = time.perf_counter() - t0
    value = group_bytes * n * args.steps / secs / 1e9
    line = {
        "impl": "reference", "metric": DECODE_METRIC, "pass": "decode", "value": value,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.decode_workload, **cfg,
                   "step": f"{n} of the {B * Hkv} (batch, kv head) groups per step, all "
                           f"{G} query heads each (bounded sample)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{args.steps} steps x {n} groups x {G} heads, window {w}"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------- GPU arm

def run_ours(args, cfg, p):
    import torch
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    import sparse_masked_attention_plan_b300 as sp
    B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    # seeded inputs drawn on the host (pinned, reused for the end-to-end leg)
    Qh, Kh, Vh = W.qkv(B, H, T, d, seed=rank, dtype=torch.bfloat16)
    Qh, Kh, Vh = (x.pin_memory() for x in (Qh, Kh, Vh))
    with torch.cuda.stream(stream):
        q, k, v = (x.to(dev, non_blocking=True) for x in (Qh, Kh, Vh))
        o = torch.empty_like(q)
        lse = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    stream.synchronize()
    t_plan = time.perf_counter()
    plan = sp.Plan(T, d, **p, stream=stream)
    stream.synchronize()
    t_plan = time.perf_counter() - t_plan
    info = plan.info()
    pairs_total = info["pairs_per_head"] * B * H
    flops_step = 4.0 * d * pairs_total
    items, ents, products = plan.schedule(0)
    packing = plan.columns().size > 0 or len(p["global_pos"]) > 0
    launches_per_step = 1 + (1 if packing else 0)
    in_bytes = 3 * q.numel() * q.element_size()
    out_bytes = o.numel() * o.element_size() + lse.numel() * 4

    def step():
        sp.fwd(plan, q, k, v, scale, out=o, lse=lse, stream=stream)

    warm_up(torch, stream, step, args.warmup)
    plan.check_device(stream)
    timer = StepTimer(torch, dev, stream, args.steps, in_bytes, "Q/K/V")
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        timer.run(step)
        torch.cuda.synchronize(dev)
        barrier(world)
    plan.check_device(stream)
    per = timer.per_step_ms()
    ms_per_step, value = aggregate(sum(per), args.steps, flops_step, world)

    # end to end through the host-buffer C-ABI entry: H2D of q, k, v, the forward,
    # D2H of O and LSE, every step
    oh = torch.empty_like(Qh).pin_memory()
    lh = torch.empty(B, H, T, dtype=torch.float32).pin_memory()
    bufs = (q, k, v, o, lse)
    e2e_steps = max(2, min(args.steps, 5))
    sp.fwd_host(plan, Qh, Kh, Vh, scale, oh, lh, bufs, stream=stream)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        sp.fwd_host(plan, Qh, Kh, Vh, scale, oh, lh, bufs, stream=stream)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = world * flops_step * e2e_steps / e2e_s / 1e12

    peaks, peak_src = load_peaks()
    line = None
    secondary = None
    if world == 1 and not args.no_secondary and not args.heads:
        secondary = time_secondary(torch, sp, [n for n in SECONDARY if n != args.workload],
                                   args.steps, args.warmup, dev, stream)
    if rank == 0:
        bound, achieved, peak, r_unit = fwd_roofline(args.workload, cfg, flops_step,
                                                     statistics.mean(per), peaks)
        traffic = (TRAFFIC["bytes_per_launch"]
                   if TRAFFIC["kernel_sha"] == kernel_sha() and
                   TRAFFIC["workload"] == args.workload and not args.heads else None)
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            rate, pairs_done, nrows, secs, threads = oracle_sample_rate(cfg, p, Qh, Kh, Vh,
                                                                        args.cpu_budget)
            cpu = {"value": 4 * d * rate / 1e12, "unit": UNIT, "cores": threads,
                   "kind": "oracle",
                   "sample": f"{nrows} seeded query rows of head (0,0) ({pairs_done} allowed "
                             f"pairs, {secs:.1f} s); pairs/s = {rate:.4g}"}
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "H": H, "T": T, "d": d,
                       "mask": mask_desc(p), "pairs_per_head": info["pairs_per_head"],
                       "tiles_full_partial_empty": [info["n_full"], info["n_partial"],
                                                    info["n_empty"]],
                       "tile_products_per_head": products,
                       "l2": timer.l2,
                       "plan_build_ms": round(1e3 * t_plan, 2)},
            "pct_of_bf16_peak": 100.0 * (value / world) / peaks["bf16_tflops"],
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak,
                         "unit": r_unit, "frac": achieved / peak,
                         "traffic": traffic,
                         "peak_source": (f"{peak_src} hbm_gbs" if bound == "hbm" else
                                         f"{peak_src} bf16_tflops (burst)"),
                         "frac_of_sustained": (achieved / peaks["bf16_tflops_sustained"]
                                               if bound == "tensor" else None),
                         "kernel": "fwd_tc_kernel<%d>" % d + (" (with k_pack)" if packing else ""),
                         "kernel_ms": statistics.mean(per)},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": in_bytes,
                    "d2h_bytes_per_step": out_bytes,
                    "api": "spattn_fwd_host (pinned host buffers)"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        if secondary is not None:
            line["secondary"] = secondary
        print(json.dumps(line))
    plan.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------- backward arm

BWD_METRIC = "allowed-pair backward TFLOP/s (10·d·pairs/s), 1 GPU"
def run_ours_bwd(args, cfg, p):
    """One step = one spattn_bwd over the whole batch (dQ, dK, dV of every head) with
    q, k, v, O, LSE and dO resident in HBM.  value = 10 d B H pairs / t_step: per
    allowed pair 2d flops each for the recomputed logit, dO.v, and the dV, dK and dQ
    updates.  The tensor-core kernels execute 14 d per pair (the query-major dQ pass
    and the key-major dK/dV pass each recompute the logit and dO.v); the roofline is
    taken on the algorithmic 10 d against the measured bf16 peak."""
    import torch
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    import sparse_masked_attention_plan_b300 as sp
    B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    Qh, Kh, Vh = W.qkv(B, H, T, d, seed=rank, dtype=torch.bfloat16)
    dOh = W.grad_out(B, H, T, d, seed=rank, dtype=torch.bfloat16)
    with torch.cuda.stream(stream):
        q, k, v, do = (x.to(dev) for x in (Qh, Kh, Vh, dOh))
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    plan = sp.Plan(T, d, **p, stream=stream)
    o, lse = sp.fwd(plan, q, k, v, scale, stream=stream)
    stream.synchronize()
    info = plan.info()
    pairs_total = info["pairs_per_head"] * B * H
    flops_step = 10.0 * d * pairs_total
    n_packed_units = int((plan.schedule(4)[0][:, 3] & 1).sum())
    packing = plan.columns().size > 0 or len(p["global_pos"]) > 0
    # rowdot, [pack K/V/Q, pack dO], dQ, dK/dV (packed units, natural units)
    launches = 1 + (1 if packing else 0) + (1 if len(p["global_pos"]) else 0) + 1 + \
        (1 if n_packed_units else 0) + 1

    def step():
        sp.bwd(plan, q, k, v, o, lse, do, scale, dq, dk, dv, stream=stream)

    warm_up(torch, stream, step, args.warmup)
    timer = StepTimer(torch, dev, stream, args.steps,
                      5 * q.numel() * q.element_size() + lse.numel() * 4, "q, k, v, O, dO, LSE")
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        timer.run(step)
        torch.cuda.synchronize(dev)
        barrier(world)
    plan.check_device(stream)
    per = timer.per_step_ms()
    ms_per_step, value = aggregate(sum(per), args.steps, flops_step, world)

    # end to end: every step copies q, k, v, O, LSE and dO in from pinned host memory,
    # runs the backward and copies dQ, dK, dV back out
    host_in = [x.pin_memory() for x in (Qh, Kh, Vh)] + \
        [o.cpu().pin_memory(), lse.cpu().pin_memory(), dOh.pin_memory()]
    dev_in = (q, k, v, o, lse, do)
    host_out = [torch.empty(dq.shape, dtype=dq.dtype).pin_memory() for _ in range(3)]
    h2d = sum(x.numel() * x.element_size() for x in host_in)
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    e2e_steps = max(3, min(args.steps, 5))
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        with torch.cuda.stream(stream):
            for dst, src in zip(dev_in, host_in):
                dst.copy_(src, non_blocking=True)
        step()
        with torch.cuda.stream(stream):
            for dst, src in zip(host_out, (dq, dk, dv)):
                dst.copy_(src, non_blocking=True)
        stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e = world * flops_step * e2e_steps / e2e_s / 1e12
    plan.check_device(stream)
    if rank == 0:
        peaks, peak_src = load_peaks()
        step_ms = statistics.mean(per)
        achieved = flops_step / (step_ms / 1e3) / 1e12
        line = {
            "metric": BWD_METRIC, "pass": "bwd", "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "H": H, "T": T, "d": d,
                       "mask": mask_desc(p), "pairs_per_head": info["pairs_per_head"],
                       "l2": timer.l2},
            "roofline": {"bound": "tensor", "achieved": achieved,
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"],
                         "traffic": (BWD_TRAFFIC["bytes_per_launch"]
                                     if kernel_sha(BWD_TRAFFIC["file"]) == BWD_TRAFFIC["kernel_sha"]
                                     and args.workload == BWD_TRAFFIC["workload"]
                                     and not args.heads else None),
                         "traffic_kernel": "bwd_dkdv_tc_kernel",
                         "peak_source": f"{peak_src} bf16_tflops (burst)",
                         "executed_tflops": achieved * 1.4,
                         "kernel": "rowdot + pack + bwd_dq_tc + bwd_dkdv_tc (whole step)",
                         "kernel_ms": step_ms},
            "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "api": "spattn_bwd with q, k, v, O, LSE, dO copied in from pinned host "
                           "memory and dQ, dK, dV copied out, every step"},
            "gpu_launches": launches * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line))
    plan.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------- decode arm

DECODE_METRIC = "decode KV-cache GB/s (bytes of cached K/V read per step / step time), 1 GPU"


def run_decode(args):
    """One step = one generation step of every sequence: spattn_kv_append of the
    step's key/value rows, then spattn_decode of the step's queries against the
    ring-buffer cache (the window of every sequence is full).  Algorithmic bytes per
    step: the cached K and V rows read (B Hkv window d 2 2 bytes) plus q, the new rows
    and the output."""
    import torch
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    import sparse_masked_attention_plan_b300 as sp
    cfg = W.DECODE_WORKLOADS[args.decode_workload]
    B, Hq, Hkv, cap, w, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["cap"], cfg["window"], cfg["d"]
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    g = torch.Generator().manual_seed(rank)
    with torch.cuda.stream(stream):
        c = sp.DecodeCache(B, Hq, Hkv, cap, d, window=w, device=dev)
        c.K.copy_(torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16))
        c.V.copy_(torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16))
    qh = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16).pin_memory()
    kh = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).pin_memory()
    vh = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).pin_memory()
    pos0 = torch.from_numpy(W.decode_positions(B, cap, rank))
    q, kn, vn = (x.to(dev) for x in (qh, kh, vh))
    out = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    steps_total = args.warmup + args.steps
    pos_all = torch.stack([pos0 + s for s in range(steps_total)]).to(dev)  # [steps, B]
    stream.synchronize()
    kv_bytes = B * Hkv * w * d * 2 * 2
    step_bytes = kv_bytes + (2 * q.numel() + 2 * kn.numel()) * 2 + lse.numel() * 4
    scale = 1.0 / math.sqrt(d)

    def step(s):  # append the step's rows and decode, one call (two launches for bf16)
        c.append_step(kn, vn, q, pos_all[s], scale, out=out, lse=lse, stream=stream)

    for s in range(args.warmup):
        step(s)
    stream.synchronize()
    c.check(stream)
    # The timed steps run as one captured CUDA graph, the way a generation loop
    # launches its steps: every step still appends its rows, decodes at its own
    # position and merges the splits (two kernels: the decode kernel appends), with no
    # host work in between.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for s in range(args.steps):
            step(args.warmup + s)
    # the graph's first launches (upload, and the clocks up from idle); replaying it
    # again rewrites the same rows at the same positions, so the timed launch repeats it
    t_w = time.perf_counter()
    while True:
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        if time.perf_counter() - t_w >= 0.2:
            break
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        ev[0].record(stream)
        with torch.cuda.stream(stream):
            graph.replay()
        ev[1].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    c.check(stream)
    ms = max_over_ranks(ev[0].elapsed_time(ev[1]), world) / args.steps
    value = world * step_bytes / (ms / 1e3) / 1e9

    # end to end: this step's q, k, v from pinned host memory, append + decode, the
    # output back to the host, every step
    oh = torch.empty_like(qh).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    barrier(world)
    t0 = time.perf_counter()
    for s in range(e2e_steps):
        with torch.cuda.stream(stream):
            q.copy_(qh, non_blocking=True)
            kn.copy_(kh, non_blocking=True)
            vn.copy_(vh, non_blocking=True)
        step(s % steps_total)
        with torch.cuda.stream(stream):
            oh.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e = world * step_bytes * e2e_steps / e2e_s / 1e9
    if rank == 0:
        peaks, src = load_peaks()
        step_ms = ev[0].elapsed_time(ev[1]) / args.steps
        achieved = step_bytes / (step_ms / 1e3) / 1e9
        line = {
            "metric": DECODE_METRIC, "pass": "decode", "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.decode_workload, **cfg,
                       "tokens_per_step": B,
                       "launch": "timed steps replayed from one captured CUDA graph",
                       "l2": (f"cache larger than L2 ({kv_bytes / 1e6:.0f} MB of K/V)"
                              if kv_bytes > L2_BYTES else
                              f"cache of {kv_bytes / 1e6:.0f} MB fits in L2 (not flushed: the "
                              f"steps run back to back from one graph)")},
            "tokens_per_s": world * B / (ms / 1e3),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": (DEC_TRAFFIC["bytes_per_launch"].get(args.decode_workload)
                                     if kernel_sha(DEC_TRAFFIC["file"]) == DEC_TRAFFIC["kernel_sha"]
                                     else None),
                         "traffic_kernel": "decode_mma_kernel",
                         "peak_source": f"{src} hbm_gbs",
                         "kernel": "decode (with the append) + combine (whole step)",
                         "kernel_ms": step_ms},
            "e2e": {"value": e2e, "unit": "GB/s",
                    "h2d_bytes_per_step": (q.numel() + 2 * kn.numel()) * 2,
                    "d2h_bytes_per_step": out.numel() * 2,
                    "api": "DecodeCache.append_step (spattn_decode_append) with pinned host "
                           "q/k/v and output"},
            "gpu_launches": 2 * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd", "decode"],
                    help="time the forward (default, the headline), the backward pass, or "
                         "one decode step")
    ap.add_argument("--decode-workload", default="decode_b32_w4096",
                    choices=sorted(W.DECODE_WORKLOADS))
    ap.add_argument("--no-secondary", action="store_true",
                    help="time the named workload only (no secondary forward workloads)")
    ap.add_argument("--heads", type=int, default=0,
                    help="override H (smaller profiling captures; the line then names it)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = dict(W.WORKLOADS[args.workload])
    if args.heads:
        cfg["H"] = args.heads
    p = W.mask_params(args.workload)
    if args.impl == "reference":
        if args.which == "bwd":
            return run_reference_bwd(args, cfg, p)
        if args.which == "decode":
            return run_reference_decode(args)
        return run_reference(args, cfg, p)
    if args.which == "bwd":
        return run_ours_bwd(args, cfg, p)
    if args.which == "decode":
        return run_decode(args)
    return run_ours(args, cfg, p)


if __name__ == "__main__":
    sys.exit(main())

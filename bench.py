#!/usr/bin/env python3
"""Benchmark of the W4A8 skinny linear on GB300: the 27B-class decode step.

One step = the 257 decode linears of a 27B-class decoder, in order: 64 layers
of (QKV 5120->7168, O 5120->5120, gate+up 5120->34816, down 17408->5120) and
the LM head 5120->152064, each one launch of the fused bf16 -> int8 -> W4A8
GEMV entry point (woq_w4a8_linear_bf16), captured once in a CUDA graph.
Weights are distinct synthetic tensors per linear (11.3 GB packed, far larger
than the 129 MB L2, so every step streams them from HBM); activations are
seeded bf16 N(0,1) with 1 % x20 outlier channels (synthetic.py).

Prints one JSON line (rank 0).  `value` is the achieved algorithmic HBM
bandwidth of the step in GB/s (packed int4 weights + fp16 group scales +
bf16 activations read once), summed over ranks; ms_per_step and the M = 3 / 4
step times ride along.  `--impl reference` times the CPU oracle instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A8 skinny-GEMV HBM GB/s & % of GB300 peak at M=1,3; µs per 27B-class step"
WORKLOAD = ("27B-class decode step, W4A8: 64 x (QKV 5120->7168, O 5120->5120, gate+up 5120->34816, "
            "down 17408->5120) + LM head 5120->152064 = 257 linears")
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--m", type=int, default=1, help="activation rows of the headline step")
    ap.add_argument("--extra-m", default="3,4", help="also time the step at these M (comma list, '' for none)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prologue-fusion", dest="prologue_fusion", action="store_false",
                    help="skip the RMSNorm / SwiGLU prologue-fusion step (fused against unfused)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-div", type=int, default=8, help="oracle sample: 1/div of every linear's rows")
    ap.add_argument("--linear", default="", help="time one 27B-class linear (qkv, o, gate_up, down, lm_head) "
                                                 "instead of the step: a graph of launches over distinct weight copies")
    ap.add_argument("--int8", action="store_true", help="with --linear: the int8 entry (act_quant once, then GEMV)")
    ap.add_argument("--bits", type=int, default=4, choices=[4, 6], help="with --linear: int4 or int6 weights")
    ap.add_argument("--prologue", default="none", choices=["none", "rmsnorm", "swiglu"],
                    help="with --linear: the bf16 entry with the RMSNorm prologue, or the SwiGLU entry")
    ap.add_argument("--tree-planner", action="store_true",
                    help="time one re-plan of the draft-tree planner (host code) against its oracle")
    ap.add_argument("--relayout", action="store_true",
                    help="time the in-place relayout of 27B-class matrices instead of the step")
    ap.add_argument("--path", type=int, default=0, choices=[0, 1, 2],
                    help="with --linear: int4 consumer (0 launch table, 1 dp4a, 2 tensor-core MMA)")
    ap.add_argument("--shape", default="27b", choices=["27b", "9b"], help="with --linear: 27B- or 9B-class shapes")
    ap.add_argument("--suite", action="store_true",
                    help="time the 1024 x 1024 linear, the 9B W4A8 linears (M = 1, 3) and the 9B W6A8 linears "
                         "(M = 1 .. 4) instead of the step")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the per-linear config suite on the headline line")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers

def algorithmic_bytes(linears, M, bits=4):
    """Packed weights + fp16 group scales + bf16 activations read once, per step."""
    tot = 0
    for _, K, N in linears:
        tot += N * K * bits // 8 + 2 * N * (K // 128) + 2 * M * K
    return tot


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic():
    """Per-step DRAM bytes of the GEMV kernel from the committed ncu summary (None if absent)."""
    p = os.path.join(ROOT, "profiles", "gemv_w4a8_27b_step_m1.md")
    try:
        with open(p) as f:
            for line in f:
                if line.startswith("dram_bytes_per_step:"):
                    return int(line.split(":")[1].strip())
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self, util_floor_mhz=0):
        sms, maxes, reasons, powers = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx, pw = float(f[1]), float(f[2]), float(f[3])
            except ValueError:
                continue
            powers.append(pw)
            sms.append(sm)
            maxes.append(mx)
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        # samples taken while the GPU was busy: the top half by power draw
        pw_cut = statistics.median(powers)
        loaded = [s for s, p in zip(sms, powers) if p >= pw_cut] or sms
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms), "power_w_max": max(powers)}


# ----------------------------------------------------------------------------- ranks

class RankGroup:
    """The N replicas of a multi-GPU run: a barrier around the timed region and the maximum
    of a per-rank time (no collective on the data path; replicas only).  device: where the
    reduction tensor lives (the GPU under NCCL, the CPU under gloo)."""

    def __init__(self, world, device):
        self.world, self.device = world, device

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max(self, v):
        if self.world == 1:
            return v
        import torch
        import torch.distributed as dist
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())


def job_value(world, bytes_per_step, ms_per_step):
    """Whole-job throughput in GB/s: every replica streams bytes_per_step per step, and the
    step time is the slowest replica's."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


# ----------------------------------------------------------------------------- our arm

class Step:
    """The 27B-class decode step on one GPU: weights packed in HBM, one CUDA graph per M."""

    def __init__(self, device, seed=2, cpu_sample_div=0):
        import torch

        import synthetic
        import weight_only_quantised_gb300 as woq
        self.torch, self.woq, self.synthetic = torch, woq, synthetic
        self.device = device
        self.linears = synthetic.step_27b()
        self.packed = []
        self.cpu_sample = []  # (K, N rows, canonical w rows, scale rows) for the oracle baseline
        for name, K, N in self.linears:
            w, s = synthetic.weights(4, N, K, synthetic.sub_seed(seed, name), device=device)
            p = torch.empty(woq.woq_packed_bytes(4, N, K), dtype=torch.uint8, device=device)
            woq.woq_pack_device(4, w, s.view(torch.int16), N, K, p)
            self.packed.append(p)
            if cpu_sample_div:
                rows = max(1, N // cpu_sample_div)
                self.cpu_sample.append((K, rows, w[:rows].cpu().numpy(),
                                        synthetic.to_numpy_u16(s[:rows])))
            del w, s
        torch.cuda.synchronize()
        self.graphs = {}
        self.prefetch_next_kb = 0  # next-linear L2 prefetch per CTA (KiB, 0 = library default, -1 = off)

    def buffers(self, M, seed=2):
        torch, synthetic, woq = self.torch, self.synthetic, self.woq
        xs = {K: synthetic.activations(M, K, synthetic.sub_seed(seed, "x", M, K), outliers=True,
                                       device=self.device) for K in sorted({K for _, K, _ in self.linears})}
        ys = {N: torch.empty((M, N), dtype=torch.float32, device=self.device)
              for N in sorted({N for _, _, N in self.linears})}
        wsb = max(woq.woq_workspace_bytes(4, M, N, K) for _, K, N in self.linears)
        ws = torch.zeros(wsb, dtype=torch.uint8, device=self.device)
        return xs, ys, ws

    def launch_all(self, xs, ys, ws):
        woq = self.woq
        n = len(self.linears)
        for i, ((name, K, N), p) in enumerate(zip(self.linears, self.packed)):
            if self.prefetch_next_kb >= 0 and i + 1 < n:
                _, K2, N2 = self.linears[i + 1]
                woq.woq_prefetch_next(self.packed[i + 1], 4, N2, K2, self.prefetch_next_kb)
            woq.woq_w4a8_linear_bf16(p, xs[K], N, K, ys[N], ws)

    def time_prologue_chain(self, M, steps, warmup, fused):
        """The step as a dependency chain with the prologue fusions of "Optimizing the Linear
        Kernel": qkv and gate_up behind an RMSNorm, down behind the SwiGLU of the gate_up output
        (its fp32 y is the down projection's input), o on the bf16 entry, the LM head behind
        the final RMSNorm.  fused: one launch per linear; else the unfused twins
        (woq_rmsnorm_act_quant_int8 / woq_swiglu_act_quant_int8) then the int8 GEMV."""
        torch, synthetic, woq = self.torch, self.synthetic, self.woq
        xs, ys, ws = self.buffers(M)
        K = 5120
        gamma = synthetic.rmsnorm_weight(K, 9, device=self.device)
        qs = {Kl: torch.empty((M, Kl), dtype=torch.int8, device=self.device) for Kl in (5120, 17408)}
        a = torch.empty((M,), dtype=torch.float32, device=self.device)

        def launch():
            for (name, Kl, N), p in zip(self.linears, self.packed):
                kind = name.split(".")[-1]
                y = ys[N]
                if kind in ("qkv", "gate_up", "lm_head"):
                    if fused:
                        woq.woq_w4a8_linear_rmsnorm_bf16(p, xs[Kl], gamma, 1e-6, N, Kl, y, ws)
                    else:
                        woq.woq_rmsnorm_act_quant_int8(xs[Kl], gamma, 1e-6, qs[Kl], a)
                        woq.woq_w4a8_gemv(p, qs[Kl], a, N, Kl, y, ws)
                elif kind == "down":
                    gu = ys[2 * Kl]  # the gate_up output of this layer
                    if fused:
                        woq.woq_w4a8_linear_swiglu_f32(p, gu, N, Kl, y, ws)
                    else:
                        woq.woq_swiglu_act_quant_int8(gu, qs[Kl], a)
                        woq.woq_w4a8_gemv(p, qs[Kl], a, N, Kl, y, ws)
                else:
                    woq.woq_w4a8_linear_bf16(p, xs[Kl], N, Kl, y, ws)

        stream = torch.cuda.Stream(device=self.device)
        ys[34816].zero_()
        with torch.cuda.stream(stream):
            launch()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launch()
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        assert self.woq.woq_read_status(ws) == 0
        return e0.elapsed_time(e1) / steps

    def capture(self, M):
        torch = self.torch
        xs, ys, ws = self.buffers(M)
        stream = torch.cuda.Stream(device=self.device)
        with torch.cuda.stream(stream):
            self.launch_all(xs, ys, ws)  # warm-up outside the capture (sets kernel attributes)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.launch_all(xs, ys, ws)
        torch.cuda.synchronize()
        assert self.woq.woq_read_status(ws) == 0
        self.graphs[M] = (g, xs, ys, ws)
        return self.graphs[M]

    def time_device(self, M, steps, warmup, barrier, sampler_gpu=None):
        torch = self.torch
        g, xs, ys, ws = self.graphs.get(M) or self.capture(M)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        clocks = None
        barrier()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        sampler = ClockSampler(sampler_gpu) if sampler_gpu is not None else None
        if sampler:
            sampler.__enter__()
        start.record()
        for _ in range(steps):
            g.replay()
        end.record()
        torch.cuda.synchronize()
        if sampler:
            sampler.__exit__(None, None, None)
            clocks = sampler.summary()
        barrier()
        assert self.woq.woq_read_status(ws) == 0
        return start.elapsed_time(end), clocks

    def time_e2e(self, M, steps, warmup):
        """Per step: pinned host -> device copy of the step's activations, the graph, and a
        device -> pinned host read of the LM-head output; synchronised every step."""
        torch = self.torch
        g, xs, ys, ws = self.graphs.get(M) or self.capture(M)
        xh = {K: x.cpu().pin_memory() for K, x in xs.items()}
        n_out = self.linears[-1][2]
        yh = torch.empty((M, n_out), dtype=torch.float32).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in xh.values())
        d2h = yh.numel() * yh.element_size()

        def one():
            for K, x in xs.items():
                x.copy_(xh[K], non_blocking=True)
            g.replay()
            yh.copy_(ys[n_out], non_blocking=True)
            torch.cuda.current_stream().synchronize()

        for _ in range(warmup):
            one()
        t0 = time.perf_counter()
        for _ in range(steps):
            one()
        dt = (time.perf_counter() - t0) / steps
        return dt, h2d, d2h


def host_cores():
    """CPU cores this process may run on (sched_getaffinity), or the CPU count."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline_oracle(sample, M, threads=1, seed=2):
    """The oracle, as it stands, on 1/div of every linear's rows, M activation rows.  threads > 1
    splits each linear's rows into that many slices run by Python threads (the oracle is C
    called through ctypes, which releases the GIL, so the slices run in parallel)."""
    import concurrent.futures as cf

    import oracle
    import synthetic
    xs = {}
    for K, *_ in sample:
        if K not in xs:
            xs[K] = synthetic.to_numpy_u16(synthetic.activations(M, K, synthetic.sub_seed(seed, "x", M, K)))
    jobs = []
    total_bytes = 0
    for K, rows, wn, sn in sample:
        total_bytes += rows * K // 2 + 2 * rows * (K // 128) + 2 * M * K
        n = max(1, min(threads, rows))
        for t in range(n):
            r0, r1 = rows * t // n, rows * (t + 1) // n
            if r1 > r0:
                jobs.append((K, r1 - r0, wn[r0:r1], sn[r0:r1]))
    t0 = time.perf_counter()
    if threads == 1:
        for K, r, wn, sn in jobs:
            oracle.linear_bf16(4, wn, sn, r, K, xs[K])
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda j: oracle.linear_bf16(4, j[2], j[3], j[1], j[0], xs[j[0]]), jobs))
    dt = time.perf_counter() - t0
    return total_bytes / dt / 1e9, dt, total_bytes


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    group = RankGroup(world, device)
    barrier, max_over_ranks = group.barrier, group.max

    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    step = Step(device, cpu_sample_div=args.cpu_sample_div if do_cpu else 0)
    M = args.m
    bytes_step = algorithmic_bytes(step.linears, M)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    gpu_index = vis.split(",")[local].strip() if vis else str(local)

    ms_total, clocks = step.time_device(M, args.steps, args.warmup, barrier, sampler_gpu=gpu_index)
    ms_total = max_over_ranks(ms_total)
    ms_step = ms_total / args.steps
    value = job_value(world, bytes_step, ms_step)

    extra = {}
    for em in [int(v) for v in args.extra_m.split(",") if v.strip()]:
        if em == M:
            continue
        k = min(args.steps, 300)
        ms_e, _ = step.time_device(em, k, min(args.warmup, 5), barrier)
        ms_e = max_over_ranks(ms_e) / k
        b_e = algorithmic_bytes(step.linears, em)
        extra[f"m{em}"] = {"ms_per_step": round(ms_e, 4), "us_per_step": round(ms_e * 1e3, 1),
                           "gbs": round(b_e / (ms_e * 1e-3) / 1e9, 1),
                           "vs_m1_time": round(ms_e / ms_step, 4)}

    prologue = None
    if args.prologue_fusion:
        k = min(args.steps, 200)
        f_ms = max_over_ranks(step.time_prologue_chain(M, k, min(args.warmup, 5), fused=True))
        u_ms = max_over_ranks(step.time_prologue_chain(M, k, min(args.warmup, 5), fused=False))
        prologue = {"fused_ms_per_step": round(f_ms, 4), "unfused_ms_per_step": round(u_ms, 4),
                    "fused_launches": len(step.linears), "unfused_launches": len(step.linears) + 3 * 64 + 1,
                    "what": "qkv, gate_up, lm_head behind RMSNorm; down behind SwiGLU of the gate_up output"}

    e2e = None
    if not args.no_e2e:
        k = min(args.steps, 200)
        dt, h2d, d2h = step.time_e2e(M, k, min(args.warmup, 5))
        dt = max_over_ranks(dt)
        e2e = {"value": round(world * bytes_step / dt / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(dt * 1e3, 4)}

    configs = None
    if args.configs and rank == 0:
        configs = config_suite(steps=30, warmup=3)

    cpu = None
    if do_cpu:
        cores = host_cores()
        v1, dt1, nbytes = cpu_baseline_oracle(step.cpu_sample, M, threads=1)
        vn, dtn, _ = cpu_baseline_oracle(step.cpu_sample, M, threads=cores)
        what = (f"first 1/{args.cpu_sample_div} of the rows of all 257 linears of the step, M={M} "
                f"({nbytes / 1e9:.2f} GB of weights+scales)")
        cpu = {"value": round(vn, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{what}; {cores} threads (one per core from sched_getaffinity), {dtn:.1f} s",
               "single_thread": {"value": round(v1, 4), "unit": "GB/s", "cores": 1, "seconds": round(dt1, 1)}}

    peak, peak_kind = measured_peak()
    achieved = bytes_step / (ms_step * 1e-3) / 1e9
    traffic = profiled_traffic()
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "us_per_step": round(ms_step * 1e3, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "s8xs4->s32, f32 scale",
        "data": "synthetic (seeded; random weights of the 27B-class shapes)",
        "config": {"workload": WORKLOAD, "m": M, "linears": len(step.linears),
                   "bytes_per_step": bytes_step, "entry": "woq_w4a8_linear_bf16 (fused bf16 quant + GEMV)",
                   "cuda_graph": True, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: 11.3 GB of distinct weights streamed per step"},
        "pct_of_peak": round(100.0 * achieved / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": peak_kind, "kernel": "woq::kern::gemv_kernel<4, M, fused, dp4a>",
                     "per": "step (257 launches)"},
        "extra_m": extra,
        "prologue_fusion": prologue,
        "configs": configs,
        "e2e": e2e,
        "gpu_launches": len(step.linears) * args.steps,
        "prefetch_next": {"kb_per_cta": "library default", "what": "each launch prefetches the next linear's "
                                                                  "first weights into L2 (woq_prefetch_next)"},
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle on the host cores: each step is a bounded row sample of one of the
    step's linears (cycling through all 257), sized so the whole run takes about a minute; the
    sample's rows are split over one thread per core (the C oracle runs without the GIL)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import synthetic
    linears = synthetic.step_27b()
    M = args.m
    # calibrate the oracle's rate on this host
    K0, N0 = 5120, 64
    w, s = synthetic.weights(4, N0, K0, 0)
    x = synthetic.to_numpy_u16(synthetic.activations(M, K0, 0))
    t0 = time.perf_counter()
    oracle.linear_bf16(4, w.numpy(), synthetic.to_numpy_u16(s), N0, K0, x)
    rate = N0 * K0 / max(time.perf_counter() - t0, 1e-6)  # weights per second
    budget = 60.0 / max(1, args.steps + args.warmup)
    cores = host_cores()
    import concurrent.futures as cf
    pool = cf.ThreadPoolExecutor(max_workers=cores)
    cache = {}
    total_b, total_t = 0, 0.0
    for i in range(args.warmup + args.steps):
        name, K, N = linears[i % len(linears)]
        rows = int(min(N, max(cores, budget * rate * cores / K)))
        key = (name, rows)
        if key not in cache:
            wt, st = synthetic.weights(4, rows, K, synthetic.sub_seed(2, name, rows))
            xk = synthetic.to_numpy_u16(synthetic.activations(M, K, synthetic.sub_seed(2, "x", M, K)))
            cache = {key: (wt.numpy(), synthetic.to_numpy_u16(st), xk)}
        wn, sn, xk = cache[key]
        cuts = [rows * t // cores for t in range(cores + 1)]
        t0 = time.perf_counter()
        list(pool.map(lambda t: oracle.linear_bf16(4, wn[cuts[t]:cuts[t + 1]], sn[cuts[t]:cuts[t + 1]],
                                                   cuts[t + 1] - cuts[t], K, xk),
                      [t for t in range(cores) if cuts[t + 1] > cuts[t]]))
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            total_t += dt
            total_b += rows * K // 2 + 2 * rows * (K // 128) + 2 * M * K
    value = total_b / total_t / 1e9
    ms_step = total_t / args.steps * 1e3
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int64 dots, f32 terms, f64 sum",
        "data": "synthetic (seeded; random weights of the 27B-class shapes)",
        "config": {"workload": WORKLOAD, "m": M, "linears": len(linears),
                   "sample": "each step: a row sample of one linear of the step, cycling through all 257"},
        "cpu_baseline": {"kind": "oracle", "cores": cores, "value": round(value, 4), "unit": "GB/s",
                         "sample": f"{args.steps} steps of row samples (~{budget:.2f} s each), {cores} threads "
                                   f"(one per core from sched_getaffinity)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    pool.shutdown()
    print(json.dumps(line), flush=True)


L2_BYTES = 129 * 2 ** 20  # GB300 L2


def time_linear_chain(bits, M, K, N, entry="bf16", seed=2, steps=50, warmup=3, path=0, name="linear",
                      rotation_bytes=int(1.2e9)):
    """One linear launched back to back over distinct packed copies of its weights whose total is
    at least rotation_bytes (>= 4 x L2 by default: every launch streams its weights from HBM, the
    cold-L2 rule), captured in one CUDA graph and replayed steps times.  entry: "bf16" (fused
    quant + GEMV), "int8" (act_quant once, then the GEMV), "rmsnorm" or "swiglu" (the prologue
    fusions).  Returns a dict with the time per launch and the algorithmic bandwidth."""
    import torch

    import synthetic
    import weight_only_quantised_gb300 as woq
    assert rotation_bytes >= 4 * L2_BYTES
    dev = torch.device("cuda", torch.cuda.current_device())
    woq.woq_tune_path(path)
    pb = woq.woq_packed_bytes(bits, N, K)
    copies = max(4, -(-rotation_bytes // pb))
    w, s = synthetic.weights(bits, N, K, synthetic.sub_seed(seed, name, bits), device=dev)
    bufs = []
    for _ in range(copies):
        p = torch.empty(pb, dtype=torch.uint8, device=dev)
        woq.woq_pack_device(bits, w, s.view(torch.int16), N, K, p)
        bufs.append(p)
    del w, s
    x = synthetic.activations(M, K, synthetic.sub_seed(seed, "x", M, K), device=dev)
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    a = torch.empty((M,), dtype=torch.float32, device=dev)
    woq.woq_act_quant_int8(x, q, a)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    ws = torch.zeros(woq.woq_workspace_bytes(bits, M, N, K), dtype=torch.uint8, device=dev)
    gamma = synthetic.rmsnorm_weight(K, 9, device=dev)
    gu = synthetic.gate_up_output(M, K, 9, device=dev)
    w4 = bits == 4

    def launch(p):
        if entry == "int8":
            (woq.woq_w4a8_gemv if w4 else woq.woq_w6a8_gemv)(p, q, a, N, K, y, ws)
        elif entry == "rmsnorm":
            (woq.woq_w4a8_linear_rmsnorm_bf16 if w4 else woq.woq_w6a8_linear_rmsnorm_bf16)(p, x, gamma, 1e-6, N, K,
                                                                                         y, ws)
        elif entry == "swiglu":
            (woq.woq_w4a8_linear_swiglu_f32 if w4 else woq.woq_w6a8_linear_swiglu_f32)(p, gu, N, K, y, ws)
        else:
            (woq.woq_w4a8_linear_bf16 if w4 else woq.woq_w6a8_linear_bf16)(p, x, N, K, y, ws)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        launch(bufs[0])
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for p in bufs:
            launch(p)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    assert woq.woq_read_status(ws) == 0
    woq.woq_tune_path(0)
    us = e0.elapsed_time(e1) * 1e3 / (steps * copies)
    act_bytes = {"bf16": 2 * M * K, "rmsnorm": 2 * M * K + 2 * K, "swiglu": 8 * M * K, "int8": M * K + 4 * M}[entry]
    nbytes = N * K * bits // 8 + 2 * N * (K // 128) + act_bytes
    peak, kind = measured_peak()
    del bufs
    torch.cuda.empty_cache()
    return {"linear": name, "K": K, "N": N, "m": M, "bits": bits, "entry": entry,
            "us_per_launch": round(us, 3), "gbs": round(nbytes / us / 1e3, 1),
            "frac_of_peak": round(nbytes / us / 1e3 / peak, 4), "peak_kind": kind, "bytes_per_launch": nbytes,
            "rotation": {"copies": copies, "bytes": copies * pb}}


def config_suite(steps=30, warmup=3):
    """The single 1024 x 1024 linear, the 9B-class layer's linears at M = 1 and 3 (W4A8), and the
    9B-class linears in W6A8 at M = 1 .. 4 through the fused bf16 entry; each timed as a chain over
    a cold-L2 rotation of distinct weight copies (>= 4 x L2)."""
    import synthetic
    out = {"w4a8_1024x1024": [time_linear_chain(4, 1, 1024, 1024, seed=0, steps=steps, warmup=warmup,
                                                name="single_1024")]}
    rows = []
    for M in (1, 3):
        for name, (K, N) in synthetic.LINEARS_9B.items():
            rows.append(time_linear_chain(4, M, K, N, seed=1, steps=steps, warmup=warmup, name=name))
    out["9b_w4a8"] = rows
    rows = []
    for M in (1, 2, 3, 4):
        for name, (K, N) in synthetic.LINEARS_9B.items():
            rows.append(time_linear_chain(6, M, K, N, seed=4, steps=steps, warmup=warmup, name=name))
    out["9b_w6a8_fused"] = rows
    for key, rows in out.items():
        for r in rows:
            r.pop("peak_kind", None)
    return out


def run_linear(args):
    """One 27B-class linear (or, with --shape 9b, a 9B-class one), launched back to back over
    distinct packed copies whose total exceeds 1 GB (every launch streams its weights from HBM)."""
    import torch

    import synthetic
    shapes = dict(synthetic.LINEARS_9B if args.shape == "9b" else synthetic.LINEARS_27B)
    shapes["lm_head"] = synthetic.LM_HEAD_27B
    K, N = shapes[args.linear]
    torch.cuda.set_device(torch.device("cuda", 0))
    entry = "int8" if args.int8 else {"none": "bf16", "rmsnorm": "rmsnorm", "swiglu": "swiglu"}[args.prologue]
    r = time_linear_chain(args.bits, args.m, K, N, entry=entry, seed=2, steps=args.steps, warmup=args.warmup,
                          path=args.path, name=args.linear)
    r["consumer"] = {0: "table", 1: "dp4a", 2: "mma"}[args.path]
    print(json.dumps(r), flush=True)


def run_suite(args):
    """The configs other than the 27B step (see config_suite), one JSON line."""
    import torch
    torch.cuda.set_device(torch.device("cuda", 0))
    peak, kind = measured_peak()
    print(json.dumps({"metric": "per-linear time and algorithmic HBM GB/s, cold L2", "peak": peak, "peak_kind": kind,
                      "configs": config_suite(steps=max(10, min(args.steps, 100)), warmup=args.warmup)}), flush=True)


def run_tree_planner(args):
    """Draft-tree planner re-plan time: all 64 shapes scored (library), and the oracle's."""
    import random

    import weight_only_quantised_gb300 as woq
    from oracle import tree as T
    rng = random.Random(3)
    lib, ora = woq.TreePlanner(replan_every=10 ** 9), T.Planner(replan_every=10 ** 9)
    probs = []
    for _ in range(7):
        w = [rng.random() for _ in range(8)]
        probs.append([x / sum(w) for x in w])
    for _ in range(256):  # synthetic acceptance statistics
        _, ranks = T.simulate_step(probs, ora.shape, rng)
        lib.observe(ranks, 0.08, 1.0)
        ora.observe(ranks, 0.08, 1.0)
    n = max(1000, args.steps)
    t0 = time.perf_counter()
    for _ in range(n):
        lib.replan()
    lib_us = (time.perf_counter() - t0) / n * 1e6
    m = 200
    t0 = time.perf_counter()
    for _ in range(m):
        ora.replan()
    ora_us = (time.perf_counter() - t0) / m * 1e6
    print(json.dumps({"metric": "draft-tree planner re-plan time (64 shapes)", "value": round(lib_us, 3), "unit": "us",
                      "higher_is_better": False, "calls": n, "note": "host code, called through ctypes",
                      "cpu_baseline": {"value": round(ora_us, 2), "unit": "us", "cores": 1, "kind": "oracle",
                                       "sample": f"{m} re-plans"}}), flush=True)


def run_relayout(args):
    """In-place relayout (woq_relayout_inplace) of 27B-class int4 / int6 matrices, timed per call
    with CUDA events; beside it the out-of-place device packer (woq_pack_device) on the same input."""
    import torch

    import synthetic
    import weight_only_quantised_gb300 as woq
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_peak()
    rows = []
    for bits, name, (K, N) in [(4, "gate_up", synthetic.LINEARS_27B["gate_up"]), (4, "lm_head", synthetic.LM_HEAD_27B),
                               (6, "gate_up", synthetic.LINEARS_27B["gate_up"])]:
        w, s = synthetic.weights(bits, N, K, seed=9, device=dev)
        nbytes = woq.woq_packed_bytes(bits, N, K)
        buf = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
        ref = torch.empty_like(buf)
        algo = w.numel() + 2 * s.numel() + nbytes  # canonical bytes read + packed bytes written
        times = {"relayout_inplace": [], "pack_device": []}
        for it in range(args.warmup + max(3, min(args.steps, 10))):
            woq.canonical_into_buffer(bits, w, s.view(torch.int16), buf)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            woq.woq_relayout_inplace(bits, buf, N, K)
            b.record()
            torch.cuda.synchronize()
            c, d = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c.record()
            woq.woq_pack_device(bits, w, s.view(torch.int16), N, K, ref)
            d.record()
            torch.cuda.synchronize()
            if it >= args.warmup:
                times["relayout_inplace"].append(a.elapsed_time(b))
                times["pack_device"].append(c.elapsed_time(d))
        assert torch.equal(buf, ref), "relayout differs from the device packer"
        row = {"matrix": f"27B {name} int{bits} (N={N}, K={K})", "algorithmic_bytes": algo}
        for key, v in times.items():
            ms = float(statistics.median(v))
            row[key] = {"ms": round(ms, 4), "gbs": round(algo / (ms * 1e-3) / 1e9, 1),
                        "frac": round(algo / (ms * 1e-3) / 1e9 / peak, 4)}
        rows.append(row)
        del w, s, buf, ref
        torch.cuda.empty_cache()
    print(json.dumps({"metric": "in-place relayout throughput", "unit": "GB/s", "higher_is_better": True,
                      "peak": peak, "peak_kind": peak_kind, "rows": rows,
                      "note": "median over calls; woq_relayout_inplace includes its header memset and "
                              "read-back; pack_device writes into a second buffer"}), flush=True)


def main():
    args = parse_args()
    if args.tree_planner:
        run_tree_planner(args)
        return
    if args.relayout:
        run_relayout(args)
        return
    if args.linear:
        run_linear(args)
        return
    if args.suite:
        run_suite(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

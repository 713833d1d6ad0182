#!/usr/bin/env python3
"""MoE layer forward benchmark on GB300 (prints ONE JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extras]

A step is one whole MoE layer forward (route -> metadata -> dispatch
gather -> w13 GEMM + activation -> w2 GEMM + gate scale + scatter ->
combine) through the C ABI, on synthetic seeded inputs already resident in
HBM. Default workload: the GPT-OSS-shaped prefill (8192 tokens, hidden
2880, 32 experts, top-4, intermediate 2880, SwiGLU-OAI, interleaved w13).

value        tokens/s over all ranks (each rank runs its own batch: weak scaling)
roofline     the stage with the largest device time, algorithmic FLOPs or
             bytes per launch / its mean CUDA-event duration, against the
             measured peak in MEASURED_PEAKS.json ("ffn": both expert
             contractions, where they run as one launch)
e2e          the same metric with host (pinned) buffers: x and logits copied
             host->device and the output device->host inside the timed region
cpu_baseline the CPU oracle timed on this host's cores on a bounded sample
also         routing + metadata us/call at 16384 tokens (E = 128 and 32, top-4) and
             the MiniMind-shaped layer (E = 4, 16), timed by CUDA-graph replay
             (their steps are too short for eager launches to keep the GPU busy)

--impl reference times the CPU oracle (the reference for this method) on
the same workload and prints its line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))

import numpy as np  # noqa: E402

import moe_inputs as I  # noqa: E402

METRIC = "MoE-layer tokens/s and routing-metadata µs/call on 1 GB300; % of roofline"
WORKLOADS = {
    "gptoss_prefill_n8192": I.GPTOSS.with_n(8192),
    "gptoss_prefill_n2048": I.GPTOSS.with_n(2048),
    "gptoss_prefill_n4096": I.GPTOSS.with_n(4096),
    "minimind_e4": I.MINIMIND_E4,
    "minimind_e8": I.MINIMIND_E8,
    "minimind_e16": I.MINIMIND_E16,
    "skewed_n16384": I.SKEWED,
    "gptoss_decode_n1": I.GPTOSS.with_n(1),
    "gptoss_decode_n8": I.GPTOSS.with_n(8),
    "gptoss_decode_n64": I.GPTOSS.with_n(64),
}
DEFAULT_WORKLOAD = "gptoss_prefill_n8192"
# routing-only workloads (--profile-only): one moe_route_metadata call per step
ROUTING_WORKLOADS = {"routing_n16384_e128": (16384, 128, 4), "routing_n16384_e32": (16384, 32, 4)}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------- setup --
def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(ROUTING_WORKLOADS),
                   default=DEFAULT_WORKLOAD)
    p.add_argument("--no-extras", action="store_true", help="skip the routing / MiniMind extras")
    p.add_argument("--ffn-kernel", choices=["auto", "tiled", "swap"], default="auto",
                   help="grouped-GEMM kernel of the expert FFN (auto: by batch size)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile-only", action="store_true",
                   help="only the warm-up and timed steps (for ncu): no e2e, extras, "
                        "CPU baseline or clock sampling")
    a = p.parse_args()
    a.warmup = max(a.warmup, 3)
    return a


def dist_setup(args):
    """One process per GPU under torchrun (RANK / LOCAL_RANK / WORLD_SIZE /
    MASTER_* from the environment). NCCL for the GPU arm; gloo for the CPU
    reference arm and wherever no GPU is visible (the multi-rank CPU tests)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch
        import torch.distributed as dist
        use_nccl = args.impl == "ours" and torch.cuda.is_available()
        if use_nccl:
            torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl" if use_nccl else "gloo")
        pg = dist
    return rank, world, local, pg


def max_over_ranks(pg, value: float) -> float:
    """The slowest rank's value (every rank gets it); value itself when alone."""
    if pg is None:
        return value
    import torch
    on_gpu = pg.get_backend() == "nccl"
    t = torch.tensor([value], dtype=torch.float64,
                     device=torch.device("cuda", torch.cuda.current_device()) if on_gpu else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def rank_case(c: I.LayerCase, rank: int, r: int) -> I.LayerCase:
    """Token set r of rank `rank`: every rank draws its own batches (weak
    scaling: per-rank work is fixed, ranks never exchange data)."""
    return dataclasses.replace(c, seed=c.seed + 1000 * rank + r)


def job_tokens_per_s(world: int, n: int, ms_per_step: float) -> float:
    """Whole-job throughput: all ranks' tokens over the slowest rank's step."""
    return world * n / (ms_per_step * 1e-3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, \
            "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms in the background."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        rows = self.samples
        if self.window:
            inside = [r for t, r in rows if self.window[0] <= t <= self.window[1]]
            rows_used = inside if inside else [r for _, r in rows]
        else:
            rows_used = [r for _, r in rows]
        if not rows_used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows_used if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows_used if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows_used for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows_used)}


def workload_config(c: I.LayerCase, world: int) -> dict:
    """The workload a line is measured on (both arms print the same dict)."""
    return {"workload": c.name, "n_tokens": c.n, "hidden": c.H, "n_experts": c.E,
            "topk": c.k, "intermediate": c.I, "gating": c.gating, "activation": c.act,
            "w13_layout": c.layout,
            "l2": "inputs of consecutive steps exceed L2 (rotated input sets)",
            "parallelism": f"replicas x{world} (token batches per rank)"}


# ---------------------------------------------------------- algorithmic --
def stage_work(c: I.LayerCase, touched: float = None, pk: dict = None) -> dict:
    """Algorithmic work of one launch of each stage kernel: ("hbm", bytes) or
    ("tensor", FLOPs). A contraction is bound by whichever of its FLOPs (at
    the bf16 peak) and its bytes (at the HBM peak) takes longer; its bytes
    are the weights of the `touched` experts (those that receive a slot)
    plus its activations in and out."""
    n, E, k, H, Idim = c.n, c.E, c.k, c.H, c.I
    N = n * k
    touched = E if touched is None else touched
    ffn1_bytes = touched * 2 * Idim * H * 2 + N * H * 2 + N * Idim * 2
    ffn2_bytes = touched * H * Idim * 2 + N * Idim * 2 + N * H * 2 + N * (4 + 2)
    ffn1_flops, ffn2_flops = 2.0 * N * H * 2 * Idim, 2.0 * N * Idim * H

    def contraction(flops, nbytes):
        if pk is not None and nbytes / (pk["hbm_gbs"] * 1e9) > flops / (pk["bf16_tflops"] * 1e12):
            return ("hbm", nbytes)
        return ("tensor", flops)

    return {
        "route": ("hbm", n * E * 4 + N * (4 + 2)),
        "metadata": ("hbm", N * (4 + 2) + N * (4 + 4 + 2) + (2 * E + 1) * 4),
        "gather": ("hbm", n * H * 2 + N * H * 2),
        "ffn1": contraction(ffn1_flops, ffn1_bytes),
        "ffn2": contraction(ffn2_flops, ffn2_bytes),
        # both contractions as one launch (moe_ffn_plan's "fused")
        "ffn": contraction(ffn1_flops + ffn2_flops, ffn1_bytes + ffn2_bytes),
        "combine": ("hbm", (N * H * 2 + n * H * 2) if k > 1 else 0),
    }


def dominant_stage(stage_ms: dict, fused: bool):
    """The stage kernel with the largest device time, and that time. Where
    both contractions run in one launch, the ffn1 stage's events bracket
    that launch (ffn2's bracket nothing): they count as one kernel, "ffn"."""
    ms = dict(stage_ms)
    if fused:
        ms["ffn"] = ms.pop("ffn1") + ms.pop("ffn2")
    dom = max(ms, key=ms.get)
    return dom, ms[dom]


def touched_experts(dc) -> float:
    """Mean number of experts that receive at least one slot over the case's
    token sets, read back from the library's own routing (untimed)."""
    import torch
    import mixture_experts_routing_warp_gb300 as moe
    c = dc.c
    counts = []
    for lg in dc.logits:
        _, _, meta = moe.route_metadata(lg, c.k, gating=c.gating, ws=dc.ws)
        counts.append(int((meta["col_sum"] > 0).sum().item()))
    torch.cuda.synchronize()
    return float(np.mean(counts))


def roofline_entry(bound, work, seconds, pk, source, sustained=False):
    """achieved = algorithmic work per launch / mean launch time. A tensor
    kernel timed inside a long loop of steps (power cap engaged) is set
    against the measured sustained bf16 peak, one timed in short bursts
    against the burst peak; frac_of_burst is given either way."""
    if bound == "tensor":
        achieved = work / seconds / 1e12
        peak = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
        return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "frac_of_burst": round(achieved / pk["bf16_tflops"], 4),
                "peak_source": f"{'bf16_tflops_sustained' if sustained else 'bf16_tflops'} "
                               f"({source}, {'sustained' if sustained else 'burst'})"}
    achieved = work / seconds / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / pk["hbm_gbs"], 4), "peak_source": f"hbm_gbs ({source})"}


# The sources that define each stage's kernel (its file and the headers it
# includes): a committed ncu figure stays valid while these are unchanged.
STAGE_SOURCES = {
    "ffn1": ("grouped_gemm_swap.cu", "tc_ptx.cuh", "moe_internal.cuh"),
    "ffn2": ("grouped_gemm_swap.cu", "tc_ptx.cuh", "moe_internal.cuh"),
    "ffn": ("grouped_gemm_swap.cu", "tc_ptx.cuh", "moe_internal.cuh"),
}


def kernel_source_digest(stage: str = None) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixture_experts_routing_warp_gb300", "csrc")
    names = STAGE_SOURCES.get(stage) or sorted(n for n in os.listdir(csrc)
                                               if n.endswith((".cu", ".cuh")))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(stage: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(f"{workload}:{stage}")
    if not ent or ent.get("source_digest") != kernel_source_digest(stage):
        return None
    return ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------ GPU arm --
class DeviceCase:
    """A workload's inputs on the device, with R rotated (x, logits) sets and
    W rotated weight sets so that the inputs of consecutive steps exceed L2."""

    def __init__(self, c: I.LayerCase, device, l2_bytes: int, rank: int = 0, weights=None,
                 ffn_kernel: str = "auto"):
        import torch
        import mixture_experts_routing_warp_gb300 as moe

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
                torch.bfloat16).to(device)

        self.c = c
        weights_bytes = 2 * c.E * 3 * c.H * c.I
        act_bytes = c.n * c.H * 2 + c.n * c.E * 4
        self.n_wsets = max(1, min(16, -(-2 * l2_bytes // max(weights_bytes, 1))))
        self.n_xsets = max(2, min(8, -(-2 * l2_bytes // max(act_bytes, 1))))
        self.x, self.logits, self.host_x, self.host_logits = [], [], [], []
        for r in range(self.n_xsets):
            cr = rank_case(c, rank, r)
            hx = I.layer_x(cr)
            hl = I.layer_logits(cr, hx)
            self.x.append(bf16(hx))
            self.logits.append(torch.from_numpy(hl).to(device))
            self.host_x.append(torch.from_numpy(hx.view(np.int16)).view(torch.bfloat16)
                               .pin_memory())
            self.host_logits.append(torch.from_numpy(hl).pin_memory())
        self.w13, self.w2 = [], []
        if weights is not None:  # another case's weight sets (same E, H, I)
            self.n_wsets = weights.n_wsets
            self.w13, self.w2 = weights.w13, weights.w2
        for r in range(len(self.w13), self.n_wsets):
            cw = dataclasses.replace(c, seed=c.seed + r)
            self.w13.append(bf16(I.all_w13(cw)))
            self.w2.append(bf16(I.all_w2(cw)))
        self.params = moe.make_params(c.gating, c.act, c.layout, ffn_kernel=ffn_kernel)
        self.ws = moe.workspace(c.n, c.E, c.k, c.H, c.I, device)
        self.out = torch.empty((c.n, c.H), dtype=torch.bfloat16, device=device)
        self.host_out = torch.empty((c.n, c.H), dtype=torch.bfloat16).pin_memory()

    def args(self, i):
        return (self.x[i % self.n_xsets], self.logits[i % self.n_xsets],
                self.w13[i % self.n_wsets], self.w2[i % self.n_wsets])


def time_layer(dc: DeviceCase, steps, warmup, pg, sampler=None, timed_stages=True):
    import torch
    import mixture_experts_routing_warp_gb300 as moe
    c = dc.c
    S = len(moe.STAGES)
    for i in range(warmup):
        moe.forward(*dc.args(i), c.k, dc.params, dc.ws, out=dc.out)
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(S + 1)] for _ in range(steps)]
    for ev in events:   # torch creates each CUDA event on its first record
        for e in ev:
            e.record()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record()
    for i in range(steps):
        if timed_stages:
            moe.forward_timed(*dc.args(warmup + i), c.k, dc.params, dc.ws, events[i], out=dc.out)
        else:
            moe.forward(*dc.args(warmup + i), c.k, dc.params, dc.ws, out=dc.out)
    end.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if pg is not None:
        pg.barrier()
    if sampler is not None:
        sampler.mark(t0, t1)
    total_ms = start.elapsed_time(end)
    stage_ms = None
    if timed_stages:
        stage_ms = {name: sum(ev[j].elapsed_time(ev[j + 1]) for ev in events) / steps
                    for j, name in enumerate(moe.STAGES)}
    status = moe.read_status(dc.ws)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    return total_ms, stage_ms


def time_e2e(dc: DeviceCase, steps, warmup):
    """Same forward with host buffers: H2D x + logits, forward, D2H out."""
    import torch
    import mixture_experts_routing_warp_gb300 as moe
    c = dc.c
    xd = torch.empty_like(dc.x[0])
    ld = torch.empty_like(dc.logits[0])

    def step(i):
        j = i % dc.n_xsets
        xd.copy_(dc.host_x[j], non_blocking=True)
        ld.copy_(dc.host_logits[j], non_blocking=True)
        moe.forward(xd, ld, dc.w13[i % dc.n_wsets], dc.w2[i % dc.n_wsets], c.k, dc.params, dc.ws,
                    out=dc.out)
        dc.host_out.copy_(dc.out, non_blocking=True)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(steps):
        step(warmup + i)
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    h2d = dc.host_x[0].numel() * 2 + dc.host_logits[0].numel() * 4
    d2h = dc.host_out.numel() * 2
    return ms, h2d, d2h


def time_e2e_pipelined(dc: DeviceCase, steps, warmup):
    """The same calls with the copies on their own streams, as a serving
    loop would run them: step i's H2D (x, logits) on one stream, its forward
    on a second, its D2H (out) on a third, two device buffer sets, events
    ordering each step's copies against its forward and the buffer reuse two
    steps later. Every step still copies its inputs in and its result out
    inside the timed region; the copies of neighbouring steps overlap the
    forward. Returns ms per step."""
    import torch
    import mixture_experts_routing_warp_gb300 as moe
    c = dc.c
    slots = 2
    xd = [torch.empty_like(dc.x[0]) for _ in range(slots)]
    ld = [torch.empty_like(dc.logits[0]) for _ in range(slots)]
    od = [torch.empty_like(dc.out) for _ in range(slots)]
    host_out = [dc.host_out] + [torch.empty_like(dc.host_out).pin_memory()
                                for _ in range(slots - 1)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(slots)]
    comp_done = [torch.cuda.Event() for _ in range(slots)]
    out_done = [torch.cuda.Event() for _ in range(slots)]
    for e in comp_done + out_done:   # recorded once so that the first waits are no-ops
        e.record()

    def step(i):
        b, j = i % slots, i % dc.n_xsets
        with torch.cuda.stream(s_in):
            s_in.wait_event(comp_done[b])        # slot b's inputs no longer read
            xd[b].copy_(dc.host_x[j], non_blocking=True)
            ld[b].copy_(dc.host_logits[j], non_blocking=True)
            in_done[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_done[b])
            s_comp.wait_event(out_done[b])       # slot b's output already copied out
            moe.forward(xd[b], ld[b], dc.w13[i % dc.n_wsets], dc.w2[i % dc.n_wsets], c.k,
                        dc.params, dc.ws, out=od[b])
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            host_out[b].copy_(od[b], non_blocking=True)
            out_done[b].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    start.record(cur)
    for s_ in (s_in, s_comp, s_out):
        s_.wait_stream(cur)
    for i in range(steps):
        step(warmup + i)
    for s_ in (s_in, s_comp, s_out):
        cur.wait_stream(s_)
    end.record(cur)
    torch.cuda.synchronize()
    if moe.read_status(dc.ws) != 0:
        raise RuntimeError("device status after the end-to-end loop")
    return start.elapsed_time(end) / steps


def graph_time_ms(fn, reps: int, replays: int = 5) -> float:
    """Capture reps calls of fn(i) in one CUDA graph, replay it, and return
    the device time per call (median over replays)."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(3):
            fn(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(replays):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / reps)
    del g
    return float(np.median(times))


def time_route_gemm(n, E, H, k, device, l2_bytes, pk, source):
    """moe_route_gemm (router matmul x . w_gate^T with the top-k in its
    epilogue, logits never written) per call: CUDA-graph replays, x rotated
    over more than 2 x L2. Bound: x's bytes (a small GEMM: 2nHE FLOP)."""
    import torch
    import mixture_experts_routing_warp_gb300 as moe
    case = I.LayerCase("router", n=n, H=H, E=E, k=k, I=64)
    sets = max(2, min(16, -(-2 * l2_bytes // (n * H * 2))))

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(
            device)

    xs = [bf16(I.layer_x(dataclasses.replace(case, seed=s))) for s in range(sets)]
    wg = bf16(I.router_weight(case))
    indx = torch.empty((n, k), dtype=torch.int32, device=device)
    vals = torch.empty((n, k), dtype=torch.bfloat16, device=device)
    ws = moe.workspace(n, E, k, 64, 64, device)
    L = moe.lib()

    def call(i):
        L.moe_route_gemm(xs[i % sets].data_ptr(), wg.data_ptr(), n, E, H, k, 0, indx.data_ptr(),
                         vals.data_ptr(), None, ws.data_ptr(), ws.numel(),
                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))

    ms = graph_time_ms(call, 2 * sets)
    assert moe.read_status(ws) == 0
    alg = n * H * 2 + E * H * 2 + n * k * 6
    return {"workload": f"moe_route_gemm n{n} E{E} H{H} k{k} (x rotated over {sets} sets; "
                        f"CUDA-graph replay of {2 * sets} calls)",
            "us_per_call": round(ms * 1e3, 3), "algorithmic_bytes": alg,
            "roofline": roofline_entry("hbm", alg, ms * 1e-3, pk, source),
            "tflops": round(2.0 * n * H * E / (ms * 1e-3) / 1e12, 2)}


def time_routing(n, E, k, device, l2_bytes, pk, source):
    """moe_route + moe_build_metadata per call: CUDA-graph replays of back-to-
    back calls (so host launch overhead is not counted), logits rotated over
    more than 2 x L2."""
    import torch
    import mixture_experts_routing_warp_gb300 as moe
    sets = max(2, min(64, -(-2 * l2_bytes // (n * E * 4))))
    logits = [torch.from_numpy(I.route_logits(n, E, seed=s)).to(device) for s in range(sets)]
    indx = torch.empty((n, k), dtype=torch.int32, device=device)
    vals = torch.empty((n, k), dtype=torch.bfloat16, device=device)
    ws = moe.workspace(n, E, k, 64, 64, device)
    meta = moe.empty_meta(n * k, E, device)
    L = moe.lib()
    ms = moe._binding._meta_struct(meta)

    def stream():
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def route(i):
        L.moe_route(logits[i % sets].data_ptr(), n, E, k, 0, indx.data_ptr(), vals.data_ptr(),
                    stream())

    def metadata(i):
        L.moe_build_metadata(indx.data_ptr(), vals.data_ptr(), n, E, k, ctypes.byref(ms),
                             ws.data_ptr(), ws.numel(), stream())

    def fused(i):
        L.moe_route_metadata(logits[i % sets].data_ptr(), n, E, k, 0, indx.data_ptr(),
                             vals.data_ptr(), ctypes.byref(ms), ws.data_ptr(), ws.numel(),
                             stream())

    reps = 2 * sets
    route_ms = graph_time_ms(route, reps)
    both_ms = graph_time_ms(fused, reps)
    meta_ms = graph_time_ms(metadata, reps)   # same indices each call (L2-warm input)
    assert moe.read_status(ws) == 0
    total_us = both_ms * 1e3
    w = stage_work(I.LayerCase("routing", n=n, H=64, E=E, k=k, I=64))
    alg = n * E * 4 + n * k * (4 + 2 + 4 + 4 + 2) + (2 * E + 1) * 4
    return {"workload": f"moe_route_metadata n{n} E{E} k{k} (fp32 N(0,1) logits, {sets} "
                        f"rotated sets; CUDA-graph replay of {reps} calls)",
            "us_per_call": round(total_us, 3), "route_us": round(route_ms * 1e3, 3),
            "metadata_us_warm_input": round(meta_ms * 1e3, 3), "algorithmic_bytes": alg,
            "achieved_gbs": round(alg / (total_us * 1e-6) / 1e9, 1),
            "frac_of_hbm": round(alg / (total_us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
            "frac_of_8tbs": round(alg / (total_us * 1e-6) / 8e12, 4),
            "route_roofline": roofline_entry("hbm", w["route"][1], route_ms * 1e-3, pk, source)}


def time_layer_graph(dc, reps, pk, source):
    """Whole-layer steps replayed from a CUDA graph (stage events captured as
    event-record nodes): for workloads whose step is too short for eager
    launches to keep the GPU busy."""
    import torch
    import mixture_experts_routing_warp_gb300 as moe
    c = dc.c
    S = len(moe.STAGES)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(S + 1)] for _ in range(reps)]
    for ev in events:
        for e in ev:
            e.record()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(3):
            moe.forward(*dc.args(i), c.k, dc.params, dc.ws, out=dc.out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            moe.forward_timed(*dc.args(i), c.k, dc.params, dc.ws, events[i], out=dc.out)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    total_events_ms = a.elapsed_time(b) / reps
    # the same steps without event-record nodes: the step time reported
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        for i in range(reps):
            moe.forward(*dc.args(i), c.k, dc.params, dc.ws, out=dc.out)
    g2.replay()
    torch.cuda.synchronize()
    a.record()
    g2.replay()
    b.record()
    torch.cuda.synchronize()
    total_ms = a.elapsed_time(b) / reps
    del g2
    stage_ms = {name: sum(ev[j].elapsed_time(ev[j + 1]) for ev in events) / reps
                for j, name in enumerate(moe.STAGES)}
    assert moe.read_status(dc.ws) == 0
    touched = touched_experts(dc)
    work = stage_work(c, touched, pk)
    dom, dom_ms = dominant_stage(stage_ms, moe.ffn_plan(c.n, c.E, c.k, c.H, c.I, dc.params)["fused"])
    roof = roofline_entry(work[dom][0], work[dom][1], dom_ms * 1e-3, pk, source)
    roof["kernel"] = dom
    roof["touched_experts"] = touched
    del g
    return {"workload": c.name, "tokens_per_s": round(c.n / (total_ms * 1e-3), 1),
            "ms_per_step": round(total_ms, 4), "timing": f"CUDA-graph replay of {reps} steps",
            "ms_per_step_with_stage_events": round(total_events_ms, 4),
            "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()}, "roofline": roof}


# ------------------------------------------------------------ CPU arm --
def oracle_inputs(c: I.LayerCase) -> dict:
    hx = I.layer_x(c)
    return {"x": hx, "logits": I.layer_logits(c, hx), "w13": I.all_w13(c), "w2": I.all_w2(c)}


def oracle_sample(c: I.LayerCase, d: dict, budget_s: float = 12.0, max_tokens: int = 4096):
    """Time the CPU oracle on a bounded sample of the workload: routing and
    metadata over all n tokens plus the FFN and combine on the first m tokens,
    m grown until about budget_s of CPU work. Returns the layer's tokens/s
    (routing + metadata time prorated per token)."""
    import oracle
    t = time.perf_counter()
    indx, vals = oracle.route(d["logits"], c.k, c.gating)
    oracle.metadata(indx, vals, c.E)
    route_meta_s = time.perf_counter() - t
    m, spent = 8, 0.0
    while True:
        toks = np.arange(min(m, c.n), dtype=np.int64)
        t = time.perf_counter()
        oracle.ffn(d["x"], indx, vals, d["w13"], d["w2"], tokens=toks, act=c.act,
                   layout=c.layout)
        dt = time.perf_counter() - t
        spent += dt
        rate = 1.0 / (dt / toks.size + route_meta_s / c.n)
        if dt >= budget_s * 0.4 or toks.size >= min(c.n, max_tokens) or spent >= budget_s:
            break
        m = int(min(c.n, max_tokens, max(2 * m, toks.size * budget_s * 0.5 / max(dt, 1e-3))))
    return {"value": round(rate, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
            "affinity_cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"route+metadata over all {c.n} tokens, FFN+combine over the first "
                      f"{toks.size} tokens ({dt:.1f} s); float64 C oracle, OpenMP over tokens",
            "ffn_tokens": int(toks.size), "sample_s": round(route_meta_s + dt, 3)}


def oracle_sample_with_output(c: I.LayerCase, d: dict, budget_s: float = 12.0,
                              max_tokens: int = 4096):
    """oracle_sample, plus the oracle's layer output for the first m tokens
    (recomputed untimed) so that the GPU's output can be checked against it."""
    import oracle
    rec = oracle_sample(c, d, budget_s, max_tokens)
    m = rec["ffn_tokens"]
    indx, vals = oracle.route(d["logits"], c.k, c.gating)
    toks = np.arange(m, dtype=np.int64)
    ref = oracle.ffn(d["x"], indx, vals, d["w13"], d["w2"], tokens=toks, act=c.act,
                     layout=c.layout)
    return rec, toks, ref


def parity_vs_oracle(got_bits: np.ndarray, ref_bits: np.ndarray) -> dict:
    """|gpu - ref| <= 3e-2 + 2e-2 |ref| elementwise, cosine > 0.99 and relative
    L2 <= 1e-2 over the sampled rows (the tolerance the parity tests use)."""
    def f64(b):
        return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(
            np.float32).astype(np.float64)
    got, ref = f64(got_bits), f64(ref_bits)
    err = np.abs(got - ref)
    nref = float(np.linalg.norm(ref))
    cos = float(np.dot(got.ravel(), ref.ravel()) / (np.linalg.norm(got) * nref)) if nref else 0.0
    rel = float(np.linalg.norm(got - ref) / nref) if nref else 0.0
    n_bad = int((err > 3e-2 + 2e-2 * np.abs(ref)).sum())
    return {"rows": int(got.shape[0]), "max_abs": float(err.max()) if err.size else 0.0,
            "cos": round(cos, 6), "rel_l2": rel, "n_bad": n_bad,
            "ok": bool(n_bad == 0 and cos > 0.99 and rel <= 1e-2)}


def run_reference(args, rank, world, pg):
    if rank != 0:
        return 0
    c = WORKLOADS[args.workload]
    d = oracle_inputs(c)
    budget = max(1.0, 90.0 / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        oracle_sample(c, d, budget_s=budget, max_tokens=64)
    steps_v, steps_s = [], []
    t0 = time.time()
    for i in range(args.steps):
        t = time.perf_counter()
        r = oracle_sample(c, d, budget_s=budget, max_tokens=512)
        steps_s.append(time.perf_counter() - t)
        steps_v.append(r["value"])
    wall = time.time() - t0
    value = float(np.median(steps_v))
    # a step is one bounded sample of the workload (routing of every token,
    # the FFN of the first tokens); ms_per_step is the time such a step took
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * float(np.mean(steps_s)), 1),
            "step": "one bounded sample of the workload (see cpu_baseline.sample)",
            "ms_per_layer_extrapolated": round(1e3 * c.n / value, 1) if value else None,
            "extrapolated": True,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(c, world),
            "l2_note": "CPU run: the GPU arm's input rotation does not apply",
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "kind": "oracle",
                             "cores": r["cores"], "affinity_cores": r["affinity_cores"],
                             "sample": r["sample"]},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0, "wall_s": round(wall, 1)}
    print(json.dumps(line), flush=True)
    return 0


def profile_routing(args, device, l2):
    """--profile-only on a routing workload: warm-up + timed moe_route_metadata calls."""
    import torch
    import mixture_experts_routing_warp_gb300 as moe
    n, E, k = ROUTING_WORKLOADS[args.workload]
    sets = max(2, min(64, -(-2 * l2 // (n * E * 4))))
    logits = [torch.from_numpy(I.route_logits(n, E, seed=s)).to(device) for s in range(sets)]
    ws = moe.workspace(n, E, k, 64, 64, device)
    meta = moe.empty_meta(n * k, E, device)
    topk = (torch.empty((n, k), dtype=torch.int32, device=device),
            torch.empty((n, k), dtype=torch.bfloat16, device=device))
    for i in range(args.warmup + args.steps):
        moe.route_metadata(logits[i % sets], k, ws=ws, meta=meta, topk=topk)
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    print(json.dumps({"profile_only": True, "workload": args.workload}), flush=True)
    return 0


def run_ours(args, rank, world, local, pg):
    import torch
    import mixture_experts_routing_warp_gb300 as moe
    moe.lib()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or 132 * 1024 * 1024)
    pk, source = peaks()
    if args.workload in ROUTING_WORKLOADS:
        if not args.profile_only:
            raise SystemExit("routing workloads are for --profile-only runs")
        return profile_routing(args, device, l2)
    c = WORKLOADS[args.workload]
    dc = DeviceCase(c, device, l2, rank, ffn_kernel=args.ffn_kernel)
    if args.profile_only:
        total_ms, _ = time_layer(dc, args.steps, args.warmup, pg, None, timed_stages=False)
        if rank == 0:
            print(json.dumps({"profile_only": True, "workload": c.name,
                              "ms_per_step": round(total_ms / args.steps, 4)}), flush=True)
        return 0
    sampler = ClockSampler(local)
    sampler.start()
    total_ms, stage_ms = time_layer(dc, args.steps, args.warmup, pg, sampler)
    sampler.stop()
    total_ms = max_over_ranks(pg, total_ms)
    ms_per_step = total_ms / args.steps
    value = job_tokens_per_s(world, c.n, ms_per_step)
    touched = touched_experts(dc)
    work = stage_work(c, touched, pk)
    dom, dom_ms = dominant_stage(stage_ms, moe.ffn_plan(c.n, c.E, c.k, c.H, c.I, dc.params)["fused"])
    bound, w = work[dom]
    roof = roofline_entry(bound, w, dom_ms * 1e-3, pk, source, sustained=total_ms > 100.0)
    roof["kernel"] = dom
    roof["touched_experts"] = touched
    # the committed counters are of the swap-operand kernel (the default)
    roof["traffic"] = ncu_traffic(dom, args.workload) if args.ffn_kernel != "tiled" else None
    kernels_per_step = moe.forward_launch_count(c.n, c.E, c.k, c.H, c.I)
    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded numpy PCG64, N(0,1) tokens, N(0,0.02) weights)",
            "config": workload_config(c, world),
            "ffn_kernel": args.ffn_kernel,
            "l2_sets": {"token_sets": dc.n_xsets, "weight_sets": dc.n_wsets,
                        "how": "x / logits and the weights rotated so that consecutive steps' "
                               "inputs total more than 2x L2"},
            "roofline": roof,
            "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
            "gpu_launches": kernels_per_step * args.steps,
            "clocks": sampler.summary()}
    if rank == 0:
        e2e_steps = max(3, min(args.steps, 50))
        serial_ms, h2d, d2h = time_e2e(dc, e2e_steps, args.warmup)
        e2e_ms = time_e2e_pipelined(dc, e2e_steps, args.warmup)
        line["e2e"] = {"value": round(job_tokens_per_s(world, c.n, e2e_ms), 1),
                       "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                       "how": "moe.forward from pinned host buffers: per step H2D x + logits, "
                              "forward, D2H out; copies on their own streams, overlapping the "
                              "neighbouring steps' forwards (2 buffer sets)",
                       "serial": {"value": round(job_tokens_per_s(world, c.n, serial_ms), 1),
                                  "ms_per_step": round(serial_ms, 4),
                                  "how": "the same three operations back to back on one stream"}}
        if not args.no_extras:
            also = {"routing_metadata_16k_e128": time_routing(16384, 128, 4, device, l2, pk,
                                                              source),
                    "router_gemm_topk_n8192_e32_h2880": time_route_gemm(8192, 32, 2880, 4,
                                                                        device, l2, pk, source),
                    "routing_metadata_16k_e32": time_routing(16384, 32, 4, device, l2, pk,
                                                             source)}
            for name in ("minimind_e4", "minimind_e8", "minimind_e16"):
                if WORKLOADS[name] != c:
                    mm = DeviceCase(WORKLOADS[name], device, l2)
                    also[name] = time_layer_graph(mm, 64, pk, source)
                    del mm
            if (c.E, c.H, c.I) == (I.GPTOSS.E, I.GPTOSS.H, I.GPTOSS.I):
                for nd in I.GPTOSS_DECODE_N:  # decode batches on the same weights
                    for fk in ("auto", "tiled"):
                        cd = DeviceCase(I.GPTOSS.with_n(nd), device, l2, weights=dc,
                                        ffn_kernel=fk)
                        key = f"gptoss_decode_n{nd}" + ("" if fk == "auto" else "_tiled")
                        also[key] = time_layer_graph(cd, 64, pk, source)
                        del cd
                if c.n != 2048:
                    cp = DeviceCase(I.GPTOSS.with_n(2048), device, l2, weights=dc)
                    also["gptoss_prefill_n2048"] = time_layer_graph(cp, 32, pk, source)
                    del cp
            if WORKLOADS["skewed_n16384"] != c:
                del dc.w13, dc.w2   # make room for the 128 experts' weights
                torch.cuda.empty_cache()
                sk = DeviceCase(WORKLOADS["skewed_n16384"], device, l2)
                also["skewed_n16384"] = time_layer_graph(sk, 16, pk, source)
                del sk
                torch.cuda.empty_cache()
            also["host_sync_roundtrip_us"] = host_sync_roundtrip_us(device)
            line["also"] = also
        if not args.no_cpu_baseline:
            rec, toks, ref = oracle_sample_with_output(c, oracle_inputs(c))
            line["cpu_baseline"] = rec
        else:
            import oracle
            d0 = oracle_inputs(c)
            toks = np.arange(min(c.n, 64), dtype=np.int64)
            ix, vx = oracle.route(d0["logits"], c.k, c.gating)
            ref = oracle.ffn(d0["x"], ix, vx, d0["w13"], d0["w2"], tokens=toks, act=c.act,
                             layout=c.layout)
        line["parity"] = check_timed_output(c, device, l2, toks, ref, args.ffn_kernel)
        print(json.dumps(line), flush=True)
        if not line["parity"]["ok"]:
            log(f"parity against the oracle failed: {line['parity']}")
            return 1
    return 0


def host_sync_roundtrip_us(device, reps: int = 100) -> dict:
    """What one device->host synchronisation costs on this host: a one-element
    reduction whose result the host reads (.item()), repeated; the cost a
    layer pays per readback in a loop that syncs ([P2] Measurement: the
    per-sync ruler)."""
    import torch
    flag = torch.zeros(1, dtype=torch.bool, device=device)
    for _ in range(20):
        flag.any().item()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        t = time.perf_counter()
        flag.any().item()
        ts.append(time.perf_counter() - t)
    return {"us_median": round(1e6 * float(np.median(ts)), 2),
            "us_mean": round(1e6 * float(np.mean(ts)), 2), "reps": reps,
            "syncs_per_layer_here": 0,
            "how": "1-element bool any() + .item(), 100 times after 20 warm-up calls"}


def check_timed_output(c: I.LayerCase, device, l2, toks, ref, ffn_kernel) -> dict:
    """One more forward of the benchmarked call on token set 0 / weight set 0
    (the oracle's inputs) and its first rows against the oracle's output."""
    import torch
    import mixture_experts_routing_warp_gb300 as moe
    hx = I.layer_x(c)
    x = torch.from_numpy(hx.view(np.int16)).view(torch.bfloat16).to(device)
    lg = torch.from_numpy(I.layer_logits(c, hx)).to(device)
    w13 = torch.from_numpy(I.all_w13(c).view(np.int16)).view(torch.bfloat16).to(device)
    w2 = torch.from_numpy(I.all_w2(c).view(np.int16)).view(torch.bfloat16).to(device)
    params = moe.make_params(c.gating, c.act, c.layout, ffn_kernel=ffn_kernel)
    ws = moe.workspace(c.n, c.E, c.k, c.H, c.I, device)
    out = moe.forward(x, lg, w13, w2, c.k, params, ws)
    torch.cuda.synchronize()
    status = moe.read_status(ws)
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)[toks]
    rec = parity_vs_oracle(got, ref)
    rec["status"] = int(status)
    rec["ok"] = rec["ok"] and status == 0
    rec["what"] = f"output rows of the first {toks.size} tokens vs the CPU oracle"
    del x, lg, w13, w2, ws, out
    torch.cuda.empty_cache()
    return rec


def main():
    args = parse_args()
    rank, world, local, pg = dist_setup(args)
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world, pg)
        return run_ours(args, rank, world, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())

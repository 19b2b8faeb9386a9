"""Benchmark of the routed INT4-expert MoE FFN on GB300.

Default workload: OLMoE-shaped decode -- 16 MoE layers, hidden 2048, 64
experts per layer, top-8 without renormalisation, expert intermediate 1024,
SwiGLU, INT4 group 128 with FP16 scale and zero point, one token per step,
all experts resident. One step = one decode token through all 16 layers:
per layer route (moe_route) then the routed expert FFN (moe_expert_forward),
each layer reading the previous layer's output.

Prints one JSON line (rank 0). Metric: MoE-layer decode tokens/s, with the
expert-weight HBM GB/s and its fraction of the measured copy bandwidth in
``roofline``. ``--impl reference`` times the CPU oracle instead.
"""
from __future__ import annotations

import os

# The CPU oracle legs run single-threaded; pin BLAS before numpy loads.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from int4_routed_expert_moe_gb300 import synth  # noqa: E402

METRIC = "MoE-layer decode tokens/s (expert-weight HBM GB/s in roofline)"
METRIC_PREFILL = "MoE-layer prefill tokens/s (tensor-core TFLOP/s in roofline)"
# DRAM bytes (read + written) per algorithmic byte of one layer call, from
# ncu captures (dram__bytes_read.sum + dram__bytes_write.sum) of the current
# kernel build on a parity-test layer of the workload's shape; the bench
# scales them by its own calls' algorithmic bytes (distinct experts x block
# bytes). A workload without an entry reports null.
DECODE_DRAM_RATIO = {
    # decode_stream_kernel, one OLMoE layer, T = 1: 26,856,960 B for 8 experts
    "olmoe_decode": 26_856_960 / 26_738_688,
    # decode_stream_kernel, 512 experts, T = 1: 16,834,304 B for 10 experts
    "large_fanout_b1": 16_834_304 / 16_711_680,
    # decode_stream_kernel, 512 experts, T = 16: 145,702,912 + 3,361,536 B for 87 experts
    "large_fanout_b16": (145_702_912 + 3_361_536) / 145_391_616,
    # grouped path, 512 experts, T = 256 (route, sort, gather, two GEMMs, combine):
    # 686,205,184 B for 377 experts
    "large_fanout_b256": 686_205_184 / 630_030_336,
}
TRAFFIC_SOURCE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of a parity-test layer of this shape "
                  "(current kernel build), scaled to this call by its distinct-expert bytes")
# Prefill: DRAM bytes of the gate/up and down grouped GEMMs of one layer call
# from an ncu capture (gate/up 159.49 MB read + 5.61 MB written, down 79.79 +
# 6.74 MB).
PREFILL_GEMM_DRAM_BYTES = 251_635_456


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="olmoe_decode",
                    choices=["olmoe_decode", "qwen_decode", "olmoe_partial", "olmoe_prefill",
                             "large_fanout_b1", "large_fanout_b16", "large_fanout_b256"])
    ap.add_argument("--graph-window", type=int, default=128)
    ap.add_argument("--policy", default="decay", choices=["decay", "lru", "pinned"],
                    help="residency victim policy (olmoe_partial, --mode copy)")
    ap.add_argument("--mode", default="copy", choices=["copy", "zerocopy"],
                    help="olmoe_partial: copy misses into slots, or read them in place over the CPU-GPU link")
    ap.add_argument("--slots", type=int, default=None, help="olmoe_partial: experts resident per layer")
    ap.add_argument("--prefetch", type=int, default=0,
                    help="olmoe_partial --mode copy: spare slots per layer filled with predicted misses")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# --------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (every 50 ms) with host timestamps."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        self.windows = []

    def mark(self):
        return time.time()

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.strip().split(", ") for r in self.f.read().splitlines() if r.strip()]
        self.f.close()
        os.unlink(self.f.name)
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        import datetime
        def ts(s):
            try:
                return datetime.datetime.strptime(s, "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None
        inside = [r for r in rows if len(r) >= 9 and ts(r[0]) is not None and t0 <= ts(r[0]) <= t1]
        used = inside if inside else [r for r in rows if len(r) >= 9]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in used if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in used if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(used), "samples_in_timed_region": len(inside)}


def smi_index():
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    first = vis.split(",")[0].strip() if vis else ""
    return first if first.isdigit() else str(torch.cuda.current_device())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback 6.8 TB/s"


def measured_tensor_peak(sustained):
    """Dense FP16 tensor peak in TFLOP/s: the measured cuBLAS bf16 figure
    (FP16 and BF16 run at the same nominal rate)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d[key]), f"measured (MEASURED_PEAKS.json {key}; fp16 = bf16 nominal rate)"
    return (1700.0, "fallback 1.7 PFLOP/s sustained") if sustained else (1900.0, "fallback 1.9 PFLOP/s")


# --------------------------------------------------------------------------
class DecodeWorkload:
    """A decode stack (OLMoE-shaped by default), resident on the device."""

    def __init__(self, moe, seed, steps_total, rank=0, name="olmoe_decode"):
        wl = synth.WORKLOADS[name]
        self.name = name
        self.moe = moe
        self.L, self.H, self.I, self.E = wl["L"], wl["H"], wl["I"], wl["E"]
        self.k, self.g, self.T, self.renorm = wl["k"], wl["g"], wl["T"], wl["renorm"]
        self.shape = (self.H, self.I, self.g)
        dev = torch.device("cuda")
        self.bb = moe.moe_expert_block_bytes(self.shape)
        assert self.bb == synth.block_layout(*self.shape)["total"]
        # One pool per layer, expert e in slot e (all resident).
        self.pool = synth.device_pool(self.L * self.E, self.H, self.I, self.g, seed + rank)
        self.slot_of = torch.arange(self.E, dtype=torch.int32, device=dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed + 1000 + rank)
        self.n = steps_total
        self.x0 = torch.randn((steps_total, self.T, self.H), generator=gen, device=dev).half()
        self.logits = torch.randn((steps_total, self.L, self.T, self.E), generator=gen, device=dev)
        self.ids = torch.empty((self.L, self.T, self.k), dtype=torch.int32, device=dev)
        self.w = torch.empty((self.L, self.T, self.k), dtype=torch.float32, device=dev)
        self.y = torch.empty((self.L, self.T, self.H), dtype=torch.float16, device=dev)
        wsb = moe.moe_forward_workspace_bytes(self.shape, self.T, self.k, self.E, moe.MOE_PATH_GEMV)
        self.ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)

    def layer_pool(self, l):
        return self.pool[l * self.E:(l + 1) * self.E]

    def step(self, s, x0=None, logits=None):
        moe = self.moe
        for l in range(self.L):
            lg = self.logits[s, l] if logits is None else logits[l]
            x = (self.x0[s] if x0 is None else x0) if l == 0 else self.y[l - 1]
            moe.moe_layer_forward(self.shape, x, lg, self.k, self.renorm, self.ids[l], self.w[l],
                                  self.layer_pool(l), self.slot_of, self.E, None, self.y[l], self.ws,
                                  moe.MOE_PATH_GEMV)

    def launches_per_step(self):
        return self.L  # one decode kernel per layer (routing inside)

    def expert_bytes_per_step(self):
        # T = 1: the k chosen experts of every layer are read once each.
        return self.L * self.k * self.bb


def timed_blocks(graph_blocks, warm_graphs, world, stream):
    """Replays the warm-up graphs, then each block of graphs bracketed by
    CUDA events on the launching stream (barrier + synchronize around the
    whole timed region). Returns (total ms, [ms per block], host t0, t1)."""
    for g in warm_graphs:
        g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(graph_blocks) + 1)]
    t_host0 = time.time()
    evs[0].record(stream)
    for i, blk in enumerate(graph_blocks):
        for g in blk:
            g.replay()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier(world)
    block_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(len(graph_blocks))]
    return sum(block_ms), block_ms, t_host0, t_host1


def split_blocks(K, n_blocks=3):
    """[(first step, steps)] of n_blocks nearly equal blocks of K steps."""
    sizes = [K // n_blocks + (1 if i < K % n_blocks else 0) for i in range(n_blocks)]
    out, s0 = [], 0
    for n in sizes:
        if n:
            out.append((s0, n))
        s0 += n
    return out


def run_ours(args, world, rank, local, name="olmoe_decode"):
    from int4_routed_expert_moe_gb300 import moe
    seed = synth.BASE_SEED + (1 if name == "olmoe_decode" else 6)
    K = args.steps or 512
    W = max(3, args.warmup if args.warmup is not None else 128)
    wl = DecodeWorkload(moe, seed, K + W, rank, name)
    stream = torch.cuda.current_stream()
    win = max(1, args.graph_window)

    wl.step(0)  # eager pass: sets up kernel attributes before capture
    torch.cuda.synchronize()

    def capture(s0, s1):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for s in range(s0, s1):
                wl.step(s)
        return g

    # Warm-up, then the timed steps as 3 blocks (the pages pool their decode
    # rate over blocks and report the spread between them), each block one or
    # more CUDA graphs of at most `win` steps.
    warm_graphs = [capture(s, min(W, s + win)) for s in range(0, W, win)]
    graph_blocks = [[capture(W + b0 + s, W + b0 + min(n, s + win)) for s in range(0, n, win)]
                    for b0, n in split_blocks(K)]
    torch.cuda.synchronize()

    sampler = ClockSampler(smi_index())
    time.sleep(0.2)
    ms, block_ms, t_host0, t_host1 = timed_blocks(graph_blocks, warm_graphs, world, stream)
    rows = sampler.stop()
    clocks = ClockSampler.summarize(rows, t_host0, t_host1)
    assert moe.moe_workspace_flags(wl.ws) == 0
    ms_max = max_over_ranks(ms, world)

    tokens = K * wl.T * world
    value = tokens / (ms_max / 1e3)
    peak, peak_src = measured_peaks()
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms_max / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded; random-init INT4 experts of the workload's shape)",
        "config": {"workload": wl.name, "layers": wl.L, "hidden": wl.H, "experts": wl.E,
                   "top_k": wl.k, "inter": wl.I, "group": wl.g, "tokens_per_step": wl.T,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "arithmetic": "INT4 weights, FP16 products (<= 8 terms), FP32 accumulation",
                   "l2": f"inputs larger than L2: {wl.expert_bytes_per_step() / 1e6:.1f} MB of expert weights "
                         f"per step from a {wl.L * wl.E * wl.bb / 1e9:.2f} GB pool",
                   "launch": f"CUDA graphs of <= {win} steps, one kernel per layer, PDL between layers"},
        "blocks": block_stats(block_ms, [n for _, n in split_blocks(K)], wl.T),
        "roofline": decode_roofline(wl, ms / K, peak, peak_src),
        "gpu_launches": wl.launches_per_step() * K,
        "clocks": clocks,
    }
    if not args.no_e2e:
        out["e2e"] = run_e2e(moe, wl, min(K, 256), W)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl)
    return out


def block_stats(block_ms, block_steps, T):
    """Rate of each timed block and the spread between blocks ((max - min) /
    pooled rate), as the pages report their decode blocks."""
    rates = [n * T / (ms / 1e3) for ms, n in zip(block_ms, block_steps)]
    pooled = sum(block_steps) * T / (sum(block_ms) / 1e3)
    return {"n": len(rates), "tokens_per_s": [round(r, 2) for r in rates],
            "spread": round((max(rates) - min(rates)) / pooled, 5) if rates else None,
            "pooled_tokens_per_s": round(pooled, 2)}


def decode_roofline(wl, step_ms, peak, peak_src):
    """Roofline of the decode kernel (one launch = one layer): the expert
    bytes a launch reads (k blocks at one token) over the launch's average
    duration in the timed region, i.e. the step time over the layers (the
    launches run back to back on one stream, so L x launch time = step time)."""
    bytes_per_launch = wl.expert_bytes_per_step() / wl.L
    launch_s = step_ms / 1e3 / wl.L
    assert wl.L * launch_s * 1e3 <= step_ms * (1 + 1e-9)
    achieved = bytes_per_launch / launch_s / 1e9
    ratio = DECODE_DRAM_RATIO.get(wl.name)
    traffic = int(round(ratio * wl.expert_bytes_per_step() / wl.L)) if ratio else None
    return {"bound": "hbm", "kernel": "decode_stream_kernel (routing, gate/up + SwiGLU, down + combine; one layer)",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "traffic_source": TRAFFIC_SOURCE if traffic else "not captured for this kernel build",
            "bytes_per_launch": int(bytes_per_launch), "avg_launch_us": round(launch_s * 1e6, 3),
            "peak_source": peak_src,
            "timing": "CUDA events over the timed region on the launching stream; launch time = step time / layers"}


def base_line(metric, value, unit, world, K, W, ms, config, hib=True):
    return {"metric": metric, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": round(ms / K, 5), "higher_is_better": hib, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16",
            "data": "synthetic (seeded; random-init INT4 experts)", "config": config}


def time_model_line(full, low, main, K, Ktm, E, lo):
    """The declared time model t_token = t_calc + bytes_out / bandwidth
    (lucashiago explainer, etapa 5) fitted on two runs of Ktm steps -- all E
    experts resident (`full`) and `lo` resident (`low`) -- and the rate it
    predicts for the main run of K steps, beside the measured one (one rank's
    tokens). Each run: {"ms": device time, "bytes_out": bytes read or copied
    from host memory}."""
    t_full, t_low = full["ms"] / 1e3 / Ktm, low["ms"] / 1e3 / Ktm
    b_full, b_low = full["bytes_out"] / Ktm, low["bytes_out"] / Ktm
    per_byte = (t_low - t_full) / max(1.0, b_low - b_full)
    t_calc = t_full - b_full * per_byte
    b_main = main["bytes_out"] / K
    t_pred = t_calc + b_main * per_byte
    measured = K / (main["ms"] / 1e3)
    return {"form": "t_token = t_calc + bytes_out / bandwidth (lucashiago explainer, etapa 5)",
            "fit": f"two runs of {Ktm} steps in the same mode: all {E} experts resident and {lo} resident",
            "t_calc_us": round(t_calc * 1e6, 2),
            "bandwidth_gbs": round(1.0 / per_byte / 1e9, 2) if per_byte > 0 else None,
            "bytes_out_per_token": int(b_main), "predicted_tok_s": round(1.0 / t_pred, 2),
            "measured_tok_s": round(measured, 2), "pred_over_meas": round((1.0 / t_pred) / measured, 4),
            "endpoints_tok_s": {str(E): round(1.0 / t_full, 2), str(lo): round(1.0 / t_low, 2)}}


class PartialStack:
    """Inputs shared by the partial-residency runs of the OLMoE shape: the
    complete pinned host source of all L x E expert blocks, each layer's
    Zipf(alpha) popularity ranks, and per-step router logits and layer-0
    inputs for n steps (all on the device)."""

    def __init__(self, moe, rank, n):
        wl = synth.WORKLOADS["olmoe_partial"]
        self.wl = wl
        self.L, self.H, self.I, self.E, self.k, self.g = (wl[key] for key in ("L", "H", "I", "E", "k", "g"))
        self.shape = (self.H, self.I, self.g)
        self.bb = moe.moe_expert_block_bytes(self.shape)
        self.seed = synth.BASE_SEED + 3 + rank
        dev = torch.device("cuda")
        self.src = torch.empty((self.L, self.E, self.bb), dtype=torch.uint8).pin_memory()
        for l in range(self.L):  # generated on the device, kept as the pinned host source
            self.src[l].copy_(synth.device_pool(self.E, self.H, self.I, self.g, self.seed * 100 + l))
        self.ranks = np.stack([synth.zipf_ranks(self.seed, l, self.E) for l in range(self.L)])  # [L][E]
        gen = torch.Generator(device=dev)
        gen.manual_seed(self.seed)
        gum = -torch.log(-torch.log(torch.rand((n, self.L, 1, self.E), generator=gen, device=dev).clamp_min(1e-20)))
        self.logits = (-wl["alpha"] * torch.log(torch.from_numpy(self.ranks).float().to(dev)))[None, :, None, :] + gum
        self.x0 = torch.randn((n, 1, self.H), generator=gen, device=dev).half()
        self.n = n

    def profile(self):
        return 1.0 / self.ranks.astype(np.float64) ** self.wl["alpha"]


def partial_copy(moe, ps, C, policy, K, W, world, steps_from=0, prefetch=0):
    """Residency by copies: per layer and step the router runs on the GPU, its
    ids reach the host, the residency manager decides and streams misses from
    pinned host RAM on a side stream into the layer's C slots, then the experts
    run from the managed pool. With prefetch = S > 0 the layer has S spare
    slots and, once a layer's experts are enqueued, the next layer's S
    non-resident experts with the highest decayed counts are copied into them
    on the side stream, overlapping this layer. Returns the device time of K
    steps after W."""
    L, E, k, bb = ps.L, ps.E, ps.k, ps.bb
    dev = torch.device("cuda")
    pool = torch.zeros((L, C + prefetch, bb), dtype=torch.uint8, device=dev)
    slot_of = torch.full((L, E), -1, dtype=torch.int32, device=dev)
    copy = torch.cuda.Stream()
    # Pinned policy: the profile is the popularity the stream is drawn from
    # (a perfect measurement pass); C - k experts pinned, k slots follow LRU.
    pinned = C - k if policy == "pinned" else 0
    h = moe.moe_residency_create(dict(layers=L, experts=E, slots=C, spares=prefetch, max_ids_per_step=k,
                                      block_bytes=bb, decay=ps.wl["decay"], policy=policy, pinned=pinned,
                                      profile=ps.profile() if policy == "pinned" else None),
                                 ps.src, pool, slot_of, torch.cuda.current_stream(), copy)
    ids = torch.empty((L, 1, k), dtype=torch.int32, device=dev)
    w = torch.empty((L, 1, k), dtype=torch.float32, device=dev)
    y = torch.empty((L, 1, ps.H), dtype=torch.float16, device=dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(ps.shape, 1, k, E, moe.MOE_PATH_GEMV), dtype=torch.uint8,
                     device=dev)
    ids_host = torch.empty((k,), dtype=torch.int32).pin_memory()
    id_trace = [[] for _ in range(L)]  # every step's ids per layer, as the manager saw them

    def step(s):
        for l in range(L):
            moe.moe_route(ps.logits[s, l], k, ps.wl["renorm"], ids[l], w[l])
            ids_host.copy_(ids[l].view(-1), non_blocking=True)
            torch.cuda.current_stream().synchronize()  # the step's ids reach the host
            id_trace[l].append(ids_host.numpy().tolist())
            moe.moe_residency_prepare(h, l, ids_host.numpy())
            x = ps.x0[s] if l == 0 else y[l - 1]
            moe.moe_expert_forward(ps.shape, x, ids[l], w[l], E, pool[l], slot_of[l], C + prefetch, None, y[l],
                                   ws, moe.MOE_PATH_GEMV)
            if prefetch:
                nl = (l + 1) % L
                counts = moe.moe_residency_counts(h, nl, E)
                table = moe.moe_residency_slot_table(h, nl, E)
                out = [e for e in np.lexsort((np.arange(E), -counts)) if table[e] < 0][:prefetch]
                moe.moe_residency_prefetch(h, nl, out)

    try:
        for s in range(steps_from, steps_from + W):
            step(s)
        torch.cuda.synchronize()
        st0 = moe.moe_residency_get_stats(h)
        barrier(world)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        t0 = time.perf_counter()
        for s in range(steps_from + W, steps_from + W + K):
            step(s)
        ev1.record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        ms = max_over_ranks(ev0.elapsed_time(ev1), world)
        st1 = moe.moe_residency_get_stats(h)
        assert moe.moe_workspace_flags(ws) == 0
    finally:
        moe.moe_residency_destroy(h)
    hits, misses = st1["hits"] - st0["hits"], st1["misses"] - st0["misses"]
    return {"ms": ms, "wall_s": wall, "hits": hits, "misses": misses, "pinned": pinned,
            "id_trace": id_trace, "total_hits": st1["hits"], "total_misses": st1["misses"],
            "bytes_out": st1["h2d_bytes"] - st0["h2d_bytes"], "launches_per_step": L * 7,
            "prefetched": st1["prefetched"] - st0["prefetched"],
            "prefetch_copies": st1["prefetch_copies"] - st0["prefetch_copies"]}


def partial_zero_copy(moe, ps, C, K, W, world, graph=True, steps_from=0):
    """Zero-copy residency: each layer keeps a fixed set of C experts in HBM
    (the C most popular by the profile); the rest are read in place from the
    pinned host source by the expert kernels over the CPU-GPU link. No host
    round trip, so the 16 layers of a step are enqueued (and, with graph=True,
    captured once into a CUDA graph and replayed per step)."""
    L, E, k, bb = ps.L, ps.E, ps.k, ps.bb
    dev = torch.device("cuda")
    n_slots = max(1, C)
    pool = torch.zeros((L, n_slots, bb), dtype=torch.uint8, device=dev)
    slot_table = np.full((L, E), -1, dtype=np.int32)
    for l in range(L):
        resident = sorted(np.argsort(ps.ranks[l], kind="stable")[:C].tolist())
        for s_i, e in enumerate(resident):
            slot_table[l, e] = s_i
            pool[l, s_i].copy_(ps.src[l, e])
    slot_of = torch.from_numpy(slot_table).to(dev)
    ids = torch.empty((L, 1, k), dtype=torch.int32, device=dev)
    w = torch.empty((L, 1, k), dtype=torch.float32, device=dev)
    y = torch.empty((L, 1, ps.H), dtype=torch.float16, device=dev)
    lg_cur = torch.empty((L, 1, E), dtype=torch.float32, device=dev)
    x_cur = torch.empty((1, ps.H), dtype=torch.float16, device=dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(ps.shape, 1, k, E, moe.MOE_PATH_GEMV_UNFUSED),
                     dtype=torch.uint8, device=dev)
    hist = torch.empty((ps.n, L, k), dtype=torch.int32, device=dev)

    def layers():
        for l in range(L):
            moe.moe_route(lg_cur[l], k, ps.wl["renorm"], ids[l], w[l])
            x = x_cur if l == 0 else y[l - 1]
            moe.moe_expert_forward_zero_copy(ps.shape, x, ids[l], w[l], E, pool[l], slot_of[l], n_slots,
                                             ps.src[l], None, y[l], ws)

    g = None
    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            layers()  # warm the binding and the kernels before capture
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            layers()

    def step(s):
        lg_cur.copy_(ps.logits[s])
        x_cur.copy_(ps.x0[s])
        if g is not None:
            g.replay()
        else:
            layers()
        hist[s].copy_(ids.view(L, k))

    for s in range(steps_from, steps_from + W):
        step(s)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    t0 = time.perf_counter()
    for s in range(steps_from + W, steps_from + W + K):
        step(s)
    ev1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    assert moe.moe_workspace_flags(ws) == 0
    used = hist[steps_from + W:steps_from + W + K].cpu().numpy()  # [K][L][k]
    resident = slot_table[np.arange(L)[None, :, None], used] >= 0
    hits = int(resident.sum())
    misses = int(resident.size - hits)
    return {"ms": ms, "wall_s": wall, "hits": hits, "misses": misses, "bytes_out": misses * bb,
            "launches_per_step": L * 3, "graph": graph}


def copy_engine_gbs(ps, n=48):
    """Host-to-device bandwidth of block-sized copies from the pinned source
    (one cudaMemcpyAsync per block on a side stream), for context."""
    dev = torch.device("cuda")
    dst = torch.empty((n, ps.bb), dtype=torch.uint8, device=dev)
    flat = ps.src.view(-1, ps.bb)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for i in range(8):
            dst[i].copy_(flat[i], non_blocking=True)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(st)
        for i in range(n):
            dst[i].copy_(flat[(7 * i + 3) % flat.shape[0]], non_blocking=True)
        ev1.record(st)
    st.synchronize()
    return n * ps.bb / (ev0.elapsed_time(ev1) / 1e3) / 1e9


def run_partial(args, world, rank):
    """OLMoE shape with partial residency: C of 64 experts per layer in HBM
    (default 30), Zipf(1.0) popularity per layer, one token per step through
    16 layers. --mode copy: misses are copied into slots chosen by the victim
    policy (decayed counts 0.9 per step, LRU, or profile-pinned) before the
    experts run. --mode zerocopy: a fixed profile set stays in HBM and misses
    are read in place over the CPU-GPU link. The line adds the time model
    t_token = t_calc + bytes_out / bandwidth fitted on the two extreme
    residencies of the same mode and compared with the measured rate."""
    from int4_routed_expert_moe_gb300 import moe
    wl = synth.WORKLOADS["olmoe_partial"]
    L, H, I, E, k, g = wl["L"], wl["H"], wl["I"], wl["E"], wl["k"], wl["g"]
    C = args.slots if args.slots is not None else wl["C"]
    if not (0 if args.mode == "zerocopy" else k) <= C <= E:
        raise SystemExit(f"--slots must be in [{0 if args.mode == 'zerocopy' else k}, {E}] for --mode {args.mode}")
    K = args.steps or wl["seqs"] * wl["steps"]
    W = args.warmup if args.warmup is not None else wl["warm_seqs"] * wl["steps"]
    Ktm, Wtm = min(K, 256), min(W, 32)
    ps = PartialStack(moe, rank, max(W + K, 2 * (Wtm + Ktm)))
    lo = 0 if args.mode == "zerocopy" else k

    def run(c, steps, warm, graph=True):
        r = (partial_zero_copy(moe, ps, c, steps, warm, world, graph=graph) if args.mode == "zerocopy"
             else partial_copy(moe, ps, c, args.policy, steps, warm, world, prefetch=args.prefetch))
        torch.cuda.empty_cache()
        return r

    main_run = run(C, K, W)
    eager = run(C, Ktm, Wtm, graph=False) if args.mode == "zerocopy" else None
    full = run(E, Ktm, Wtm)
    low = run(lo, Ktm, Wtm)
    ms = main_run["ms"]
    value = K * world / (ms / 1e3)
    cfg = {"workload": "olmoe_partial", "layers": L, "hidden": H, "experts": E, "top_k": k,
           "inter": I, "group": g, "slots": C, "zipf_alpha": wl["alpha"], "mode": args.mode,
           "tokens_per_step": 1}
    if args.mode == "copy":
        cfg.update({"policy": args.policy, "pinned": main_run["pinned"], "decay": wl["decay"],
                    "prefetch_spares": args.prefetch,
                    "launch": "eager; per layer: route, D2H of ids, host decision, H2D misses, experts"})
    else:
        cfg.update({"resident_set": "the C most popular experts of each layer (profile), fixed",
                    "launch": "one CUDA graph per step: per layer route + two-kernel GEMV reading misses "
                              "from pinned host memory"})
    out = base_line(METRIC, value, "tokens/s", world, K, W, ms, cfg)
    hits, misses = main_run["hits"], main_run["misses"]
    out["residency"] = {"hit_rate": round(hits / max(1, hits + misses), 4), "misses_per_token": round(misses / K, 3),
                        "bytes_out_gb": round(main_run["bytes_out"] / 1e9, 3),
                        "bytes_out_gbs": round(main_run["bytes_out"] / (ms / 1e3) / 1e9, 2),
                        "wall_s": round(main_run["wall_s"], 3)}
    if args.mode == "copy" and args.prefetch:
        out["residency"]["prefetched_per_token"] = round(main_run["prefetched"] / K, 3)
        out["residency"]["prefetch_copies_per_token"] = round(main_run["prefetch_copies"] / K, 3)
    if eager is not None:
        out["residency"]["eager_value"] = round(Ktm * world / (eager["ms"] / 1e3), 2)
    out["time_model"] = time_model_line(full, low, main_run, K, Ktm, E, lo)
    if args.mode == "copy":
        out["time_model"]["copy_engine_gbs"] = round(copy_engine_gbs(ps), 2)
        if rank == 0:
            out["residency_oracle"] = residency_oracle_timing(ps, C, args.policy, args.prefetch, main_run)
    out["gpu_launches"] = main_run["launches_per_step"] * K
    return out


def residency_oracle_timing(ps, C, policy, spares, run):
    """The oracle's residency simulator (the decision model the library
    implements) on the run's full id trace -- every layer, warm-up and timed
    steps -- single-threaded on the host, with its hit and miss totals beside
    the library's. With spare slots the library also served prefetches the
    trace does not hold, so only the time is reported."""
    from oracle import moe_oracle
    pinned = run["pinned"]
    profile = ps.profile() if policy == "pinned" else None
    t0 = time.perf_counter()
    hits = misses = 0
    for l, steps in enumerate(run["id_trace"]):
        r = moe_oracle.residency_sim(steps, ps.E, C, 0, ps.wl["decay"], policy,
                                     None if profile is None else profile[l], pinned)
        hits += r["hits"]
        misses += r["misses"]
    dt = time.perf_counter() - t0
    n_steps = sum(len(st) for st in run["id_trace"])
    out = {"layers": len(run["id_trace"]), "layer_steps": n_steps, "seconds": round(dt, 3), "cores": 1,
           "layer_steps_per_s": round(n_steps / dt, 1), "kind": "oracle"}
    if not spares:
        out.update({"hits": hits, "misses": misses,
                    "matches_library": hits == run["total_hits"] and misses == run["total_misses"]})
    return out


def run_fanout(args, world, rank, T):
    """Large fan-out stack: 48 layers x 512 experts (hidden 2048, inter 512,
    top-10 renormalised, Zipf(1.1) popularity), ~41 GB of INT4 experts all
    resident; T tokens per step through all 48 layers on the path
    MOE_PATH_AUTO picks (the streamed decode kernel up to 16 tokens, the
    grouped tensor-core path above). The roofline bytes of a step are the
    distinct experts each layer reads, counted from the routing of every
    timed step."""
    from int4_routed_expert_moe_gb300 import moe
    wl = synth.WORKLOADS["large_fanout"]
    L, H, I, E, k, g = wl["L"], wl["H"], wl["I"], wl["E"], wl["k"], wl["g"]
    shape = (H, I, g)
    K = args.steps or (24 if T >= 256 else 96)
    W = max(3, args.warmup if args.warmup is not None else 8)
    dev = torch.device("cuda")
    bb = moe.moe_expert_block_bytes(shape)
    seed = synth.BASE_SEED + 5 + rank
    pool = synth.device_pool(L * E, H, I, g, seed, chunk=256)
    slot_of = torch.arange(E, dtype=torch.int32, device=dev)
    n = W + K
    ranks = np.stack([synth.zipf_ranks(seed, l, E) for l in range(L)])
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    base = (-wl["alpha"] * torch.log(torch.from_numpy(ranks).float().to(dev)))[:, None, :]
    x0 = torch.randn((n, T, H), generator=gen, device=dev).half()
    ids = torch.empty((n, L, T, k), dtype=torch.int32, device=dev)  # every step's routing is kept
    w = torch.empty((L, T, k), dtype=torch.float32, device=dev)
    y = torch.empty((L, T, H), dtype=torch.float16, device=dev)
    path = moe.MOE_PATH_AUTO
    ws = torch.zeros(moe.moe_forward_workspace_bytes(shape, T, k, E, path), dtype=torch.uint8, device=dev)
    logits = torch.empty((n, L, T, E), device=dev)  # drawn before the timed region
    for s in range(n):
        u = torch.rand((L, T, E), generator=gen, device=dev).clamp_min(1e-20)
        logits[s] = base - torch.log(-torch.log(u))

    def step(s):
        for l in range(L):
            x = x0[s] if l == 0 else y[l - 1]
            moe.moe_layer_forward(shape, x, logits[s, l], k, wl["renorm"], ids[s, l], w[l],
                                  pool[l * E:(l + 1) * E], slot_of, E, None, y[l], ws, path)

    step(0)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def capture(steps):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for s in steps:
                step(s)
        return gr

    warm = [capture(range(W))]
    blocks = [[capture(range(W + b0, W + b0 + nb))] for b0, nb in split_blocks(K)]
    torch.cuda.synchronize()
    sampler = ClockSampler(smi_index())
    time.sleep(0.2)
    ms, block_ms, t_host0, t_host1 = timed_blocks(blocks, warm, world, stream)
    rows = sampler.stop()
    clocks = ClockSampler.summarize(rows, t_host0, t_host1)
    assert moe.moe_workspace_flags(ws) == 0
    ms_max = max_over_ranks(ms, world)
    # Distinct experts read per layer, from the timed steps' routing.
    idc = ids[W:].reshape(K, L, T * k).cpu().numpy()
    uniq = np.array([[len(np.unique(idc[s, l][idc[s, l] >= 0])) for l in range(L)] for s in range(K)])
    bytes_step = float(uniq.sum(axis=1).mean()) * bb
    peak, peak_src = measured_peaks()
    step_s = ms / 1e3 / K
    achieved = bytes_step / step_s / 1e9
    streamed = T <= 16
    launch_s = step_s / L
    out = base_line(METRIC, K * T * world / (ms_max / 1e3), "tokens/s", world, K, W, ms_max,
                    {"workload": f"large_fanout_b{T}", "layers": L, "hidden": H, "experts": E, "top_k": k,
                     "inter": I, "group": g, "tokens_per_step": T, "zipf_alpha": wl["alpha"],
                     "path": "streamed decode kernel" if streamed else "grouped tensor-core path",
                     "launch": f"CUDA graphs (one per block of steps), {L} moe_layer_forward calls per step",
                     "l2": f"inputs larger than L2: {L * E * bb / 1e9:.1f} GB pool"})
    out["blocks"] = block_stats(block_ms, [nb for _, nb in split_blocks(K)], T)
    out["unique_experts_per_layer"] = round(float(uniq.mean()), 2)
    out["roofline"] = {"bound": "hbm",
                       "kernel": ("decode_stream_kernel, one layer" if streamed else
                                  "moe_layer_forward grouped path (route, sort, gather, 2 GEMMs, combine), one layer"),
                       "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                       "frac": round(achieved / peak, 4),
                       "traffic": (int(round(DECODE_DRAM_RATIO[f"large_fanout_b{T}"] * bytes_step / L))
                                   if f"large_fanout_b{T}" in DECODE_DRAM_RATIO else None),
                       "traffic_source": (TRAFFIC_SOURCE if f"large_fanout_b{T}" in DECODE_DRAM_RATIO
                                          else "not captured for this kernel build"),
                       "bytes_per_launch": int(bytes_step / L), "avg_launch_us": round(launch_s * 1e6, 3),
                       "bytes_rule": "distinct experts of each layer x expert block bytes, from the timed steps' ids",
                       "peak_source": peak_src,
                       "timing": "CUDA events over the timed region; layer time = step time / layers"}
    out["gpu_launches"] = L * K * (1 if streamed else 6)  # grouped: route, sort, gather, 2 GEMMs, combine
    out["clocks"] = clocks
    return out


def run_prefill(args, world, rank):
    """OLMoE-shaped prefill: 512 tokens through 16 routed layers (uniform
    router logits, 4096 (token, choice) pairs per layer over all 64 experts),
    grouped tensor-core path, layers chained; then the non-routed FP16 SwiGLU
    FFN of 2048 tokens (H 2048, Is 4096) as its own leg."""
    from int4_routed_expert_moe_gb300 import moe
    wl = synth.WORKLOADS["olmoe_prefill"]
    L, H, I, E, k, g, T = wl["L"], wl["H"], wl["I"], wl["E"], wl["k"], wl["g"], wl["T"]
    Ts, Is = wl["Ts"], wl["Is"]
    shape = (H, I, g)
    K = args.steps or 20
    W = max(3, args.warmup if args.warmup is not None else 3)
    dev = torch.device("cuda")
    seed = synth.BASE_SEED + 4 + rank
    pool = synth.device_pool(L * E, H, I, g, seed)
    bb = moe.moe_expert_block_bytes(shape)
    slot_of = torch.arange(E, dtype=torch.int32, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    n = W + K
    x0 = torch.randn((n, T, H), generator=gen, device=dev).half()
    logits = torch.rand((n, L, T, E), generator=gen, device=dev)
    ids = torch.empty((L, T, k), dtype=torch.int32, device=dev)
    w = torch.empty((L, T, k), dtype=torch.float32, device=dev)
    y = torch.empty((L, T, H), dtype=torch.float16, device=dev)
    path = moe.MOE_PATH_GROUPED
    ws = torch.zeros(moe.moe_forward_workspace_bytes(shape, T, k, E, path), dtype=torch.uint8, device=dev)

    def layer(s, l):
        x = x0[s] if l == 0 else y[l - 1]
        moe.moe_layer_forward(shape, x, logits[s, l], k, wl["renorm"], ids[l], w[l], pool[l * E:(l + 1) * E],
                              slot_of, E, None, y[l], ws, path)

    def step(s):
        for l in range(L):
            layer(s, l)

    step(0)  # eager: kernel attributes, tensor-map entry point
    torch.cuda.synchronize()
    graphs = []
    for s in range(n):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            step(s)
        graphs.append(gr)
    torch.cuda.synchronize()
    sampler = ClockSampler(smi_index())
    time.sleep(0.2)
    for s in range(W):
        graphs[s].replay()
    torch.cuda.synchronize()
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    ev0.record()
    for s in range(W, n):
        graphs[s].replay()
    ev1.record()
    torch.cuda.synchronize()
    t_host1 = time.time()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    assert moe.moe_workspace_flags(ws) == 0

    # One layer call = the routing kernel and the six grouped-path kernels,
    # back to back on one stream: its average duration is the step time over
    # the layers (an upper bound of the dominant GEMM kernel's own time, so
    # the fraction below is a lower bound for that kernel).
    layer_ms = ms / K / L

    # Shared FFN leg.
    sw = {kk: torch.from_numpy(v).to(dev) for kk, v in synth.shared_weights(seed, H, Is).items()}
    xs = torch.randn((Ts, H), generator=gen, device=dev).half()
    ys = torch.empty((Ts, H), dtype=torch.float16, device=dev)
    wss = torch.zeros(moe.moe_shared_workspace_bytes(Ts, H, Is), dtype=torch.uint8, device=dev)
    moe.moe_shared_forward(xs, sw["wg"], sw["wu"], sw["wd"], ys, wss)
    torch.cuda.synchronize()
    reps = 20
    g_sh = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_sh):
        for _ in range(reps):
            moe.moe_shared_forward(xs, sw["wg"], sw["wu"], sw["wd"], ys, wss)
    for _ in range(3):
        g_sh.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g_sh.replay()
    e1.record()
    torch.cuda.synchronize()
    sh_s = e0.elapsed_time(e1) / 1e3 / reps
    assert moe.moe_workspace_flags(wss) == 0
    rows = sampler.stop()
    clocks = ClockSampler.summarize(rows, t_host0, t_host1)

    P = T * k
    flops_layer = 6.0 * H * I * P
    peak_t, peak_t_src = measured_tensor_peak(sustained=True)
    peak_h, peak_h_src = measured_peaks()
    achieved = flops_layer / (layer_ms / 1e3) / 1e12
    weight_gbs = E * bb / (layer_ms / 1e3) / 1e9
    sh_flops = 6.0 * Ts * H * Is
    out = base_line(METRIC_PREFILL, K * T * world / (ms / 1e3), "tokens/s", world, K, W, ms,
                    {"workload": "olmoe_prefill", "layers": L, "hidden": H, "experts": E, "top_k": k,
                     "inter": I, "group": g, "tokens_per_step": T, "logits": "uniform",
                     "l2": "inputs larger than L2: 3.42 GB of expert weights per step",
                     "launch": "one CUDA graph per step (16 x (route + 6 grouped-path kernels))"})
    out["roofline"] = {"bound": "tensor", "kernel": "moe_layer_forward grouped path, one layer (route, sort, "
                                                    "tiles, gather, tcgen05 gate/up GEMM, tcgen05 down GEMM, combine)",
                       "achieved": round(achieved, 1), "peak": peak_t, "unit": "TFLOP/s",
                       "frac": round(achieved / peak_t, 4), "traffic": PREFILL_GEMM_DRAM_BYTES,
                       "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of the gate/up and "
                                         "down GEMM kernels of one layer call (the small kernels not included)",
                       "flops_per_launch": flops_layer, "avg_launch_us": round(layer_ms * 1e3, 2),
                       "peak_source": peak_t_src,
                       "weight_gbs": round(weight_gbs, 1), "weight_hbm_frac": round(weight_gbs / peak_h, 4),
                       "timing": "CUDA events over the timed region; layer time = step time / layers"}
    out["shared_ffn"] = {"tokens": Ts, "hidden": H, "inter": Is, "us_per_call": round(sh_s * 1e6, 2),
                         "tflops": round(sh_flops / sh_s / 1e12, 1),
                         "frac_of_tensor_peak": round(sh_flops / sh_s / 1e12 / peak_t, 4)}
    out["gpu_launches"] = (L * 7) * K
    out["clocks"] = clocks
    return out


def run_e2e(moe, wl, n, W):
    """Same metric through the public API with host buffers: per step the
    token's activations and every layer's router logits are copied from
    pinned host memory, the layers run, and the output is read back
    (synchronising). The per-layer moe_layer_forward calls are captured once
    into a CUDA graph through the binding (as a latency-minded caller would)
    and replayed per step; the eager per-call variant is reported beside it."""
    x_h = wl.x0[W:W + n].cpu().pin_memory()
    lg_h = wl.logits[W:W + n].cpu().pin_memory()
    x_d = torch.empty_like(wl.x0[0])
    lg_d = torch.empty_like(wl.logits[0])
    y_h = torch.empty((wl.T, wl.H), dtype=torch.float16).pin_memory()
    stream = torch.cuda.current_stream()

    def timed(run_layers):
        for s in range(min(8, n)):  # warm-up
            x_d.copy_(x_h[s], non_blocking=True)
            lg_d.copy_(lg_h[s], non_blocking=True)
            run_layers()
            y_h.copy_(wl.y[wl.L - 1], non_blocking=True)
            stream.synchronize()
        t0 = time.perf_counter()
        for s in range(n):
            x_d.copy_(x_h[s], non_blocking=True)
            lg_d.copy_(lg_h[s], non_blocking=True)
            run_layers()
            y_h.copy_(wl.y[wl.L - 1], non_blocking=True)
            stream.synchronize()
        return n * wl.T / (time.perf_counter() - t0)

    eager = timed(lambda: wl.step(0, x0=x_d, logits=lg_d))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        wl.step(0, x0=x_d, logits=lg_d)
    torch.cuda.synchronize()
    graphed = timed(g.replay)
    return {"value": round(graphed, 2), "unit": "tokens/s",
            "h2d_bytes_per_step": int(x_h[0].numel() * 2 + lg_h[0].numel() * 4),
            "d2h_bytes_per_step": int(y_h.numel() * 2), "steps": n,
            "eager_value": round(eager, 2),
            "how": f"per step: pinned H2D of x and the {wl.L} layers' logits, the {wl.L} moe_layer_forward "
                   "calls (captured once into a CUDA graph through the binding and replayed; eager_value: "
                   "called one by one), D2H of the last layer's y, stream sync"}


def oracle_layer_sample(wl, s, l, x16, experts_from_device):
    from oracle import moe_oracle
    lg = wl.logits[s, l].cpu().numpy()
    return moe_oracle.moe_layer(x16, lg, experts_from_device, wl.k, wl.renorm, wl.g)


def physical_cores():
    """Physical cores available to this process: distinct SMT sibling sets of
    the allowed CPUs (each CPU its own core where the kernel gives no
    topology)."""
    try:
        cpus = sorted(os.sched_getaffinity(0))
    except AttributeError:
        cpus = list(range(os.cpu_count() or 1))
    cores = set()
    for c in cpus:
        try:
            with open(f"/sys/devices/system/cpu/cpu{c}/topology/thread_siblings_list") as f:
                cores.add(f.read().strip())
        except OSError:
            cores.add(str(c))
    return max(1, len(cores))


def _oracle_expert_task(args):
    """One routed expert of one token through the oracle (dequantise the
    block's arrays in FP64, SwiGLU FFN, weighted by the routing weight):
    the unit of the parallel CPU-baseline leg, run in worker processes."""
    from oracle import moe_oracle
    arrs, group, x, w = args
    return w * moe_oracle.expert_ffn(x, *moe_oracle.dequantize_expert(arrs, group))


def cpu_baseline(wl, budget_s=10.0):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    decode workload, at 1 thread and at the physical core count:
    * 1 thread: one decode token through as many of the layers as fit in
      ~budget_s (at least one): routing, FP64 dequantisation of each chosen
      expert, SwiGLU FFN, weighted sum;
    * all physical cores: the same per-expert work of as many (token, layer)
      pairs as fit in ~budget_s, one expert per task on a pool of worker
      processes (spawned; the oracle is unchanged, only its per-expert calls
      run side by side).
    Expert arrays are read out of the device pool before the clock starts."""
    import multiprocessing as mp
    from oracle import moe_oracle
    t_total, layers = 0.0, 0
    s = 0
    samples = []
    for l in range(wl.L):
        lg = wl.logits[s, l].cpu().numpy()
        ids, wts = moe_oracle.route(lg, wl.k, wl.renorm)
        pool = wl.layer_pool(l)
        blocks = {int(e): pool[int(e)].cpu().numpy() for e in ids.reshape(-1)}
        experts = {e: synth.arrays_from_block(b, *wl.shape) for e, b in blocks.items()}
        x16 = synth.activations(7, l, wl.T, wl.H)
        samples.append((x16, ids, wts, experts))
        t0 = time.perf_counter()
        moe_oracle.moe_layer(x16, lg, experts, wl.k, wl.renorm, wl.g)
        t_total += time.perf_counter() - t0
        layers += 1
        if t_total >= budget_s:
            break
    one = wl.T * layers / wl.L / t_total
    ncores = physical_cores()
    tasks = []
    for x16, ids, wts, experts in samples:
        for j in range(wl.k):
            e = int(ids[0, j])
            tasks.append((experts[e], wl.g, x16[0].astype(np.float64), float(wts[0, j])))
    per_task = t_total / max(1, len(tasks))
    n_tasks = min(len(tasks) * 8, max(ncores, int(budget_s * ncores / max(per_task, 1e-6))))
    work = [tasks[i % len(tasks)] for i in range(n_tasks)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(ncores) as pool_p:
        pool_p.map(_oracle_expert_task, work[:ncores])  # start-up outside the clock
        t0 = time.perf_counter()
        pool_p.map(_oracle_expert_task, work, chunksize=1)
        t_par = time.perf_counter() - t0
    many = n_tasks / (wl.L * wl.k) / t_par
    return {"value": round(one, 5), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"1 decode token through {layers} of {wl.L} layers ({layers * wl.k} experts "
                      f"dequantised in FP64), {t_total:.1f} s single-threaded",
            "all_cores": {"value": round(many, 5), "unit": "tokens/s", "cores": ncores,
                          "sample": f"{n_tasks} routed experts (= {n_tasks / (wl.L * wl.k):.2f} decode tokens) "
                                    f"on {ncores} worker processes, {t_par:.1f} s"},
            "nproc": os.cpu_count(), "cpu": cpu_model()}


def device_info():
    """Where the line was measured (best effort, never raises): GPU name, SM
    count and memory, host core count and CPU model."""
    info = {"host_cores": os.cpu_count(), "cpu": cpu_model()}
    try:
        if torch.cuda.is_available():
            p = torch.cuda.get_device_properties(torch.cuda.current_device())
            info.update({"gpu": p.name, "sms": int(p.multi_processor_count),
                         "gpu_mem_gib": round(p.total_memory / 2 ** 30, 1)})
    except Exception:  # metadata only
        pass
    return info


# Arm "CPU part" numbers of /proc/cpuinfo (implementer 0x41) seen on these hosts.
ARM_PARTS = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
             "0xd49": "Arm Neoverse N2"}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.lower()
                if key.startswith("model name"):
                    return line.split(":", 1)[1].strip()
                if key.startswith("cpu part"):
                    part = line.split(":", 1)[1].strip()
                    return f"{ARM_PARTS[part]} (CPU part {part})" if part in ARM_PARTS else f"CPU part {part}"
    except OSError:
        pass
    return "unknown"


# --------------------------------------------------------------------------
def run_reference(args):
    """The CPU oracle on the same workload and metric: each step is a bounded
    sample -- one routed expert of one (token, layer) pair of the OLMoE decode
    stack (routing plus FP64 dequantisation and SwiGLU FFN) -- i.e. 1/128 of a
    decode token. Inputs are the seeded host generator's."""
    from oracle import moe_oracle
    wl = synth.WORKLOADS["olmoe_decode"]
    H, I, E, k, g, L = wl["H"], wl["I"], wl["E"], wl["k"], wl["g"], wl["L"]
    K = args.steps or 512
    W = args.warmup if args.warmup is not None else 128
    seed = synth.BASE_SEED + 2

    def one(s):
        lg = synth.logits_normal(seed, s, 1, E)
        ids, w = moe_oracle.route(lg, k, wl["renorm"])
        e = int(ids[0, s % k])
        arrs = synth.expert_arrays(seed, s % L, e, H, I, g)
        x = synth.activations(seed, s, 1, H)[0]
        t0 = time.perf_counter()
        ids, w = moe_oracle.route(lg, k, wl["renorm"])
        mats = moe_oracle.dequantize_expert(arrs, g)
        o = w[0, s % k] * moe_oracle.expert_ffn(x, *mats)
        return time.perf_counter() - t0, o

    for s in range(W):
        one(s)
    total = 0.0
    for s in range(W, W + K):
        dt, _ = one(s)
        total += dt
    frac = 1.0 / (L * k)
    value = K * frac / total
    return {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": K, "warmup": W, "ms_per_step": round(total / K * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": "olmoe_decode", "layers": L, "hidden": H, "experts": E, "top_k": k,
                       "inter": I, "group": g, "tokens_per_step": 1},
            "cpu_baseline": {"value": round(value, 5), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": "per step one routed expert of one (token, layer) pair = 1/128 "
                                       "of a decode token", "cpu": cpu_model()},
            "e2e": {"value": round(value, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        if rank == 0:  # the other ranks exit without work
            line = run_reference(args)
            line["device"] = device_info()
            print(json.dumps(line), flush=True)
        barrier(world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    if args.workload == "olmoe_partial":
        out = run_partial(args, world, rank)
    elif args.workload == "olmoe_prefill":
        out = run_prefill(args, world, rank)
    elif args.workload.startswith("large_fanout_b"):
        out = run_fanout(args, world, rank, int(args.workload.split("_b")[1]))
    else:
        out = run_ours(args, world, rank, local, args.workload)
    if rank == 0:
        out["device"] = device_info()
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

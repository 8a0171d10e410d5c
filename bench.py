#!/usr/bin/env python
"""Benchmark of the sparse MoE FFN layer on GB300: MoE-layer tokens/s and the expert FFN's
HBM roofline fraction.

Default workload: the decode-shaped GLM-style layer (hidden 6144, 256 routed experts, top-8,
d_ff 2048, one shared expert d_ff 2048, routed_scaling_factor 2.5) at a batch of 32 tokens.
A step is one moe_layer_forward call (router, batch-union, routed + shared expert FFN,
combine) on a batch of synthetic tokens; the batches rotate over 5 seeded inputs so that
the set of experts read changes from step to step.  Every step reads about 2 GB of expert
weights (95 unique experts and the shared one at 21 MB each), far above the 129 MB L2, so
nothing is served from L2 across steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--tokens T] [--no-sweep] [--no-configs]
                    [--no-cpu-baseline]

Under torchrun (N > 1) every rank runs the same workload on its own GPU and its own
batches (weak scaling, no collective on the data path); rank 0 prints the JSON line with
the whole-job tokens/s over the slowest rank's time.  ``--impl reference`` times the CPU
oracle (the slow reference program) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s at 1 GB300 (expert-weight HBM GB/s as % of roofline in 'roofline')"
UNIT = "tokens/s"
N_BATCHES = 5
PROFILE_DIR = os.path.join(ROOT, "profiles")


# --------------------------------------------------------------------------- ranks

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(v: float, world: int, device=None) -> float:
    """Maximum of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while active."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [c.strip() for c in line.split(",")]
                if len(f) >= 9:
                    rows.append(f)
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------------- peaks

def tensor_peak():
    """Dense bf16 TFLOP/s of this GPU as measured by the driver: the sustained figure (a
    kernel timed inside a long layer step), else the recipe's fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured (bf16 sustained)"
    except (OSError, KeyError, ValueError):
        return 1700.0, "fallback (bf16 sustained)"


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


PATH_NAMES = {0: "warp GEMV", 1: "tcgen05 grouped GEMM", 2: "row GEMV"}


def stage_path(cfg, T: int, stage: str) -> int:
    """The kernel that runs an FFN stage ("gate_up" or "down")."""
    import sparse_expert_ffn_route_gb300 as moe
    return moe.moe_ffn_path(cfg, T) if stage == "gate_up" else moe.moe_ffn_path_down(cfg, T)


def ffn_kernel_name(cfg, T: int) -> str:
    import sparse_expert_ffn_route_gb300 as moe
    gu, dn = moe.moe_ffn_path(cfg, T), moe.moe_ffn_path_down(cfg, T)
    if gu == dn:
        return PATH_NAMES.get(gu, "?")
    return "%s (gate/up) + %s (down)" % (PATH_NAMES.get(gu, "?"), PATH_NAMES.get(dn, "?"))


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded by an ncu capture of this kernel (profiles/), or None
    when the kernel's source changed since the capture."""
    import hashlib
    path = os.path.join(PROFILE_DIR, "%s_%s.md" % (kernel, workload))
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if line.startswith("<!-- ") and "=" in line:
            k, v = line[5:].split("-->")[0].strip().split("=", 1)
            vals[k.strip()] = v.strip()
    src = os.path.join(ROOT, "sparse_expert_ffn_route_gb300", "csrc", vals.get("source", ""))
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    if digest != vals.get("source_sha256_16"):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------- our arm

def workload_of(args) -> synth.Workload:
    from dataclasses import replace
    wl = synth.WORKLOADS[args.workload]
    if args.n_experts:
        # smaller expert count of the same shapes (profiling captures of a few GB)
        wl = replace(wl, name="%s_E%d" % (wl.name, args.n_experts), n_experts=args.n_experts)
    return wl


def expert_bytes_gate_up(wl, shared=False):
    F = wl.d_ff_shared if shared else wl.d_ff
    return 2 * (F * wl.hidden // 2 + F * wl.hidden // 64 * 4)


def expert_bytes_down(wl, shared=False):
    F = wl.d_ff_shared if shared else wl.d_ff
    return F * wl.hidden // 2 + F * wl.hidden // 64 * 4


def algorithmic_bytes(wl, T, U, pairs):
    """Bytes per layer call each stage must move at least (weights of the unique experts
    read once, activations in, results out)."""
    ns = wl.n_shared
    H, F = wl.hidden, wl.d_ff
    rows = pairs + T * ns
    gu = U * expert_bytes_gate_up(wl) + ns * expert_bytes_gate_up(wl, True) \
        + T * H + T * (H // 32) * 4 + rows * F * 4
    dn = U * expert_bytes_down(wl) + ns * expert_bytes_down(wl, True) \
        + rows * F + rows * (F // 32) * 4 + rows * H * 4
    layer = U * wl.expert_bytes() + ns * wl.expert_bytes(True) + wl.n_experts * H * 4 \
        + T * H * 4 * 2
    return {"gate_up": gu, "down": dn, "layer": layer}


def algorithmic_flops(wl, T, pairs):
    """Multiply-add FLOPs (2 per MAC) of the expert FFN per layer call: every routed pair and
    shared-expert row against its expert's matrices, no padding counted."""
    ns = wl.n_shared
    H, F, Fs = wl.hidden, wl.d_ff, wl.d_ff_shared
    gu = 2.0 * (pairs * 2 * F * H + T * ns * 2 * Fs * H)
    dn = 2.0 * (pairs * F * H + T * ns * Fs * H)
    return {"gate_up": gu, "down": dn}


def run_ours(args, world, rank, local):
    import sparse_expert_ffn_route_gb300 as moe
    from sparse_expert_ffn_route_gb300 import build as moe_build

    moe_build.build()
    moe.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workload_of(args)
    T = args.tokens or max(wl.tokens)
    cfg = moe.MoeConfig.make(wl.hidden, wl.n_experts, wl.top_k, wl.d_ff, wl.n_shared,
                             wl.d_ff_shared, wl.norm_topk_prob, wl.routed_scaling_factor,
                             wl.top_p)
    routed = synth.gen_experts(wl, device=dev)
    shared = synth.gen_experts(wl, shared=True, device=dev) if wl.n_shared else None
    wr, bias = synth.gen_router(wl)
    wr, bias = wr.to(dev), bias.to(dev)

    def batches(Tb):
        xs = [synth.gen_x(wl, Tb, batch=rank * N_BATCHES + b) for b in range(N_BATCHES)]
        return xs, [x.to(dev) for x in xs]

    def routing_stats(xd, Tb, ws):
        """(unique experts, pairs) of each batch, from the library's own router + permute."""
        out = []
        K, E = wl.top_k, wl.n_experts
        ids = torch.empty(Tb, K, dtype=torch.int32, device=dev)
        w = torch.empty(Tb, K, dtype=torch.float32, device=dev)
        keff = torch.empty(Tb, dtype=torch.int32, device=dev)
        bufs = [torch.empty(n, dtype=torch.int32, device=dev)
                for n in (E, E + 1, Tb * K, Tb * K, E, 1)]
        for x in xd:
            moe.moe_route(cfg, x, wr, bias, ids, w, keff, ws)
            moe.moe_permute(cfg, ids, keff, *bufs, ws)
            out.append((int(bufs[5].item()), int(bufs[1][-1].item())))
        return out

    def time_layer(xd, Tb, ws, y, steps, flags=0):
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for k in range(steps):
            moe.moe_layer_forward(cfg, xd[k % N_BATCHES], wr, bias, routed, shared, y, ws,
                                  flags=flags)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1)

    ws = moe.alloc_workspace(cfg, T, device=dev)
    xh, xd = batches(T)
    y = torch.empty(T, wl.hidden, device=dev)
    stats = routing_stats(xd, T, ws)

    for k in range(args.warmup):
        moe.moe_layer_forward(cfg, xd[k % N_BATCHES], wr, bias, routed, shared, y, ws,
                              flags=moe.MOE_FLAG_SYNC_CHECK if k == 0 else 0)
    torch.cuda.synchronize()

    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local
    with ClockSampler(gpu_index) as clk:
        ms = time_layer(xd, T, ws, y, args.steps)
    clocks = clk.summary()
    ms_max = max_over_ranks(ms, world, dev)
    value = T * args.steps * world / (ms_max / 1e3)

    # per-stage device time over a second pass of the same K steps (events between stages)
    moe.moe_stage_times(reset=True)
    ms_ev = time_layer(xd, T, ws, y, args.steps, flags=moe.MOE_FLAG_STAGE_EVENTS)
    st = moe.moe_stage_times(reset=True)
    tot_bytes = {"gate_up": 0.0, "down": 0.0, "layer": 0.0}
    for k in range(args.steps):
        U, P = stats[k % N_BATCHES]
        for key, v in algorithmic_bytes(wl, T, U, P).items():
            tot_bytes[key] += v
    dom = max(("gate_up", "down"), key=lambda s: st[s][0])
    peak, peak_kind = hbm_peak()
    achieved = tot_bytes[dom] / (st[dom][0] / 1e3) / 1e9
    traffic = recorded_traffic("ffn_" + dom, "%s_T%d" % (wl.name, T))
    if stage_path(cfg, T, dom) == moe.MOE_FFN_TENSOR:
        # a dense contraction: tensor-pipe roofline on the useful FLOPs (the stage also holds
        # the x-code gather launch, so this is a lower bound on the GEMM kernel's own rate)
        tot_flops = {"gate_up": 0.0, "down": 0.0}
        for k in range(args.steps):
            _, P = stats[k % N_BATCHES]
            for key, v in algorithmic_flops(wl, T, P).items():
                tot_flops[key] += v
        tpeak, tpeak_kind = tensor_peak()
        tf = tot_flops[dom] / (st[dom][0] / 1e3) / 1e12
        roofline = {"bound": "tensor", "kernel": "ffn_" + dom, "achieved": round(tf, 1),
                    "peak": tpeak, "peak_kind": tpeak_kind, "unit": "TFLOP/s",
                    "frac": round(tf / tpeak, 4), "traffic": traffic,
                    "algorithmic_flops_per_launch": round(tot_flops[dom] / args.steps),
                    "launch_ms": round(st[dom][0] / args.steps, 4),
                    "hbm_achieved_gbs": round(achieved, 1), "hbm_peak": peak,
                    "layer_hbm_frac": round(tot_bytes["layer"] / (ms / 1e3) / 1e9 / peak, 4)}
    else:
        roofline = {"bound": "hbm", "kernel": "ffn_" + dom, "achieved": round(achieved, 1),
                    "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "traffic": traffic,
                    "algorithmic_bytes_per_launch": round(tot_bytes[dom] / args.steps),
                    "launch_ms": round(st[dom][0] / args.steps, 4),
                    "layer_frac": round(tot_bytes["layer"] / (ms / 1e3) / 1e9 / peak, 4)}
    stages = {s: round(v[0] / args.steps, 4) for s, v in st.items()}
    launches = sum(v[1] for v in st.values())

    # end to end through the host-buffer call (moe_layer_forward_host): every step copies its
    # x in from pinned host memory and its y out, inside the timed region.  Two streams, each
    # with its own workspace, take alternate batches, so that one batch's copies overlap the
    # other's compute, as a serving loop with two batches in flight does.
    e2e = None
    if world >= 1:
        pin_x = [x.pin_memory() for x in xh]
        pin_y = [torch.empty(T, wl.hidden).pin_memory() for _ in range(2)]
        streams = [torch.cuda.current_stream(), torch.cuda.Stream()]
        wss = [ws, moe.alloc_workspace(cfg, T, device=dev)]
        for k in range(2):
            moe.moe_layer_forward_host(cfg, pin_x[k % N_BATCHES], wr, bias, routed, shared,
                                       pin_y[k], wss[k], stream=streams[k])
        k2 = args.steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        done1 = torch.cuda.Event()
        barrier(world)
        torch.cuda.synchronize()
        e0.record(streams[0])
        streams[1].wait_event(e0)
        for k in range(k2):
            moe.moe_layer_forward_host(cfg, pin_x[k % N_BATCHES], wr, bias, routed, shared,
                                       pin_y[k % 2], wss[k % 2], stream=streams[k % 2])
        done1.record(streams[1])
        streams[0].wait_event(done1)
        e1.record(streams[0])
        torch.cuda.synchronize()
        barrier(world)
        ms_e2e = max_over_ranks(e0.elapsed_time(e1), world, dev)
        nbytes = T * wl.hidden * 4
        del wss
        e2e = {"value": round(T * k2 * world / (ms_e2e / 1e3), 1), "unit": UNIT,
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
               "call": "moe_layer_forward_host", "pipeline": "2 streams, alternate batches"}

    # router look-ahead ["MoE 路由与专家流式加载" §5]: RMSNorm of a residual state + the next
    # layer's router, timed alone at the workload's batch (HBM-bound: the router weights)
    lookahead = None
    if rank == 0 and world == 1:
        hh, gg, wn, bn = synth.gen_lookahead(wl, T, batch=rank)
        hh, gg, wn, bn = hh.to(dev), gg.to(dev), wn.to(dev), bn.to(dev)
        ids_p = torch.empty(T, wl.top_k, dtype=torch.int32, device=dev)
        w_p = torch.empty(T, wl.top_k, dtype=torch.float32, device=dev)
        k_p = torch.empty(T, dtype=torch.int32, device=dev)
        # copies of the router weights cycled call by call, twice the L2 size in all, so every
        # call reads its weights from HBM
        n_copies = max(1, min(64, -(-2 * 129 * 2 ** 20 // wn.numel() // 4)))
        wns = [wn.clone() for _ in range(n_copies)]
        for k in range(5):
            moe.moe_route_lookahead(cfg, hh, gg, 1e-5, wns[k % n_copies], bn, ids_p, w_p, k_p, ws)
        n_la = 200
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for k in range(n_la):
            moe.moe_route_lookahead(cfg, hh, gg, 1e-5, wns[k % n_copies], bn, ids_p, w_p, k_p, ws)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / n_la
        la_bytes = wl.n_experts * wl.hidden * 4 + wl.hidden * 4 + 2 * T * wl.hidden * 4
        lookahead = {"tokens": T, "us_per_call": round(us, 2),
                     "algorithmic_bytes": la_bytes,
                     "hbm_frac": round(la_bytes / (us / 1e6) / 1e9 / peak, 4),
                     "l2": "router weights cycled over %d copies (> 2x L2)" % n_copies}
        del wns

    # offline fp32 -> int4-gs64 weight quantiser (HBM-bound: 4 bytes in, 0.5625 out per weight)
    quantiser = None
    if rank == 0 and world == 1:
        wq = synth.gen_dense_weights(wl, 4 * wl.d_ff, wl.hidden).to(dev)   # > L2
        pq = torch.empty(wq.shape[0], wq.shape[1] // 2, dtype=torch.uint8, device=dev)
        sq = torch.empty(wq.shape[0], wq.shape[1] // 64, dtype=torch.float32, device=dev)
        for _ in range(3):
            moe.moe_quantize_int4_gs64(wq, pq, sq)
        n_q = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n_q):
            moe.moe_quantize_int4_gs64(wq, pq, sq)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / n_q
        qbytes = wq.numel() * 4 + pq.numel() + sq.numel() * 4
        quantiser = {"weights": wq.numel(), "us_per_call": round(us, 1),
                     "algorithmic_bytes": qbytes,
                     "achieved_gbs": round(qbytes / (us / 1e6) / 1e9, 1),
                     "hbm_frac": round(qbytes / (us / 1e6) / 1e9 / peak, 4)}
        del wq, pq, sq

    sweep = None
    if not args.no_sweep and rank == 0 and world == 1 and len(wl.tokens) > 1:
        sweep = {}
        for Tb in wl.tokens:
            wsb = moe.alloc_workspace(cfg, Tb, device=dev)
            _, xdb = batches(Tb)
            yb = torch.empty(Tb, wl.hidden, device=dev)
            sb = routing_stats(xdb, Tb, wsb)
            steps_b = max(50, min(args.steps, 400))
            time_layer(xdb, Tb, wsb, yb, 10)
            msb = time_layer(xdb, Tb, wsb, yb, steps_b)
            moe.moe_stage_times(reset=True)
            time_layer(xdb, Tb, wsb, yb, steps_b, flags=moe.MOE_FLAG_STAGE_EVENTS)
            stb = moe.moe_stage_times(reset=True)
            lb = sum(algorithmic_bytes(wl, Tb, *sb[k % N_BATCHES])["layer"] for k in range(steps_b))
            sweep["T%d" % Tb] = {"tokens_per_s": round(Tb * steps_b / (msb / 1e3), 1),
                                 "us_per_layer": round(msb / steps_b * 1e3, 2),
                                 "layer_hbm_frac": round(lb / (msb / 1e3) / 1e9 / peak, 4),
                                 "unique_experts_mean": round(float(np.mean([s[0] for s in sb])), 1),
                                 "stage_us": {k: round(v[0] / steps_b * 1e3, 1) for k, v in stb.items()}}
            del wsb, xdb, yb

    configs = None
    if not args.no_configs and rank == 0 and world == 1 and wl.name == "glm_decode":
        configs = measure_other_configs(moe, args, dev, peak, wl, routed, shared)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "i4xi8->i32,f32",
        "data": "synthetic (seeded SplitMix64 inputs of the workload's shapes and distributions)",
        "config": {"workload": "%s_T%d" % (wl.name, T), "hidden": wl.hidden,
                   "n_experts": wl.n_experts, "top_k": wl.top_k, "d_ff": wl.d_ff,
                   "n_shared": wl.n_shared, "d_ff_shared": wl.d_ff_shared, "tokens": T,
                   "routed_scaling_factor": wl.routed_scaling_factor, "top_p": wl.top_p,
                   "unique_experts_mean": round(float(np.mean([s[0] for s in stats])), 1),
                   "batches_rotated": N_BATCHES,
                   "ffn_kernel": ffn_kernel_name(cfg, T),
                   "l2": "inputs larger than L2: each step reads %.2f GB of expert weights"
                         % (np.mean([algorithmic_bytes(wl, T, *s)["layer"] for s in stats]) / 1e9),
                   "parallelism": "dp%d (replicas, no collective)" % world},
        "roofline": roofline, "stage_ms_per_step": stages,
        "stage_timing_overhead_ms_per_step": round((ms_ev - ms) / args.steps, 5),
        "gpu_launches": launches, "clocks": clocks, "e2e": e2e,
    }
    if sweep:
        out["sweep"] = sweep
    if configs:
        out["configs"] = configs
    if lookahead:
        out["router_lookahead"] = lookahead
    if quantiser:
        out["weight_quantiser"] = quantiser
    return out


# --------------------------------------------------------------------------- other configs

# The other layer shapes the metric is reported on, each measured in the default run:
# (workload, batch sizes, top_p override or None).  The A3B-style layer is also routed with
# top-p off, for the count of experts top-p saves ("MoE 路由与专家流式加载" §1.2).
OTHER_CONFIGS = (("a3b_decode", (64,), None), ("a3b_decode", (64,), 0.0), ("prefill", (4096,), None),
                 ("wide", (1, 8, 64, 512, 8192), None))
L2_BYTES = 129 * 2 ** 20


def same_experts(a: synth.Workload, b: synth.Workload) -> bool:
    """Do two workloads draw identical expert tensors (same shapes, seed and scale range)?"""
    return (a.hidden, a.n_experts, a.d_ff, a.d_ff_shared, a.seed, a.scale_lo, a.scale_hi) == \
        (b.hidden, b.n_experts, b.d_ff, b.d_ff_shared, b.seed, b.scale_lo, b.scale_hi)


def measure_layer(moe, wl, T, routed, shared, dev, steps, warmup, peak, rank=0):
    """One layer configuration: tokens/s over `steps` timed calls (CUDA events on the launch
    stream), the stages' device time from a second pass with stage events, the routing
    statistics (unique experts, kept experts per token, tokens per routed expert) and the
    roofline of the dominant FFN stage.  When one call reads less than four times the L2
    size, L2 is flushed (a 256 MB write) before every call and each call is timed alone."""
    cfg = moe.MoeConfig.make(wl.hidden, wl.n_experts, wl.top_k, wl.d_ff, wl.n_shared,
                             wl.d_ff_shared, wl.norm_topk_prob, wl.routed_scaling_factor, wl.top_p)
    wr, bias = synth.gen_router(wl)
    wr, bias = wr.to(dev), bias.to(dev)
    xd = [synth.gen_x(wl, T, batch=rank * N_BATCHES + b).to(dev) for b in range(N_BATCHES)]
    ws = moe.alloc_workspace(cfg, T, device=dev)
    y = torch.empty(T, wl.hidden, device=dev)
    K, E = wl.top_k, wl.n_experts
    ids = torch.empty(T, K, dtype=torch.int32, device=dev)
    w = torch.empty(T, K, dtype=torch.float32, device=dev)
    keff = torch.empty(T, dtype=torch.int32, device=dev)
    bufs = [torch.empty(n, dtype=torch.int32, device=dev) for n in (E, E + 1, T * K, T * K, E, 1)]
    stats, keffs, tpe_max, tpe_mean = [], [], [], []
    for x in xd:
        moe.moe_route(cfg, x, wr, bias, ids, w, keff, ws)
        moe.moe_permute(cfg, ids, keff, *bufs, ws)
        cnt = bufs[0].cpu().numpy()
        stats.append((int(bufs[5].item()), int(bufs[1][-1].item())))
        keffs.append(float(keff.float().mean().item()))
        tpe_max.append(int(cnt.max()))
        tpe_mean.append(float(cnt[cnt > 0].mean()))
    layer_bytes = float(np.mean([algorithmic_bytes(wl, T, *s)["layer"] for s in stats]))
    flush = layer_bytes < 4 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None
    stream = torch.cuda.current_stream()

    def run(n, flags=0):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n if flush else 1)]
        torch.cuda.synchronize()
        if not flush:
            evs[0][0].record(stream)
        for k in range(n):
            if flush:
                scratch.zero_()
                evs[k][0].record(stream)
            moe.moe_layer_forward(cfg, xd[k % N_BATCHES], wr, bias, routed, shared, y, ws, flags=flags)
            if flush:
                evs[k][1].record(stream)
        if not flush:
            evs[0][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs)

    run(warmup)
    ms = run(steps)
    moe.moe_stage_times(reset=True)
    run(steps, flags=moe.MOE_FLAG_STAGE_EVENTS)
    st = moe.moe_stage_times(reset=True)
    tot = {"gate_up": 0.0, "down": 0.0, "layer": 0.0}
    fl = {"gate_up": 0.0, "down": 0.0}
    for k in range(steps):
        U, P = stats[k % N_BATCHES]
        for key, v in algorithmic_bytes(wl, T, U, P).items():
            tot[key] += v
        for key, v in algorithmic_flops(wl, T, P).items():
            fl[key] += v
    dom = max(("gate_up", "down"), key=lambda s_: st[s_][0])
    gbs = tot[dom] / (st[dom][0] / 1e3) / 1e9
    traffic = recorded_traffic("ffn_" + dom, "%s_T%d" % (wl.name, T))
    path = ffn_kernel_name(cfg, T)
    if stage_path(cfg, T, dom) == moe.MOE_FFN_TENSOR:
        tpeak, tkind = tensor_peak()
        tf = fl[dom] / (st[dom][0] / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": "ffn_" + dom, "achieved": round(tf, 1), "peak": tpeak,
                "peak_kind": tkind, "unit": "TFLOP/s", "frac": round(tf / tpeak, 4), "traffic": traffic,
                "algorithmic_flops_per_launch": round(fl[dom] / steps),
                "launch_ms": round(st[dom][0] / steps, 4), "hbm_achieved_gbs": round(gbs, 1),
                "int8_tensor": "none on sm_103a (ptxas: tcgen05.mma .kind::i8 not supported); "
                               "the contraction runs exactly on kind::f16"}
    else:
        roof = {"bound": "hbm", "kernel": "ffn_" + dom, "achieved": round(gbs, 1), "peak": peak,
                "peak_kind": "measured", "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": traffic,
                "algorithmic_bytes_per_launch": round(tot[dom] / steps),
                "launch_ms": round(st[dom][0] / steps, 4)}
    return {"tokens": T, "ffn_kernel": path, "tokens_per_s": round(T * steps / (ms / 1e3), 1),
            "us_per_layer": round(ms / steps * 1e3, 2),
            "layer_hbm_frac": round(tot["layer"] / (ms / 1e3) / 1e9 / peak, 4),
            "roofline": roof,
            "stage_us": {k: round(v[0] / steps * 1e3, 1) for k, v in st.items()},
            "unique_experts_mean": round(float(np.mean([s_[0] for s_ in stats])), 1),
            "keff_mean": round(float(np.mean(keffs)), 3),
            "tokens_per_routed_expert": {"mean": round(float(np.mean(tpe_mean)), 1),
                                         "max": int(max(tpe_max))},
            "timed_steps": steps,
            "l2": ("flushed (256 MB write) before each call; calls timed one by one" if flush else
                   "inputs larger than L2 (%.2f GB of expert weights per call)" % (layer_bytes / 1e9))}


def measure_other_configs(moe, args, dev, peak, base_wl, base_routed, base_shared):
    """Every other layer configuration of the metric, on this GPU, one after the other."""
    out = {}
    cache = {}
    for name, tokens, top_p in OTHER_CONFIGS:
        wl = synth.WORKLOADS[name]
        if top_p is not None:
            wl = replace(wl, top_p=top_p)
        if same_experts(wl, base_wl):
            routed, shared = base_routed, base_shared
        else:
            key = name
            if key not in cache:
                cache.clear()
                torch.cuda.empty_cache()
                cache[key] = (synth.gen_experts(wl, device=dev),
                              synth.gen_experts(wl, shared=True, device=dev) if wl.n_shared else None)
            routed, shared = cache[key]
        for T in tokens:
            steps = max(5, min(args.steps, 50 if T <= 512 else 20))
            r = measure_layer(moe, wl, T, routed, shared, dev, steps, 3, peak)
            if top_p is not None:
                r["top_p"] = top_p
                r["parity"] = "parity unpinned: the pages' fewer experts under top-p rest on trained routers"
            label = "%s_T%d%s" % (name, T, "" if top_p is None else "_top_p_off")
            out[label] = r
    cache.clear()
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- oracle arm

def oracle_sample_run(wl, T, pairs_budget, steps=1, time_budget_s=None):
    """Time the CPU oracle on a bounded sample of the workload: the first tokens of batch 0
    routed by the oracle, each taken whole (its kept experts plus the shared expert) until
    ``pairs_budget`` expert applications per step.  Returns (tokens per second, cores, text)."""
    import oracle
    oracle.build()
    cfg = oracle.config_of(wl)
    x = synth.gen_x(wl, T, batch=0).numpy()
    wr, bias = synth.gen_router(wl)
    r = oracle.route(cfg, x, wr, bias)
    per_tok = r["keff"] + wl.n_shared
    ntok = int(max(1, np.searchsorted(np.cumsum(per_tok), pairs_budget, side="right")))
    ntok = min(ntok, T)
    rows = list(range(ntok))
    used = sorted({int(e) for t in rows for e in r["ids"][t, :r["keff"][t]]})
    remap = {e: i for i, e in enumerate(used)}
    from dataclasses import replace
    wl_c = replace(wl, n_experts=len(used), top_k=min(wl.top_k, len(used)))
    cfg_c = oracle.config_of(wl_c)
    R = {k: v.numpy() for k, v in synth.gen_experts(wl, experts=used).items()}
    S = ({k: v[0].numpy() for k, v in synth.gen_experts(wl, shared=True).items()}
         if wl.n_shared else None)
    ids_c = np.full((ntok, wl_c.top_k), -1, np.int32)
    for t in rows:
        for i in range(r["keff"][t]):
            ids_c[t, i] = remap[int(r["ids"][t, i])]
    keff = r["keff"][:ntok].copy()
    w = r["w"][:ntok, :wl_c.top_k].copy()
    xs = np.ascontiguousarray(x[:ntok])
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.route(cfg, xs, wr, bias)                        # routing of the sample
        perm = oracle.permute(cfg_c, ids_c, keff)
        ffn = oracle.expert_ffn(cfg_c, xs, R, perm["offsets"], perm["tok"])
        ys = oracle.shared_ffn(cfg_c, xs, S) if S is not None else None
        oracle.combine(cfg_c, ffn["y_pairs"], perm["slot"], perm["offsets"], w, keff, ys)
        times.append(time.perf_counter() - t0)
        if time_budget_s is not None and sum(times) > time_budget_s:
            break
    tot = sum(times)
    text = ("oracle on the first %d token(s) of batch 0 (%d expert applications incl. shared, "
            "full routing of those tokens), %d timed run(s)" % (ntok, int(per_tok[:ntok].sum()),
                                                                len(times)))
    return ntok * len(times) / tot, oracle.threads(), text, tot, len(times)


def run_reference(args, world, rank):
    if rank != 0:
        return None
    wl = workload_of(args)
    T = args.tokens or max(wl.tokens)
    # size each step so that warmup + steps end within about two minutes
    rate, cores, text, tot, n = oracle_sample_run(wl, T, pairs_budget=wl.top_k + wl.n_shared,
                                                  steps=1)
    per_step = tot / n
    budget = 120.0 / max(1, args.steps + args.warmup)
    pairs = (wl.top_k + wl.n_shared) * max(1, int(budget / per_step))
    oracle_sample_run(wl, T, pairs_budget=pairs, steps=max(0, args.warmup))
    rate, cores, text, tot, n = oracle_sample_run(wl, T, pairs_budget=pairs, steps=args.steps)
    return {"metric": METRIC, "value": round(rate, 4), "unit": UNIT, "n_gpus": world,
            "steps": n, "warmup": args.warmup, "ms_per_step": round(tot / n * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "i4xi8->i32,f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "%s_T%d" % (wl.name, T), "sample": text},
            "cpu_baseline": {"value": round(rate, 4), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": text},
            "e2e": {"value": round(rate, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="glm_decode", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=0, help="batch size (default: the largest)")
    ap.add_argument("--n-experts", type=int, default=0,
                    help="override the routed expert count (for small profiling captures)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other layer configurations (A3B, prefill, wide)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    try:
        if args.impl == "reference":
            out = run_reference(args, world, rank)
        else:
            out = run_ours(args, world, rank, local)
            if out is not None and rank == 0 and world == 1 and not args.no_cpu_baseline:
                wl = workload_of(args)
                T = args.tokens or max(wl.tokens)
                rate, cores, text, tot, n = oracle_sample_run(
                    wl, T, pairs_budget=4 * (wl.top_k + wl.n_shared), steps=3, time_budget_s=20)
                out["cpu_baseline"] = {"value": round(rate, 4), "unit": UNIT, "cores": cores,
                                       "kind": "oracle", "sample": text}
        if rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the weight-only INT4 MoE expert MLP on GB300.

One step = one moe_int4_forward per token count M of the workload's sweep
(default: the K2.6-shaped decode workload, 384 experts, top-8, hidden 7168,
intermediate 2048, M in {1, 9, 90}).  Weights are resident in HBM; every call
gets a routing from a rotating pool and an L2 flush (a 512 MB device write)
runs before it, outside its timed interval.  Times are CUDA events on the
launching stream.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle on
the host cores instead (bounded samples of the same workload).  Under torchrun
each rank runs an independent replica on its own GPU (the layer does not shard).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from weight_only_int4_moe_gb300 import inputs  # noqa: E402

METRIC = ("fused INT4 MoE µs/call & tokens/s vs M; HBM GB/s and tensor-pipe % of "
          "roofline")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(inputs.WORKLOADS), default="k26_decode")
    ap.add_argument("--ms", type=str, default=None, help="comma-separated token counts")
    ap.add_argument("--pool", type=int, default=8, help="routings per M")
    ap.add_argument("--flush-mb", type=int, default=512)
    ap.add_argument("--out-dtype", choices=["f32", "bf16"], default="f32")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--routed", action="store_true",
                    help="time moe_int4_forward_routed: routing from router logits in the call")
    ap.add_argument("--format", choices=["int4", "mxfp4"], default="int4",
                    help="expert weight format (mxfp4: E2M1 codes, E8M0 scale per 32)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (a smaller case of the same kernels, for ncu captures)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the verify, prefill and mid-size blocks of the default run")
    ap.add_argument("--extra-calls", type=int, default=20,
                    help="timed calls per M of each extra workload")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def expert_bytes(H, I, fmt="int4"):
    """Algorithmic bytes of one expert: 4-bit codes plus one scale per 32
    (bf16 for INT4, one E8M0 byte for MXFP4)."""
    sb = 2 if fmt == "int4" else 1
    w13 = 2 * I * H // 2 + 2 * I * (H // 32) * sb
    w2 = H * I // 2 + H * (I // 32) * sb
    return w13, w2


def make_weights(cfg, fmt):
    if fmt == "mxfp4":
        return inputs.make_weights_mxfp4(cfg.E, cfg.H, cfg.I, cfg.weight_seed)
    return inputs.make_weights(cfg.E, cfg.H, cfg.I, cfg.weight_seed)


GEMM_SOURCES = ("gemm.cu", "dequant.cuh", "kernels.cuh", "common.cuh")


def kernel_source_hash():
    """sha256 of the GEMM kernel sources without their // comments and blank
    lines: a code change invalidates a stored ncu capture, a comment edit does
    not (the sources have no block comments and no // inside strings)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "weight_only_int4_moe_gb300", "csrc", name)) as f:
            for line in f:
                code = re.sub(r"//.*$", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()


def kernel_traffic(kernel, workload, bytes_per_launch):
    """DRAM traffic per launch of `kernel`, from the committed ncu summary of a
    smaller case of the same kernel, scaled by algorithmic bytes.  None when no
    summary exists or the kernel's source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.json")
    if not os.path.exists(path):
        return None, "no ncu summary for this kernel and workload"
    with open(path) as f:
        d = json.load(f)
    if kernel_source_hash() != d.get("kernel_source_sha256"):
        return None, "kernel changed since the ncu capture"
    if d.get("traffic_per_algorithmic_byte") is None:  # no single ratio applies
        return None, d.get("reason", "no single traffic ratio for this workload")
    ratio = float(d["traffic_per_algorithmic_byte"])
    return ratio * bytes_per_launch, (f"ncu dram bytes of {d['captured_case']}: "
                                      f"{ratio:.4f} x algorithmic bytes, scaled")


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, enabled=True):
        self.index = index
        self.proc = None
        self.path = None
        self.enabled = enabled

    def start(self):
        if not self.enabled:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[1]) for r in rows]
        smax = max(num(r[2]) for r in rows)
        power = [num(r[3]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "sm_mhz_min": min(sm), "power_w_max": max(power), "samples": len(rows),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------- distributed --
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, local, use_gpu):
    if world <= 1:
        return None
    import torch
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    if use_gpu:
        torch.cuda.set_device(local)
    dist.init_process_group("nccl" if use_gpu else "gloo")
    return dist


def barrier(dist, use_gpu):
    if dist is None:
        return
    if use_gpu:
        import torch
        dist.barrier(device_ids=[torch.cuda.current_device()])
    else:
        dist.barrier()


def allreduce_max(dist, value, use_gpu):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if use_gpu else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_step, step_seconds_max):
    """Whole-job throughput of `world` replicas that each process units_per_step
    per step: every rank's units over the slowest rank's step time."""
    return world * units_per_step / step_seconds_max


# ------------------------------------------------------------ CPU oracle --
def time_oracle(w, cfg, Ms, target_s, threads, state=None, fmt="int4"):
    """Times the oracle on a bounded sample: rounds of `threads` tokens (one per
    thread) taken in turn from the largest call of the sweep, until about
    target_s seconds have passed.  Returns (tokens, seconds, M sampled)."""
    import oracle
    oracle.build()
    M = max(Ms)
    t = inputs.make_tokens(cfg, M)
    state = state if state is not None else {"next": 0}
    toks_done, t_total, rounds = 0, 0.0, 0
    while rounds == 0 or (t_total < target_s and rounds < 100):
        n = min(threads, M)
        tk = np.array(sorted({(state["next"] + j) % M for j in range(n)}))
        state["next"] = (state["next"] + n) % M
        t0 = time.perf_counter()
        oracle.moe_forward(t["x"], w["q13"], w["s13"], w["q2"], w["s2"], t["topk_ids"],
                           t["topk_weights"], tokens=tk, threads=threads, fmt=fmt)
        t_total += time.perf_counter() - t0
        toks_done += len(tk)
        rounds += 1
    return toks_done, t_total, M


def run_reference(args, cfg, Ms, world, rank):
    if rank != 0:
        return
    threads = host_threads()
    w = make_weights(cfg, args.format)
    per_step_s = max(0.5, args.cpu_seconds / max(1, args.steps))
    state = {"next": 0}
    for _ in range(args.warmup):
        time_oracle(w, cfg, Ms, 0.0, threads, state, fmt=args.format)
    toks, secs = 0, 0.0
    step_ms = []
    for _ in range(args.steps):
        n, s, Msamp = time_oracle(w, cfg, Ms, per_step_s, threads, state, fmt=args.format)
        toks += n
        secs += s
        step_ms.append(s * 1e3)
    value = toks / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(step_ms), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "E": cfg.E, "top_k": cfg.top_k, "hidden": cfg.H,
                   "inter": cfg.I, "weight_format": args.format, "Ms": list(Ms)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{toks} tokens of the M={Msamp} call ({args.steps} "
                                   f"steps of rounds of {threads} tokens), fp64 oracle, "
                                   f"{threads} threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- GPU arm --
def roofline_of(recs, w13_b, w2_b, top_k, H, I, hbm_peak, tc_peak, peak_src, workload):
    """Roofline position of the dominant kernel over profiled calls: of the fused
    decode kernel (both GEMMs in one launch, where the forward ran it), the
    gate/up GEMM and the down GEMM or the per-block down kernel (where it ran
    them separately) and the two small-batch matrix-vector kernels (where it
    ran those), the one with the
    largest share of the per-kernel event time, over the calls that ran it.
    Algorithmic bytes (touched experts x packed weights + scales) or FLOPs
    (2 x pairs x the kernel's weights) per launch over its CUDA-event duration,
    whichever bound is the slower at the peaks."""
    mult = {"fused": 3, "gate_up": 2, "down": 1, "block_down": 1, "gemv_gate_up": 2,
            "gemv_down": 1}
    wbytes = {"fused": w13_b + w2_b, "gate_up": w13_b, "down": w2_b, "block_down": w2_b,
              "gemv_gate_up": w13_b, "gemv_down": w2_b}

    def launches(kernel):  # (ms, record) of every launch of the kernel
        if kernel == "fused":
            return [(r["stages"][1], r) for r in recs if r["fused"]]
        gemv = kernel.startswith("gemv_")
        col = 1 if kernel.endswith("gate_up") else 2
        rs = [r for r in recs if not r["fused"] and r["gemv"] == gemv]
        if kernel in ("down", "block_down"):  # the separate plan's two down kernels
            rs = [r for r in rs if r["block_down"] == (kernel == "block_down")]
        return [(r["stages"][col], r) for r in rs]

    dominant = max(mult, key=lambda k: sum(ms for ms, _ in launches(k)))
    lr = launches(dominant)
    k_ms = [ms for ms, _ in lr]
    k_bytes = [r["touched"] * wbytes[dominant] for _, r in lr]
    k_flops = [2.0 * r["M"] * top_k * H * I * mult[dominant] for _, r in lr]
    t_hbm = sum(k_bytes) / (hbm_peak * 1e9)
    t_tc = sum(k_flops) / (tc_peak * 1e12)
    bytes_mean = statistics.mean(k_bytes)
    traffic, traffic_src = kernel_traffic(dominant, workload, bytes_mean)
    if t_hbm >= t_tc:  # weight streaming bound
        ach = sum(k_bytes) / (sum(k_ms) / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                "frac": ach / hbm_peak, "peak_source": f"{peak_src} (hbm_gbs)"}
    else:  # tensor bound; fp16 operands run at the bf16 dense rate
        ach = sum(k_flops) / (sum(k_ms) / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": ach / tc_peak,
                "peak_source": f"{peak_src} (bf16_tflops; fp16 has the same dense rate)"}
    roof.update({"traffic": traffic, "kernel": dominant, "traffic_source": traffic_src,
                 "bytes_per_launch_mean": bytes_mean,
                 "flops_per_launch_mean": statistics.mean(k_flops),
                 "launch_ms_mean": statistics.mean(k_ms)})
    return roof


class Workload:
    """Device inputs of one workload: a routing pool per M, x, the output and a
    shared workspace; one_call() runs one timed forward after an L2 flush."""

    def __init__(self, args, cfg, Ms, pw, dev, flush):
        import torch
        from weight_only_int4_moe_gb300 import ops
        self.args, self.cfg, self.Ms, self.pw, self.flush = args, cfg, Ms, pw, flush
        shape = pw.shape
        self.shape = shape
        ws_bytes = max(ops.moe_int4_workspace_bytes(M, shape) for M in Ms)
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        self.data = {}
        for M in Ms:
            t = inputs.make_tokens(cfg, M)
            pool = ([(t["topk_ids"], t["topk_weights"])]
                    + inputs.routing_pool(cfg, M, args.pool - 1))
            x = torch.from_numpy(t["x"].view(np.int16)).to(dev).view(torch.bfloat16)
            routes = []
            for ids, tw in pool:
                n = len(inputs.touched_experts(ids, cfg.E))
                routes.append((torch.from_numpy(ids).to(dev), torch.from_numpy(tw).to(dev), n))
            out = torch.empty((M, cfg.H), dtype=shape.torch_out_dtype, device=dev)
            d = {"x": x, "routes": routes, "out": out, "host": t}
            if args.routed:
                d["logits"] = [torch.from_numpy(lg).to(dev)
                               for lg in inputs.router_logits_pool(cfg, M, args.pool - 1)]
                d["rids"] = torch.empty((M, cfg.top_k), dtype=torch.int32, device=dev)
                d["rw"] = torch.empty((M, cfg.top_k), dtype=torch.float32, device=dev)
            self.data[M] = d

    def one_call(self, M, r, rec, stream, profiled=False):
        import torch
        from weight_only_int4_moe_gb300 import ops
        d = self.data[M]
        pw, shape = self.pw, self.shape
        ids, tw, n_touched = d["routes"][r % len(d["routes"])]
        self.flush.zero_()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        if self.args.routed:
            ops.moe_int4_forward_routed(d["x"], pw.w13, pw.w13_scales, pw.w2, pw.w2_scales,
                                        d["logits"][r % len(d["logits"])], shape, out=d["out"],
                                        topk_ids=d["rids"], topk_weights=d["rw"],
                                        workspace=self.ws, stream=stream)
        else:
            ops.moe_int4_forward(d["x"], pw.w13, pw.w13_scales, pw.w2, pw.w2_scales, ids, tw,
                                 shape, out=d["out"], workspace=self.ws, stream=stream)
        ev1.record(stream)
        launches = ops.moe_int4_last_launch_count()
        if rec is not None:
            stages = ops.moe_int4_profile_read() if profiled else None  # waits for the events
            ev1.synchronize()
            rec.append({"M": M, "ms": ev0.elapsed_time(ev1), "stages": stages,
                        "touched": n_touched, "launches": launches,
                        "fused": ops.moe_int4_fused(M, shape),
                        "gemv": ops.moe_int4_gemv(M, shape),
                        "block_down": ops.moe_int4_block_down(M, shape)})

    def profiled(self, steps, first, stream):
        """The same calls again with CUDA events between the kernels, on the
        launching stream (for the stage split and the roofline)."""
        import torch
        from weight_only_int4_moe_gb300 import ops
        ops.moe_int4_profile_enable(True)
        prec = []
        for s in range(steps):
            for M in self.Ms:
                self.one_call(M, first + s, prec, stream, profiled=True)
        torch.cuda.synchronize()
        ops.moe_int4_profile_enable(False)
        return prec

    def per_m(self, rec, prec, hbm_peak, tc_peak, fmt):
        cfg = self.cfg
        w13_b, w2_b = expert_bytes(cfg.H, cfg.I, fmt)
        out = {}
        for M in self.Ms:
            rs = [r for r in rec if r["M"] == M]
            us = [r["ms"] * 1e3 for r in rs]
            touched = statistics.mean(r["touched"] for r in rs)
            bytes_w = touched * (w13_b + w2_b)
            flops = 2.0 * M * cfg.top_k * 3 * cfg.H * cfg.I
            t_med = statistics.median(us)
            t_hbm = bytes_w / (hbm_peak * 1e9) * 1e6
            t_tc = flops / (tc_peak * 1e12) * 1e6
            st = np.mean([r["stages"] for r in prec if r["M"] == M], axis=0)
            fused = all(r["fused"] for r in rs)
            gemv = all(r["gemv"] for r in rs)
            block_down = all(r["block_down"] for r in rs)
            out[str(M)] = {
                "us_per_call": t_med, "us_mean": statistics.mean(us), "calls": len(us),
                "tokens_per_s": M / (t_med / 1e6),
                "touched_experts": touched,
                "weight_bytes": bytes_w,
                "hbm_gbs": bytes_w / (t_med / 1e6) / 1e9,
                "frac_hbm": bytes_w / (t_med / 1e6) / 1e9 / hbm_peak,
                "tflops": flops / (t_med / 1e6) / 1e12,
                "frac_tensor": flops / (t_med / 1e6) / 1e12 / tc_peak,
                "ideal_us": {"hbm": t_hbm, "tensor": t_tc},
                "bound": "hbm" if t_hbm >= t_tc else "tensor",
                "roofline_frac": max(t_hbm, t_tc) / t_med,
                "kernels": "gemv" if gemv else ("fused" if fused else (
                    "separate, block down" if block_down else "separate")),
                "stage_us": ({"route": st[0] * 1e3, "gate_up": st[1] * 1e3, "down": st[2] * 1e3,
                              "finalize": st[3] * 1e3} if gemv else
                             {"align": st[0] * 1e3, "fused": st[1] * 1e3, "finalize": st[3] * 1e3}
                             if fused else
                             {"align+gather": st[0] * 1e3, "gate_up": st[1] * 1e3,
                              "down": st[2] * 1e3, "finalize": st[3] * 1e3}),
            }
        return out


def extra_workloads(args, base_cfg):
    """The other workloads of the default run, each measured in a few calls per M
    (their own per-M numbers and roofline position): verify and prefill on the
    decode workload's weights, the mid-size MoE on its own."""
    if args.no_extra or args.workload != "k26_decode" or args.experts or args.ms:
        return []
    return [(inputs.WORKLOADS[n], n != "mid") for n in ("k26_verify", "k26_prefill", "mid")]


def run_ours(args, cfg, Ms, world, rank, local):
    import torch
    from weight_only_int4_moe_gb300 import ops

    dist = dist_init(world, local, True)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    out_dtype = ops.MOE_OUT_F32 if args.out_dtype == "f32" else ops.MOE_OUT_BF16

    w = make_weights(cfg, args.format)
    pw = ops.PackedWeights(w, cfg.E, cfg.H, cfg.I, cfg.top_k, device=dev, out_dtype=out_dtype,
                           fmt=args.format)
    shape = pw.shape
    Mmax = max(Ms)
    flush = torch.empty(args.flush_mb << 20, dtype=torch.uint8, device=dev)
    w13_b, w2_b = expert_bytes(cfg.H, cfg.I, args.format)
    wl = Workload(args, cfg, Ms, pw, dev, flush)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    # warm-up
    for s in range(args.warmup):
        for M in Ms:
            wl.one_call(M, s, None, stream)
    torch.cuda.synchronize()

    # timed region: whole calls, no events between the kernels (they would
    # hold back the overlap of each kernel's set-up with the previous one)
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    barrier(dist, True)
    torch.cuda.synchronize()
    clocks.start()
    rec = []
    wall0 = time.perf_counter()
    for s in range(args.steps):
        for M in Ms:
            wl.one_call(M, args.warmup + s, rec, stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(dist, True)
    clk = clocks.stop()
    prec = wl.profiled(args.steps, args.warmup, stream)

    ms_per_step = sum(r["ms"] for r in rec) / args.steps
    ms_per_step_max = allreduce_max(dist, ms_per_step, True)
    tokens_per_step = sum(Ms)
    value = job_rate(world, tokens_per_step, ms_per_step_max / 1e3)
    per_m = wl.per_m(rec, prec, hbm_peak, tc_peak, args.format)
    roofline = roofline_of(prec, w13_b, w2_b, cfg.top_k, cfg.H, cfg.I, hbm_peak, tc_peak,
                           peak_src, cfg.name)

    # the other workloads: a few calls per M each, same timing rules
    workloads = {}
    for xcfg, shared in extra_workloads(args, cfg):
        if shared:
            xpw = pw
        else:
            xw = make_weights(xcfg, args.format)
            xpw = ops.PackedWeights(xw, xcfg.E, xcfg.H, xcfg.I, xcfg.top_k, device=dev,
                                    out_dtype=out_dtype, fmt=args.format)
            del xw
        xpw.shape.top_k = xcfg.top_k
        xl = Workload(args, xcfg, xcfg.Ms, xpw, dev, flush)
        for s in range(3):
            for M in xcfg.Ms:
                xl.one_call(M, s, None, stream)
        xrec = []
        for s in range(args.extra_calls):
            for M in xcfg.Ms:
                xl.one_call(M, 3 + s, xrec, stream)
        torch.cuda.synchronize()
        xprec = xl.profiled(max(3, args.extra_calls // 2), 3, stream)
        xb13, xb2 = expert_bytes(xcfg.H, xcfg.I, args.format)
        workloads[xcfg.name] = {
            "config": {"E": xcfg.E, "top_k": xcfg.top_k, "hidden": xcfg.H, "inter": xcfg.I,
                       "Ms": list(xcfg.Ms), "routing": xcfg.routing,
                       "block_m": {str(M): ops.moe_int4_block_m(M, xpw.shape)
                                   for M in xcfg.Ms}},
            "per_m": xl.per_m(xrec, xprec, hbm_peak, tc_peak, args.format),
            "roofline": roofline_of(xprec, xb13, xb2, xcfg.top_k, xcfg.H, xcfg.I, hbm_peak,
                                    tc_peak, peak_src, xcfg.name),
        }
        del xl
        if not shared:
            del xpw
        torch.cuda.empty_cache()

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        ws_io = ops.alloc_workspace(Mmax, shape, flags=ops.MOE_WS_HOST_IO, device=dev)
        hosts = {}
        h2d = d2h = 0
        for M in Ms:
            t = wl.data[M]["host"]
            hx = torch.from_numpy(t["x"].view(np.int16)).pin_memory()
            hids = torch.from_numpy(t["topk_ids"]).pin_memory()
            htw = torch.from_numpy(t["topk_weights"]).pin_memory()
            hout = torch.empty((M, cfg.H), dtype=shape.torch_out_dtype).pin_memory()
            hosts[M] = (hx, hids, htw, hout)
            h2d += hx.numel() * 2 + hids.numel() * 4 + htw.numel() * 4
            d2h += hout.numel() * hout.element_size()
        for _ in range(max(1, args.warmup)):
            for M in Ms:
                ops.moe_int4_forward_host(hosts[M][0], pw.w13, pw.w13_scales, pw.w2,
                                          pw.w2_scales, hosts[M][1], hosts[M][2], hosts[M][3],
                                          shape, ws_io)
        torch.cuda.synchronize()
        e2e_s = 0.0
        for _ in range(args.steps):
            for M in Ms:
                flush.zero_()
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                ops.moe_int4_forward_host(hosts[M][0], pw.w13, pw.w13_scales, pw.w2,
                                          pw.w2_scales, hosts[M][1], hosts[M][2], hosts[M][3],
                                          shape, ws_io)
                e2e_s += time.perf_counter() - t0
        e2e_step = allreduce_max(dist, e2e_s / args.steps, True)
        e2e = {"value": job_rate(world, tokens_per_step, e2e_step), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_step * 1e3}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = host_threads()
        n, secs, Msamp = time_oracle(w, cfg, Ms, args.cpu_seconds, threads, fmt=args.format)
        cpu = {"value": n / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} tokens of the M={Msamp} call, fp64 oracle, {threads} threads, "
                         f"{secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": {"workload": cfg.name, "E": cfg.E, "top_k": cfg.top_k, "hidden": cfg.H,
                       "inter": cfg.I, "group": 32, "weight_format": args.format, "Ms": list(Ms),
                       "step": "one moe_int4_forward per M",
                       "l2": f"flushed by a {args.flush_mb} MB device write before every call; "
                             f"routing rotates over {args.pool} seeded routings per M",
                       "out_dtype": args.out_dtype, "parallelism": f"replicas x{world}",
                       "routing": ("router logits -> top-k in the call (moe_int4_forward_routed)"
                                   if args.routed else "precomputed top-k ids and weights"),
                       "block_m": {str(M): ops.moe_int4_block_m(M, shape) for M in Ms}},
            "per_m": per_m, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(sum(r["launches"] for r in rec)),
            "clocks": clk, "wall_s_timed": wall,
            "workloads": workloads,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse_args()
    cfg = inputs.WORKLOADS[args.workload]
    if args.experts:
        cfg = dataclasses.replace(cfg, E=args.experts, name=f"{cfg.name}_E{args.experts}")
    if args.format != "int4":
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}_{args.format}")
    Ms = tuple(int(m) for m in args.ms.split(",")) if args.ms else cfg.Ms
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, cfg, Ms, world, rank)
        return
    run_ours(args, cfg, Ms, world, rank, local)


if __name__ == "__main__":
    main()

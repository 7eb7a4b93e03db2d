#!/usr/bin/env python3
"""Benchmark of the PLX attention hot path on B300.

One step = one pass of the whole hot path on HBM-resident synthetic inputs:
  * plx_fwd on the prefill workload B=4, H=16, N=2048, d=128 (bf16, causal,
    rho = W_R x), outputs o and lse in fp32 (bf16 storage of o would add
    rounding beyond the parity tolerance on rows where |o| is far above its RMS);
  * plx_fwd on the long-sequence prefill B=2, H=16, N=8192, d=128 (bf16,
    planted keys, rho ~ N(0, 0.1^2)), fp32 o and lse, reported in its own
    block with its own roofline;
  * plx_decode on the decode workload B=64, H=16, d=128, bf16 KV cache with
    every length 4096 (split-KV + LSE combine).
The headline value is prefill TFLOP/s, counting 8*d flop per causal
(query, key) pair (four GEMMs: QK^T, rho K^T, PV, (P o R)V).  Decode is
reported beside it in GB/s of K/V read (sum of lengths * H * d * 2 tensors
* 2 bytes, plus q, rho, out).  Kernel durations come from CUDA events on the
launching stream; L2 is flushed (a 256 MiB write) before every timed launch,
outside the events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --impl reference the fp64 CPU oracle is timed on the host cores on a
bounded sample of the same prefill workload (it is the reference arm: this
method has no runnable reference implementation).  Under torchrun (N > 1)
every rank runs the same per-GPU workload (weak scaling, no data-path
collective) and rank 0 prints one JSON line.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "PLX prefill TFLOP/s and decode KV GB/s vs B300 roofline, 1 GPU"
PREFILL = "prefill_b4_h16_n2048_d128"
PREFILL_LONG = "prefill_b2_h16_n8192_d128_planted"
DECODE = "decode_b64_h16_ctx4096_d128"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def prefill_flops(B, H, N, d, plx=True):
    pairs = B * H * N * (N + 1) / 2
    return pairs * (8 if plx else 4) * d


def decode_bytes(seqlens, H, d, plx=True):
    kv = float(np.sum(seqlens)) * H * d * 2 * 2
    small = len(seqlens) * H * d * 2 * (3 if plx else 2)      # q, (rho), out (bf16)
    return kv + small


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


def kernel_source_hash():
    """sha256 over the CUDA sources (file name + bytes, sorted by name)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "parameterized_local_linear_02_b300", "csrc", "*"))):
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def read_traffic():
    """Per-launch DRAM bytes of the timed kernels from the committed ncu
    summary (profiles/traffic.json).  An entry taken from other kernel
    sources than the ones built now is stale and dropped, so the caller
    reports null for it."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        data = json.load(f)
    now = kernel_source_hash()
    return {k: v for k, v in data.items() if isinstance(v, dict) and v.get("source_sha256") == now}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def hold_device(us=100.0):
    """Queue a spin kernel of about `us` microseconds on the current stream.
    A CUDA-event pair recorded on an idle device also times the host's work
    to issue the launch between them (argument checks, tensor-map encoding,
    the launch call): the start event fires at once and the device then
    waits for the kernel.  With the device busy for longer than that, the
    launch is queued before the start event fires, and the pair times the
    kernel alone.  It is queued before the L2 flush, outside every timed
    pair."""
    import torch
    torch.cuda._sleep(int(us * 2000))    # clock64 cycles, about 2 GHz


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The largest x over all ranks (the slowest rank's time); x itself at N=1.
    Uses a host tensor under the gloo backend and a device tensor under NCCL."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(units_per_rank, ms_per_rank, world):
    """Whole-job throughput when every rank processes its own fixed share:
    all ranks' units divided by the slowest rank's time (units per second)."""
    slowest = max_over_ranks(ms_per_rank, world)
    return world * units_per_rank / (slowest * 1e-3)


def rank_seed(seed, rank):
    """Seed of a rank's shard: ranks draw distinct inputs of the same shape."""
    return seed + 1000003 * rank


# ------------------------------------------------------------------ CPU oracle
def oracle_prefill_sample(cfg, budget_s=12.0, x=None, per_batch=4):
    """Time the fp64 oracle (streaming form, all host threads) on whole heads
    of the prefill workload, ``per_batch`` heads at a time, until ``budget_s``
    has elapsed or every head is done.  Returns (TFLOP/s, seconds,
    description, threads)."""
    import oracle
    import plx_inputs
    if x is None:
        x = plx_inputs.prefill(cfg["B"], cfg["H"], cfg["N"], cfg["d"], seed=cfg["seed"], dtype="bf16",
                               rho=cfg["rho"], keys=cfg["keys"])
    heads = [(b, h) for b in range(cfg["B"]) for h in range(cfg["H"])]
    done, flops, t0 = 0, 0.0, time.perf_counter()
    threads = oracle.n_threads()
    while done < len(heads) and time.perf_counter() - t0 < budget_s:
        batch = heads[done:done + per_batch]
        oracle.prefill("stream", x.q, x.k, x.v, x.rho, x.scale, heads=batch, threads=threads)
        done += len(batch)
        flops += len(batch) * prefill_flops(1, 1, cfg["N"], cfg["d"])
    dt = time.perf_counter() - t0
    desc = f"{done} of {len(heads)} heads (all {cfg['N']} rows each) of the prefill workload, stream form"
    return flops / dt / 1e12, dt, desc, threads


def oracle_decode_sample(budget_s=5.0):
    """Time the fp64 oracle (streaming form, all host threads) on host-drawn
    (b, h) rows of the decode workload's shape (context 4096, d=128) until
    ``budget_s`` has elapsed.  Returns (GB/s of K/V processed, seconds,
    description, threads)."""
    import oracle
    import plx_inputs
    dc = plx_inputs.CONFIGS[DECODE]
    H, d, S = dc["H"], dc["d"], dc["S_cap"]
    x = plx_inputs.decode(1, H, d, S, seed=dc["seed"], seqlens="full", rho_std=dc["rho_std"])
    threads = oracle.n_threads()
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        oracle.decode("stream", x.q, x.rho, x.k_cache, x.v_cache, x.seqlens, x.scale, threads=threads)
        done += H
    dt = time.perf_counter() - t0
    gbs = done * S * d * 2 * 2 / dt / 1e9
    desc = f"{done} (b, h) rows of length {S} (one batch row of the decode workload, repeated), stream form"
    return gbs, dt, desc, threads


def step_config(do_pf=True, do_long=True, do_dec=True, decode_batch=None):
    """The workload a bench step times (the same dict on both arms)."""
    import plx_inputs
    pc = plx_inputs.CONFIGS[PREFILL]
    cfg = {"workload": PREFILL if do_pf else (PREFILL_LONG if do_long else DECODE), "B": pc["B"], "H": pc["H"],
           "N": pc["N"], "d": pc["d"], "causal": True, "rho": "W_R x", "out": "fp32 o + fp32 lse",
           "l2": "flushed (256 MiB write) before every launch"}
    if do_long:
        cfg["long_prefill_workload"] = PREFILL_LONG
    if do_dec:
        cfg.update({"decode_workload": DECODE,
                    "decode_batch": decode_batch or plx_inputs.CONFIGS[DECODE]["B"]})
    return cfg


def run_reference(args, world, rank):
    import plx_inputs
    if rank != 0:
        return 0
    cfg = plx_inputs.CONFIGS[PREFILL]
    x = plx_inputs.prefill(cfg["B"], cfg["H"], cfg["N"], cfg["d"], seed=cfg["seed"], dtype="bf16",
                           rho=cfg["rho"], keys=cfg["keys"])
    per_step_budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_prefill_sample(cfg, budget_s=min(per_step_budget, 2.0), x=x)
    vals, times, desc, threads = [], [], "", 1
    for _ in range(args.steps):
        v, dt, desc, threads = oracle_prefill_sample(cfg, budget_s=per_step_budget, x=x)
        vals.append(v)
        times.append(dt)
    value = float(np.median(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * float(np.median(times)), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(args.only in ("both", "prefill"), args.only in ("both", "long") and not args.no_long,
                              args.only in ("both", "decode"), args.decode_batch),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU path
def run_ours(args, world, rank, local):
    import torch
    import parameterized_local_linear_02_b300 as plx
    import plx_inputs

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks = read_peaks()
    do_pf = args.only in ("both", "prefill")
    do_long = args.only in ("both", "long") and not args.no_long
    do_dec = args.only in ("both", "decode")
    extras = not args.no_extras

    pc = plx_inputs.CONFIGS[PREFILL]
    dc = plx_inputs.CONFIGS[DECODE]
    B, H, N, d = pc["B"], pc["H"], pc["N"], pc["d"]
    Bd, Hd, S_cap = (args.decode_batch or dc["B"]), dc["H"], dc["S_cap"]
    x = None
    if do_pf:
        x = plx_inputs.prefill(B, H, N, d, seed=rank_seed(pc["seed"], rank), dtype="bf16", rho=pc["rho"],
                               keys=pc["keys"])
        t = x.device_tensors(dev)
        out = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    lc = plx_inputs.CONFIGS[PREFILL_LONG]
    Bl, Hl, Nl, dl = lc["B"], lc["H"], lc["N"], lc["d"]
    if do_long:
        xl = plx_inputs.prefill(Bl, Hl, Nl, dl, seed=rank_seed(lc["seed"], rank), dtype="bf16", rho=lc["rho"],
                                rho_std=lc["rho_std"], keys=lc["keys"])
        tl = xl.device_tensors(dev)
        if world > 1 or args.no_cpu_baseline:
            del xl
            xl = None
        out_l = torch.empty((Bl, Hl, Nl, dl), dtype=torch.float32, device=dev)
        lse_l = torch.empty((Bl, Hl, Nl), dtype=torch.float32, device=dev)
    if do_dec:
        dd = plx_inputs.decode_device(Bd, Hd, dc["d"], S_cap, seed=rank_seed(dc["seed"], rank), seqlens=dc["seqlens"],
                                      rho_std=dc["rho_std"], device=dev)
        dout = torch.empty((Bd, Hd, dc["d"]), dtype=torch.bfloat16, device=dev)
        dlse = torch.empty((Bd, Hd), dtype=torch.float32, device=dev)
        splits = plx.plx_decode_num_splits(Bd, Hd, dc["d"], S_cap)
        ws_bytes = plx.plx_decode_workspace_size(Bd, Hd, dc["d"], S_cap, splits)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def fwd(rho=True):
        plx.plx_fwd(t["q"], t["k"], t["v"], t["rho"] if rho else None, out=out, lse=lse)

    def fwd_long(rho=True):
        plx.plx_fwd(tl["q"], tl["k"], tl["v"], tl["rho"] if rho else None, out=out_l, lse=lse_l)

    def dec(rho=True):
        plx.plx_decode(dd["q"], dd["rho"] if rho else None, dd["k_cache"], dd["v_cache"], dd["seqlens"],
                       num_splits=splits, workspace=ws, out=dout, lse=dlse)

    launches_per_step = (1 if do_pf else 0) + (1 if do_long else 0) + ((2 if splits > 1 else 1) if do_dec else 0)

    def timed(fn, k):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        return evs

    # the clock sampler starts (and gets its first sample) before the warm-up,
    # so the GPU does not idle between the warm-up and the timed region (an
    # idle GPU drops its clocks, and the first timed launches would run while
    # they ramp back up)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        flush.zero_()
        if do_pf:
            fwd()
        if do_long:
            fwd_long()
        if do_dec:
            dec()
    torch.cuda.synchronize()
    if plx.plx_last_device_error() != 0:
        raise RuntimeError("device status set during warm-up")

    # ---- timed region: K steps of (prefill, decode)
    barrier(world)
    torch.cuda.synchronize()
    ev_f, ev_l, ev_d = [], [], []
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # the device works through this while the host queues the first steps; a
    # step's launches then run well behind the host, so no timed pair
    # contains the time to issue a launch
    hold_device(1000.0)
    t_start.record(stream)
    for _ in range(args.steps):
        if do_pf:
            ev_f += timed(fwd, 1)
        if do_long:
            ev_l += timed(fwd_long, 1)
        if do_dec:
            ev_d += timed(dec, 1)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    wall_ms = t_start.elapsed_time(t_end)
    status = plx.plx_last_device_error()
    line = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic"}
    traffic = read_traffic()

    if do_pf:
        f_avg = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev_f])), world)
        flops = prefill_flops(B, H, N, d)
        value = world * flops / (f_avg * 1e-3) / 1e12
        line.update({"value": value, "unit": "TFLOP/s"})
        line["roofline"] = {
            "bound": "tensor", "achieved": value / world, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": value / world / peaks["bf16_tflops"],
            "traffic": traffic.get("plx_fwd", {}).get("bytes_per_launch"),
            "peak_source": f"{peaks['source']} bf16 dense (burst)",
            "frac_of_sustained": value / world / peaks["bf16_tflops_sustained"],
            "kernel": "plx_fwd_tc_kernel<128,true>", "flop_per_launch": flops, "avg_launch_ms": f_avg}
    if do_long:
        l_avg = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev_l])), world)
        l_flops = prefill_flops(Bl, Hl, Nl, dl)
        l_val = world * l_flops / (l_avg * 1e-3) / 1e12
        lroof = {"bound": "tensor", "achieved": l_val / world, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                 "frac": l_val / world / peaks["bf16_tflops"],
                 "traffic": traffic.get("plx_fwd_long", {}).get("bytes_per_launch"),
                 "peak_source": f"{peaks['source']} bf16 dense (burst)",
                 "frac_of_sustained": l_val / world / peaks["bf16_tflops_sustained"],
                 "kernel": "plx_fwd_tc_kernel<128,true>", "flop_per_launch": l_flops, "avg_launch_ms": l_avg}
        line["prefill_long"] = {"workload": PREFILL_LONG, "value": l_val, "unit": "TFLOP/s", "ms": l_avg,
                                "B": Bl, "H": Hl, "N": Nl, "d": dl, "keys": "planted (64 centres + N(0, 0.05^2))",
                                "rho": "N(0, 0.1^2)", "out": "fp32 o + fp32 lse",
                                "l2": "flushed (256 MiB write) before every launch", "roofline": lroof}
        if not do_pf:
            line.update({"value": l_val, "unit": "TFLOP/s", "roofline": lroof})
    if do_dec:
        d_avg = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev_d])), world)
        dbytes = decode_bytes(dd["seqlens_host"], Hd, dc["d"])
        d_gbs = world * dbytes / (d_avg * 1e-3) / 1e9
        droof = {"bound": "hbm", "achieved": d_gbs / world, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                 "frac": d_gbs / world / peaks["hbm_gbs"],
                 "traffic": traffic.get("plx_decode", {}).get("bytes_per_launch"),
                 "peak_source": f"{peaks['source']} HBM copy", "bytes_per_launch": dbytes,
                 "avg_launch_ms": d_avg,
                 "kernel": "plx_decode_split_kernel<128,true>" + (" + combine" if splits > 1 else "")}
        line["decode"] = {"value": d_gbs, "unit": "GB/s", "ms": d_avg, "batch": Bd, "splits": splits,
                          "tokens_per_s": world * Bd / (d_avg * 1e-3), "roofline": droof}
        if not do_pf and not do_long:
            line.update({"value": d_gbs, "unit": "GB/s", "roofline": droof})
    line["ms_per_step"] = ((f_avg if do_pf else 0.0) + (l_avg if do_long else 0.0)
                           + (d_avg if do_dec else 0.0))
    line["config"] = step_config(do_pf, do_long, do_dec, Bd)

    if extras and do_pf:
        # the same launches back to back, no L2 flush between them (sustained clocks)
        bb_n = max(20, args.steps)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(bb_n):
            fwd()
        e1.record(stream)
        torch.cuda.synchronize()
        bb_ms = e0.elapsed_time(e1) / bb_n
        line["roofline"]["back_to_back"] = {"launches": bb_n, "avg_launch_ms": bb_ms,
                                            "achieved": prefill_flops(B, H, N, d) / bb_ms / 1e9,
                                            "frac_of_sustained": prefill_flops(B, H, N, d) / bb_ms / 1e9
                                            / peaks["bf16_tflops_sustained"]}
    if extras:
        sa = {}
        hold_device(1000.0)
        if do_pf:
            sa_f = timed(lambda: fwd(False), max(5, args.steps // 2))
        if do_long:
            sa_l = timed(lambda: fwd_long(False), max(3, args.steps // 4))
        if do_dec:
            sa_d = timed(lambda: dec(False), max(5, args.steps // 2))
        torch.cuda.synchronize()
        if do_pf:
            sa_f_ms = float(np.mean([a.elapsed_time(b) for a, b in sa_f]))
            sa.update({"prefill_ms": sa_f_ms,
                       "prefill_tflops_4d": prefill_flops(B, H, N, d, False) / sa_f_ms / 1e9,
                       "plx_over_sa_time": f_avg / sa_f_ms})
        if do_long:
            sa_l_ms = float(np.mean([a.elapsed_time(b) for a, b in sa_l]))
            sa.update({"prefill_long_ms": sa_l_ms,
                       "prefill_long_tflops_4d": prefill_flops(Bl, Hl, Nl, dl, False) / sa_l_ms / 1e9,
                       "prefill_long_plx_over_sa_time": l_avg / sa_l_ms})
        if do_dec:
            sa_d_ms = float(np.mean([a.elapsed_time(b) for a, b in sa_d]))
            sa.update({"decode_ms": sa_d_ms,
                       "decode_gbs": decode_bytes(dd["seqlens_host"], Hd, dc["d"], False) / sa_d_ms / 1e6})
        line["softmax_attention_same_kernel"] = sa
        if do_pf:
            # end to end through the C ABI with host buffers: plx_fwd_host copies
            # the pinned q, k, v, rho in and out, lse back in chunks of heads,
            # overlapping the copies with the kernels
            pin = {n: t[n].cpu().pin_memory() for n in ("q", "k", "v", "rho")}
            h_out = torch.empty((B, H, N, d), dtype=torch.float32).pin_memory()
            h_lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
            h_ws = torch.empty(plx.plx_fwd_host_workspace_size(B, H, N, d, torch.float32), dtype=torch.uint8,
                               device=dev)
            h2d = sum(v.numel() * v.element_size() for v in pin.values())
            d2h = h_out.numel() * 4 + h_lse.numel() * 4

            def e2e_step():
                plx.plx_fwd_host(pin["q"], pin["k"], pin["v"], pin["rho"], h_out, h_lse, workspace=h_ws,
                                 stream=stream)

            for _ in range(2):
                e2e_step()
            torch.cuda.synchronize()
            e_steps = max(5, args.steps // 2)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(e_steps):
                e2e_step()
            e1.record(stream)
            torch.cuda.synchronize()
            e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world)
            # the same transfers and launch without the overlap, for comparison
            d_in = {n: torch.empty_like(t[n]) for n in pin}

            def serial_step():
                for n in pin:
                    d_in[n].copy_(pin[n], non_blocking=True)
                plx.plx_fwd(d_in["q"], d_in["k"], d_in["v"], d_in["rho"], out=out, lse=lse)
                h_out.copy_(out, non_blocking=True)
                h_lse.copy_(lse, non_blocking=True)

            serial_step()
            torch.cuda.synchronize()
            e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e2.record(stream)
            for _ in range(e_steps):
                serial_step()
            e3.record(stream)
            torch.cuda.synchronize()
            s_ms = e2.elapsed_time(e3) / e_steps
            line["e2e"] = {"value": world * flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
                           "path": "plx_fwd_host: pinned host q, k, v, rho -> device in chunks of heads, "
                                   "plx_fwd per chunk, out + lse -> pinned host, copies overlapping the kernels",
                           "serial_ms_per_step": s_ms,
                           "pcie_gbs": (h2d + d2h) / (e_ms * 1e-3) / 1e9}
    line["gpu_launches"] = launches_per_step * args.steps
    line["clocks"] = clocks
    line["wall_ms_timed_region"] = wall_ms
    line["device_status"] = status
    if rank == 0 and world == 1 and do_pf and not args.no_cpu_baseline:
        v, dt, desc, threads = oracle_prefill_sample(pc, budget_s=args.cpu_budget, x=x)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": desc, "seconds": dt}
        if do_long and xl is not None:
            lv, ldt, ldesc, lthreads = oracle_prefill_sample(lc, budget_s=min(6.0, args.cpu_budget), x=xl,
                                                             per_batch=1)
            line["cpu_baseline"]["prefill_long"] = {"value": lv, "unit": "TFLOP/s", "cores": lthreads,
                                                    "kind": "oracle", "sample": ldesc, "seconds": ldt}
        if do_dec:
            gbs, ddt, ddesc, dthreads = oracle_decode_sample(min(5.0, args.cpu_budget))
            line["cpu_baseline"]["decode"] = {"value": gbs, "unit": "GB/s", "cores": dthreads, "kind": "oracle",
                                              "sample": ddesc, "seconds": ddt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_decode_sweep(args, world, rank, local):
    """Decode over a sweep of batch x context (per-sequence lengths drawn
    uniformly from [ctx/2, ctx]), H=16, d=128, bf16 cache; cells whose K+V
    cache would exceed the 180 GB cap are listed as not run.  Each cell times
    PLX and the rho = NULL (softmax attention) instantiation of the same
    kernels; L2 is flushed (256 MiB write) before every timed launch, outside
    the events.  Prints one JSON line."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    import plx_inputs

    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    cfg = plx_inputs.CONFIGS["decode_sweep"]
    H, d = cfg["H"], cfg["d"]
    cap = 180e9
    peaks = read_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cells = []
    sampler = ClockSampler(local)
    sampler.start()
    for B in cfg["batches"]:
        for ctx in cfg["contexts"]:
            cache_bytes = 2 * B * H * ctx * d * 2
            cell = {"batch": B, "context": ctx, "cache_gb": cache_bytes / 1e9}
            if cache_bytes > cap:
                cell["status"] = "does not fit (180 GB cap)"
                cells.append(cell)
                continue
            seed = cfg["seed"] + 100 * B + ctx // 1024
            t = plx_inputs.decode_device(B, H, d, ctx, seed=seed, seqlens="ragged", rho_std=cfg["rho_std"],
                                         device=dev)
            splits = plx.plx_decode_num_splits(B, H, d, ctx)
            ws = torch.empty(max(plx.plx_decode_workspace_size(B, H, d, ctx, splits), 16), dtype=torch.uint8,
                             device=dev)
            out = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((B, H), dtype=torch.float32, device=dev)
            res = {}
            for name, rho in (("plx", t["rho"]), ("sa", None)):
                def call():
                    plx.plx_decode(t["q"], rho, t["k_cache"], t["v_cache"], t["seqlens"], num_splits=splits,
                                   workspace=ws, out=out, lse=lse)
                for _ in range(3):
                    call()
                ms = []
                for _ in range(args.sweep_iters):
                    hold_device()
                    flush.zero_()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    call()
                    b.record(stream)
                    torch.cuda.synchronize()
                    ms.append(a.elapsed_time(b))
                med = float(np.median(ms))
                nbytes = decode_bytes(t["seqlens_host"], H, d, plx=(rho is not None))
                res[name] = {"ms": med, "gbs": nbytes / (med * 1e-3) / 1e9,
                             "frac_hbm": nbytes / (med * 1e-3) / 1e9 / peaks["hbm_gbs"],
                             "tokens_per_s": B / (med * 1e-3)}
            cell.update({"splits": splits, "kv_bytes": float(decode_bytes(t["seqlens_host"], H, d)),
                         "mean_len": float(np.mean(t["seqlens_host"])), "plx": res["plx"], "sa": res["sa"]})
            status = plx.plx_last_device_error()
            cell["device_status"] = status
            cells.append(cell)
            print(f"# B={B:4d} ctx={ctx:6d} splits={splits:4d} PLX {res['plx']['ms']:.4f} ms "
                  f"{res['plx']['gbs']:7.1f} GB/s  SA {res['sa']['ms']:.4f} ms {res['sa']['gbs']:7.1f} GB/s",
                  file=sys.stderr, flush=True)
            del t, ws, out, lse
            torch.cuda.empty_cache()
    clocks = sampler.stop()
    line = {"metric": "PLX decode KV GB/s over batch x context (ragged lengths), 1 GPU", "unit": "GB/s",
            "higher_is_better": True, "n_gpus": 1, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "decode_sweep", "H": H, "d": d, "lengths": "U[ctx/2, ctx] per sequence",
                       "l2": "flushed (256 MiB write) before every launch", "iters_per_cell": args.sweep_iters},
            "peak_hbm_gbs": peaks["hbm_gbs"], "cells": cells, "clocks": clocks}
    print(json.dumps(line), flush=True)
    return 0


def run_backward_bench(args, world, rank, local):
    """plx_bwd (tensor cores, bf16 inputs) on the prefill workload's shape
    (B=4, H=16, N=2048, d=128) with a seeded bf16 dL/do.  TFLOP/s counts 14 d
    flop per causal pair: S, R and dO V^T once (3 x 2d), dq, drho (2 x 2d),
    dk (4d), dv (2d); the implementation runs 28 d (S, R, G in each of its three
    passes: the row statistics, dq/drho, dk/dv).  The
    roofline is the measured dense bf16 tensor rate.  plx_bwd_f32 (CUDA
    cores) is timed beside it on the same values widened to fp32, with its o
    and lse from plx_fwd_f32 (not timed).  Prints one JSON line."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    import plx_inputs

    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    pc = plx_inputs.CONFIGS[PREFILL]
    B, H, N, d = pc["B"], pc["H"], pc["N"], pc["d"]
    x = plx_inputs.prefill(B, H, N, d, seed=pc["seed"], dtype="bf16", rho=pc["rho"], keys=pc["keys"])
    tb = x.device_tensors(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    dout = torch.randn((B, H, N, d), generator=g, device=dev).to(torch.bfloat16)
    grads = tuple(torch.empty((B, H, N, d), dtype=torch.float32, device=dev) for _ in range(4))
    ws = torch.empty(plx.plx_bwd_bf16_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn, steps, warmup):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(steps):
            hold_device()
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return float(np.median(ms)), len(ms)

    def call():
        plx.plx_bwd(tb["q"], tb["k"], tb["v"], tb["rho"], dout, scale=x.scale, workspace=ws, grads=grads)

    # the sampler's first readings come in before the warm-up (as in the main step)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    med, nsteps = timed(call, max(3, args.steps), 0)
    clocks = sampler.stop()
    # the fp32 path on the same values
    t32 = {n: tb[n].float() for n in ("q", "k", "v", "rho")}
    out32, lse32 = plx.plx_fwd_f32(t32["q"], t32["k"], t32["v"], t32["rho"], scale=x.scale)
    ws32 = torch.empty(plx.plx_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    dout32 = dout.float()
    f32_ms, _ = timed(lambda: plx.plx_bwd_f32(t32["q"], t32["k"], t32["v"], t32["rho"], out32, lse32, dout32,
                                              scale=x.scale, workspace=ws32, grads=grads), 3, 1)
    pairs = B * H * N * (N + 1) / 2
    flops = pairs * 14 * d
    value = flops / (med * 1e-3) / 1e12
    peaks = read_peaks()
    peak = peaks["bf16_tflops"]
    peak_s = peaks["bf16_tflops_sustained"]
    props = torch.cuda.get_device_properties(dev)
    sm_max = clocks.get("sm_max_mhz") or 2032.0
    alu_peak = props.multi_processor_count * 128 * 2 * sm_max * 1e6 / 1e12
    line = {"metric": "PLX backward (dq, dk, dv, drho) TFLOP/s, bf16 inputs on the tensor cores, 1 GPU",
            "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": nsteps, "warmup": max(3, args.warmup),
            "ms_per_step": med, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": PREFILL, "B": B, "H": H, "N": N, "d": d, "causal": True, "rho": "W_R x",
                       "inputs": "bf16 q, k, v, rho, dout (lse and the row statistics recomputed by the statistics pass)",
                       "l2": "flushed (256 MiB write) before every launch"},
            "roofline": {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s", "frac": value / peak,
                         "peak_source": f"{peaks['source']} bf16 dense (burst)",
                         "frac_of_sustained": value / peak_s,
                         "flop_per_launch": flops, "flop_per_pair": 14 * d, "implementation_flop_per_pair": 28 * d,
                         "implementation_tflops": pairs * 28 * d / (med * 1e-3) / 1e12},
            "f32_path": {"ms": f32_ms, "value": flops / (f32_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                         "roofline": {"bound": "alu", "peak": alu_peak,
                                      "frac": flops / (f32_ms * 1e-3) / 1e12 / alu_peak}},
            "speedup_over_f32_path": f32_ms / med,
            "gpu_launches": 3 * nsteps, "clocks": clocks}
    # the training pair: plx_fwd_train saves vbar and c beside o and lse, and
    # plx_bwd_saved forms the row statistics from them (a bandwidth-bound
    # kernel) instead of the statistics pass
    o_t = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    lse_t = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    vbar_t = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    c_t = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fwd_train = lambda: plx.plx_fwd_train(tb["q"], tb["k"], tb["v"], tb["rho"], scale=x.scale, out=o_t, lse=lse_t,
                                          vbar=vbar_t, c=c_t)
    fwd_plain = lambda: plx.plx_fwd(tb["q"], tb["k"], tb["v"], tb["rho"], scale=x.scale, out=o_t, lse=lse_t)
    fp_ms, _ = timed(fwd_plain, max(3, args.steps), 3)
    ft_ms, _ = timed(fwd_train, max(3, args.steps), 3)
    sv_ms, sv_steps = timed(lambda: plx.plx_bwd_saved(tb["q"], tb["k"], tb["v"], tb["rho"], dout, o_t, lse_t, vbar_t,
                                                      c_t, scale=x.scale, workspace=ws, grads=grads),
                            max(3, args.steps), 3)
    sv_val = flops / (sv_ms * 1e-3) / 1e12
    fwd_flops = pairs * 8 * d
    line["saved_path"] = {
        "bwd_ms": sv_ms, "value": sv_val, "unit": "TFLOP/s", "frac": sv_val / peak,
        "implementation_flop_per_pair": 20 * d,
        "fwd_train_ms": ft_ms, "fwd_ms": fp_ms, "fwd_train_tflops": fwd_flops / (ft_ms * 1e-3) / 1e12,
        "train_step_ms": ft_ms + sv_ms, "recompute_train_step_ms": fp_ms + med,
        "inputs": "plx_fwd_train's o (fp32), lse, vbar (fp32), c; bf16 q, k, v, rho, dout",
        "l2": "flushed (256 MiB write) before every launch"}
    line["gpu_launches"] += 3 * sv_steps
    line["device_status"] = plx.plx_last_device_error()
    print(json.dumps(line), flush=True)
    return 0


def run_cached_bench(args, world, rank, local):
    """plx_fwd_cached (T new tokens per sequence on the tensor cores) on the
    decode workload's cache (B=64, H=16, every length 4096, d=128), for T in
    (1, 16, 64, 128), beside plx_decode on the same cache.  The cache is read
    once per (b, h) whatever T is, so the roofline is HBM bandwidth over the
    K/V bytes; tokens/s = B * T / time.  L2 is flushed before every launch.
    Prints one JSON line."""
    import torch
    import parameterized_local_linear_02_b300 as plx
    import plx_inputs

    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    dc = plx_inputs.CONFIGS[DECODE]
    B, H, d, S = dc["B"], dc["H"], dc["d"], dc["S_cap"]
    g = torch.Generator(device=dev)
    g.manual_seed(dc["seed"])
    kc = torch.randn((B, H, S, d), generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn((B, H, S, d), generator=g, device=dev).to(torch.bfloat16)
    seqlens = torch.full((B,), S, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    peaks = read_peaks()

    def timed(fn, steps):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(steps):
            hold_device()
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return float(np.median(ms))

    kv_bytes = B * H * S * d * 2 * 2
    q1 = torch.randn((B, H, d), generator=g, device=dev).to(torch.bfloat16)
    r1 = (0.1 * torch.randn((B, H, d), generator=g, device=dev)).to(torch.bfloat16)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    dec_ms = timed(lambda: plx.plx_decode(q1, r1, kc, vc, seqlens), max(3, args.steps))
    rows = []
    for T in (1, 16, 64, 128):
        q = torch.randn((B, H, T, d), generator=g, device=dev).to(torch.bfloat16)
        r = (0.1 * torch.randn((B, H, T, d), generator=g, device=dev)).to(torch.bfloat16)
        out = torch.empty((B, H, T, d), dtype=torch.bfloat16, device=dev)
        ms = timed(lambda: plx.plx_fwd_cached(q, r, kc, vc, seqlens, out=out, with_lse=False), max(3, args.steps))
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        rows.append({"T": T, "ms": ms, "kv_gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
                     "tokens_per_s": B * T / (ms * 1e-3), "vs_T_decode_calls": T * dec_ms / ms})
    clocks = sampler.stop()
    line = {"metric": "PLX multi-token decode against a KV cache (plx_fwd_cached), K/V GB/s and tokens/s, 1 GPU",
            "unit": "GB/s", "value": rows[1]["kv_gbs"], "n_gpus": 1, "steps": max(3, args.steps),
            "warmup": max(3, args.warmup), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": DECODE, "B": B, "H": H, "S": S, "d": d, "value_at_T": 16,
                       "l2": "flushed (256 MiB write) before every launch"},
            "roofline": {"bound": "hbm", "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "peak_source": f"{peaks['source']} HBM copy"},
            "plx_decode_ms": dec_ms, "plx_decode_kv_gbs": kv_bytes / (dec_ms * 1e-3) / 1e9, "by_T": rows,
            "clocks": clocks,
            "gpu_launches": (4 + 1) * max(3, args.steps), "device_status": plx.plx_last_device_error()}
    print(json.dumps(line), flush=True)
    return 0


def run_proj_bench(args, world, rank, local):
    """plx_probe_proj (tcgen05 GEMM rho = W_R x written in the [B, H, N, d]
    layout) on the prefill workload's probe: x [4, 2048, 1024] bf16, W_R
    [16 * 128, 1024] bf16.  flop = 2 B N (H d) Dx; the roofline is the
    measured dense bf16 tensor rate.  For context, torch's matmul (cuBLAS) of
    the same operands, alone and followed by the [B, N, H, d] -> [B, H, N, d]
    copy the PLX kernels need.  L2 is flushed before every launch.  Prints
    one JSON line."""
    import torch
    import parameterized_local_linear_02_b300 as plx

    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    B, N, H, d, Dx = 4, 2048, 16, 128, 1024
    g = torch.Generator(device=dev)
    g.manual_seed(13)
    x = torch.randn((B, N, Dx), generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn((H * d, Dx), generator=g, device=dev) / math.sqrt(Dx)).to(torch.bfloat16)
    rho = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn, steps):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(steps):
            hold_device()
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return float(np.median(ms)), len(ms)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for _ in range(max(3, args.warmup)):
        plx.plx_probe_proj(x, w, heads=H, out=rho)
    torch.cuda.synchronize()
    med, nsteps = timed(lambda: plx.plx_probe_proj(x, w, heads=H, out=rho), max(3, args.steps))
    clocks = sampler.stop()
    y = torch.empty((B * N, H * d), dtype=torch.bfloat16, device=dev)
    x2 = x.view(B * N, Dx)
    mm_ms, _ = timed(lambda: torch.matmul(x2, w.t(), out=y), max(3, args.steps))
    mmp_ms, _ = timed(lambda: rho.copy_(torch.matmul(x2, w.t(), out=y).view(B, N, H, d).permute(0, 2, 1, 3)),
                      max(3, args.steps))
    flops = 2.0 * B * N * H * d * Dx
    value = flops / (med * 1e-3) / 1e12
    peaks = read_peaks()
    peak, peak_s = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    hbm_bytes = (B * N * Dx + H * d * Dx + B * H * N * d) * 2
    line = {"metric": "probe projection rho = W_R x (plx_probe_proj) TFLOP/s, bf16 on the tensor cores, 1 GPU",
            "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": nsteps, "warmup": max(3, args.warmup),
            "ms_per_step": med, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "probe_proj_b4_n2048_dx1024_h16_d128", "B": B, "N": N, "Dx": Dx, "H": H, "d": d,
                       "l2": "flushed (256 MiB write) before every launch"},
            "roofline": {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s", "frac": value / peak,
                         "peak_source": f"{peaks['source']} bf16 dense (burst)", "frac_of_sustained": value / peak_s,
                         "flop_per_launch": flops, "hbm_bytes_per_launch": hbm_bytes,
                         "hbm_gbs_at_this_time": hbm_bytes / (med * 1e-3) / 1e9},
            "torch_matmul_ms": mm_ms, "torch_matmul_tflops": flops / (mm_ms * 1e-3) / 1e12,
            "torch_matmul_plus_head_transpose_ms": mmp_ms,
            "gpu_launches": nsteps, "clocks": clocks, "device_status": plx.plx_last_device_error()}
    print(json.dumps(line), flush=True)
    return 0


def run_lla_bench(args, world, rank, local):
    """plx_lla_f32 (local linear attention, probe solved by fp32 conjugate
    gradients) on the prefill workload's shape B=4, H=16, N=2048, d=128 with
    fp32 q, k, v ~ N(0, 1), ridge lambda = 0.1, at most 48 steps per row,
    relative tolerance 1e-4.  Work: the softmax weights of the CG steps once
    (q.k, 2 d flop per causal pair), then each CG step of row i streams its
    i + 1 keys at 4 d flop per key (p.k and the update of Sigma p); the softmax
    pass for kbar costs 4 d and the output pass 8 d per causal pair.  The timed
    call keeps the weights across the steps (the kept-weights workspace), and
    its steps after the first run on the tensor cores in split tf32; the path
    that recomputes the weights in every step on the CUDA cores (the minimal
    workspace, 2 d more per key and step) is timed beside it.  The roofline is
    that of the dominant kernel, the tensor-core CG step: its time is the
    solve's minus that of the same call with one CG step (the k-bar pass, the
    first step and the output pass), its work 4 d per key of the steps after
    the first, its peak the dense tf32 rate (the measured bf16 burst rate x
    the nominal tf32 / bf16 ratio 1.1 / 2.25); each product costs 3 tf32 MMA
    products.  L2 is flushed before every launch sequence.  Prints one JSON
    line."""
    import torch
    import parameterized_local_linear_02_b300 as plx

    if rank != 0:
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    B, H, N, d = 4, 16, 2048, 128
    lam, iters, tol = 0.1, 48, 1e-4
    g = torch.Generator(device=dev)
    g.manual_seed(17)
    q, k, v = (torch.randn((B, H, N, d), generator=g, device=dev) for _ in range(3))
    ws = torch.empty(plx.plx_lla_kept_weights_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    ws_min = torch.empty(plx.plx_lla_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    out = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    steps = torch.empty((B, H, N), dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call(workspace=ws, n_iters=iters):
        plx.plx_lla_f32(q, k, v, lam=lam, max_iters=n_iters, tol=tol, workspace=workspace, out=out, lse=lse,
                        steps=steps, with_rho=False)

    def timed(workspace, n_iters=iters):
        for _ in range(max(3, args.warmup)):
            call(workspace, n_iters)
        torch.cuda.synchronize()
        ms = []
        for _ in range(max(3, args.steps)):
            hold_device()
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call(workspace, n_iters)
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return ms

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ms = timed(ws)
    clocks = sampler.stop()
    med = float(np.median(ms))
    st = steps.double()
    n_max, n_at_max = int(steps.max()), int((steps == iters).sum())
    keys = torch.arange(1, N + 1, device=dev, dtype=torch.float64)
    cg_flops = float((st * keys).sum()) * 4 * d
    tc_flops = float((torch.clamp(st - 1, min=0) * keys).sum()) * 4 * d     # the steps after the first
    pairs = B * H * N * (N + 1) / 2
    flops = cg_flops + pairs * (2 + 12) * d
    value = flops / (med * 1e-3) / 1e12
    med_min = float(np.median(timed(ws_min)))
    med_one = float(np.median(timed(ws, 1)))       # k-bar, init, the first step (CUDA cores), output
    tc_ms = med - med_one
    tc_value = tc_flops / (tc_ms * 1e-3) / 1e12
    peaks = read_peaks()
    tf32_peak = peaks["bf16_tflops"] * 1.1 / 2.25
    props = torch.cuda.get_device_properties(dev)
    sm_max = clocks.get("sm_max_mhz") or 2032.0
    alu_peak = props.multi_processor_count * 128 * 2 * sm_max * 1e6 / 1e12
    line = {"metric": "LLA (probe solved by conjugate gradients) TFLOP/s, 1 GPU",
            "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": len(ms), "warmup": max(3, args.warmup),
            "ms_per_step": med, "higher_is_better": True, "dtype": "f32, tf32x3", "data": "synthetic",
            "config": {"workload": "lla_b4_h16_n2048_d128", "B": B, "H": H, "N": N, "d": d, "lambda": lam,
                       "max_iters": iters, "tol": tol, "l2": "flushed (256 MiB write) before every launch sequence"},
            "cg_steps": {"max": n_max, "mean": float(st.mean()), "rows_at_max": n_at_max, "rows": B * H * N},
            "roofline": {"bound": "tensor", "kernel": "plx_lla_cg_tc_kernel<128> (CG steps 2 ..)",
                         "achieved": tc_value, "peak": tf32_peak, "unit": "TFLOP/s", "frac": tc_value / tf32_peak,
                         "peak_source": f"dense tf32: measured bf16 burst {peaks['bf16_tflops']} x 1.1 / 2.25 "
                                        f"({peaks['source']})",
                         "mma_products_per_product": 3, "ms_per_solve": tc_ms, "flop_per_solve": tc_flops,
                         "ms_rest_of_solve": med_one},
            "solve_vs_fp32_fma_peak": {"frac": value / alu_peak, "peak": alu_peak,
                                       "peak_source": f"{props.multi_processor_count} SMs x 128 fp32 lanes x 2 flop x "
                                                      f"{sm_max:.0f} MHz"},
            "flop_per_launch_sequence": flops, "cg_flop": cg_flops,
            "weights": {"kept": "softmax weights of the CG steps stored by the first step (B H N^2 fp32 of workspace)",
                        "recomputed_ms_per_step": med_min,
                        "recomputed_value": flops / (med_min * 1e-3) / 1e12},
            "gpu_launches": (iters + 3) * len(ms), "clocks": clocks, "device_status": plx.plx_last_device_error()}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=("both", "prefill", "long", "decode"), default="both",
                    help="run one leg only (profiling of a single kernel); 'both' runs every leg")
    ap.add_argument("--no-long", action="store_true", help="leave the long-sequence prefill out of the step")
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="decode batch (default: the decode workload's 64); smaller for profiling")
    ap.add_argument("--decode-sweep", action="store_true",
                    help="time plx_decode over the batch x context sweep instead of the step")
    ap.add_argument("--sweep-iters", type=int, default=10)
    ap.add_argument("--backward", action="store_true",
                    help="time plx_bwd (and plx_bwd_f32) on the prefill workload's shape instead of the step")
    ap.add_argument("--cached", action="store_true",
                    help="time plx_fwd_cached (T new tokens per sequence) on the decode workload's cache")
    ap.add_argument("--proj", action="store_true",
                    help="time plx_probe_proj (rho = W_R x) on the prefill workload's probe")
    ap.add_argument("--lla", action="store_true",
                    help="time plx_lla_f32 (local linear attention, CG-solved probe) on the prefill workload's shape")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the softmax-attention comparison and the end-to-end leg")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)     # at least 3 untimed warm-up steps, always
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.decode_sweep:
        return run_decode_sweep(args, world, rank, local)
    if args.backward:
        return run_backward_bench(args, world, rank, local)
    if args.cached:
        return run_cached_bench(args, world, rank, local)
    if args.proj:
        return run_proj_bench(args, world, rank, local)
    if args.lla:
        return run_lla_bench(args, world, rank, local)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())

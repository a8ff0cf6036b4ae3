#!/usr/bin/env python
"""Throughput of the mHC hot path (mhc_pre + mhc_post) on GB300.

One step = mhc_pre then mhc_post over one M=16384-row chunk of the residual
R[M,4,5120] (the prefill-chunk workload), with synthetic seeded inputs
already resident in HBM; fn is prepared once (mhc_prepare_weights), as at
model load, and the step calls mhc_pre_prepared.  Prints one JSON line
(rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mhc|reference]

Multi-GPU (torchrun): rows are independent, so every rank runs its own
16384-row chunk (weak scaling) with no collective on the data path; a barrier
and a max-over-ranks of the elapsed time bracket the timed region.
--impl reference times the CPU oracle (the deliberately slow reference arm)
on a bounded sample of rows per step.
"""
from __future__ import annotations

import argparse
import hashlib
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

import synth  # noqa: E402
from hyper_connection_residual_mhc_gb300.shard import max_over_ranks  # noqa: E402

METRIC = "mHC pre+post rows/s and achieved HBM GB/s (% of GB300 peak) at M=16384"
HC, H, K, MIX = 4, 5120, 20480, 24
ROWS = 16384
SEED = 4
# algorithmic HBM bytes: pre reads R and writes x_norm/post/comb; post reads
# R/y/post/comb and writes R'.  Per call, fn (fp32), scale, base, norm_w once.
PRE_BYTES_ROW = K * 2 + H * 2 + HC * 4 + HC * HC * 4          # 51,280
POST_BYTES_ROW = K * 2 + H * 2 + HC * 4 + HC * HC * 4 + K * 2  # 92,240
PRE_BYTES_CALL = MIX * K * 4 + H * 2 + 3 * 4 + MIX * 4         # fn, norm_w, scale, base
PRE_LAUNCHES, POST_LAUNCHES = 1, 1                             # kernels per call
KERNEL_SRC = {"mhc_post": ["post.cu", "mhc_common.cuh"],
              "mhc_pre": ["pre_onepass.cu", "tc_ptx.cuh", "mhc_common.cuh"]}
KERNEL_NAME = {"mhc_post": "post_kernel", "mhc_pre": "pre_onepass_kernel<false, 8, true>"}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def src_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "hyper_connection_residual_mhc_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[kernel]
    except Exception:
        return None
    try:
        if t.get("src_sha256_16") != src_hash(KERNEL_SRC[kernel]):
            return None
    except (KeyError, OSError):
        return None
    return t.get("dram_bytes_per_launch_full_size")


class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.path = index, None, None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            self.proc.wait()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if not self.path or not os.path.exists(self.path):
            return out
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sms.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if sms:
            out.update(sm_mhz=statistics.median(sms), sm_max_mhz=mx, reasons=sorted(reasons),
                       samples=len(sms))
        return out


# --------------------------------------------------------------------------- CPU oracle timing
def oracle_rows_per_s(R, y, W, rows, threads):
    """Oracle pre+post on the first `rows` rows, row blocks spread over threads."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    oracle.build()
    blk = 8
    spans = [(lo, min(rows, lo + blk)) for lo in range(0, rows, blk)]

    def one(span):
        lo, hi = span
        o = oracle.pre(R[lo:hi], W.fn, W.scale, W.base, W.norm_w)
        oracle.post(R[lo:hi], y[lo:hi], o["post"].astype(np.float32), o["comb"].astype(np.float32))

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, spans))
    return rows / (time.perf_counter() - t0)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    R = synth.residual(SEED, 512)
    y = synth.sublayer_out(SEED, 512)
    W = synth.weights(SEED)
    # ~25 ms of CPU per row for pre+post: size the per-step sample so the whole
    # run stays around two minutes of wall time.
    per_step = int(max(threads, min(512, 120.0 * threads / 0.025 / max(1, args.steps + args.warmup))))
    per_step = max(1, per_step // threads * threads)
    for _ in range(args.warmup):
        oracle_rows_per_s(R, y, W, per_step, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_rows_per_s(R, y, W, per_step, threads)
    dt = time.perf_counter() - t0
    v = per_step * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"M={ROWS} rows of R[M,4,5120] bf16 (seed {SEED}); "
                               f"each step the CPU oracle on the first {per_step} rows"},
        "cpu_baseline": {"value": v, "unit": "rows/s", "cores": threads, "kind": "oracle",
                         "sample": f"{per_step} rows per step, {args.steps} steps"},
        "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm
def run_mhc(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import hyper_connection_residual_mhc_gb300 as m
    from hyper_connection_residual_mhc_gb300 import build as b
    b.build()
    m.lib()

    M = args.rows
    row0 = rank * M                      # each rank: its own chunk of rows
    Rh = synth.residual(SEED, M, row0=row0)
    yh = synth.sublayer_out(SEED, M, row0=row0)
    W = synth.weights(SEED)

    dev = torch.device("cuda", local)

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    R = bf(Rh).to(dev)
    y = bf(yh).to(dev)
    fn = torch.from_numpy(W.fn).to(dev)
    scale = torch.from_numpy(W.scale).to(dev)
    base = torch.from_numpy(W.base).to(dev)
    w = bf(W.norm_w).to(dev)
    xn = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    post = torch.empty((M, HC), dtype=torch.float32, device=dev)
    comb = torch.empty((M, HC, HC), dtype=torch.float32, device=dev)
    R2 = torch.empty_like(R)
    ws = torch.empty((max(1, m.mhc_pre_workspace_bytes(M)),), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    # fn prepared once, as at model load (outside every timed region)
    wh = m.mhc_prepare_weights(fn)
    torch.cuda.synchronize(dev)

    def step():
        m.mhc_pre_prepared(R, wh, scale, base, w, logical_rows=M, workspace=ws, x_norm=xn,
                           post=post, comb=comb, stream=stream)
        m.mhc_post(R, y, post, comb, logical_rows=M, out=R2, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    K_ = args.steps
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        # events only around the K steps: an event between two launches would
        # cut the programmatic launch dependency between them
        start.record(stream)
        for _ in range(K_):
            step()
        end.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
    clocks = clk.summary()
    ms = start.elapsed_time(end)
    ms = max_over_ranks(ms, dist if world > 1 else None, dev)
    # the pre / post split, from a second loop with events around each call
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K_)]
    for i in range(K_):
        ev[i][0].record(stream)
        m.mhc_pre_prepared(R, wh, scale, base, w, logical_rows=M, workspace=ws, x_norm=xn,
                           post=post, comb=comb, stream=stream)
        ev[i][1].record(stream)
        m.mhc_post(R, y, post, comb, logical_rows=M, out=R2, stream=stream)
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    pre_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    post_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)

    # ---- end to end: host buffers, copies inside the timed region ----------
    e2e = None
    if not args.no_e2e:
        def make_bufs():
            return {"R": torch.empty_like(R), "y": torch.empty_like(y), "xn": torch.empty_like(xn),
                    "post": torch.empty_like(post), "comb": torch.empty_like(comb),
                    "R2": torch.empty_like(R2), "ws": torch.empty_like(ws)}

        def step_on(B, st):
            m.mhc_pre_prepared(B["R"], wh, scale, base, w, logical_rows=M, workspace=B["ws"],
                               x_norm=B["xn"], post=B["post"], comb=B["comb"], stream=st)
            m.mhc_post(B["R"], B["y"], B["post"], B["comb"], logical_rows=M, out=B["R2"], stream=st)

        e2e = run_e2e(m, torch, dist, world, dev, step_on, make_bufs, Rh, yh, bf, M, K_)

    # ---- the other prefill sizes, each with L2 evicted before every step
    # (rank 0, N=1; outside the timed region) ---------------------------------
    per_config = None
    if rank == 0 and world == 1 and not args.no_configs:
        flush = torch.empty((FLUSH_BYTES,), dtype=torch.uint8, device=dev)
        per_config = {}
        for seed_c, M_c in SWEEP:
            if M_c == M:
                continue
            line_c = measure_config(m, torch, dev, stream, flush, seed_c, M_c, 20, 3, local)
            per_config[f"M={M_c}"] = config_summary(line_c)
        del flush
        torch.cuda.empty_cache()

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N=1) --------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        # the whole chunk: ~1 ms of fp64 oracle work a row, so ~15-30 core-seconds
        sample = M
        t0 = time.perf_counter()
        v = oracle_rows_per_s(Rh, yh, W, sample, threads)
        wall = time.perf_counter() - t0
        # the single-threaded oracle on the first 1024 rows (about a second)
        one = oracle_rows_per_s(Rh, yh, W, min(M, 1024), 1)
        cpu = {"value": v, "unit": "rows/s", "cores": threads, "kind": "oracle",
               "sample": f"oracle pre+post on all {sample} rows of the M={M} workload "
                         f"({wall:.1f} s wall on {threads} threads); single-threaded on "
                         f"the first {min(M, 1024)} rows: {one:.0f} rows/s",
               "single_thread_value": one}
    return finish(args, m, world, rank, M, K_, ms, pre_ms, post_ms, clocks, e2e, cpu, dist,
                  per_config)


def run_e2e(m, torch, dist, world, dev, step_on, make_bufs, Rh, yh, bf, M, K_, lanes=1):
    """The step through the public API with host buffers: every step copies its
    inputs from pinned host memory and its results back inside the timed
    region.  Two device buffer sets pipeline the steps: step k's compute
    overlaps step k+1's host-to-device copies and step k-1's device-to-host
    copies.  Each direction's copies can be split by rows over `lanes`
    streams; on GB300 more lanes did not help (the host link is the limit)."""
    e2e_steps = max(4, min(K_, 20))
    Rp = bf(Rh).pin_memory()
    yp = bf(yh).pin_memory()
    xn_h = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
    R2_h = torch.empty((M, HC, H), dtype=torch.bfloat16).pin_memory()
    post_h = torch.empty((M, HC), dtype=torch.float32).pin_memory()
    comb_h = torch.empty((M, HC, HC), dtype=torch.float32).pin_memory()
    bufs = [make_bufs() for _ in range(2)]
    s_in = [torch.cuda.Stream(dev) for _ in range(lanes)]
    s_out = [torch.cuda.Stream(dev) for _ in range(lanes)]
    s_cmp = torch.cuda.Stream(dev)
    cuts = [M * i // lanes for i in range(lanes + 1)]
    E = lambda: torch.cuda.Event()

    def run(n):
        cmp_done = [None, None]
        out_done = [[], []]
        for k in range(n):
            b = k % 2
            B = bufs[b]
            ins = []
            for L, st in enumerate(s_in):
                lo, hi = cuts[L], cuts[L + 1]
                with torch.cuda.stream(st):
                    if cmp_done[b] is not None:
                        st.wait_event(cmp_done[b])       # step k-2 is done reading B
                    B["R"][lo:hi].copy_(Rp[lo:hi], non_blocking=True)
                    B["y"][lo:hi].copy_(yp[lo:hi], non_blocking=True)
                    ev = E(); ev.record(st); ins.append(ev)
            for ev in ins + out_done[b]:               # inputs here; step k-2's results home
                s_cmp.wait_event(ev)
            step_on(B, s_cmp)
            cmp_done[b] = E(); cmp_done[b].record(s_cmp)
            out_done[b] = []
            for L, st in enumerate(s_out):
                lo, hi = cuts[L], cuts[L + 1]
                st.wait_event(cmp_done[b])
                with torch.cuda.stream(st):
                    xn_h[lo:hi].copy_(B["xn"][lo:hi], non_blocking=True)
                    R2_h[lo:hi].copy_(B["R2"][lo:hi], non_blocking=True)
                    post_h[lo:hi].copy_(B["post"][lo:hi], non_blocking=True)
                    comb_h[lo:hi].copy_(B["comb"][lo:hi], non_blocking=True)
                    ev = E(); ev.record(st); out_done[b].append(ev)

    run(2)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(s_cmp)
    for st in s_in + s_out:
        st.wait_event(s2)
    run(e2e_steps)
    for st in s_in + s_out:
        s_cmp.wait_stream(st)
    e2.record(s_cmp)
    torch.cuda.synchronize(dev)
    e2e_ms = s2.elapsed_time(e2)
    e2e_ms = max_over_ranks(e2e_ms, dist if world > 1 else None, dev)
    h2d = (Rp.numel() + yp.numel()) * 2
    d2h = (xn_h.numel() + R2_h.numel()) * 2 + (post_h.numel() + comb_h.numel()) * 4
    return {"value": world * M * e2e_steps / (e2e_ms / 1e3), "unit": "rows/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
            "pipelined": f"2 buffer sets; compute stream; {lanes} H2D and {lanes} D2H streams"}


def finish(args, m, world, rank, M, K_, ms, pre_ms, post_ms, clocks, e2e, cpu, dist,
           per_config=None):
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    hbm_peak, peak_src = peaks()
    step_bytes = M * (PRE_BYTES_ROW + POST_BYTES_ROW) + PRE_BYTES_CALL
    rows_per_s = world * M * K_ / (ms / 1e3)
    gbs = step_bytes * K_ / (ms / 1e3) / 1e9
    pre_gbs = (M * PRE_BYTES_ROW + PRE_BYTES_CALL) / (pre_ms / 1e3) / 1e9
    post_gbs = M * POST_BYTES_ROW / (post_ms / 1e3) / 1e9
    # the dominant kernel is the call with the larger share of the step (each
    # call is one launch at this size); the other is reported beside it
    calls = {"mhc_pre": (pre_ms, pre_gbs, M * PRE_BYTES_ROW + PRE_BYTES_CALL),
             "mhc_post": (post_ms, post_gbs, M * POST_BYTES_ROW)}
    dom = max(calls, key=lambda k: calls[k][0])

    def kernel_roofline(name):
        t, g, nb = calls[name]
        return {"kernel": name, "kernel_name": KERNEL_NAME[name], "launches": 1, "ms": t,
                "achieved": g, "frac": g / hbm_peak, "algorithmic_bytes_per_launch": nb,
                "traffic": traffic_for(name)}
    line = {
        "metric": METRIC,
        "value": rows_per_s,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": K_,
        "warmup": args.warmup,
        "ms_per_step": ms / K_,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"M={M} rows per GPU: R[M,4,5120] bf16, fn[24,20480] f32, y[M,5120] bf16 "
                        f"(seed {SEED}); one step = mhc_pre + mhc_post",
            "rows_per_gpu": M,
            "weights": "fn prepared once with mhc_prepare_weights before the timed regions (as "
                       "at model load); the step calls mhc_pre_prepared + mhc_post",
            "l2": f"inputs larger than L2 (R alone is {M * K * 2 / 1e6:.0f} MB per step); no flush",
            "achieved_gbs": gbs,
            "frac_of_hbm": gbs / hbm_peak,
            "pre_ms": pre_ms,
            "post_ms": post_ms,
            "pre_gbs": pre_gbs,
            "post_gbs": post_gbs,
            "algorithmic_bytes_per_step": step_bytes,
            "per_config": per_config,
        },
        "roofline": {
            "bound": "hbm",
            "kernel": dom,
            "kernel_name": KERNEL_NAME[dom],
            "achieved": calls[dom][1],
            "peak": hbm_peak,
            "peak_source": f"{peak_src} (hbm_gbs)",
            "unit": "GB/s",
            "frac": calls[dom][1] / hbm_peak,
            "traffic": traffic_for(dom),
            "algorithmic_bytes_per_launch": calls[dom][2],
            "timing": "CUDA events on the launching stream around each call, mean over the "
                      "steps of a second loop",
            "pre_call": kernel_roofline("mhc_pre"),
            "post_call": kernel_roofline("mhc_post"),
        },
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K_ * ((PRE_LAUNCHES if M > 48 else 1) + POST_LAUNCHES),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# --------------------------------------------------------------------------- other entry points
HEAD_BYTES_ROW = K * 2 + H * 2                 # read R, write y
HEAD_BYTES_CALL = HC * K * 4 + HC * 4 + 4      # fn, base, scale


def run_op(args):
    """Time one of the library's other entry points alone (1 GPU, inputs in
    HBM): prints one JSON line in the same shape as the step's."""
    import torch
    import hyper_connection_residual_mhc_gb300 as m
    from hyper_connection_residual_mhc_gb300 import build as b
    b.build()
    m.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    M = args.rows

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    R = bf(synth.residual(SEED, M))
    stream = torch.cuda.current_stream(dev)
    if args.op == "hc_head":
        hw = synth.head_weights(SEED)
        fn = torch.from_numpy(hw.fn).to(dev)
        scale = torch.from_numpy(hw.scale).to(dev)
        base = torch.from_numpy(hw.base).to(dev)
        y = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty((max(1, m.mhc_pre_workspace_bytes(M)),), dtype=torch.uint8, device=dev)

        def step():
            m.mhc_hc_head(R, fn, scale, base, logical_rows=M, workspace=ws, out=y, stream=stream)
        # one launch at every size (above 256 rows the tiled kernel)
        nbytes, launches = M * HEAD_BYTES_ROW + HEAD_BYTES_CALL, 1
        metric = "mhc_hc_head rows/s (final stream collapse) and achieved HBM GB/s"
        workload = f"M={M} rows: R[M,4,5120] bf16, hc_head fn[4,20480] f32 (seed {SEED})"
    elif args.op == "fused_post_pre":
        # hc_post of one sublayer + hc_pre of the next on its result, fused,
        # against the same work as mhc_post then mhc_pre (timed the same way)
        W = synth.weights(SEED)
        Wn = synth.weights(SEED + 100)
        t_ = lambda a: torch.from_numpy(a).to(dev)
        fn, scale, base, w = t_(Wn.fn), t_(Wn.scale), t_(Wn.base), bf(Wn.norm_w)
        yv = bf(synth.sublayer_out(SEED, M))
        _, post, comb = m.mhc_pre(R, t_(W.fn), t_(W.scale), t_(W.base), bf(W.norm_w))
        R2 = torch.empty_like(R)
        xn = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        po = torch.empty((M, HC), dtype=torch.float32, device=dev)
        co = torch.empty((M, HC, HC), dtype=torch.float32, device=dev)
        ws = torch.empty((max(256, m.mhc_pre_workspace_bytes(M)),), dtype=torch.uint8, device=dev)
        wh = m.mhc_prepare_weights(fn)          # the next sublayer's fn, as at model load

        def step():
            m.mhc_fused_post_pre_prepared(R, yv, post, comb, wh, scale, base, w, logical_rows=M,
                                          workspace=ws, R_out=R2, x_norm=xn, post_out=po,
                                          comb_out=co, stream=stream)

        def unfused():
            m.mhc_post(R, yv, post, comb, logical_rows=M, out=R2, stream=stream)
            m.mhc_pre_prepared(R2, wh, scale, base, w, logical_rows=M, workspace=ws, x_norm=xn,
                               post=po, comb=co, stream=stream)
        for _ in range(args.warmup):
            unfused()
        torch.cuda.synchronize(dev)
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        for _ in range(args.steps):
            unfused()
        b_.record(stream)
        torch.cuda.synchronize(dev)
        unfused_ms = a_.elapsed_time(b_) / args.steps
        # minimal traffic of the pair: read R, y, post, comb; write R', x_norm,
        # post', comb' (the fused launch reads R' once more, for the combine)
        # (2 launches: the fused kernel and the combine; fn is not converted per call)
        nbytes = M * (2 * (K * 2 + H * 2 + HC * 4 + HC * HC * 4)) + PRE_BYTES_CALL
        launches = 2 if M > 48 else 1      # decode sizes: one launch of the decode kernel
        metric = "mhc_fused_post_pre rows/s (hc_post + next hc_pre) and achieved HBM GB/s"
        workload = (f"M={M} rows: R[M,4,5120], y[M,5120] bf16, next fn[24,20480] f32 "
                    f"(seed {SEED}), prepared once; unfused mhc_post+mhc_pre: {unfused_ms:.4f} "
                    "ms/step")
    elif args.op == "pre_mxfp8":
        # mhc_pre with x_norm's MXFP8 codes and scales written beside it, timed
        # against mhc_pre_prepared alone (the same inputs, the same way)
        W = synth.weights(SEED)
        t_ = lambda a: torch.from_numpy(a).to(dev)
        scale, base, w = t_(W.scale), t_(W.base), bf(W.norm_w)
        wh = m.mhc_prepare_weights(t_(W.fn))
        xn = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        xq = torch.empty((M, H), dtype=torch.uint8, device=dev)
        xs = torch.empty((M, H // 32), dtype=torch.uint8, device=dev)
        po = torch.empty((M, HC), dtype=torch.float32, device=dev)
        co = torch.empty((M, HC, HC), dtype=torch.float32, device=dev)
        ws = torch.empty((max(256, m.mhc_pre_workspace_bytes(M)),), dtype=torch.uint8, device=dev)

        def step():
            m.mhc_pre_mxfp8(R, wh, scale, base, w, logical_rows=M, workspace=ws, x_norm=xn,
                            x_q=xq, x_s=xs, post=po, comb=co, stream=stream)

        def plain():
            m.mhc_pre_prepared(R, wh, scale, base, w, logical_rows=M, workspace=ws, x_norm=xn,
                               post=po, comb=co, stream=stream)
        for _ in range(args.warmup):
            plain()
        torch.cuda.synchronize(dev)
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        for _ in range(args.steps):
            plain()
        b_.record(stream)
        torch.cuda.synchronize(dev)
        plain_ms = a_.elapsed_time(b_) / args.steps
        # mhc_pre's bytes plus the codes (1 B per x_norm value) and scales (1 B
        # per 32 values)
        nbytes = M * (PRE_BYTES_ROW + H + H // 32) + PRE_BYTES_CALL
        launches = 1 if M > 48 else 2   # the one-pass launch; at decode sizes decode kernel + quantizer
        metric = "mhc_pre_mxfp8 rows/s (mhc_pre + MXFP8 x_norm) and achieved HBM GB/s"
        workload = (f"M={M} rows: R[M,4,5120] bf16, fn[24,20480] f32 (seed {SEED}), prepared "
                    f"once; mhc_pre_prepared alone: {plain_ms:.4f} ms/step")
    elif args.op == "latency":
        # decode-size rows: one step = mhc_pre + mhc_post; latency per step,
        # launched eagerly and replayed from a CUDA graph
        W = synth.weights(SEED)
        fn = torch.from_numpy(W.fn).to(dev)
        scale = torch.from_numpy(W.scale).to(dev)
        base = torch.from_numpy(W.base).to(dev)
        w = bf(W.norm_w)
        yv = bf(synth.sublayer_out(SEED, M))
        xn = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        post = torch.empty((M, HC), dtype=torch.float32, device=dev)
        comb = torch.empty((M, HC, HC), dtype=torch.float32, device=dev)
        R2 = torch.empty_like(R)
        ws = torch.empty((max(256, m.mhc_pre_workspace_bytes(M)),), dtype=torch.uint8, device=dev)
        side = torch.cuda.Stream(dev)

        LM = args.logical_rows or M
        wh = m.mhc_prepare_weights(fn)          # as at model load
        if args.fused:
            # one sublayer boundary of a decode loop: hc_post of this sublayer
            # and hc_pre of the next in one call (gates from a pre of R)
            m.mhc_pre(R, fn, scale, base, w, x_norm=xn, post=post, comb=comb)
            po2, co2 = torch.empty_like(post), torch.empty_like(comb)

        def launch(st):
            if args.fused:
                m.mhc_fused_post_pre_prepared(R, yv, post, comb, wh, scale, base, w,
                                              logical_rows=LM, workspace=ws, R_out=R2, x_norm=xn,
                                              post_out=po2, comb_out=co2, stream=st)
                return
            m.mhc_pre_prepared(R, wh, scale, base, w, logical_rows=LM, workspace=ws, x_norm=xn,
                               post=post, comb=comb, stream=st)
            m.mhc_post(R, yv, post, comb, logical_rows=LM, out=R2, stream=st)

        def timed(fn_, n):
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(side)
            for _ in range(n):
                fn_()
            b.record(side)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) / n * 1e3          # us per step

        with torch.cuda.stream(side):
            for _ in range(args.warmup):
                launch(side)
            eager_us = timed(lambda: launch(side), args.steps)
            # the graph holds --chain consecutive steps, so each step after the
            # first can overlap its predecessor's tail
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(args.chain):
                    launch(side)
            for _ in range(args.warmup):
                g.replay()
            graph_us = timed(g.replay, args.steps) / args.chain
        nbytes = M * (PRE_BYTES_ROW + POST_BYTES_ROW) + PRE_BYTES_CALL
        line = {
            "metric": (f"mhc_fused_post_pre latency at M={M} rows (one decode sublayer boundary)"
                       if args.fused else
                       f"mhc_pre + mhc_post latency at M={M} rows (decode-size step)"),
            "value": graph_us, "unit": "us/step", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": graph_us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"M={M} rows of R[M,4,5120] bf16 (seed {SEED}); inputs "
                                   "L2-resident between steps (decode-size, latency-bound)",
                       "op": "latency", "fused": bool(args.fused), "rows": M,
                       "logical_rows": LM, "eager_us": eager_us,
                       "graph_us": graph_us, "graph_chain": args.chain},
            "roofline": {"bound": "latency", "algorithmic_bytes_per_step": nbytes,
                         "achieved_gbs_graph": nbytes / (graph_us * 1e-6) / 1e9},
            # per step: prefill sizes 2 (the one-pass pre, post) or, fused with
            # fn prepared, 2 (fused kernel, combine); decode sizes 2, or 1 fused
            "gpu_launches": (2 if LM > 48 else (1 if args.fused else 2)) * args.steps * args.chain,
        }
        print(json.dumps(line), flush=True)
        return
    else:
        raise SystemExit(f"unknown --op {args.op}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        torch.cuda.synchronize(dev)
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize(dev)
    clocks = clk.summary()
    ms = start.elapsed_time(end)
    hbm_peak, peak_src = peaks()
    gbs = nbytes * args.steps / (ms / 1e3) / 1e9
    line = {
        "metric": metric, "value": M * args.steps / (ms / 1e3), "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload, "op": args.op, "rows": M,
                   "l2": f"inputs larger than L2 (R is {M * K * 2 / 1e6:.0f} MB); no flush"},
        "roofline": {"bound": "hbm", "kernel": args.op, "achieved": gbs, "peak": hbm_peak,
                     "peak_source": f"{peak_src} (hbm_gbs)", "unit": "GB/s",
                     "frac": gbs / hbm_peak, "traffic": None,
                     "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


SWEEP = [(0, 128), (1, 1500), (2, 2048), (3, 4096), (4, 16384)]   # (seed, M)
FLUSH_BYTES = 512 << 20                                           # > 129 MB of L2


def measure_config(m, torch, dev, stream, flush, seed, M, steps, warmup, clock_index=0):
    """mhc_pre + mhc_post on the M-row workload of `seed` (fn prepared once).
    Before each timed step a 512 MB memset evicts L2, so R never starts
    L2-resident (fn and norm_w are re-read from L2 or HBM as they fall);
    events bracket each step alone and the figures are medians over the
    steps.  At M=4096 mhc_post is also timed alone on a second-seed y.
    Returns one JSON-ready line."""
    hbm_peak, peak_src = peaks()

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    def per_step(fns):
        """Median ms of each of fns (run back to back) and of their sum."""
        for _ in range(warmup):
            for f in fns:
                f()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)]
              for _ in range(steps)]
        torch.cuda.synchronize(dev)
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            for j, f in enumerate(fns):
                f()
                ev[i][j + 1].record(stream)
        torch.cuda.synchronize(dev)
        parts = [statistics.median(e[j].elapsed_time(e[j + 1]) for e in ev)
                 for j in range(len(fns))]
        total = statistics.median(e[0].elapsed_time(e[-1]) for e in ev)
        return total, parts

    W = synth.weights(seed)
    R = bf(synth.residual(seed, M))
    y = bf(synth.sublayer_out(seed, M))
    t_ = lambda a: torch.from_numpy(a).to(dev)
    fn, scale, base, w = t_(W.fn), t_(W.scale), t_(W.base), bf(W.norm_w)
    xn = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    post = torch.empty((M, HC), dtype=torch.float32, device=dev)
    comb = torch.empty((M, HC, HC), dtype=torch.float32, device=dev)
    R2 = torch.empty_like(R)
    ws = torch.empty((max(256, m.mhc_pre_workspace_bytes(M)),), dtype=torch.uint8, device=dev)
    wh = m.mhc_prepare_weights(fn)          # as at model load, outside the timing

    def pre():
        m.mhc_pre_prepared(R, wh, scale, base, w, logical_rows=M, workspace=ws, x_norm=xn,
                           post=post, comb=comb, stream=stream)

    def post_(yy=y):
        m.mhc_post(R, yy, post, comb, logical_rows=M, out=R2, stream=stream)

    with ClockSampler(clock_index) as clk:
        ms, (pre_ms, post_ms) = per_step([pre, post_])
        extra = {}
        if M == 4096:
            y2 = bf(synth.sublayer_out(seed + 1, M))
            alone, _ = per_step([lambda: post_(y2)])
            a_gbs = M * POST_BYTES_ROW / (alone / 1e3) / 1e9
            extra = {"post_alone_ms": alone, "post_alone_gbs": a_gbs,
                     "post_alone_frac": a_gbs / hbm_peak}
    torch.cuda.synchronize(dev)
    wh.release()
    nbytes = M * (PRE_BYTES_ROW + POST_BYTES_ROW) + PRE_BYTES_CALL
    gbs = nbytes / (ms / 1e3) / 1e9
    pre_gbs = (M * PRE_BYTES_ROW + PRE_BYTES_CALL) / (pre_ms / 1e3) / 1e9
    post_gbs = M * POST_BYTES_ROW / (post_ms / 1e3) / 1e9
    return {
        "metric": f"mHC pre+post rows/s and achieved HBM GB/s at M={M}",
        "value": M / (ms / 1e3), "unit": "rows/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"M={M} rows: R[M,4,5120] bf16, fn[24,20480] f32, "
                               f"y[M,5120] bf16 (seed {seed}); one step = mhc_pre + "
                               "mhc_post (fn prepared once); median of per-step event "
                               "times",
                   "op": "sweep", "rows": M,
                   "l2": "512 MB memset before every timed step (outside the events)",
                   "pre_ms": pre_ms, "post_ms": post_ms,
                   "pre_gbs": pre_gbs, "post_gbs": post_gbs,
                   "pre_frac": pre_gbs / hbm_peak, "post_frac": post_gbs / hbm_peak, **extra},
        "roofline": {"bound": "hbm", "kernel": "mhc_pre+mhc_post", "achieved": gbs,
                     "peak": hbm_peak, "peak_source": f"{peak_src} (hbm_gbs)",
                     "unit": "GB/s", "frac": gbs / hbm_peak, "traffic": None,
                     "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": (PRE_LAUNCHES if M > 48 else 1) * steps + POST_LAUNCHES * steps,
        "clocks": clk.summary(),
    }


def config_summary(line):
    """The figures of one measure_config line that the headline line carries."""
    c = line["config"]
    out = {"seed_rows": c["workload"].split(";")[0], "rows_per_s": line["value"],
           "ms_per_step": line["ms_per_step"], "achieved_gbs": line["roofline"]["achieved"],
           "frac_of_hbm": line["roofline"]["frac"], "pre_ms": c["pre_ms"],
           "pre_frac": c["pre_frac"], "post_ms": c["post_ms"], "post_frac": c["post_frac"],
           "steps": line["steps"], "sm_mhz": line["clocks"]["sm_mhz"],
           "throttle_reasons": line["clocks"]["reasons"]}
    for k in ("post_alone_ms", "post_alone_gbs", "post_alone_frac"):
        if k in c:
            out[k] = c[k]
    return out


def run_sweep(args):
    """mhc_pre + mhc_post at every prefill size (M = 128, 1500, 2048, 4096,
    16384; seeds 0..4), one JSON line per size (see measure_config)."""
    import torch
    import hyper_connection_residual_mhc_gb300 as m
    from hyper_connection_residual_mhc_gb300 import build as b
    b.build()
    m.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty((FLUSH_BYTES,), dtype=torch.uint8, device=dev)
    for seed, M in SWEEP:
        line = measure_config(m, torch, dev, stream, flush, seed, M, max(20, args.steps),
                              args.warmup)
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mhc", "reference"], default="mhc")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config figures (M = 128, 1500, 2048, 4096) of the "
                         "headline line")
    ap.add_argument("--op", choices=["step", "hc_head", "latency", "fused_post_pre", "sweep",
                                     "pre_mxfp8"],
                    default="step",
                    help="step: mhc_pre + mhc_post (the headline); others time one entry "
                         "point alone")
    ap.add_argument("--fused", action="store_true",
                    help="--op latency: time mhc_fused_post_pre (one decode sublayer boundary)")
    ap.add_argument("--chain", type=int, default=1,
                    help="--op latency: consecutive steps captured in one CUDA graph "
                         "(the graph figure is per step)")
    ap.add_argument("--logical-rows", type=int, default=0,
                    help="--op latency: the chunk's row count (default: --rows)")
    ap.add_argument("--rows", type=int, default=ROWS,
                    help="rows per GPU (default: the 16384-row chunk); other sizes are "
                         "for profiling runs")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.chain < 1:
        ap.error("--chain must be >= 1")
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "sweep":
        run_sweep(args)
    elif args.op != "step":
        run_op(args)
    else:
        run_mhc(args)


if __name__ == "__main__":
    main()

"""Benchmark of paged split-KV decode attention (stage 1 + stage 2 per call).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pda_decode call (all of stage 1 and stage 2) over the
fp8_decode workload: bs 128, R 1, 64 query / 8 kv heads, head_dim 128,
ctx 2048, page 64, Q/K/V E4M3 with per-tensor scales, bf16 output. The call is
captured once in a CUDA graph and replayed; before every step L2 is flushed by
a memset of twice its size followed by a read of another buffer of twice its
size (which writes the memset's dirty lines back), both outside the CUDA
events that time the step, so each step starts from a cold, clean L2.
`value` is the algorithmic HBM bytes of the call (paged_split_kv_03_gb300.
traffic) over its measured time, summed over ranks; the line also carries the
R = 1 / 4 / 8 sweep at bs 1 and bs 16 of the two workloads at 16 query / 2 kv
heads and head_dim 256 (bf16 ctx 32768 and E4M3 per-(token, head) ctx 131072)
with their R8 / R1 time ratios, the mixed batch (bs 64, 48 / 2 heads, R 1..8,
ctx 1K..64K, half windowed), and the int8, head_dim 512 and MLA workloads.

`--impl reference` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of (row, q head) items per step, scaled to the same metric.
With N > 1 (torchrun) every rank runs an independent replica: the path needs
no collective.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("paged decode attn µs/call and achieved HBM GB/s (% of GB300 peak) at R=1/4/8")
HEADLINE = "fp8_decode"
HEADLINE_DESC = ("fp8_decode: bs128, R1, 64 q / 8 kv heads, head_dim 128, ctx 2048 each, "
                 "page 64, Q/K/V e4m3 per-tensor scales, bf16 out")
PAGES_NUMBER = {"value": 3672.1, "unit": "GB/s",
                "source": "hpc-ops FP8 decode on H200 (other hardware; context only)"}
SWEEP = [("mtp_verify_bf16", bs, R) for bs in (1, 16) for R in (1, 4, 8)] + \
        [("longctx_fp8_pth", bs, R) for bs in (1, 16) for R in (1, 4, 8)] + \
        [("mixed", 64, None)] + \
        [("longctx_int8_pth", 16, R) for R in (1, 8)] + \
        [("d512_mtp_bf16", 1, R) for R in (1, 4, 8)] + \
        [("d512_mtp_fp8", 1, R) for R in (1, 4, 8)] + \
        [("mla_bf16", 64, 1), ("mla_fp8", 64, 1), ("mla_fp8", 64, 2), ("mla_fp8_mixed", 64, 1),
         ("mla_fp8_mixed", 64, 2)]
# the same FP8 decode batch with the cache in HND order (one kv head's page
# contiguous) beside the NHD headline: the access-pattern check
LAYOUT_SWEEP = [("fp8_decode", dict(layout="HND"), "fp8_decode bs128 R1 HND")]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = {"stage1": ("pda_tc.cu", "pda_internal.h")}


def source_sha(kernel: str = "stage1") -> str:
    """Hash of the sources a kernel is built from: ncu traffic figures apply
    only to that code."""
    h = hashlib.sha256()
    cs = os.path.join(ROOT, "paged_split_kv_03_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(f.encode())
        h.update(open(os.path.join(cs, f), "rb").read())
    return h.hexdigest()[:12]


def recorded_traffic(kernel: str, workload: str):
    """dram read+write bytes per launch from the committed ncu summary, or
    None when the summary is for other sources."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    sha = source_sha(kernel)
    for line in open(path):
        m = re.match(r"\s*(\S+)\s+(\S+)\s+(\S+)\s+(\d+)", line)
        if m and m.group(1) == kernel and m.group(2) == workload and m.group(3) == sha:
            return int(m.group(4))
    return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


THROTTLE_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_ok(summary) -> bool:
    """False when the clock record of a timed region disqualifies its number:
    a hardware or thermal slowdown was active, or the median SM clock sat
    below 90 % of its maximum with no reason given (a clock lock left by
    someone else). sw_power_cap alone is kept. No record (no nvidia-smi):
    nothing to judge, True."""
    if not summary:
        return True
    if any(r in THROTTLE_REASONS for r in summary.get("reasons", ())):
        return False
    mx = summary.get("sm_max_mhz") or 0.0
    if mx > 0 and summary.get("sm_mhz", mx) < 0.9 * mx and not summary.get("reasons"):
        return False
    return True


# ------------------------------------------------------------------ GPU arm
def make_flush(dev):
    """L2 flush for timing: a memset of 2x L2, then a read of another 2x L2
    buffer, so the timed step neither hits in L2 nor pays for write-backs of
    the memset's dirty lines."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n = max(2 * l2, 256 << 20)
    wbuf = torch.empty(n, dtype=torch.uint8, device=dev)
    rbuf = torch.zeros(n // 8, dtype=torch.int64, device=dev)

    def flush():
        wbuf.zero_()
        rbuf.max()

    return flush


# Quantise-on-append of one decode step's new rows, timed like a call:
# (workload, sizes) -- per-tensor E4M3 (bs 128, R 1, 8 kv heads, D 128),
# per-(token, head) E4M3 and int8 (bs 16, R 8, 2 kv heads, D 256), bf16 (same shape).
APPEND_SWEEP = [("fp8_decode", {}), ("longctx_fp8_pth", dict(bs=16, R=8)),
                ("longctx_int8_pth", dict(bs=16, R=8)), ("mtp_verify_bf16", dict(bs=16, R=8))]


def append_time(name, kw, dev, steps, flush, peak):
    """Median time of one pda_append_kv (graph-replayed, L2 flushed) and its
    algorithmic bytes: the new rows' bf16 K and V read, their cache bytes and
    per-(token, head) scales written, one page-table entry per row and the
    index arrays."""
    import torch
    from paged_split_kv_03_gb300 import binding as B
    from paged_split_kv_03_gb300.synth import config_workload
    wl = config_workload(name, device=dev, **kw)
    dec = B.Decoder(B.params_for(wl, device=dev.index or 0), device=dev)
    rows, H, D = wl.total_rows, wl.num_kv_heads, wl.head_dim
    g = torch.Generator(device=dev).manual_seed(11)
    k_new = torch.randn(rows, H, D, generator=g, device=dev).to(torch.bfloat16)
    v_new = torch.randn(rows, H, D, generator=g, device=dev).to(torch.bfloat16)
    mq = max(1, wl.max_q_len)
    s = torch.cuda.Stream(device=dev)

    def call():
        B.pda_append_kv(dec.plan, k_new, v_new, wl.page_table, wl.kv_indptr, wl.kv_len,
                        wl.qo_indptr, mq, wl.k_pages, wl.v_pages, wl.k_scale, wl.v_scale,
                        dec.scratch, stream=s)

    with torch.cuda.stream(s):
        call()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    med = statistics.median(time_graph(graph.replay, steps, 3, flush, s))
    elt = 1 if (wl.kv_e4m3 or getattr(wl, "kv_int8", False)) else 2
    nbytes = 2 * rows * H * D * (2 + elt) + rows * 4 + 4 * (3 * wl.batch + 2)
    if wl.scale_mode == 2:
        nbytes += 2 * rows * H * 4
    elif wl.scale_mode == 1:
        nbytes += 8
    status = dec.status()
    del graph, dec, k_new, v_new, wl
    return {"workload": f"{name} {kw}".strip(), "us_per_call": med * 1e3,
            "GB_s": nbytes / (med * 1e-3) / 1e9, "frac_of_peak": nbytes / (med * 1e-3) / 1e9 / peak,
            "bytes": nbytes, "status": status}


def append_once(name, kw, dev):
    """One eager pda_append_kv on the workload (a profiler's target)."""
    import torch
    from paged_split_kv_03_gb300 import binding as B
    from paged_split_kv_03_gb300.synth import config_workload
    wl = config_workload(name, device=dev, **kw)
    dec = B.Decoder(B.params_for(wl, device=dev.index or 0), device=dev)
    g = torch.Generator(device=dev).manual_seed(11)
    shape = (wl.total_rows, wl.num_kv_heads, wl.head_dim)
    k_new = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    v_new = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    B.pda_append_kv(dec.plan, k_new, v_new, wl.page_table, wl.kv_indptr, wl.kv_len, wl.qo_indptr,
                    max(1, wl.max_q_len), wl.k_pages, wl.v_pages, wl.k_scale, wl.v_scale,
                    dec.scratch)
    torch.cuda.synchronize()
    assert dec.status() == 0


def time_graph(fn, steps, warmup, flush, stream):
    """Per-step CUDA-event times (ms) of ``fn`` replayed on ``stream``, with an
    L2 flush enqueued before every step outside the events."""
    import torch
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush()
            a.record(stream)
            fn()
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


# workloads planned from the batch's host lengths, rows and windows (their
# lengths vary; a serving step plans each batch this way), the others from
# their maxima (one plan for any lengths)
HOST_PLANNED = ("mixed",)


def setup_call(wl, dev):
    """Plan, scratch, outputs and a captured CUDA graph of one pda_decode."""
    import torch
    from paged_split_kv_03_gb300 import binding as B
    dec = B.Decoder(B.params_for(wl, device=dev.index or 0, host_plan=wl.name in HOST_PLANNED),
                    device=dev)
    dv = getattr(wl, "head_dim_v", None) or wl.head_dim
    out = torch.empty(wl.total_rows, wl.num_qo_heads, dv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(wl.total_rows, wl.num_qo_heads, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    mq = max(1, wl.max_q_len)
    with torch.cuda.stream(stream):
        dec.run(wl, out, lse, max_q_len=mq, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        dec.run(wl, out, lse, max_q_len=mq, stream=stream)
    return dec, out, lse, stream, graph


def e2e_time(wl, dec, steps, warmup, dev):
    """End to end through the C ABI: pinned host inputs copied to the device,
    pda_decode, outputs copied back, all inside the timed region."""
    import torch
    names = ["q", "k_pages", "v_pages", "k_scale", "v_scale", "page_table", "kv_indptr",
             "kv_len", "qo_indptr", "window"]
    alias = wl.v_pages is wl.k_pages  # an MLA latent is both caches: copied once
    host = {n: getattr(wl, n).cpu().pin_memory() for n in names
            if getattr(wl, n) is not None and not (alias and n == "v_pages")}
    devb = {n: torch.empty_like(getattr(wl, n)) for n in host}
    if alias:
        devb["v_pages"] = devb["k_pages"]
    dv = getattr(wl, "head_dim_v", None) or wl.head_dim
    out = torch.empty(wl.total_rows, wl.num_qo_heads, dv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(wl.total_rows, wl.num_qo_heads, dtype=torch.float32, device=dev)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    stream = torch.cuda.Stream(device=dev)

    class View:
        pass
    v = View()
    for n in names:
        setattr(v, n, devb.get(n))
    v.sm_scale, v.max_q_len = wl.sm_scale, wl.max_q_len

    def step():
        for n, t in host.items():
            devb[n].copy_(t, non_blocking=True)
        dec.run(v, out, lse, stream=stream)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, h2d, d2h


def oracle_rate(wl, budget_s: float, seed: int = 0, max_items=None):
    """Oracle GB/s on ``wl``: times a random sample of (row, q head) items
    sized to about ``budget_s`` seconds and scales to the whole call."""
    import numpy as np
    import torch

    import oracle
    from paged_split_kv_03_gb300.traffic import call_bytes
    host = wl.to("cpu")
    total = host.total_rows * host.num_qo_heads
    g = torch.Generator().manual_seed(seed)
    calib = np.sort(torch.randperm(total, generator=g)[: min(total, 32)].numpy()).astype(np.int64)
    t0 = time.perf_counter()
    oracle.attention_for(host, items=calib)
    per = (time.perf_counter() - t0) / len(calib)
    n = int(min(total, max(len(calib), budget_s / max(per, 1e-9))))
    if max_items:
        n = min(n, max_items)
    items = np.sort(torch.randperm(total, generator=g)[:n].numpy()).astype(np.int64)
    t0 = time.perf_counter()
    oracle.attention_for(host, items=items)
    dt = time.perf_counter() - t0
    full_s = dt * total / n
    gbs = call_bytes(host)["total"] / full_s / 1e9
    return gbs, full_s, n, total, oracle.max_threads()


def parse_workload(spec):
    """'name' or 'name:k=v,k=v' (integer values, else strings such as
    layout=HND) -> (name, kwargs, description)."""
    name, _, rest = spec.partition(":")
    kw = {}
    for item in filter(None, rest.split(",")):
        k, _, v = item.partition("=")
        v = v.strip()
        kw[k.strip()] = int(v) if v.lstrip("-").isdigit() else v
    if name == HEADLINE and not kw:
        return name, kw, HEADLINE_DESC
    return name, kw, f"{name} {kw}"


def max_over_ranks(ms, device):
    """The slowest replica's step time (ms): the job's time when ranks run in
    a process group (any backend), else ``ms`` itself."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (context beside the measured peak)


def step_stats(times_ms):
    """Median and interquartile mean (the mean of the middle half of the sorted
    samples) of per-step times, in microseconds."""
    xs = sorted(times_ms)
    n = len(xs)
    q = n // 4
    mid = xs[q:n - q] if n - 2 * q > 0 else xs
    return {"us_median": statistics.median(xs) * 1e3, "us_iqm": sum(mid) / len(mid) * 1e3}


def whole_job_gbs(bytes_per_rank, world, ms):
    """Whole-job throughput: the bytes every replica moved / the slowest
    replica's time (weak scaling: each rank runs the full workload)."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


def run_ours(args, rank, world, dev):
    import torch

    from paged_split_kv_03_gb300.synth import config_workload
    from paged_split_kv_03_gb300.traffic import call_bytes, call_flops
    torch.cuda.set_device(dev)
    peak, peak_kind = peaks()
    flush = make_flush(dev)

    wname, wkw, wdesc = parse_workload(args.workload)
    wl = config_workload(wname, device=dev, **wkw)
    dec, out, lse, stream, graph = setup_call(wl, dev)
    nbytes = call_bytes(wl, plan=dec.plan)
    flops = call_flops(wl)
    launches_per_step = 1 + (1 if dec.plan.max_splits > 1 else 0)

    dist = world > 1
    if dist:
        import torch.distributed as tdist
        tdist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        times = time_graph(graph.replay, args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()
    clocks = clk.summary()
    if max_over_ranks(0.0 if clocks_ok(clocks) else 1.0, dev) > 0:  # every rank agrees
        # a throttled or clock-locked timed region is taken once more; the
        # line reports the second one and keeps the first one's record
        first = clocks
        with ClockSampler(dev.index or 0) as clk:
            times = time_graph(graph.replay, args.steps, args.warmup, flush, stream)
        torch.cuda.synchronize()
        if dist:
            tdist.barrier()
        clocks = clk.summary() or {}
        clocks = dict(clocks, remeasured_after=first)
    ms = max_over_ranks(sum(times) / len(times), dev)
    value = whole_job_gbs(nbytes["total"], world, ms)
    assert dec.status() == 0, "device status bits set during the benchmark"

    # the dominant kernel: stage 1, timed on its own (a graph of the stage-1
    # launch alone, pda_decode_stages(PARTIAL), same flush and events) right
    # after the timed region; with one split it is the whole call
    if launches_per_step == 1:
        stage1_ms = ms
    else:
        from paged_split_kv_03_gb300 import binding as B
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            dec.run(wl, out, lse, max_q_len=max(1, wl.max_q_len), stream=stream,
                    stages=B.PDA_STAGE_PARTIAL)
        t1 = time_graph(g1.replay, args.steps, args.warmup, flush, stream)
        stage1_ms = sum(t1) / len(t1)
        del g1
    stage1_bytes = nbytes["total"] - nbytes["scratch"] // 2
    roof = {"bound": "hbm", "kernel": "stage1", "peak": peak, "unit": "GB/s",
            "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
            "traffic": recorded_traffic("stage1", args.workload)}
    if stage1_ms:
        roof["achieved"] = stage1_bytes / (stage1_ms * 1e-3) / 1e9
        roof["frac"] = roof["achieved"] / peak
        roof["algorithmic_bytes"] = stage1_bytes
    # the same kernel's duration without the graph-launch latency in it: four
    # stage-1 launches back to back in one graph (each reads the whole cache,
    # more than 2 x L2, from its start, so the L2 it finds holds the end of
    # the previous pass, evicted before it gets there), one flush before them
    if stage1_ms and nbytes["kv"] > 2 * torch.cuda.get_device_properties(dev).L2_cache_size:
        from paged_split_kv_03_gb300 import binding as B
        g4 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g4, stream=stream):
            for _ in range(4):
                dec.run(wl, out, lse, max_q_len=max(1, wl.max_q_len), stream=stream,
                        stages=B.PDA_STAGE_PARTIAL)
        t4 = time_graph(g4.replay, max(3, args.steps // 2), args.warmup, flush, stream)
        b2b_ms = sum(t4) / len(t4) / 4
        del g4
        roof["back_to_back"] = {"ms_per_launch": b2b_ms,
                                "achieved": stage1_bytes / (b2b_ms * 1e-3) / 1e9,
                                "frac": stage1_bytes / (b2b_ms * 1e-3) / 1e9 / peak}

    sweep = []
    if rank == 0 and not args.no_sweep:
        runs = [(name, dict(R=R, bs=bs), f"{name} bs{bs} R{R}" if R else f"{name} bs{bs} R1..8")
                for name, bs, R in SWEEP] + LAYOUT_SWEEP
        for name, kw, label in runs:
            w2 = config_workload(name, device=dev, **kw)
            d2, o2, l2_, s2, g2 = setup_call(w2, dev)
            t2 = time_graph(g2.replay, max(10, args.steps), 3, flush, s2)
            b2 = call_bytes(w2, plan=d2.plan)["total"]
            # the mean, as for the headline: calls of a few tens of us scatter
            # by 1-3 us from step to step (launch jitter and the event clock's
            # granularity), and their median jumps between clusters
            mean = sum(t2) / len(t2)
            sweep.append({"workload": label, "us_per_call": mean * 1e3,
                          "median_us": statistics.median(t2) * 1e3,
                          "GB_s": b2 / (mean * 1e-3) / 1e9,
                          "frac_of_peak": b2 / (mean * 1e-3) / 1e9 / peak, "bytes": b2,
                          "splits": d2.plan.max_splits})
            del w2, d2, o2, l2_, g2
            torch.cuda.empty_cache()
        by = {s["workload"]: s["us_per_call"] for s in sweep}
        for name in ("mtp_verify_bf16", "longctx_fp8_pth"):
            for bs in (1, 16):
                r1, r8 = by.get(f"{name} bs{bs} R1"), by.get(f"{name} bs{bs} R8")
                if r1 and r8:
                    sweep.append({"workload": f"{name} bs{bs}", "R8_over_R1": r8 / r1})

    append = []
    if rank == 0 and not args.no_sweep:
        for name, kw in APPEND_SWEEP:
            append.append(append_time(name, kw, dev, max(10, args.steps), flush, peak))
            torch.cuda.empty_cache()

    e2e = None
    if rank == 0:
        e_ms, h2d, d2h = e2e_time(wl, dec, max(5, args.steps // 2), 2, dev)
        e2e = {"value": nbytes["total"] / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, full_s, n, total, cores = oracle_rate(wl, budget_s=args.cpu_seconds)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} of {total} (row, q head) items of {wname}, timed and scaled "
                         f"to the whole call ({full_s:.1f} s per call)"}

    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "us_per_call": ms * 1e3,
        "step_stats": step_stats(times),
        "frac_of_peak": value / world / peak,
        "frac_of_nominal_8tbs": value / world / NOMINAL_HBM_GBS,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / world / PAGES_NUMBER["value"] if wdesc == HEADLINE_DESC else None,
        "vs_baseline_ref": PAGES_NUMBER,
        "dtype": ("e4m3 (tcgen05 e4m3 x e4m3 MMAs, fp32 accumulate)" if wdesc == HEADLINE_DESC
                  else ("int8" if wl.kv_int8 else "e4m3" if wl.kv_e4m3 else "bf16")),
        "data": "synthetic (seeded N(0,1), e4m3 per-tensor)" if wdesc == HEADLINE_DESC
                else "synthetic (seeded N(0,1))",
        "config": {"workload": wdesc},
        "setup": {"parallelism": f"replicas x{world}",
                  "l2": "flushed before every step (memset of 2x L2, then a read of 2x L2), outside the events",
                  "graph": "stage 1 + stage 2 captured in one CUDA graph",
                  "splits": dec.plan.max_splits, "chunk_pages": dec.plan.chunk_pages,
                  "grid_ctas": dec.plan.grid_ctas, "bytes_per_call": nbytes,
                  "flops_per_call": flops, "tflops": flops / (ms * 1e-3) / 1e12},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
        "r_sweep": sweep, "append": append, "source_sha": source_sha(),
    }


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores: each step a bounded
    sample of the headline workload scaled to the call."""
    import torch

    from paged_split_kv_03_gb300.synth import config_workload
    if rank != 0:
        return None
    wl = config_workload(HEADLINE, device="cpu")
    budget = args.reference_seconds
    for i in range(args.warmup):
        oracle_rate(wl, budget_s=min(budget, 2.0), seed=100 + i)
    rates, secs = [], []
    n = total = cores = 0
    for i in range(args.steps):
        gbs, full_s, n, total, cores = oracle_rate(wl, budget_s=budget, seed=i)
        rates.append(gbs)
        secs.append(full_s)
    value = statistics.mean(rates)
    sample = (f"per step {n} of {total} (row, q head) items of {HEADLINE}, scaled to the call")
    ms = statistics.mean(secs) * 1e3
    return {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": HEADLINE_DESC},
            "cpu_baseline": {"value": value, "unit": "GB/s", "kind": "oracle", "cores": cores,
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--workload", default=HEADLINE,
                    help="workload of the timed step, 'name' or 'name:bs=16,R=8' (default: "
                         "the FP8 decode headline); other workloads serve profiling")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=4.0)
    ap.add_argument("--profile-append", action="store_true",
                    help="profiling aid: run one pda_append_kv of each append workload and "
                         "exit (no timing, no JSON line)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.profile_append:
        import torch
        for name, kw in APPEND_SWEEP:
            append_once(name, kw, torch.device("cuda", local))
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        import torch
        if world > 1:
            import torch.distributed as tdist
            torch.cuda.set_device(local)
            tdist.init_process_group("nccl")
        res = run_ours(args, rank, world, torch.device("cuda", local))
        if world > 1:
            import torch.distributed as tdist
            tdist.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

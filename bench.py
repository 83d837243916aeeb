"""Benchmark: paged FP8 MQA logits on one GB300 (replicas on N GPUs), one JSON line.

Default workload: the decode batch (64 requests, next_n = 1, 64 heads, head_dim 128, 64-token
blocks, seq_lens uniform in [1024, 32768]).  One step = one launch of the fused logits kernel
(in-kernel schedule, logits, row_ends); for the workloads with a top-k (long_select, serving) the
step also resets the counters and thresholds and runs the threshold select with its repair.
Metric: Gscores/s, valid (query row, KV position) pairs per second.  Inputs are resident in HBM; three copies of the KV pool (each larger than
L2) are used in rotation so no step finds its pool in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|mtp|long_select|serving]
  python bench.py --impl reference ...   # the CPU oracle on the host cores, same metric

Multi-GPU: the path shards by request with no exchange step; each rank runs an independent
replica of the workload ("scaling": "weak") and rank 0 reports the sum over ranks.
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

import torch  # noqa: E402

import paged_fp8_mqa_gb300 as idx  # noqa: E402
from paged_fp8_mqa_gb300 import synth  # noqa: E402

METRIC = "Gscores/s (query row x KV pos) and % of HBM/FP8 roofline, paged MQA logits"
UNIT = "Gscores/s"
POOL_COPIES = 3


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained",
                                                     p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def load_fp8_peak() -> dict | None:
    """The dense e4m3 tensor peak measured on the GB300s (``--measure-fp8-peak``,
    committed under profiles/), or None."""
    path = os.path.join(ROOT, "profiles", "fp8_peak.json")
    if not os.path.exists(path):
        return None
    return json.load(open(path))


def measure_fp8_peak(dev, seconds: float = 4.0) -> dict:
    """Dense e4m3 x e4m3 -> bf16 GEMM throughput of the library GEMM (torch._scaled_mm,
    8192^3, 2*N^3 flops): best of 10 single calls (burst) and the mean over a loop of about
    `seconds` (sustained, under the power cap), with the clocks sampled meanwhile."""
    n = 8192
    g = torch.Generator(device=dev).manual_seed(0)
    a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    one = torch.ones((), device=dev, dtype=torch.float32)

    def mm():
        return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16,
                                use_fast_accum=True)

    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    iters = max(10, int(seconds * 1e3 / best))
    e0.record()
    for _ in range(iters):
        mm()
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    sustained = e0.elapsed_time(e1) / iters
    flops = 2.0 * n ** 3
    return {"fp8_tflops": flops / (best * 1e-3) / 1e12,
            "fp8_tflops_sustained": flops / (sustained * 1e-3) / 1e12,
            "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, 8192^3 (2*N^3 flops), use_fast_accum; "
                   f"best of 10 (burst) and the mean of {iters} back-to-back calls (sustained)",
            "gpu": torch.cuda.get_device_name(dev), "torch": torch.__version__,
            "clocks_sustained": clocks}


def algorithmic(w: synth.Workload) -> dict:
    """Per-launch algorithmic work: KV values + scales of every valid position (132 B each),
    the logits written (4 B per valid score), q and w; MMA flops 2*64*128 per score."""
    P = int(w.seq_lens.to(torch.int64).sum())
    scores = w.valid_scores()
    kv = 132 * P
    out = 4 * scores
    qw = w.q.numel() + 4 * w.weights.numel()
    return {"positions": P, "scores": scores, "kv_bytes": kv, "bytes": kv + out + qw,
            "flops": 2 * 64 * 128 * w.next_n * P}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        self.device = device
        self.t0 = self.t1 = None

    def start(self):
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(self.device).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which: str):
        setattr(self, which, time.time())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm, mx, reasons = [], None, set()
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for name, col in (("hw_slowdown", 5), ("hw_thermal_slowdown", 6),
                                  ("sw_thermal_slowdown", 7), ("sw_power_cap", 8)):
                    if r[col].strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# Sources compiled into the logits kernel: the committed traffic figures hold only for them.
KERNEL_SOURCES = ("logits.cu", "logits_kernel.cuh", "ptx.cuh", "split.cuh", "slots.cuh",
                  "internal.h", "mx_convert.cuh")


def kernel_sources_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "paged_fp8_mqa_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


def measured_traffic(workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the committed
    ncu capture, if it was taken on the kernel sources as they stand; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(workload)
    if not rec or rec.get("kernel_sources_sha256") != kernel_sources_digest():
        return None
    return rec["bytes_per_launch"]


def device_inputs(w: synth.Workload, dev):
    pools = [w.kv_fused.to(dev)]
    for _ in range(POOL_COPIES - 1):
        pools.append(pools[0].clone())
    return dict(q=w.q.to(dev), pools=pools, weights=w.weights.to(dev),
                bt=w.block_tables.to(dev), seq_lens=w.seq_lens.to(dev))


def launch(w, t, pool, out, row_ends, stream):
    sel = t.get("select")
    if sel is not None:
        # The caller's part of the select contract: zeroed counters, this step's thresholds.
        sel["counters"].zero_()
        sel["thr"].copy_(sel["thr0"])
    idx.logits_fp8(t["q"], pool, t["weights"], t["bt"], t["seq_lens"], w.max_seq_len, out=out,
                   row_ends_out=row_ends, stream=stream)
    if sel is not None:
        idx.threshold_select(out, row_ends, sel["thr"], sel["counters"], sel["cand"], w.top_k,
                             w.capacity, w.max_seq_len, arrivals=sel["arrivals"],
                             ranges=sel["ranges"], stream=stream)


def selection_inputs(w: synth.Workload, t: dict, dev) -> dict:
    """Select buffers and this workload's thresholds, derived (outside any timed region) from
    the logits of one untimed launch: each row's K'-th largest value, perturbed as the workload
    prescribes (below the K'-th value with forced +inf rows, or x U[0.9, 1.1])."""
    rows, pad = w.rows, idx.idx_padded_seq_len(w.max_seq_len)
    out = torch.empty(rows, pad, device=dev)
    row_ends = torch.empty(rows, dtype=torch.int32, device=dev)
    idx.logits_fp8(t["q"], t["pools"][0], t["weights"], t["bt"], t["seq_lens"], w.max_seq_len,
                   out=out, row_ends_out=row_ends)
    torch.cuda.synchronize()
    kth = torch.full((rows,), float("nan"), dtype=torch.float64)
    ends = row_ends.cpu()
    for r in range(rows):
        e = int(ends[r])
        k = min(e, w.top_k)
        if k:
            kth[r] = float(torch.topk(out[r, :e], k).values[-1])
    if w.name == "serving":
        thr0 = synth.thresholds_scaled_kth(w, kth)
    else:
        thr0 = synth.thresholds_below_kth(w, kth)
    del out
    # Thresholds at which every row fits (each row's K'-th largest score itself): the steady
    # state of a serving loop whose thresholds carry over from step to step.
    thr_fit = torch.nan_to_num(kth, nan=0.0).to(torch.float32)
    return dict(thr0=thr0.to(dev), thr=thr0.to(dev).clone(), thr_fit=thr_fit.to(dev),
                counters=torch.zeros(rows, 2, dtype=torch.int32, device=dev),
                cand=torch.zeros(rows, w.top_k + w.capacity, 2, dtype=torch.int32, device=dev),
                arrivals=torch.zeros(rows, dtype=torch.int32, device=dev),
                ranges=torch.zeros(2, rows, dtype=torch.int32, device=dev))


def time_select(w, t, stream, launches: int = 200) -> dict:
    """Diagnostic: the select launch alone, each bracketed by its own events, on logits that
    stay in L2 between launches (the situation inside a step)."""
    sel = t["select"]
    rows, pad = w.rows, idx.idx_padded_seq_len(w.max_seq_len)
    out = torch.empty(rows, pad, device=t["q"].device)
    row_ends = torch.empty(rows, dtype=torch.int32, device=t["q"].device)
    with torch.cuda.stream(stream):
        idx.logits_fp8(t["q"], t["pools"][0], t["weights"], t["bt"], t["seq_lens"],
                       w.max_seq_len, out=out, row_ends_out=row_ends, stream=stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(launches)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)
        for a, b in ev:
            sel["counters"].zero_()
            sel["thr"].copy_(sel["thr0"])
            a.record(stream)
            idx.threshold_select(out, row_ends, sel["thr"], sel["counters"], sel["cand"],
                                 w.top_k, w.capacity, w.max_seq_len, arrivals=sel["arrivals"],
                                 ranges=sel["ranges"], stream=stream)
            b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    keys = int(w.row_ends().to(torch.int64).sum())
    return {"ms_per_launch": ms, "keys": keys, "keys_per_s": keys / (ms * 1e-3),
            "logits_gbs": 4 * keys / (ms * 1e-3) / 1e9,
            "note": "two launches (classification; fit rule and repair); reads each row's "
                    "logits (L2-resident after the logits kernel) once, and rows that do not "
                    "fit again in their radix repair"}


def time_device(w, t, steps, warmup, stream, sampler=None):
    """The timed region: K launches back to back on the launching stream, bracketed by CUDA
    events (and a barrier plus a device synchronize on both sides).  Returns the milliseconds
    per launch over the region.  The host enqueues ahead of the device (a short device-side
    spin opens the region), so the figure is the device's own launch-to-launch time."""
    dev = t["q"].device
    out = torch.empty(w.rows, idx.idx_padded_seq_len(w.max_seq_len), device=dev)
    row_ends = torch.empty(w.rows, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            launch(w, t, t["pools"][i % POOL_COPIES], out, row_ends, stream)
    torch.cuda.synchronize()
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t0")
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)  # ~1 ms: the host's enqueueing runs ahead of the device
        region0.record(stream)
        h0 = time.perf_counter()
        for i in range(steps):
            launch(w, t, t["pools"][i % POOL_COPIES], out, row_ends, stream)
        host_ms = (time.perf_counter() - h0) * 1e3 / steps
        region1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t1")
    barrier()
    return region0.elapsed_time(region1) / steps, host_ms


def time_fused(w, t, steps, warmup, stream) -> dict:
    """The same step through the fused score + select (no logits written; the rescoring and
    repair launches run when a row needs them), timed like the two-stage step."""
    sel = t["select"]
    dev = t["q"].device
    arrivals = torch.zeros(w.batch, dtype=torch.int32, device=dev)
    scratch = torch.empty(w.rows, idx.idx_padded_seq_len(w.max_seq_len), device=dev)

    def step(pool):
        sel["counters"].zero_()
        sel["thr"].copy_(sel["thr0"])
        idx.indexer_threshold_select(t["q"], pool, t["weights"], t["bt"], t["seq_lens"],
                                     w.max_seq_len, thresholds=sel["thr"],
                                     counters=sel["counters"], candidates=sel["cand"],
                                     top_k=w.top_k, arrivals=arrivals, ranges=sel["ranges"],
                                     scratch=scratch, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(t["pools"][i % POOL_COPIES])
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)
        e0.record(stream)
        for i in range(steps):
            step(t["pools"][i % POOL_COPIES])
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"ms_per_step": ms, "launches_per_step": 3,
            "note": "one pass scores and classifies without writing logits; rows that do not "
                    "fit are rescored into a scratch buffer and repaired by two further launches "
                    "(launched every step, empty when nothing needs a repair)"}


def time_selecting(name: str, dev, steps: int, warmup: int, stream, peaks: dict) -> dict:
    """A workload with a top-k (long_select or serving), timed like the headline: the two-stage
    step (counter and threshold reset, logits, threshold select with its repair) over K
    back-to-back steps; the select launch alone; the fused score + select step with the
    workload's thresholds; and both steps again with thresholds at which every row fits."""
    w = make(name)
    t = device_inputs(w, dev)
    t["select"] = selection_inputs(w, t, dev)
    alg = algorithmic(w)
    two, _ = time_device(w, t, steps, warmup, stream)
    single = time_launch_events(w, t, min(steps, 100), stream)
    sel = time_select(w, t, stream, min(steps, 200))
    fused = time_fused(w, t, steps, warmup, stream)
    s = t["select"]
    saved, s["thr0"] = s["thr0"], s["thr_fit"]
    two_fit, _ = time_device(w, t, steps, warmup, stream)
    fused_fit = time_fused(w, t, steps, warmup, stream)
    s["thr0"] = saved
    t_roof = alg["kv_bytes"] / (peaks["hbm_gbs"] * 1e9) * 1e3
    return {"value": alg["scores"] / (two * 1e-3) / 1e9, "unit": UNIT,
            "config": workload_config(w), "ms_per_step": two,
            "single_step_ms": single, "select_ms_per_launch": sel["ms_per_launch"],
            "fused_ms_per_step": fused["ms_per_step"],
            "all_rows_fit": {"ms_per_step": two_fit, "fused_ms_per_step": fused_fit["ms_per_step"],
                             "thresholds": "each row's K'-th largest score"},
            "kv_roofline_time_ms": t_roof, "kv_roofline_frac": t_roof / two,
            "note": "step = counter/threshold reset + logits + select (3 kernels, plus 2 small "
                    "torch fills); fused = the same outputs through idx_indexer_threshold_select "
                    "(3 kernels)"}


def time_mxfp4(w: synth.Workload, dev, steps: int, warmup: int, stream, peaks: dict) -> dict:
    """The MXFP4 variant on the same lengths, pages and weights (q and K drawn anew and
    quantized): q staging + the MXFP4 logits kernel per step, three MXFP4 pools in rotation
    (each below L2 on its own, together above it).  Roofline: the MXFP4 bytes of every valid position (D/2 + D/32
    per token), the logits written, q, q_sf and w."""
    m = synth.make_mxfp4(w)
    pools = [m.kv_fused.to(dev)]
    for _ in range(POOL_COPIES - 1):
        pools.append(pools[0].clone())
    q, qsf = m.q.to(dev), m.q_sf.to(dev)
    wt, bt, sl = w.weights.to(dev), w.block_tables.to(dev), w.seq_lens.to(dev)
    ws = torch.empty(idx.idx_mxfp4_workspace_bytes(w.num_blocks, w.block_size, w.batch,
                                                   w.next_n, w.num_heads, w.head_dim),
                     dtype=torch.uint8, device=dev)
    out = torch.empty(w.rows, idx.idx_padded_seq_len(w.max_seq_len), device=dev)

    def step(i):
        idx.logits_mxfp4(q, qsf, pools[i % POOL_COPIES], wt, bt, sl, w.max_seq_len, out=out,
                         workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)
        e0.record(stream)
        for i in range(steps):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    D = w.head_dim
    P = int(w.seq_lens.to(torch.int64).sum())
    scores = w.valid_scores()
    nbytes = P * (D // 2 + D // 32) + 4 * scores + m.q.numel() + m.q_sf.numel() + 4 * wt.numel()
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    return {"value": scores / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_launch": ms,
            "launches_per_step": 2, "algorithmic_bytes": nbytes,
            "hbm_gbs": nbytes / (ms * 1e-3) / 1e9, "roofline_time_ms": t_hbm * 1e3,
            "roofline_frac": t_hbm * 1e3 / ms,
            "note": "q staged in the FP8 layout by a small kernel, then the logits kernel with "
                    "converter warps turning each tile's MXFP4 pages into e4m3 in shared memory "
                    "(no staged KV pool in HBM)"}


def time_launch_events(w, t, steps, stream):
    """Diagnostic: the same launches each bracketed by its own pair of events (which keeps the
    device from overlapping one launch's start with the previous one's end)."""
    dev = t["q"].device
    out = torch.empty(w.rows, idx.idx_padded_seq_len(w.max_seq_len), device=dev)
    row_ends = torch.empty(w.rows, dtype=torch.int32, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)
        for i, (a, b) in enumerate(ev):
            a.record(stream)
            launch(w, t, t["pools"][i % POOL_COPIES], out, row_ends, stream)
            b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def time_e2e(w, dev, steps, stream, sel=None):
    """Same metric through the public calls with host buffers: every step copies its inputs
    from pinned host memory, runs the step and copies its result back (the logits, or for a
    selecting workload the selection: candidates, counters, ranges and thresholds).  The steps
    are pipelined as a serving loop would run them: step i + 1's inputs are copied (into the
    second of two device input sets, on a copy stream) while step i computes, and step i's
    result is copied back on another copy stream."""
    host = dict(q=w.q.pin_memory(), kv=w.kv_fused.pin_memory(),
                weights=w.weights.pin_memory(), bt=w.block_tables.pin_memory(),
                seq_lens=w.seq_lens.pin_memory())
    if sel is not None:
        host["thr"] = sel["thr0"].cpu().pin_memory()
    devb = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    pad = idx.idx_padded_seq_len(w.max_seq_len)
    out = torch.empty(w.rows, pad, device=dev)
    row_ends = torch.empty(w.rows, dtype=torch.int32, device=dev)

    def results(j):
        if sel is None:
            return {"out": out}
        return {"cand": sel["cand"], "counters": sel["counters"], "ranges": sel["ranges"],
                "thr": devb[j]["thr"]}
    back = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in results(0).items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in back.values())
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # set j's inputs landed
    ev_used = [torch.cuda.Event() for _ in range(2)]  # the step computing on set j finished
    ev_back = torch.cuda.Event()                      # the last result copy finished
    ev_used[0].record(stream)
    ev_used[1].record(stream)
    ev_back.record(stream)

    def copy_in(i):
        j = i % 2
        s_in.wait_event(ev_used[j])
        with torch.cuda.stream(s_in):
            for k in host:
                devb[j][k].copy_(host[k], non_blocking=True)
        ev_in[j].record(s_in)

    def compute(i):
        j = i % 2
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_back)  # the result buffers are free again
        d = devb[j]
        idx.logits_fp8(d["q"], d["kv"], d["weights"], d["bt"], d["seq_lens"], w.max_seq_len,
                       out=out, row_ends_out=row_ends, stream=stream)
        if sel is not None:
            with torch.cuda.stream(stream):
                sel["counters"].zero_()
            idx.threshold_select(out, row_ends, d["thr"], sel["counters"], sel["cand"],
                                 w.top_k, w.capacity, w.max_seq_len, arrivals=sel["arrivals"],
                                 ranges=sel["ranges"], stream=stream)
        ev_used[j].record(stream)
        s_out.wait_event(ev_used[j])
        with torch.cuda.stream(s_out):
            for k, v in results(j).items():
                back[k].copy_(v, non_blocking=True)
        ev_back.record(s_out)

    def run(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
        stream.wait_event(ev_back)

    run(3)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    ev_used[0].record(stream)  # the copies start after e0
    ev_used[1].record(stream)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, h2d, d2h


def _first_requests(w: synth.Workload, nreq: int) -> synth.Workload:
    return synth.Workload(**{**w.__dict__, "batch": nreq, "seq_lens": w.seq_lens[:nreq],
                             "block_tables": w.block_tables[:nreq],
                             "q": w.q[:nreq].contiguous(),
                             "weights": w.weights[:nreq * w.next_n].contiguous()})


def cpu_baseline(w: synth.Workload, budget_s: float = 15.0) -> dict:
    """The float64 oracle, as it stands, on this host's cores, over a bounded sample of the
    workload: its first requests, as many as a one-request probe says fit the time budget."""
    import oracle
    lib = oracle.load()
    threads = oracle.max_threads(lib)

    def run(sub):
        t0 = time.perf_counter()
        oracle.paged_logits(sub.q, sub.kv_fused, sub.weights, sub.block_tables, sub.seq_lens,
                            sub.max_seq_len, block_size=sub.block_size, with_tol=False, lib=lib)
        return time.perf_counter() - t0

    probe = _first_requests(w, 1)
    per_score = run(probe) / max(probe.valid_scores(), 1)
    re = w.row_ends().to(torch.int64).view(w.batch, w.next_n).sum(1).cumsum(0)
    nreq = max(1, int((re.to(torch.float64) * per_score <= budget_s).sum()))
    sub = _first_requests(w, nreq)
    dt = run(sub)
    return {"value": sub.valid_scores() / dt / 1e9, "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": f"first {nreq} of {w.batch} requests of the {w.name} workload "
                      f"({sub.valid_scores()} scores in {dt:.1f} s wall; float64, exact e4m3 "
                      f"decode, OpenMP over rows and 256-position chunks)"}


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def _reduce(x: float, op) -> float:
    """All-reduce of one float over the replicas (on the GPU under NCCL, on the host under
    gloo); x itself without a process group."""
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=op)
        return float(t.item())
    return x


def reduce_max(x: float) -> float:
    return _reduce(x, torch.distributed.ReduceOp.MAX)


def reduce_sum(x: float) -> float:
    return _reduce(x, torch.distributed.ReduceOp.SUM)


def make(name: str) -> synth.Workload:
    return synth.WORKLOADS[name]()


def run_reference(args, rank: int, world: int) -> None:
    """The oracle on the host cores: each step is a bounded sample of the workload."""
    if rank != 0:
        return
    import oracle
    w = make(args.workload)
    lib = oracle.load()
    threads = oracle.max_threads(lib)
    nreq = max(1, min(w.batch, 4))
    sub = _first_requests(w, nreq)

    def step():
        oracle.paged_logits(sub.q, sub.kv_fused, sub.weights, sub.block_tables, sub.seq_lens,
                            sub.max_seq_len, block_size=sub.block_size, with_tol=False, lib=lib)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = sub.valid_scores() / dt / 1e9
    sample = (f"first {nreq} of {w.batch} requests of the {w.name} workload "
              f"({sub.valid_scores()} scores per step), float64 oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def workload_config(w: synth.Workload) -> dict:
    return {"workload": f"{w.name}: B={w.batch}, next_n={w.next_n}, heads={w.num_heads}, "
                        f"head_dim={w.head_dim}, block_size={w.block_size}, "
                        f"max_seq_len={w.max_seq_len}, seed={w.seed}",
            "batch": w.batch, "next_n": w.next_n, "max_seq_len": w.max_seq_len,
            "valid_scores": w.valid_scores(),
            "l2": f"inputs larger than L2: {POOL_COPIES} KV-pool copies "
                  f"({w.kv_fused.numel() / 1e6:.0f} MB each) used in rotation",
            "parallelism": "replicas"}


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--measure-fp8-peak", action="store_true",
                    help="print the dense e4m3 GEMM peak of this GPU as one JSON line and exit")
    args = ap.parse_args()
    if args.measure_fp8_peak:
        print(json.dumps(measure_fp8_peak(torch.device("cuda", 0))), flush=True)
        return
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(dev)
    peaks = load_peaks()

    w = make(args.workload)
    t = device_inputs(w, dev)
    if w.top_k is not None:
        t["select"] = selection_inputs(w, t, dev)
    alg = algorithmic(w)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    mean_ms, host_ms = time_device(w, t, args.steps, args.warmup, stream, sampler)
    clocks = sampler.stop() if sampler else None
    step_ms = reduce_max(mean_ms)
    event_ms = time_launch_events(w, t, min(args.steps, 200), stream)
    select_diag = time_select(w, t, stream) if "select" in t else None
    fused_diag = None
    if "select" in t and not args.no_secondary:
        n_fused = max(3, min(500, args.steps))
        fused_diag = time_fused(w, t, n_fused, args.warmup, stream)
        fused_diag["value"] = alg["scores"] / (fused_diag["ms_per_step"] * 1e-3) / 1e9
        fused_diag["unit"] = UNIT
        fused_diag["two_stage_ms_per_step"] = mean_ms
        # The same comparison with thresholds at which every row fits (no repair runs).
        sel = t["select"]
        saved, sel["thr0"] = sel["thr0"], sel["thr_fit"]
        two_fit, _ = time_device(w, t, n_fused, args.warmup, stream)
        fit = time_fused(w, t, n_fused, args.warmup, stream)
        sel["thr0"] = saved
        fused_diag["all_rows_fit"] = {"ms_per_step": fit["ms_per_step"],
                                      "two_stage_ms_per_step": two_fit,
                                      "thresholds": "each row's K'-th largest score"}
    value = reduce_sum(alg["scores"] / (mean_ms * 1e-3) / 1e9)
    status = idx.device_status(clear=True)

    e2e_ms, h2d, d2h = time_e2e(w, dev, max(3, min(20, args.steps)), stream, t.get("select"))
    e2e_value = reduce_sum(alg["scores"] / (e2e_ms * 1e-3) / 1e9)

    hbm_ach = alg["bytes"] / (mean_ms * 1e-3) / 1e9
    fp8 = load_fp8_peak()
    if fp8 is not None:
        fp8_peak, fp8_source = fp8["fp8_tflops"], "measured e4m3 GEMM burst (profiles/fp8_peak.json)"
    else:
        fp8_peak, fp8_source = 2.0 * peaks["bf16_tflops"], peaks["source"] + " bf16 x 2 (nominal ratio)"
    t_hbm = alg["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_mma = alg["flops"] / (fp8_peak * 1e12)
    bound = "hbm" if t_hbm >= t_mma else "tensor"
    roof = {"bound": bound, "achieved": hbm_ach if bound == "hbm" else
            alg["flops"] / (mean_ms * 1e-3) / 1e12,
            "peak": peaks["hbm_gbs"] if bound == "hbm" else fp8_peak,
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "traffic": measured_traffic(args.workload),
            "peak_source": (peaks["source"] + " copy bandwidth (MEASURED_PEAKS.json)")
            if bound == "hbm" else fp8_source,
            "fp8_peak_tflops": fp8_peak, "fp8_peak_source": fp8_source,
            "algorithmic_bytes": alg["bytes"], "kv_bytes": alg["kv_bytes"],
            "flops": alg["flops"],
            "roofline_time_ms": max(t_hbm, t_mma) * 1e3,
            "roofline_frac": max(t_hbm, t_mma) * 1e3 / mean_ms}
    roof["frac"] = roof["achieved"] / roof["peak"]
    # The survey's definition: KV bytes only (132 B per position) against the FP8 MMA time;
    # and the same for a launch timed on its own (no overlap with a neighbouring launch).
    t_kv = max(alg["kv_bytes"] / (peaks["hbm_gbs"] * 1e9), t_mma) * 1e3
    roof["kv_roofline_time_ms"] = t_kv
    roof["frac_kv"] = t_kv / mean_ms
    roof["frac_kv_single_launch"] = t_kv / event_ms

    secondary = {}
    if not args.no_secondary and args.workload == "decode":
        # The next_n = 4 workload, timed the same way (a context figure, not the headline).
        w2 = make("mtp")
        t2 = device_inputs(w2, dev)
        m2, _ = time_device(w2, t2, max(3, min(500, args.steps)), args.warmup, stream)
        a2 = algorithmic(w2)
        e2 = time_launch_events(w2, t2, min(args.steps, 200), stream)
        r2 = max(a2["bytes"] / (peaks["hbm_gbs"] * 1e9), a2["flops"] / (fp8_peak * 1e12)) * 1e3
        k2 = max(a2["kv_bytes"] / (peaks["hbm_gbs"] * 1e9), a2["flops"] / (fp8_peak * 1e12)) * 1e3
        secondary["mtp"] = {"value": a2["scores"] / (m2 * 1e-3) / 1e9, "unit": UNIT,
                            "ms_per_launch": m2, "single_launch_ms": e2,
                            "roofline_time_ms": r2, "roofline_frac": r2 / m2,
                            "kv_roofline_time_ms": k2, "frac_kv": k2 / m2,
                            "bound_kv": "hbm" if a2["kv_bytes"] / (peaks["hbm_gbs"] * 1e9) >=
                            a2["flops"] / (fp8_peak * 1e12) else "tensor",
                            "hbm_gbs": a2["bytes"] / (m2 * 1e-3) / 1e9,
                            "tflops": a2["flops"] / (m2 * 1e-3) / 1e12}
        del t2
        # The workloads with a top-k: long context (8 x 131072, next_n 2) and the serving mix.
        for name in ("long_select", "serving"):
            secondary[name] = time_selecting(name, dev, max(3, min(200, args.steps)),
                                             args.warmup, stream, peaks)
        # The MXFP4 variant on the decode workload's shape.
        secondary["mxfp4"] = time_mxfp4(w, dev, max(3, min(300, args.steps)), args.warmup,
                                        stream, peaks)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32",
            "data": "synthetic", "config": workload_config(w),
            "launch_event_ms": event_ms, "host_enqueue_ms": host_ms,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "note": "every step copies its inputs from pinned host memory and its result "
                            "back; the next step's input copy overlaps the current step's "
                            "compute and result copy (two device input sets, two copy streams)"},
            "gpu_launches": args.steps * (2 if select_diag else 1), "device_status": status,
            "clocks": clocks, "roofline": roof, "cpu_baseline": cpu,
        }
        if secondary:
            line["secondary"] = secondary
        if select_diag:
            line["select"] = select_diag
        if fused_diag:
            line["fused"] = fused_diag
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

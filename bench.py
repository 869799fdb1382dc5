"""Benchmark of the calibration-Hessian hot path on one GB300.

One step = reset the accumulator, add every batch of the workload through
the C ABI (the queue fuses them into split-K SYRK passes), and materialize
the damped fp32 Hessian.  Inputs are synthetic, seeded and resident in HBM
before the timed region; they are larger than L2, so no flush is needed.

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle instead, on a bounded sample of the same workload.
"""

from __future__ import annotations

import os

# The CPU baseline's BLAS thread count is set explicitly, before numpy loads
# its BLAS: every host core unless the caller chose otherwise.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(os.cpu_count() or 1))

import argparse
import hashlib
import json
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Hessian-accum TFLOP/s & tokens/s at d=4096 (1 GB300); % of BF16/HBM roofline"

F32_MMAS = 3  # tf32 MMAs per product in the fp32-input kernel

# DRAM bytes (read + write) per SYRK launch of one step of a workload, from an
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum), with the SHA-256
# of the kernel sources it was taken on.  When the sources differ the figure
# no longer describes the kernel and the line reports traffic as null.
SYRK_SOURCES = ["syrk_bf16.cu", "syrk_common.cuh", "schedule.cuh", "ptx.cuh", "kernels.cuh"]
SYRK_DRAM_BYTES_PER_LAUNCH = {
    # workload: (bytes per launch, sources hash)
    "d4096_ragged360_loguniform": (1.512e9, "57755913f75836f3"),
}


def syrk_source_hash():
    h = hashlib.sha256()
    for f in SYRK_SOURCES:
        with open(os.path.join(ROOT, "gptq_qqq_calibration_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def syrk_traffic(workload):
    rec = SYRK_DRAM_BYTES_PER_LAUNCH.get(workload)
    if rec is None:
        return None, "no capture for this workload"
    nbytes, src = rec
    cur = syrk_source_hash()
    if src != cur:
        return None, f"stale: captured on kernel sources {src}, current {cur}"
    return nbytes, f"ncu dram bytes per launch, kernel sources {cur}"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained", p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def algo_flops(n_tokens, d):
    return float(n_tokens) * d * (d + 1)


class Clocks:
    """nvidia-smi sampling of SM clocks, power and throttle reasons around a
    region; summary() keeps the samples taken inside the region that
    region_start()/region_end() bracket (host wall clock)."""

    def __init__(self, path):
        self.path = path
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=timestamp,index,clocks.sm,clocks.max.sm,power.draw.instant,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "20", "-i", str(self._index())],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def region_start(self):
        self.t0 = time.time()

    def region_end(self):
        self.t1 = time.time()

    @staticmethod
    def _index():
        import torch
        return torch.cuda.current_device()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        import datetime
        try:
            rows = [[x.strip() for x in r.split(",")]
                    for r in open(self.path).read().strip().splitlines() if r.strip()]
            stamp = [datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp() for r in rows]
            inside = [r for r, t in zip(rows, stamp)
                      if self.t0 is not None and self.t1 is not None and self.t0 <= t <= self.t1]
            window = "timed region"
            if not inside:  # a region shorter than the sampling interval
                inside, window = rows, "whole sampler run (no sample inside the timed region)"
            sm = [float(r[2]) for r in inside]
            mx = [float(r[3]) for r in rows]
            pw = [float(r[4]) for r in inside if r[4] not in ("", "[N/A]")]
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i] == "Active"})
            return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": max(mx),
                    "power_w": round(statistics.median(pw), 1) if pw else None, "reasons": reasons,
                    "samples": len(inside), "window": window}
        except Exception as e:  # pragma: no cover
            return {"error": str(e)}


def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return ws, rank


def max_over_ranks(x, ws):
    """The largest of every rank's x (the timing rule: the slowest rank)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, ms, ws):
    """Whole-job rate: every rank's units over the slowest rank's time."""
    return ws * units_per_rank / (ms * 1e-3)


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------- ours


def run_ours(args):
    import torch

    from gptq_qqq_calibration_gb300 import Hessian, LocalHessian
    from gptq_qqq_calibration_gb300.hessian import hess_kernel_launches
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS

    ws, rank = dist_init()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    hbm, bf16_burst, bf16_sust, peak_src = peaks()
    wl = WORKLOADS[args.workload]
    if args.batches:
        wl = wl.scaled(n_batches=args.batches)
    d = wl.d
    in_dtype = torch.float32 if args.dtype == "f32" else torch.bfloat16
    xs = [wl.batch(b, device="cuda", dtype=in_dtype) for b in range(len(wl.token_counts))]
    n_tok = wl.n_tokens
    flops = algo_flops(n_tok, d)
    h = Hessian(d)
    out = torch.empty((d, d), dtype=torch.float32, device="cuda")

    # The queue flushes at the same calls in every step (the same batches in
    # the same order): find them once, then time each flushing call with
    # events inside the timed steps.  Only that call's SYRK launch runs on
    # the stream between its two events, so their sum is the SYRK time
    # within the step.
    flush_at = _flushing_calls(h, xs)
    n_pairs = len(flush_at) + 1  # + the remainder flush inside materialize
    marks = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_pairs)] for _ in range(args.steps)]

    def step(ev=None):
        h.reset()
        k = 0
        for i, X in enumerate(xs):
            if ev is not None and i in flush_at:
                ev[k][0].record()
                h.add_batch(X)
                ev[k][1].record()
                k += 1
            else:
                h.add_batch(X)
        if ev is not None:
            ev[k][0].record()
            h.flush()
            ev[k][1].record()
        h.materialize(wl.damp_percent, out=out, want_damp=False)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    h.sync()  # no device-side wait ran out in the warm-up
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0 = hess_kernel_launches(h.handle)  # the library's own count of its kernel launches
    with Clocks(os.path.join(tempfile.gettempdir(), f"hess_bench_clocks_rank{rank}.csv")) as clk:
        time.sleep(0.3)  # let the sampler start before the timed region
        clk.region_start()
        e0.record()
        for k in range(args.steps):
            step(marks[k])
        e1.record()
        torch.cuda.synchronize()
        clk.region_end()
    barrier(ws)
    kernels_timed = hess_kernel_launches(h.handle) - k0
    h.sync()  # raises if a device-side wait ran out in the timed steps
    ms_local = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms_local, ws)
    value = job_throughput(flops, ms, ws) / 1e12
    syrk_ms = sum(a.elapsed_time(b) for ev in marks for a, b in ev) / args.steps
    assert syrk_ms <= ms_local * 1.0001, (syrk_ms, ms_local)  # disjoint intervals of the step
    syrk_tflops = flops / (syrk_ms * 1e-3) / 1e12
    region_s = ms_local * args.steps * 1e-3
    # the burst peak for a region shorter than the sustained measurement's
    # seconds-long loop, the sustained one otherwise
    peak, peak_name = (bf16_burst, "bf16_tflops (burst)") if region_s < 2.0 else \
        (bf16_sust, "bf16_tflops_sustained")
    traffic, traffic_note = syrk_traffic(wl.name) if args.dtype == "bf16" and not args.batches \
        else (None, "no capture for this configuration")
    e2e = None if args.no_e2e else _e2e(h, wl, xs, d, args)

    res = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s",
        "tokens_per_s": round(job_throughput(n_tok, ms, ws), 1),
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic (seeded torch.randn, per-channel std log-uniform [0.1, 10], rounded to bf16)",
        "config": {"workload": wl.name, "d": d, "batches": len(xs), "tokens": n_tok,
                   "token_counts": "uniform integers [1, 2000], numpy default_rng(3)",
                   "damp_percent": wl.damp_percent, "flops_counted": "N*d*(d+1) (upper triangle)",
                   "l2": "inputs (%.2f GB) larger than L2; no flush" % (n_tok * d * 2 / 1e9),
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": round(syrk_tflops, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(syrk_tflops / peak, 4),
                     "traffic": traffic,
                     "traffic_note": traffic_note + "; algorithmic X bytes per launch %.4g"
                                     % (2.0 * n_tok * d / n_pairs),
                     "kernel": "syrk_%s_kernel" % args.dtype,
                     "syrk_ms_per_step": round(syrk_ms, 4), "launches_per_step": n_pairs,
                     "timing": "CUDA events around each flushing call inside the timed steps",
                     "peak_source": f"{peak_src} {peak_name}: timed region {region_s:.2f} s"},
        "e2e": e2e,
        "gpu_launches": kernels_timed,
        "gpu_launches_note": "the library's kernels in the timed steps (SYRK flushes, fold passes, "
                             "materializations), counted by hess_kernel_launches",
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_extra:
        res["extra"] = _extra(args, hbm, bf16_burst, bf16_sust)
    if rank == 0 and not args.no_cpu:
        res["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
    h.close()
    if rank == 0:
        print(json.dumps(res))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _flushing_calls(h, xs):
    """Indices of the add_batch calls that flush the queue in one step."""
    from gptq_qqq_calibration_gb300.hessian import hess_pending_batches
    h.reset()
    at = set()
    for i, X in enumerate(xs):
        h.add_batch(X)
        if hess_pending_batches(h.handle) == 0:
            at.add(i)
    h.flush()
    return at


def _time_syrk(h, xs, reps=3):
    import torch
    pairs = []
    for _ in range(reps):
        h.reset()
        for X in xs:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            h.add_batch(X)
            if not h._queued:
                b.record()
                pairs.append((a, b))
        if h._queued:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            h.flush()
            b.record()
            pairs.append((a, b))
    torch.cuda.synchronize()
    total = sum(a.elapsed_time(b) for a, b in pairs) * 1e-3 / reps
    return {"seconds": total, "launches": len(pairs) // reps}


def _e2e(h, wl, xs, d, args, chunk_bytes=64 << 20):
    """Same metric through the public API with host buffers: pinned-host ->
    device copies of every batch and the device -> host read of H inside the
    timed region.  The batches sit back to back in one pinned buffer and
    cross in chunks of about 64 MB on a copy stream; the compute stream
    waits for each chunk's event before handing its batches to the library,
    so later copies overlap the flushes of earlier batches."""
    import torch
    counts = [int(X.shape[0]) for X in xs]
    starts = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    total = int(starts[-1])
    # pinned at allocation, filled straight from the device copies: no
    # pageable staging buffers are made and freed before the timed steps
    host_buf = torch.empty((total, d), dtype=xs[0].dtype, pin_memory=True)
    for X, a in zip(xs, starts[:-1]):
        host_buf[int(a):int(a) + X.shape[0]].copy_(X)
    torch.cuda.synchronize()
    dev_buf = torch.empty((total, d), dtype=xs[0].dtype, device="cuda")
    views = [dev_buf[int(a):int(a) + n] for a, n in zip(starts[:-1], counts)]
    # chunks: consecutive batches up to ~chunk_bytes each
    row_bytes = d * xs[0].element_size()
    chunks, cur = [], []
    for b, n in enumerate(counts):
        cur.append(b)
        if sum(counts[i] for i in cur) * row_bytes >= chunk_bytes:
            chunks.append(cur)
            cur = []
    if cur:
        chunks.append(cur)
    events = [torch.cuda.Event() for _ in chunks]
    copy_s = torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    out = torch.empty((d, d), dtype=torch.float32, device="cuda")
    host_h = torch.empty((d, d), dtype=torch.float32, pin_memory=True)
    flops = algo_flops(wl.n_tokens, d)

    def step():
        h.reset()
        copy_s.wait_stream(comp)  # the previous step's kernels are done with dev_buf
        with torch.cuda.stream(copy_s):
            for ch, ev in zip(chunks, events):
                r0, r1 = int(starts[ch[0]]), int(starts[ch[-1] + 1])
                dev_buf[r0:r1].copy_(host_buf[r0:r1], non_blocking=True)
                ev.record(copy_s)
        for ch, ev in zip(chunks, events):
            comp.wait_event(ev)
            for b in ch:
                h.add_batch(views[b])
        h.materialize(wl.damp_percent, out=out, want_damp=False)
        host_h.copy_(out, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    # the host link's rate at this moment: the same bytes as one plain copy
    link = []
    for _ in range(2):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(copy_s)
        with torch.cuda.stream(copy_s):
            dev_buf.copy_(host_buf, non_blocking=True)
        b.record(copy_s)
        torch.cuda.synchronize()
        link.append(total * row_bytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    steps = max(3, args.steps // 2)
    # The steps run back to back, as a calibration loop streams its batches:
    # each step's copies wait for the previous step's kernels (copy_s waits
    # on comp), and one synchronisation ends the timed region.  An event
    # after each step's device -> host read gives the per-step device
    # intervals.
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ends[0].record(comp)
    for k in range(steps):
        step()
        ends[k + 1].record(comp)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    per = [ends[k].elapsed_time(ends[k + 1]) * 1e-3 for k in range(steps)]
    med = statistics.median(per)
    return {"value": round(flops / dt / 1e12, 3), "unit": "TFLOP/s",
            "median_step_ms": round(med * 1e3, 3), "median_tflops": round(flops / med / 1e12, 3),
            "stalled_steps": int(sum(t > 2 * med for t in per)),
            "longest_step_ms": round(max(per) * 1e3, 3),
            "h2d_link_gbs": round(max(link), 1),
            "h2d_bytes_per_step": int(total * row_bytes),
            "d2h_bytes_per_step": int(d * d * 4), "ms_per_step": round(dt * 1e3, 3),
            "h2d": f"one pinned buffer, {len(chunks)} chunks of ~{chunk_bytes >> 20} MB on a copy stream, "
                   "overlapped with the flushes; steps back to back, wall clock over all of them"}


# Secondary measurements, each with its own roofline; `--only NAME` runs one.
def _extra(args, hbm, bf16_burst, bf16_sust):
    out = {}
    for name, fn in EXTRAS.items():
        out[name] = fn(hbm, bf16_burst)
    return out


def _x_large_batch_gram(hbm, bf16_burst):
    import torch

    from gptq_qqq_calibration_gb300 import Hessian, LocalHessian
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS
    out = {}
    # large batches: 16 updates of 32768 tokens at d = 4096
    wl = WORKLOADS["d4096_16x32768"]
    xs = [wl.batch(b, device="cuda") for b in range(len(wl.token_counts))]
    h = Hessian(wl.d)
    Hm = torch.empty((wl.d, wl.d), dtype=torch.float32, device="cuda")

    def run():
        h.reset()
        for X in xs:
            h.add_batch(X)
        h.flush()
    run()
    torch.cuda.synchronize()
    kern = _time_syrk(h, xs, reps=3)
    fl = algo_flops(wl.n_tokens, wl.d)
    t = kern["seconds"]
    out["large_batch_gram"] = {
        "workload": wl.name, "tflops": round(fl / t / 1e12, 2), "ms": round(t * 1e3, 3),
        "tokens_per_s": round(wl.n_tokens / t, 1),
        "roofline": {"bound": "tensor", "peak": bf16_burst, "unit": "TFLOP/s",
                     "frac": round(fl / t / 1e12 / bf16_burst, 4), "peak_source": "bf16_tflops (burst)"}}
    h.close()
    return out["large_batch_gram"]


def _gpu_only(fn, reps, sleep_cycles=400_000_000):
    """Device time of the work `fn` enqueues, without the host's gaps: the
    stream is held by a sleep kernel while the host enqueues `reps` calls of
    fn behind it, and events bracket the enqueued work.  Returns (device ms,
    host ms) per call of fn."""
    import torch
    torch.cuda.synchronize()
    torch.cuda._sleep(sleep_cycles)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    t0 = time.perf_counter()
    for _ in range(reps):
        fn()
    host = time.perf_counter() - t0
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps, host * 1e3 / reps


def _flush_per_call(name, hbm, n_batches=60, reps=3):
    """The ragged stream flushed after every batch (no queue fusion): each
    call reads its X and read-modify-writes the upper triangle of H.  The
    kernels' rate is taken with the calls enqueued ahead of the device
    (_gpu_only); the wall-clock rate of the same calls through the Python
    binding is reported beside it."""
    import torch

    from gptq_qqq_calibration_gb300 import Hessian
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS
    wl = WORKLOADS[name].scaled(n_batches=n_batches)
    xs = [wl.batch(b, device="cuda") for b in range(len(wl.token_counts))]
    h = Hessian(wl.d, flush_tokens=1)

    def calls():
        for X in xs:
            h.add_batch(X)
    calls()
    dev_ms, _ = _gpu_only(calls, reps)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(reps):
        calls()
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) / reps
    h.sync()
    t = dev_ms * 1e-3
    d = wl.d
    tri = d * (d + 1) // 2
    alg_bytes = 2 * wl.n_tokens * d + len(xs) * tri * 4 * 2  # X once + fp32 upper-triangle RMW per call
    h.close()
    return {
        "workload": wl.name + f" (first {n_batches} batches, one flush per batch)",
        "us_per_call": round(t / len(xs) * 1e6, 2), "tflops": round(algo_flops(wl.n_tokens, d) / t / 1e12, 2),
        "wall_us_per_call": round(wall / len(xs) * 1e6, 2),
        "timing": "device time of the calls enqueued ahead of the GPU (events; a sleep kernel holds the "
                  "stream while the host enqueues); wall_us_per_call: the same calls timed on the host",
        "roofline": {"bound": "hbm", "achieved": round(alg_bytes / t / 1e9, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(alg_bytes / t / 1e9 / hbm, 4),
                     "bytes_counted": "2*n*d + 8*d(d+1)/2 per call (X once, fp32 upper-triangle read+write)",
                     "kernel": "syrk_bf16_kernel"}}


def _x_flush_per_call(hbm, bf16_burst):
    return _flush_per_call("d4096_ragged360_loguniform", hbm)


def _x_d2560_ragged360(hbm, bf16_burst, steps=10):
    """The width-2,560 ragged stream with 1 % outlier channels: the fused
    queue (reset, 360 adds, materialize per step; TFLOP/s and tokens/s
    against the burst bf16 peak) and the same stream flushed after every
    batch (GB/s against HBM)."""
    import torch

    from gptq_qqq_calibration_gb300 import Hessian
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS
    wl = WORKLOADS["d2560_ragged360_outlier"]
    xs = [wl.batch(b, device="cuda") for b in range(len(wl.token_counts))]
    h = Hessian(wl.d)
    out = torch.empty((wl.d, wl.d), dtype=torch.float32, device="cuda")

    def step():
        h.reset()
        for X in xs:
            h.add_batch(X)
        h.materialize(wl.damp_percent, out=out, want_damp=False)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    h.sync()
    t = e0.elapsed_time(e1) * 1e-3 / steps
    fl = algo_flops(wl.n_tokens, wl.d)
    h.close()
    return {
        "workload": wl.name, "tokens": wl.n_tokens, "ms_per_step": round(t * 1e3, 3),
        "tflops": round(fl / t / 1e12, 2), "tokens_per_s": round(wl.n_tokens / t, 1),
        "roofline": {"bound": "tensor", "peak": bf16_burst, "unit": "TFLOP/s",
                     "frac": round(fl / t / 1e12 / bf16_burst, 4),
                     "peak_source": "bf16_tflops (burst)", "timing": "whole step incl. materialize"},
        "flush_per_call": _flush_per_call(wl.name, hbm)}


def _x_d256_latency(hbm, bf16_burst, steps=200):
    """The single small layer (d = 256, 4 x 128 tokens): latency of one
    accumulate-and-materialize, on the device (events) and on the host
    (wall clock of the four add_batch calls and the materialize, which waits
    for the damping value)."""
    import torch

    from gptq_qqq_calibration_gb300 import Hessian
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS
    wl = WORKLOADS["d256_4x128"]
    xs = [wl.batch(b, device="cuda") for b in range(len(wl.token_counts))]
    h = Hessian(wl.d)
    out = torch.empty((wl.d, wl.d), dtype=torch.float32, device="cuda")

    def step(want_damp=True):
        h.reset()
        for X in xs:
            h.add_batch(X)
        return h.materialize(wl.damp_percent, out=out, want_damp=want_damp)[1]
    for _ in range(10):
        step()
    torch.cuda.synchronize()
    wall = []
    for _ in range(steps):
        t0 = time.perf_counter()
        step()
        wall.append(time.perf_counter() - t0)
    # 20 steps stay well inside the launch queue (each SYRK launch carries
    # its ~25 KB parameter block), so the host's enqueue time is its own
    # cost and not a wait for queue space behind the sleep kernel
    dev_ms, host_ms = _gpu_only(lambda: step(want_damp=False), 20)
    h.close()
    return {"workload": wl.name, "device_us_per_step": round(dev_ms * 1e3, 2),
            "wall_us_per_step": round(statistics.median(wall) * 1e6, 2),
            "host_enqueue_us_per_step": round(host_ms * 1e3, 2),
            "step": "reset, 4 x add_batch (128 tokens), materialize; wall: the damping value read back "
                    "(the call waits); device: the same work enqueued ahead of the GPU",
            "note": "latency-bound (X 262 KB, H 132 KB): no roofline grade"}


def _x_f32_input_ragged(hbm, bf16_burst):
    import torch

    from gptq_qqq_calibration_gb300 import Hessian, LocalHessian
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS
    out = {}
    # fp32-input path on the ragged d = 4096 stream (split-tf32 kernel)
    wl = WORKLOADS["d4096_ragged360_loguniform"]
    xs = [wl.batch(b, device="cuda", dtype=torch.float32) for b in range(len(wl.token_counts))]
    h = Hessian(wl.d)
    for _ in range(2):
        h.reset()
        for X in xs:
            h.add_batch(X)
        h.flush()
    torch.cuda.synchronize()
    kern = _time_syrk(h, xs, reps=2)
    fl = algo_flops(wl.n_tokens, wl.d)
    t = kern["seconds"]
    tf32_peak = bf16_burst / 2.0  # dense tf32 runs at half the bf16 rate
    # hi*hi, hi*lo and lo*hi: three tf32 MMAs of the algorithmic product each
    out["f32_input_ragged"] = {
        "workload": wl.name + " (fp32 input)", "tflops": round(fl / t / 1e12, 2), "ms": round(t * 1e3, 3),
        "tokens_per_s": round(wl.n_tokens / t, 1), "mma_per_8_tokens": F32_MMAS,
        "roofline": {"bound": "tensor", "achieved_tf32": round(F32_MMAS * fl / t / 1e12, 2), "peak": tf32_peak,
                     "unit": "TFLOP/s", "frac": round(F32_MMAS * fl / t / 1e12 / tf32_peak, 4),
                     "peak_source": "bf16_tflops (burst) x 1/2 (nominal tf32:bf16 ratio)"}}
    h.close()
    return out["f32_input_ragged"]


def _x_imatrix(hbm, bf16_burst):
    import torch

    from gptq_qqq_calibration_gb300 import Hessian, LocalHessian
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS
    out = {}
    # imatrix column sums of squares over the same local workload's batches
    wl = WORKLOADS["local_d4096_8x32768"]
    xs = [wl.batch(b, device="cuda") for b in range(len(wl.token_counts))]
    from gptq_qqq_calibration_gb300 import IMatrix
    im = IMatrix(wl.d)
    for X in xs:
        im.add_batch(X)
    torch.cuda.synchronize()
    evs = []
    for _ in range(3):
        for X in xs:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            im.add_batch(X)
            b.record()
            evs.append((a, b))
    torch.cuda.synchronize()
    per = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e-3
    nbytes = xs[0].numel() * 2
    out["imatrix"] = {
        "workload": "column sums of squares, 32768 x 4096 bf16 per update", "us_per_update": round(per * 1e6, 2),
        "roofline": {"bound": "hbm", "achieved": round(nbytes / per / 1e9, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(nbytes / per / 1e9 / hbm, 4), "kernel": "colsumsq_kernel"}}
    im.close()
    return out["imatrix"]


def _x_local_hessian(hbm, bf16_burst):
    import torch

    from gptq_qqq_calibration_gb300 import Hessian, LocalHessian
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS
    out = {}
    # local_hessian: 8 updates of 32768 tokens at d = 4096
    wl = WORKLOADS["local_d4096_8x32768"]
    xs = [wl.batch(b, device="cuda") for b in range(len(wl.token_counts))]
    lh = LocalHessian(wl.d)
    for X in xs:
        lh.add_batch(X)
    torch.cuda.synchronize()
    evs = []
    for _ in range(3):
        for X in xs:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            lh.add_batch(X)
            b.record()
            evs.append((a, b))
    torch.cuda.synchronize()
    per = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e-3
    nbytes = xs[0].numel() * 2
    out["local_hessian"] = {
        "workload": wl.name, "us_per_update": round(per * 1e6, 2),
        "roofline": {"bound": "hbm", "achieved": round(nbytes / per / 1e9, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(nbytes / per / 1e9 / hbm, 4),
                     "bytes_per_update": nbytes, "kernel": "local_gram_kernel"}}
    lh.close()
    return out["local_hessian"]


# fp32 FMA lanes of GB300: 152 SMs x 128 lanes x 2 flops at the 2,070 MHz
# maximum SM clock.
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def _quantize_pass(d=4096, rows=4096, reps=3):
    """The quantization pass on the Hessian of the first 24 batches of the
    d = 4,096 ragged stream: prepare (dead columns, damping, the factor U)
    and the 4-bit grouped quantization of a synthetic [4096, 4096] weight."""
    import torch

    from gptq_qqq_calibration_gb300 import GPTQ, Hessian
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS, make_weight
    wl = WORKLOADS["d4096_ragged360_loguniform"].scaled(n_batches=24)
    h = Hessian(d)
    for b in range(len(wl.token_counts)):
        h.add_batch(wl.batch(b, device="cuda"))
    W = make_weight(rows, d, 4096, device="cuda")
    q = GPTQ(d, rows)
    q.prepare(h, wl.damp_percent)
    q.quantize(W, 128, want_loss=False)
    torch.cuda.synchronize()
    tp, tq = [], []
    for _ in range(reps):
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record()
        q.prepare(h, wl.damp_percent)
        b.record()
        q.quantize(W, 128, want_loss=False)
        c.record()
        torch.cuda.synchronize()
        tp.append(a.elapsed_time(b) * 1e-3)
        tq.append(b.elapsed_time(c) * 1e-3)
    tp, tq = statistics.median(tp), statistics.median(tq)
    # algorithmic flops: Cholesky d^3/3, triangular inverse d^3/3, and the
    # error propagation rows * d(d-1)/2 multiply-adds
    f_prep = 2.0 * d ** 3 / 3.0
    f_quant = float(rows) * d * (d - 1)
    q.close()
    h.close()
    return {
        "workload": f"H of {wl.name} (first 24 batches), W [{rows}, {d}] N(0, 0.02^2), group 128, damp 0.01",
        "prepare_ms": round(tp * 1e3, 3), "quantize_ms": round(tq * 1e3, 3),
        "total_ms": round((tp + tq) * 1e3, 3),
        "roofline": {"bound": "alu", "unit": "TFLOP/s", "peak": round(FP32_ALU_TFLOPS, 1),
                     "achieved": round((f_prep + f_quant) / (tp + tq) / 1e12, 2),
                     "frac": round((f_prep + f_quant) / (tp + tq) / 1e12 / FP32_ALU_TFLOPS, 4),
                     "peak_source": "152 SMs x 128 fp32 lanes x 2 x 2.07 GHz",
                     "flops_counted": "2 d^3 / 3 (Cholesky + triangular inverse) + rows d (d-1)",
                     "note": "fp32 work; the large GEMMs run as split tf32 (3 MMAs per product) on the "
                             "tensor cores, the diagonal blocks and step 5's column chain on CUDA cores"}}


def _x_merge(hbm, bf16_burst, d=4096, reps=5):
    """hess_merge at d = 4,096: dst += src over the (hi, lo) fp32 upper-
    triangle tiles (69 MB each; 2 reads and 1 write per element)."""
    import torch

    from gptq_qqq_calibration_gb300 import Hessian
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS
    wl = WORKLOADS["d4096_ragged360_loguniform"].scaled(n_batches=2)
    a, b = Hessian(d), Hessian(d)
    for k in range(2):
        (a if k == 0 else b).add_batch(wl.batch(k, device="cuda"))
    a.flush()
    b.flush()
    a.merge(b)
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        a.merge(b)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3)
    t = statistics.median(ts)
    T = (d + 127) // 128
    nbytes = 3 * T * (T + 1) // 2 * 128 * 128 * 8  # 8 bytes per (hi, lo) element
    a.close()
    b.close()
    return {"workload": f"hess_merge at d={d} ((hi, lo) upper-triangle tiles)", "us_per_merge": round(t * 1e6, 2),
            "roofline": {"bound": "hbm", "achieved": round(nbytes / t / 1e9, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(nbytes / t / 1e9 / hbm, 4), "bytes_per_merge": nbytes,
                         "kernel": "add_pairs_kernel"}}


EXTRAS = {
    "d256_latency": _x_d256_latency,
    "d2560_ragged360": _x_d2560_ragged360,
    "large_batch_gram": _x_large_batch_gram,
    "flush_per_call": _x_flush_per_call,
    "f32_input_ragged": _x_f32_input_ragged,
    "imatrix": _x_imatrix,
    "local_hessian": _x_local_hessian,
    "merge": _x_merge,
    "quantize_pass": lambda hbm, bf16_burst: _quantize_pass(),
}


# --------------------------------------------------------------- reference


def cpu_baseline(wl, budget_s=15.0):
    """The float64 oracle on the host cores, over as many leading batches of
    the workload as fit the time budget."""
    import torch

    from oracle import GramOracle
    from gptq_qqq_calibration_gb300.synthetic import make_batch
    o = GramOracle(wl.d)
    t_used, n_used, nb = 0.0, 0, 0
    for b, n in enumerate(wl.token_counts):
        X = make_batch(int(n), wl.d, wl.batch_seed(b), profile=wl.profile, profile_seed=wl.seed,
                       dtype=torch.bfloat16).to(torch.float64).numpy()
        t0 = time.perf_counter()
        o.add_batch(X)
        t_used += time.perf_counter() - t0
        n_used += int(n)
        nb += 1
        if t_used >= budget_s:
            break
    t0 = time.perf_counter()
    o.materialize(wl.damp_percent)
    t_used += time.perf_counter() - t0
    return {"value": round(algo_flops(n_used, wl.d) / t_used / 1e12, 5), "unit": "TFLOP/s",
            "tokens_per_s": round(n_used / t_used, 1), "cores": _blas_threads(), "kind": "oracle",
            "host_cpus": os.cpu_count(),
            "sample": f"first {nb} of {len(wl.token_counts)} batches ({n_used} tokens) of {wl.name}, "
                      f"float64 NumPy X^T X + materialize, {t_used:.1f} s",
            "one_thread": _oracle_one_thread()}


def _blas_threads():
    """BLAS threads of the oracle: the count set in the environment before
    numpy loaded (threadpoolctl's report where it is installed)."""
    try:
        from threadpoolctl import threadpool_info
        return max(i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas")
    except Exception:
        return int(os.environ["OPENBLAS_NUM_THREADS"])


def _oracle_probe(name):
    """One oracle timing, in this process (whose BLAS thread count the parent
    fixed): `d256` is the small layer's 4 x 128 tokens plus materialize;
    `d4096_update` is one 32,768-token update at d = 4,096."""
    import torch

    from oracle import GramOracle
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS, make_batch
    wl = WORKLOADS["d256_4x128" if name == "d256" else "d4096_16x32768"]
    nb = len(wl.token_counts) if name == "d256" else 1
    xs = [make_batch(int(n), wl.d, wl.batch_seed(b), profile=wl.profile, profile_seed=wl.seed,
                     dtype=torch.bfloat16).to(torch.float64).numpy()
          for b, n in enumerate(wl.token_counts[:nb])]
    reps = 20 if name == "d256" else 1
    t0 = time.perf_counter()
    for _ in range(reps):
        o = GramOracle(wl.d)
        for X in xs:
            o.add_batch(X)
        o.materialize(wl.damp_percent)
    dt = (time.perf_counter() - t0) / reps
    n_tok = sum(x.shape[0] for x in xs)
    return {"seconds": round(dt, 6), "tokens_per_s": round(n_tok / dt, 1),
            "tflops": round(algo_flops(n_tok, wl.d) / dt / 1e12, 5), "threads": _blas_threads(),
            "sample": f"{nb} batch(es), {n_tok} tokens at d={wl.d}, with materialize"}


def _oracle_one_thread():
    """The oracle with one BLAS thread (a child process, so that the thread
    count is fixed before numpy loads) on the small layer and on one
    32,768-token update at d = 4,096."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    out = {}
    for name in ("d256", "d4096_update"):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-probe", name],
                           env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, timeout=600)
        try:
            out[name] = json.loads(r.stdout.decode().strip().splitlines()[-1])
        except Exception:
            out[name] = {"error": r.stderr.decode(errors="replace")[-300:]}
    return out


def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch

    from oracle import GramOracle
    from gptq_qqq_calibration_gb300.synthetic import WORKLOADS, make_batch
    wl = WORKLOADS[args.workload]
    per_step = max(1, args.ref_batches)
    xs = [make_batch(int(n), wl.d, wl.batch_seed(b), profile=wl.profile, profile_seed=wl.seed,
                     dtype=torch.bfloat16).to(torch.float64).numpy()
          for b, n in enumerate(wl.token_counts[:per_step])]
    n_tok = sum(x.shape[0] for x in xs)

    def step():
        o = GramOracle(wl.d)
        for X in xs:
            o.add_batch(X)
        o.materialize(wl.damp_percent)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    v = algo_flops(n_tok, wl.d) / dt / 1e12
    cores = _blas_threads()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "d": wl.d, "sample_batches": per_step,
                                        "sample_tokens": n_tok},
        "cpu_baseline": {"value": round(v, 5), "unit": "TFLOP/s", "kind": "oracle", "cores": cores,
                         "sample": f"first {per_step} batches ({n_tok} tokens) of {wl.name} per step"},
        "e2e": {"value": round(v, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="d4096_ragged360_loguniform")
    ap.add_argument("--batches", type=int, default=0, help="use only the first K batches")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f32"], help="input element type")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-batches", type=int, default=2)
    ap.add_argument("--only", default=None,
                    help="run one secondary measurement (" + ", ".join(EXTRAS) + ") and print its JSON")
    ap.add_argument("--quantize-only", action="store_true", help="same as --only quantize_pass")
    ap.add_argument("--oracle-probe", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_probe:
        print(json.dumps(_oracle_probe(args.oracle_probe)))
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        from gptq_qqq_calibration_gb300 import build as b
        b.build()
        only = "quantize_pass" if args.quantize_only else args.only
        if only:
            if only not in EXTRAS:
                raise SystemExit(f"--only: unknown measurement {only!r}; one of {sorted(EXTRAS)}")
            hbm, bf16_burst, _, _ = peaks()
            print(json.dumps({only: EXTRAS[only](hbm, bf16_burst)}))
        else:
            run_ours(args)


if __name__ == "__main__":
    main()

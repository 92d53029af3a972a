#!/usr/bin/env python
"""Benchmark of the absorbed-MLA verify-attention call on GB300.

One step = one verify call (split kernel + slice merge) over one synthetic
workload; default workload: 1 stream, 9 draft-tree queries x 64 heads over a
65536-token latent prefix (576-wide bf16 cache rows).  Prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed calls, then exactly K calls bracketed by a barrier and
torch.cuda.synchronize() on both sides, timed with CUDA events on the stream
the kernels run on.  The cache is rotated over enough copies that the working
set exceeds L2, so every call reads its cache cold from HBM.  SM clocks and
throttle reasons are sampled with nvidia-smi during the timed region.

--impl reference times the fp64 CPU oracle (the only other implementation of
this computation) on the host cores, on a bounded sample of the same workload.
With N > 1 (torchrun), every rank runs its own replica of the workload (the
path has no cross-GPU exchange; "replicas only"); the reported time is the
maximum over ranks.
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
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_verify_attention_gb300 import inputs as I  # noqa: E402

METRIC = "verify-attn us/call (q_len=9, prefix 65536)"
UNIT = "us/call"
PAGES_US = {"tree9_p65536": 19722.2}   # best sm_120 time the pages report for this workload


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="tree9_p65536", choices=sorted(I.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--configs", choices=["all", "none"], default="all",
                    help="also time every workload (the per-config table in the JSON line)")
    ap.add_argument("--config-windows", type=int, default=5,
                    help="windows of back-to-back calls per workload in that table (median)")
    ap.add_argument("--page-size", type=int, default=0,
                    help="time the paged-cache entry point with pages of this many keys "
                         "(a multiple of 64, pages in seeded random order); 0 = contiguous cache")
    return ap.parse_args()


# ----------------------------------------------------------------------- helpers

def work_of(case):
    """Algorithmic FLOPs and cache bytes of one call (cache read once)."""
    rows = case.q * case.H
    keys = int(np.sum(case.seq_lens.astype(np.int64)))
    flops = 2.0 * rows * keys * (512 + 64 + 512)
    cache_bytes = keys * 576 * 2
    return flops, cache_bytes


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            m = json.load(fh)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _code_tokens(text):
    """Source text without comments and with whitespace collapsed: edits to
    comments alone leave the hash (and the recorded traffic) valid."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_src_hash(csrc=None):
    """sha256/16 of the CUDA sources' code (comments and layout ignored)."""
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "mla_verify_attention_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn), encoding="utf-8") as fh:
            h.update(fn.encode() + _code_tokens(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes (read + write) per split-kernel launch from the committed ncu
    summary, or None when the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic_%s.json" % workload)
    try:
        with open(path) as fh:
            t = json.load(fh)
    except Exception:
        return None
    if t.get("kernel_src_sha256_16") != kernel_src_hash():
        return None
    return t.get("verify_split_kernel", {}).get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks, power and throttle reasons (every
    20 ms) for the whole run; summary(window) reports the samples that fall in
    a host wall-clock window."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _rows(self):
        import datetime
        rows = []
        try:
            with open(self.path) as fh:
                for line in fh:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 10:
                        try:
                            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        except ValueError:
                            ts = None
                        rows.append((ts, parts[1:]))
        except OSError:
            pass
        return rows

    def summary(self, window=None):
        """Samples whose timestamps fall inside `window` (host wall-clock
        seconds), widened by one sampling period on each side; all samples so
        far if none do."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        time.sleep(0.05)          # let the sample after the window be written
        all_rows = self._rows()
        inside = [r for ts, r in all_rows
                  if window and ts is not None and window[0] - 0.02 <= ts <= window[1] + 0.02]
        in_window = bool(inside)
        rows = inside if inside else [r for _, r in all_rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "in_timed_window": in_window,
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        try:
            os.unlink(self.path)
        except OSError:
            pass


def physical_gpu_index(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return int(ids[local_rank])
    return local_rank


def oracle_sample(case, budget_s, steps=1):
    """Time the oracle on whole calls if they fit the budget, else on a row
    sample; returns (us per full call, cores, sample description)."""
    import oracle
    rows = case.B * case.q * case.H
    cores = os.cpu_count() or 1
    n0 = min(rows, max(8, cores))
    t0 = time.perf_counter()
    oracle.case_reference(case, nthreads=cores, rows=(0, n0))
    per_row = (time.perf_counter() - t0) / n0
    n = rows if per_row * rows <= budget_s else max(n0, int(budget_s / per_row))
    n = min(rows, n)
    times = []
    for s in range(steps):
        start = (s * n) % rows if n < rows else 0
        cnt = min(n, rows - start)
        t0 = time.perf_counter()
        oracle.case_reference(case, nthreads=cores, rows=(start, cnt))
        times.append((time.perf_counter() - t0) * rows / cnt)
    us = statistics.median(times) * 1e6
    what = ("whole call (%d query rows)" % rows if n >= rows else
            "%d of %d query rows per step, scaled to the whole call" % (n, rows))
    return us, cores, what, times


def oracle_single_thread(case, budget_s):
    """The oracle on one host thread, on as many query rows as fit the budget;
    returns (us per full call, rows timed)."""
    import oracle
    rows = case.B * case.q * case.H
    t0 = time.perf_counter()
    oracle.case_reference(case, nthreads=1, rows=(0, 1))
    per_row = time.perf_counter() - t0
    n = max(1, min(rows, int(budget_s / max(per_row, 1e-9))))
    t0 = time.perf_counter()
    oracle.case_reference(case, nthreads=1, rows=(0, n))
    return (time.perf_counter() - t0) * rows / n * 1e6, n


# ----------------------------------------------------------------------- arms

def run_reference(args, rank):
    if rank != 0:
        return
    case = I.make_case(I.WORKLOADS[args.workload], pad="normal")
    # each step is a bounded sample so that the whole run ends within minutes
    budget = min(args.cpu_budget_s, 120.0 / max(1, args.steps + 1))
    for _ in range(max(0, min(args.warmup, 1))):
        oracle_sample(case, budget / 4)
    us, cores, what, times = oracle_sample(case, budget, steps=args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(args.workload, case),
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": what},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(value, world, device=None):
    """The largest of the ranks' values, returned on every rank (replicas run in
    lock step, so the job's time per call is its slowest rank's)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as tdist
    v = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(v, op=tdist.ReduceOp.MAX)
    return float(v.item())


def case_seed_for_pages(case):
    """Seed of the page order of a bench case (fixed per workload shape)."""
    return 0x5041 + int(case.Smax)


def config_of(name, case, extra=None):
    w = I.WORKLOADS[name]
    c = {"workload": name, "B": case.B, "q_len": case.q, "H": case.H, "Dl": 512, "Dr": 64,
         "prefix": w.prefix if not isinstance(w.prefix, tuple) else list(w.prefix),
         "seq_lens": [int(s) for s in case.seq_lens], "Smax": case.Smax,
         "tree": "chain" if w.tree == "chain" else
                 "random, depth<=%d%s" % (w.max_depth, "" if w.max_children is None
                                          else ", branching<=%d" % w.max_children),
         "inputs": "bf16 N(0,1) from seed %#x" % w.seed, "scale": "1/sqrt(192)"}
    if extra:
        c.update(extra)
    return c


class Runner:
    """One workload's inputs on the device and its verify call through the C ABI.

    The cache is rotated over enough copies that the working set exceeds
    twice the L2, so every call reads its cache from HBM."""

    def __init__(self, mva, name, dev, page_size=0):
        import torch
        self.mva, self.name, self.dev, self.page_size = mva, name, dev, page_size
        self.case = case = I.make_case(I.WORKLOADS[name], pad="normal")

        def t(a, dt):
            return torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(dev)

        self.t = t
        self.q_nope = t(case.q_nope.view(np.int16), torch.bfloat16)
        self.q_rope = t(case.q_rope.view(np.int16), torch.bfloat16)
        self.seq = t(case.seq_lens, torch.int32)
        self.mask = t(case.mask.view(np.int32), torch.int32)
        self.paged = page_size > 0
        if self.paged:
            self.pool, self.table = I.to_paged(case, page_size, seed=case_seed_for_pages(case),
                                               extra_pages=0)
            kv0 = t(self.pool.view(np.int16), torch.bfloat16)
            self.table_d = t(self.table, torch.int32)
        else:
            kv0 = t(case.kv.view(np.int16), torch.bfloat16)
        self.kv0 = kv0
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.kv_bytes = kv0.numel() * 2
        self.copies = max(2, math.ceil(2.0 * self.l2 / self.kv_bytes) + 1)
        self.kvs = [kv0] + [kv0.clone() for _ in range(self.copies - 1)]
        B, q, H, Smax = case.B, case.q, case.H, case.Smax
        if self.paged:
            Smax = self.table.shape[1] * page_size      # the paged call's key bound
        self.B, self.q, self.H, self.Smax = B, q, H, Smax
        self.out = torch.empty((B, q, H, 512), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B, q, H), dtype=torch.float32, device=dev)
        if self.paged:
            self.need = mva.paged_workspace_size(B, q, H, self.table.shape[1], page_size)
        else:
            self.need = mva.workspace_size(B, q, H, Smax)
        self.ws = torch.empty(max(self.need, 1), dtype=torch.uint8, device=dev)
        self.n_rt, self.nsplit, self.chunk = mva.plan(B, q, H, Smax)
        # split kernel; the slice merge when the keys are split; for pages that
        # are not whole 64-key tiles the copy into a contiguous cache; the
        # library's planner kernel for split calls with 2..32 streams (the
        # bench never forces the slice count)
        copied = self.paged and page_size % 64 != 0
        planned = 2 <= B <= 32 and self.nsplit > 1
        self.launches_per_call = (1 + (1 if self.nsplit > 1 else 0) + (1 if copied else 0)
                                  + (1 if planned else 0))
        self.stream = torch.cuda.current_stream(dev)
        self.sh = int(self.stream.cuda_stream)
        self.flops, self.cache_bytes = work_of(case)

    def call(self, i, stream_handle=None):
        mva, c = self.mva, self.case
        sh = self.sh if stream_handle is None else stream_handle
        if self.paged:
            st = mva.load_library().mla_verify_attn_paged(
                self.q_nope.data_ptr(), self.q_rope.data_ptr(), self.kvs[i % self.copies].data_ptr(),
                self.kv0.shape[0], self.table_d.data_ptr(), self.table_d.shape[1], self.page_size,
                self.seq.data_ptr(), self.mask.data_ptr(), self.B, self.q, self.H, float(c.scale),
                self.out.data_ptr(), self.lse.data_ptr(), self.ws.data_ptr(), self.ws.numel(), sh)
        else:
            st = mva.verify_attn_raw(self.q_nope.data_ptr(), self.q_rope.data_ptr(),
                                     self.kvs[i % self.copies].data_ptr(), self.seq.data_ptr(),
                                     self.mask.data_ptr(), self.B, self.q, self.H, self.Smax,
                                     float(c.scale), self.out.data_ptr(), self.lse.data_ptr(),
                                     self.ws.data_ptr(), self.ws.numel(), sh)
        if st != 0:
            raise mva.MLAError(st)

    def check_status(self, what):
        st = self.mva.last_device_error()
        if st != 0:
            raise self.mva.MLAError(st, what)

    def time_calls(self, n, first=0):
        """us per call of n back-to-back calls (CUDA events on the call stream)."""
        import torch
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for i in range(n):
            self.call(first + i)
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1) * 1e3 / n

    def split_kernel_us(self, n):
        """The split kernel's own duration: the library records a pair of events
        around each of its launches (the merge then starts after it ends)."""
        import torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:
            a.record(self.stream)
            b.record(self.stream)
        torch.cuda.synchronize(self.dev)
        try:
            for i in range(n):
                self.mva.set_timing_events(*evs[i])
                self.call(i)
        finally:
            self.mva.set_timing_events()
        torch.cuda.synchronize(self.dev)
        return statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)

    def roofline(self, split_us, call_us):
        hbm_gbs, bf16_tf, peak_src = measured_peaks()
        t_tensor = self.flops / (bf16_tf * 1e12)
        t_hbm = self.cache_bytes / (hbm_gbs * 1e9)
        tensor = t_tensor >= t_hbm
        tflops = self.flops / (split_us * 1e-6) / 1e12
        gbs = self.cache_bytes / (split_us * 1e-6) / 1e9
        r = {"bound": "tensor" if tensor else "hbm",
             "achieved": tflops if tensor else gbs,
             "peak": bf16_tf if tensor else hbm_gbs,
             "unit": "TFLOP/s" if tensor else "GB/s"}
        r["frac"] = r["achieved"] / r["peak"]
        r["effective_tflops"] = tflops
        r["effective_gbs"] = gbs
        r["roofline_us"] = max(t_tensor, t_hbm) * 1e6
        r["peak_source"] = ("%s (MEASURED_PEAKS.json burst)" % peak_src if peak_src == "measured"
                            else "fallback")
        r["kernel_us"] = split_us
        r["call_us"] = call_us
        r["call_frac"] = (self.flops / (call_us * 1e-6) / 1e12 / bf16_tf if tensor else
                          self.cache_bytes / (call_us * 1e-6) / 1e9 / hbm_gbs)
        r["call_tflops"] = self.flops / (call_us * 1e-6) / 1e12
        r["call_gbs"] = self.cache_bytes / (call_us * 1e-6) / 1e9
        return r

    def release(self):
        self.kvs = None
        self.kv0 = None


def config_report(mva, dev, name, args, sampler):
    """One entry of the per-workload table: median us/call over several windows
    of back-to-back calls (each window >= 50 ms, so that clock samples fall
    inside), the split kernel's own median duration, the roofline, and the
    oracle timed on the host cores."""
    import torch
    r = Runner(mva, name, dev)
    for i in range(max(3, args.warmup)):
        r.call(i)
    torch.cuda.synchronize(dev)
    r.check_status("warm-up " + name)
    probe = r.time_calls(max(3, min(50, args.steps)))
    per_window = max(args.steps, int(math.ceil(50e3 / max(probe, 1.0))))
    windows = []
    t0 = time.time()
    for w in range(args.config_windows):
        windows.append(r.time_calls(per_window, first=w * per_window))
    t1 = time.time()
    r.check_status("timed windows " + name)
    call_us = statistics.median(windows)
    split_us = r.split_kernel_us(min(200, per_window))
    r.check_status("split timing " + name)
    entry = {
        "B": r.B, "q_len": r.q, "H": r.H, "Smax": r.Smax,
        "seq_lens": [int(x) for x in r.case.seq_lens],
        "plan": {"row_tiles": r.n_rt, "nsplit": r.nsplit, "chunk_tiles": r.chunk},
        "launches_per_call": r.launches_per_call,
        "us_per_call": call_us, "us_per_call_windows": windows, "calls_per_window": per_window,
        "split_kernel_us": split_us,
        "flops_per_call": r.flops, "cache_bytes_per_call": r.cache_bytes,
        "roofline": r.roofline(split_us, call_us),
        "clocks": sampler.summary(window=(t0, t1)),
    }
    r.release()
    if not args.no_cpu_baseline:
        c_us, cores, what, _ = oracle_sample(r.case, args.cpu_budget_s)
        s_us, s_rows = oracle_single_thread(r.case, min(5.0, args.cpu_budget_s / 4))
        entry["oracle"] = {"all_cores_us_per_call": c_us, "cores": cores, "sample": what,
                           "single_thread_us_per_call": s_us,
                           "single_thread_sample": "%d query rows on one thread, scaled to the "
                                                   "whole call" % s_rows}
    torch.cuda.empty_cache()
    return entry


def run_ours(args, rank, world, local_rank):
    import torch
    import mla_verify_attention_gb300 as mva
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    mva.load_library()
    sampler = ClockSampler(physical_gpu_index(local_rank))
    sampler.start()

    # ---- every workload (rank 0, one GPU): the per-config table.
    configs = None
    if rank == 0 and world == 1 and args.configs == "all":
        configs = {}
        for name in I.WORKLOADS:
            configs[name] = config_report(mva, dev, name, args, sampler)

    # ---- the headline workload: W warm-up calls, then exactly K timed calls.
    r = Runner(mva, args.workload, dev, args.page_size)
    case = r.case
    dist = world > 1
    if dist:
        import torch.distributed as tdist
    for i in range(max(3, args.warmup)):
        r.call(i)
    torch.cuda.synchronize(dev)
    r.check_status("warm-up")
    stream = r.stream
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if dist:
        tdist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    ev0.record(stream)
    for i in range(args.steps):
        r.call(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if dist:
        tdist.barrier()
    ms = ev0.elapsed_time(ev1)
    us_call = max_over_ranks(ms * 1e3 / args.steps, world, dev)
    r.check_status("timed region")
    clocks = sampler.summary(window=(t_wall0, t_wall1))

    # ---- the dominant kernel's own duration (a second loop over the same
    # rotating inputs; the merge then starts after the split kernel ends).
    split_us = r.split_kernel_us(min(args.steps, 200))

    # ---- the same calls replayed from a CUDA graph (one call per cache copy
    # captured once): what a decode loop that captures its steps sees.  Context
    # only; `value` above is stream-launched calls.
    graph = torch.cuda.CUDAGraph()
    gstream = torch.cuda.Stream(dev)
    gstream.wait_stream(stream)
    ncap = min(r.copies, 64)
    with torch.cuda.stream(gstream):
        with torch.cuda.graph(graph, stream=gstream):
            for i in range(ncap):
                r.call(i, int(gstream.cuda_stream))
    torch.cuda.synchronize(dev)
    reps = max(1, min(args.steps, 500) // ncap)
    graph.replay()
    torch.cuda.synchronize(dev)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(reps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize(dev)
    graph_us = g0.elapsed_time(g1) * 1e3 / (reps * ncap)
    r.check_status("graph replay")
    del graph

    # ---- the same call on one cache copy, which stays in L2 between calls
    # (context: `value` rotates copies so that every call reads HBM).
    n_hot = max(1, min(args.steps, 500))
    for _ in range(3):
        r.call(0)
    h0 = torch.cuda.Event(enable_timing=True)
    h1 = torch.cuda.Event(enable_timing=True)
    h0.record(stream)
    for _ in range(n_hot):
        r.call(0)
    h1.record(stream)
    torch.cuda.synchronize(dev)
    hot_us = h0.elapsed_time(h1) * 1e3 / n_hot
    r.check_status("hot-L2 calls")

    # ---- end to end through the public API, from pinned host buffers
    paged = r.paged
    host_in = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in
               (case.q_nope.view(np.int16), case.q_rope.view(np.int16),
                (r.pool if paged else case.kv).view(np.int16), case.seq_lens, case.mask.view(np.int32))
               + ((r.table,) if paged else ())]
    B, q, H = r.B, r.q, r.H
    h_out = torch.empty((B, q, H, 512), dtype=torch.float32).pin_memory()
    h_lse = torch.empty((B, q, H), dtype=torch.float32).pin_memory()
    # Two device copies of the inputs: step i+1's inputs are copied on a second
    # stream while step i computes (each copy waits until the step that last
    # read its buffers is done); the result of each step is read back on the
    # compute stream right after it.
    d_sets = [[torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host_in] for _ in range(2)]
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = h_out.numel() * 4 + h_lse.numel() * 4
    ws = r.ws if r.need > 0 else None
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def e2e_copy(i):
        k = i % 2
        copy_stream.wait_event(consumed[k])
        with torch.cuda.stream(copy_stream):
            for d, h in zip(d_sets[k], host_in):
                d.copy_(h, non_blocking=True)
        copied[k].record(copy_stream)

    def e2e_compute(i):
        d_in = d_sets[i % 2]
        stream.wait_event(copied[i % 2])
        if paged:
            o, l = mva.verify_attn_paged(d_in[0].view(torch.bfloat16), d_in[1].view(torch.bfloat16),
                                         d_in[2].view(torch.bfloat16), d_in[5], args.page_size,
                                         d_in[3], d_in[4], float(case.scale), out=r.out, lse=r.lse,
                                         workspace=ws)
        else:
            o, l = mva.verify_attn(d_in[0].view(torch.bfloat16), d_in[1].view(torch.bfloat16),
                                   d_in[2].view(torch.bfloat16), d_in[3], d_in[4], float(case.scale),
                                   out=r.out, lse=r.lse, workspace=ws)
        consumed[i % 2].record(stream)
        h_out.copy_(o, non_blocking=True)
        h_lse.copy_(l, non_blocking=True)

    def e2e_steps(n):
        for k in range(2):
            consumed[k].record(stream)
        e2e_copy(0)
        for i in range(n):
            if i + 1 < n:
                e2e_copy(i + 1)
            e2e_compute(i)

    e2e_steps(3)
    torch.cuda.synchronize(dev)
    n_e2e = max(1, args.e2e_steps)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps(n_e2e)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_us = e0.elapsed_time(e1) * 1e3 / n_e2e
    sampler.stop()

    roof = r.roofline(split_us, us_call)
    roof["traffic"] = recorded_traffic(args.workload)
    roof["kernel"] = "verify_split_kernel (1 of %d launches per call)" % r.launches_per_call
    roof["algorithmic"] = {"flops_per_launch": r.flops, "cache_bytes_per_launch": r.cache_bytes}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if configs and args.workload in configs and "oracle" in configs[args.workload]:
            o = configs[args.workload]["oracle"]
            c_us, cores, what, s_us = (o["all_cores_us_per_call"], o["cores"], o["sample"],
                                       o["single_thread_us_per_call"])
            s_what = o["single_thread_sample"]
        else:
            c_us, cores, what, _ = oracle_sample(case, args.cpu_budget_s)
            s_us, s_rows = oracle_single_thread(case, min(5.0, args.cpu_budget_s / 4))
            s_what = "%d query rows on one thread, scaled to the whole call" % s_rows
        cpu = {"value": c_us, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": what,
               "single_thread": {"value": s_us, "unit": UNIT, "sample": s_what}}

    if rank == 0:
        ref = PAGES_US.get(args.workload)
        line = {
            "metric": METRIC if args.workload == "tree9_p65536" else
            "verify-attn us/call (%s)" % args.workload,
            "value": us_call, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": us_call / 1e3,
            "higher_is_better": False, "scaling": "weak",
            "vs_baseline": (us_call / ref) if ref else None,
            "dtype": "bf16", "data": "synthetic",
            "config": config_of(args.workload, case, {
                "l2": "inputs larger than L2: %d rotating cache copies (%.0f MB > %.0f MB L2)" % (
                    r.copies, r.copies * r.kv_bytes / 1e6, r.l2 / 1e6),
                "plan": {"row_tiles": r.n_rt, "nsplit": r.nsplit, "chunk_tiles": r.chunk},
                "cache": ("paged: %d-key pages in seeded random order" % args.page_size) if paged
                else "contiguous [B, Smax, 576]",
                "parallelism": "replicas" if world > 1 else "single GPU",
                "vs_baseline_ref": ("pages' best sm_120 time for this workload: %.1f us "
                                    "(RTX PRO 6000, fp32), context only" % ref) if ref else None}),
            "roofline": roof,
            "cpu_baseline": cpu,
            "configs": configs,
            "graph": {"us_per_call": graph_us, "calls": reps * ncap,
                      "what": "the same calls replayed from one captured CUDA graph (context)"},
            "hot_l2": {"us_per_call": hot_us, "calls": n_hot,
                       "what": "the same call on one cache copy, resident in L2 (context)"},
            "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "overlap": "step i+1's inputs copied on a second stream while step i computes"},
            "gpu_launches": args.steps * r.launches_per_call,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as tdist
            tdist.destroy_process_group()


if __name__ == "__main__":
    main()

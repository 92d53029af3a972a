"""ncu captures of the verify call and the summaries kept under ``profiles/``.

Two steps, so that the capture (which needs the GPU) and the summary (which
only reads CSV text) can run on different machines:

    python -m mla_verify_attention_gb300.ncu_report capture --workload tree9_p65536 --out DIR
    python -m mla_verify_attention_gb300.ncu_report summarize --workload tree9_p65536 --dir DIR

``capture`` first runs the bench command plainly and stops unless it exits 0.
It then runs two ncu passes, each with ``--clock-control none`` (ncu would lock
the clocks otherwise):

1. the launch list: every kernel launch of the command with its device time
   alone (``gpu__time_duration.sum``, a single-pass metric), as CSV;
2. counters of the split kernel only (``-k regex:verify_split``, ``-c 2``):
   DRAM bytes read and written, tensor-pipe activity and the device time.

The bench command is ``bench.py --workload W --configs none --steps 20
--warmup 3 --no-cpu-baseline --e2e-steps 2`` (a few hundred MB of device
memory, ~0.1 ms per launch), so that both captures end by themselves.

``summarize`` turns the two CSV files into ``profiles/traffic_W.json`` (the
split kernel's DRAM bytes per launch, which ``bench.py`` reports as
``roofline.traffic`` while the kernel sources are unchanged) and
``profiles/verify_call_W_launches.md`` (per kernel: launches, total time,
share; and the counters).  Per-launch times under ncu are cold-cache and
serialised: the shares, not the absolute times, compare with the bench.
"""
from __future__ import annotations

import argparse
import csv
import datetime
import importlib.util
import io
import json
import os
import re
import subprocess
import sys
import time

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)

COUNTERS = ("gpu__time_duration.sum", "dram__bytes_read.sum", "dram__bytes_write.sum",
            "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active",
            "sm__pipe_tensor_cycles_active.max.pct_of_peak_sustained_active",
            "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed")

KERNEL_ROLES = (
    ("verify_split_kernel", "split kernel: QK, mask, online softmax and PV of one key slice "
                            "per 2-CTA cluster"),
    ("combine_kernel", "merge of the slices' partial states"),
    ("combine_cols_kernel", "merge of the slices' partial states (few rows: 128-column blocks)"),
    ("plan_kernel", "device-side slice plan (2..32 streams)"),
    ("repack_kernel", "copy of a paged cache into a contiguous one"),
)


def bench_cmd(workload, python=sys.executable, steps=20):
    return [python, os.path.join(ROOT, "bench.py"), "--workload", workload, "--configs", "none",
            "--steps", str(steps), "--warmup", "3", "--no-cpu-baseline", "--e2e-steps", "2"]


def ncu_exe():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "ncu")
    return cand if os.path.exists(cand) else "ncu"


def _run(cmd, log):
    t0 = time.time()
    with open(log, "w") as fh:
        rc = subprocess.call(cmd, stdout=fh, stderr=subprocess.STDOUT)
    return rc, time.time() - t0


def capture(workload, out, steps=20):
    """Plain run, then the launch list and the split kernel's counters."""
    os.makedirs(out, exist_ok=True)
    cmd = bench_cmd(workload, steps=steps)
    rec = {"workload": workload, "bench_cmd": " ".join(os.path.relpath(c, ROOT) if c.startswith(ROOT)
                                                       else c for c in cmd),
           "started": datetime.datetime.now().isoformat(timespec="seconds")}
    rc, dt = _run(cmd, os.path.join(out, "plain_%s.log" % workload))
    rec["plain"] = {"rc": rc, "s": round(dt, 1)}
    if rc != 0:
        _write(os.path.join(out, "capture_%s.json" % workload), rec)
        return rc
    launches = os.path.join(out, "launches_%s.csv" % workload)
    ncu_l = [ncu_exe(), "--metrics", "gpu__time_duration.sum", "--clock-control", "none",
             "-c", "2000", "--csv", "--log-file", launches] + cmd
    rc, dt = _run(ncu_l, os.path.join(out, "ncu_launches_%s.log" % workload))
    rec["launch_list"] = {"rc": rc, "s": round(dt, 1), "cmd": _rel(ncu_l)}
    if rc != 0:
        _write(os.path.join(out, "capture_%s.json" % workload), rec)
        return rc
    counters = os.path.join(out, "counters_%s.csv" % workload)
    ncu_c = [ncu_exe(), "--metrics", ",".join(COUNTERS), "--clock-control", "none",
             "-k", "regex:verify_split", "-s", "3", "-c", "2", "--csv", "--log-file", counters] + cmd
    rc, dt = _run(ncu_c, os.path.join(out, "ncu_counters_%s.log" % workload))
    rec["counters"] = {"rc": rc, "s": round(dt, 1), "cmd": _rel(ncu_c)}
    _write(os.path.join(out, "capture_%s.json" % workload), rec)
    return rc


def _rel(cmd):
    out = []
    for c in cmd:
        if c.startswith(ROOT + os.sep):
            c = os.path.relpath(c, ROOT)
        elif os.path.isabs(c) and os.path.basename(c) in ("ncu", "python", "python3") or \
                re.match(r".*/python3(\.\d+)?$", c):
            c = os.path.basename(c)
        out.append(c)
    return " ".join(out)


def _write(path, obj):
    with open(path, "w") as fh:
        json.dump(obj, fh, indent=1)
        fh.write("\n")


def read_ncu_csv(path):
    """Rows of an ncu --csv --log-file (one row per launch and metric)."""
    with open(path) as fh:
        text = fh.read()
    i = text.find('"ID"')
    if i < 0:
        return []
    rows = []
    for r in csv.DictReader(io.StringIO(text[i:])):
        try:
            v = float(r["Metric Value"].replace(",", ""))
        except (KeyError, ValueError):
            continue
        rows.append({"id": int(r["ID"]), "kernel": r["Kernel Name"], "metric": r["Metric Name"],
                     "unit": r.get("Metric Unit", ""), "value": v})
    return rows


_SCALE = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "ns": 1e-3, "us": 1.0,
          "usecond": 1.0, "nsecond": 1e-3, "msecond": 1e3, "ms": 1e3, "%": 1.0, "": 1.0}


def _in(v, unit):
    return v * _SCALE.get(unit, 1.0)


def short_name(kernel):
    """'void mla::verify_split_kernel<0, 1>(CUtensorMap_st, ...)' -> 'verify_split_kernel<0, 1>'
    (return type, namespaces and parameter list dropped)."""
    k = kernel[5:] if kernel.startswith("void ") else kernel
    depth = 0
    for i, ch in enumerate(k):
        if ch == "<":
            depth += 1
        elif ch == ">":
            depth -= 1
        elif ch == "(" and depth == 0:
            k = k[:i]
            break
    base = k.split("<", 1)
    head = base[0].rsplit("::", 1)[-1]
    return head + ("<" + base[1] if len(base) > 1 else "")


def _role(name):
    for prefix, role in KERNEL_ROLES:
        if name.startswith(prefix):
            return role
    return ""


def _kernel_src_hash():
    spec = importlib.util.spec_from_file_location("_bench_for_hash", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.kernel_src_hash(), mod


def summarize(workload, src_dir, profiles=os.path.join(ROOT, "profiles")):
    """Write profiles/traffic_W.json and profiles/verify_call_W_launches.md."""
    launches = read_ncu_csv(os.path.join(src_dir, "launches_%s.csv" % workload))
    counters = read_ncu_csv(os.path.join(src_dir, "counters_%s.csv" % workload))
    try:
        with open(os.path.join(src_dir, "capture_%s.json" % workload)) as fh:
            cap = json.load(fh)
    except OSError:
        cap = {}
    per = {}
    for r in launches:
        if r["metric"] != "gpu__time_duration.sum":
            continue
        k = short_name(r["kernel"])
        d = per.setdefault(k, {"launches": 0, "total_us": 0.0})
        d["launches"] += 1
        d["total_us"] += _in(r["value"], r["unit"])
    total = sum(d["total_us"] for d in per.values()) or 1.0
    for d in per.values():
        d["avg_us"] = d["total_us"] / max(1, d["launches"])
        d["share"] = d["total_us"] / total
    by_launch = {}
    for r in counters:
        by_launch.setdefault(r["id"], {"kernel": short_name(r["kernel"])})[r["metric"]] = \
            _in(r["value"], r["unit"])
    split = [v for v in by_launch.values() if v["kernel"].startswith("verify_split_kernel")]

    def mean(key):
        xs = [v[key] for v in split if key in v]
        return sum(xs) / len(xs) if xs else None

    h, bench = _kernel_src_hash()
    from . import inputs as I
    case = I.make_case(I.WORKLOADS[workload], pad="normal")
    flops, cache_bytes = bench.work_of(case)
    rd, wr = mean("dram__bytes_read.sum"), mean("dram__bytes_write.sum")
    traffic = {
        "what": "DRAM bytes per launch of the split kernel (verify_split_kernel), mean of the "
                "captured launches, from ncu counters",
        "workload": "%s (B=%d, q_len=%d, H=%d, seq_lens %s, Smax %d)" % (
            workload, case.B, case.q, case.H, [int(x) for x in case.seq_lens], case.Smax),
        "command": cap.get("counters", {}).get("cmd"),
        "launch_list_command": cap.get("launch_list", {}).get("cmd"),
        "verify_split_kernel": {
            "instantiations": sorted({v["kernel"] for v in split}),
            "captured_launches": len(split),
            "us_cold": mean("gpu__time_duration.sum"),
            "dram_read_bytes": rd, "dram_write_bytes": wr,
            "dram_bytes_per_launch": (rd + wr) if rd is not None and wr is not None else None,
            "tensor_pipe_active_pct": mean("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active"),
            "tensor_pipe_active_pct_max_sm": mean(
                "sm__pipe_tensor_cycles_active.max.pct_of_peak_sustained_active"),
            "dram_throughput_pct": mean("gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed"),
        },
        "algorithmic": {"flops_per_launch": flops, "cache_bytes_per_launch": cache_bytes},
        "launch_list": {k: {kk: round(vv, 4) if isinstance(vv, float) else vv for kk, vv in d.items()}
                        for k, d in sorted(per.items(), key=lambda kv: -kv[1]["total_us"])},
        "kernel_src_sha256_16": h,
    }
    os.makedirs(profiles, exist_ok=True)
    _write(os.path.join(profiles, "traffic_%s.json" % workload), traffic)

    lines = ["# Launch list and split-kernel counters: %s" % traffic["workload"], "",
             "Written by `python -m mla_verify_attention_gb300.ncu_report summarize --workload %s` "
             "from the CSV files of `... capture --workload %s` (GB300, one GPU, after the same "
             "bench command exited 0 without ncu)." % (workload, workload), "",
             "Launch list:", "", "    %s" % traffic["launch_list_command"], "",
             "Counters (split kernel only):", "", "    %s" % traffic["command"], "",
             "Kernel sources: sha256/16 of the code in mla_verify_attention_gb300/csrc "
             "(comments ignored) = %s.  Per-launch times under ncu are cold-cache and "
             "serialised; compare shares, not absolute times." % h, "",
             "| kernel | role | launches | total us | avg us (cold) | share |",
             "|---|---|---|---|---|---|"]
    for k, d in sorted(per.items(), key=lambda kv: -kv[1]["total_us"]):
        lines.append("| %s | %s | %d | %.1f | %.2f | %.1f %% |" % (
            k, _role(k), d["launches"], d["total_us"], d["avg_us"], 100 * d["share"]))
    s = traffic["verify_split_kernel"]

    def f(x, fmt):
        return fmt % x if x is not None else "n/a"

    lines += ["", "Split kernel, %d captured launch(es) (%s):" % (
        s["captured_launches"], ", ".join(s["instantiations"]) or "none"), "",
        "| counter | value |", "|---|---|",
        "| gpu__time_duration.sum | %s us |" % f(s["us_cold"], "%.2f"),
        "| dram__bytes_read.sum | %s MB |" % f(None if rd is None else rd / 1e6, "%.2f"),
        "| dram__bytes_write.sum | %s MB |" % f(None if wr is None else wr / 1e6, "%.2f"),
        "| algorithmic cache bytes (keys x 1152 B, read once) | %.2f MB |" % (cache_bytes / 1e6),
        "| DRAM traffic / algorithmic bytes | %s |" % f(
            None if s["dram_bytes_per_launch"] is None else s["dram_bytes_per_launch"] / cache_bytes,
            "%.3f"),
        "| sm__pipe_tensor_cycles_active (avg over SMs, of active cycles) | %s %% |" % f(
            s["tensor_pipe_active_pct"], "%.1f"),
        "| same, busiest SM | %s %% |" % f(s["tensor_pipe_active_pct_max_sm"], "%.1f"),
        "| gpu__dram_throughput (of peak, elapsed) | %s %% |" % f(s["dram_throughput_pct"], "%.1f"),
        ""]
    with open(os.path.join(profiles, "verify_call_%s_launches.md" % workload), "w") as fh:
        fh.write("\n".join(lines))
    return traffic


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    sub = ap.add_subparsers(dest="cmd", required=True)
    c = sub.add_parser("capture")
    c.add_argument("--workload", required=True)
    c.add_argument("--out", required=True)
    c.add_argument("--steps", type=int, default=20)
    s = sub.add_parser("summarize")
    s.add_argument("--workload", required=True)
    s.add_argument("--dir", required=True)
    s.add_argument("--profiles", default=os.path.join(ROOT, "profiles"))
    a = ap.parse_args(argv)
    if a.cmd == "capture":
        return capture(a.workload, a.out, a.steps)
    summarize(a.workload, a.dir, a.profiles)
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark: achieved HBM GB/s and rows/s of the online softmax and fused TopK.

One step = one pass of the hot path over one batch of each headline workload:
  * softmax 4096 x 32000 fp32 -> fp32
  * softmax 8192 x 128256 bf16 -> bf16 (4 spikes at +40 per row, 1% -inf)
  * fused softmax+TopK 256 x 50257 fp32, K = 8 and K = 64
`value` is the step's compulsory HBM bytes (softmax: one read of x and one
write of y; TopK: one read of x plus K*8 bytes of output) divided by the
device time of the step, summed over all ranks' work, over the max rank time.

Timing: CUDA events on the launching stream, W untimed warm-up steps, then K
timed steps between barriers and synchronisations; inside them only the
dominant kernel is bracketed by events (its duration gives `roofline`).  The softmax inputs are
larger than L2; the TopK input (51 MB) rotates over enough copies to cover
three times the L2 size, so no timed launch reads a cache-resident input.

Also printed: `e2e` (the same metric through the public API with pinned host
buffers: host->device copy of every input and device->host copy of every
output inside the timed region), `roofline` of the dominant kernel,
`cpu_baseline` (the float64 oracle on the host cores on a bounded sample),
`clocks` (nvidia-smi samples taken during the timed region),
`per_workload` (after the timed region, each kernel of the step in a loop
of its own, with its share of the step from events recorded between the
step's launches; then the other configurations -- 64x1024 fp32, causal
1048576x128, increasing 65536x4096 --, rows that are not whole 16-byte
vectors (4096 x 50257 fp32) and the ex2.approx-free kernel on the bf16
workload, in loops of their own),
`unfused_baselines` (three-pass safe softmax against the online kernel,
softmax-then-TopK against the fused kernel), `stats_and_causal` (row
statistics; causal mask applied in the kernel), `attention` (the tensor-core
attention forward in TFLOP/s) and, inside `e2e`, the plain pinned copy rates
of the host link.

`--impl reference` times the oracle alone (the reference arm: the method's
own definition run on the host cores), on the same metric.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

SOFTMAX_STEP = ["softmax_4096x32000_f32", "softmax_8192x128256_bf16"]
TOPK_NAME = "topk_256x50257_f32"
TOPK_KS = (8, 64)
EXTRA = ["softmax_64x1024_f32", "causal_1048576x128_f32", "increasing_65536x4096_f32"]
METRIC = ("achieved HBM GB/s (compulsory bytes) of one step: softmax 4096x32000 fp32 + "
          "softmax 8192x128256 bf16 + fused softmax+TopK 256x50257 fp32 K=8 and K=64")
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ bytes
def softmax_bytes(w) -> int:
    b = 4 if w.dtype == "f32" else 2
    return w.rows * w.cols * 2 * b


def topk_bytes(w, K) -> int:
    return w.rows * w.cols * 4 + w.rows * K * 8


def step_units():
    """(label, bytes, rows) of every launch in one step."""
    out = []
    for n in SOFTMAX_STEP:
        w = workloads.WORKLOADS[n]
        out.append((n, softmax_bytes(w), w.rows))
    w = workloads.WORKLOADS[TOPK_NAME]
    for K in TOPK_KS:
        out.append((f"{TOPK_NAME}_K{K}", topk_bytes(w, K), w.rows))
    return out


# ------------------------------------------------------------------ environment
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# The sources the softmax kernels are compiled from (their translation units
# and the library headers they include; the public API header only lends
# them its types); a recorded DRAM traffic figure stands only while these are
# unchanged.
SOFTMAX_KERNEL_SOURCES = ("softmax_*.cu", "softmax_dispatch.cuh", "host_common.h", "internal.h",
                          "ctl.h", "kernels/softmax_kernels.cuh", "kernels/ops.cuh")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "softmax_topk_gb300", "csrc")
    files = sorted({f for pat in SOFTMAX_KERNEL_SOURCES for f in glob.glob(os.path.join(csrc, pat))})
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.relpath(f, csrc).encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel sources as they are now (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    @staticmethod
    def _parse(lines) -> list:
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        return rows

    def _query_once(self) -> list:
        try:
            out = subprocess.run(["nvidia-smi", f"--id={self.gpu_index}",
                                  f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits"],
                                 capture_output=True, text=True, timeout=30).stdout
        except (OSError, subprocess.TimeoutExpired):
            return []
        return self._parse(out.splitlines())

    def stop(self, t0: float, t1: float) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            rows = self._parse(f)
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 1 <= r[0] <= t1 + 1]
        window = "timed region"
        if not inside:
            inside, window = rows, "whole run"
        if not inside:  # a timed region shorter than the sampling period
            inside, window = self._query_once(), "right after the timed region"
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# ------------------------------------------------------------------ our arm
def make_step_inputs(dev, st):
    """Device inputs and outputs for one step; TopK inputs rotated over L2."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    items = []
    for n in SOFTMAX_STEP:
        w = workloads.WORKLOADS[n]
        x = workloads.make(w, device=dev)
        y = torch.empty_like(x)
        items.append(("softmax", n, [x], y, None, 0))
    w = workloads.WORKLOADS[TOPK_NAME]
    xt = workloads.make(w, device=dev)
    copies = -(-3 * l2 // (xt.numel() * 4)) + 1
    xs = [xt] + [xt.clone() for _ in range(copies - 1)]
    for j, K in enumerate(TOPK_KS):
        vals = torch.empty(w.rows, K, device=dev)
        idx = torch.empty(w.rows, K, dtype=torch.int32, device=dev)
        items.append(("topk", f"{TOPK_NAME}_K{K}", xs, (vals, idx), K, j))
    return items, copies


def step_attribution(st, items, stream, dev, steps):
    """Mean device time of each launch of the step, from events recorded
    between all launches (they add about 2 us each to the stream)."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(items) + 1)]
           for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for it in range(steps):
        evs[it][0].record(stream)
        for j, item in enumerate(items):
            launch(st, item, it)
            evs[it][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    return [sum(evs[it][j].elapsed_time(evs[it][j + 1]) for it in range(steps)) / steps
            for j in range(len(items))]


def launch(st, item, it):
    """Launch one item of step `it`.  Each TopK launch of the step reads its
    own copy of the input (copy (it * len(TOPK_KS) + j) mod copies), so none
    reads a copy that an earlier launch of the last 3 x L2 bytes read."""
    kind, _, xs, out, K, j = item
    x = xs[(it * len(TOPK_KS) + j) % len(xs)]
    if kind == "softmax":
        st.softmax(x, out=out)
    else:
        st.softmax_topk(x, K, vals=out[0], idx=out[1])


def run_ours(args):
    world, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    import softmax_topk_gb300 as st

    items, topk_copies = make_step_inputs(dev, st)
    units = step_units()
    stream = torch.cuda.current_stream(dev)

    for it in range(args.warmup):
        for item in items:
            launch(st, item, it)
    torch.cuda.synchronize(dev)

    n_items = len(items)
    # Inside the timed region only the dominant kernel (the most bytes) is
    # bracketed by events: an event recorded between two launches costs the
    # stream about 2 us, which would weigh on the short TopK launches.
    dom = max(range(n_items), key=lambda j: units[j][1])
    dom_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    clocks = ClockSampler(local) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for it in range(args.steps):
        for j, item in enumerate(items):
            if j == dom:
                dom_evs[it][0].record(stream)
            launch(st, item, it)
            if j == dom:
                dom_evs[it][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    t1 = time.time()
    clock_info = clocks.stop(t0, t1) if clocks else None

    from softmax_topk_gb300 import multi
    total_ms = multi.max_over_ranks(start.elapsed_time(end), device=dev)
    dom_ms = sum(a.elapsed_time(b) for a, b in dom_evs) / args.steps
    ms_per_step = total_ms / args.steps
    # after the timed region: each launch's share of the step (events between
    # all launches, same inputs), and each kernel in a loop of its own
    in_step_ms = step_attribution(st, items, stream, dev, args.steps)
    own_ms = [_time_ms(lambda i, item=item: launch(st, item, i), dev, max(20, args.steps))
              for item in items]
    step_bytes = sum(u[1] for u in units)
    value = multi.whole_job_rate(step_bytes, world, ms_per_step * 1e-3) / 1e9

    e2e = run_e2e(st, dev, args) if rank == 0 else None
    others = time_other_workloads(st, dev, args) if rank == 0 else None
    baselines = run_baselines(st, dev, args) if rank == 0 else None
    stats_causal = run_stats_and_causal(st, dev, args) if rank == 0 else None
    attention = run_attention(st, dev, args, False) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    per = {}
    for j, (label, b, rows) in enumerate(units):
        ms = own_ms[j]
        per[label] = {"ms": round(ms, 5), "gbs": round(b / (ms * 1e-3) / 1e9, 1),
                      "rows_per_s": round(rows / (ms * 1e-3), 1),
                      "frac_of_measured_hbm": round(b / (ms * 1e-3) / 1e9 / peak, 4),
                      "frac_of_8tbs_nominal": round(b / (ms * 1e-3) / 1e9 / 8000.0, 4),
                      "timing": "own loop of back-to-back launches, inputs as in the step",
                      "in_step_ms": round(in_step_ms[j], 5),
                      "in_step_share": round(in_step_ms[j] / sum(in_step_ms), 4)}
    per[units[dom][0]]["timed_region_ms"] = round(dom_ms, 5)
    dom_label, dom_bytes, _ = units[dom]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    kernel_name = kernel_of(st, dom_label)
    traffic = recorded_traffic(kernel_name)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded generators in workloads/, shapes and distributions of the "
                "pages' workloads)",
        "config": {"workload": "softmax 4096x32000 f32 + softmax 8192x128256 bf16 + TopK "
                               "256x50257 f32 K=8,64",
                   "l2": f"softmax inputs larger than L2; TopK input rotated over {topk_copies} "
                         "copies (> 3x L2)",
                   "parallelism": f"replicas x{world} (rows are independent; no collective)"},
        "per_workload": {**per, **(others or {})},
        "rows_per_s": {k: v["rows_per_s"] for k, v in per.items()},
        "roofline": {"kernel": kernel_name, "workload": dom_label, "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": dom_bytes, "traffic": traffic},
        "gpu_launches": n_items * args.steps,
        "e2e": e2e,
        "clocks": clock_info,
    }
    line["unfused_baselines"] = baselines
    line["stats_and_causal"] = stats_causal
    line["attention"] = attention
    if args.extra:
        line["extra_workloads"] = run_extra(st, dev, args)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            line["attention"]["cpu_baseline"] = attention_oracle_rate(
                workloads.ATTENTION_WORKLOADS["attention_4x16x4096x128_bf16"], False,
                args.cpu_seconds / 3)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


OTHER_WORKLOADS = ["softmax_64x1024_f32", "causal_1048576x128_f32", "increasing_65536x4096_f32",
                   "softmax_4096x50257_f32"]


def time_other_workloads(st, dev, args) -> dict:
    """The configurations outside the step (its parity cases) and the
    ex2.approx-free kernel on the step's bf16 workload, each timed in a loop
    of its own after the step: W warm-up launches, then K launches between
    CUDA events on the launching stream; inputs smaller than 3x L2 rotate over
    enough copies that no timed launch reads a cache-resident input."""
    out = {}
    peak, _ = measured_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    steps = max(args.steps, 10)
    cases = [(n, "auto") for n in OTHER_WORKLOADS] + [("softmax_8192x128256_bf16", "stream_poly")]
    for n, path in cases:
        w = workloads.WORKLOADS[n]
        x = workloads.make(w, device=dev)
        nbytes = x.numel() * x.element_size()
        copies = -(-3 * l2 // nbytes) + 1 if nbytes < 3 * l2 else 1
        xs = [x] + [x.clone() for _ in range(copies - 1)]
        y = torch.empty_like(x)
        ms = _time_ms(lambda i: st.softmax(xs[i % copies], out=y, path=path), dev, steps,
                      warmup=args.warmup)
        b = softmax_bytes(w)
        gbs = b / (ms * 1e-3) / 1e9
        key = n if path == "auto" else f"{n}_{path}"
        out[key] = {"ms": round(ms, 5), "gbs": round(gbs, 1), "rows_per_s": round(w.rows / (ms * 1e-3), 1),
                    "frac_of_measured_hbm": round(gbs / peak, 4),
                    "frac_of_8tbs_nominal": round(gbs / 8000.0, 4),
                    "kernel": kernel_of(st, n, path), "input_copies": copies,
                    "timing": "own loop after the step"}
        if n == "softmax_64x1024_f32":
            out[key]["note"] = ("0.5 MB per launch: bound by launch overhead, not by HBM "
                                "(no roofline target)")
        del xs, x, y
    return out


def link_rates(dev, nbytes: int = 1 << 30) -> dict:
    """Plain pinned host<->device copy rates in this process (one copy per
    direction, then both directions at once on two streams): the bound of
    the e2e leg, whose every step moves its inputs and results over this link."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h2 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize(dev)
        t = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t) / reps

    t_h2d = timed(lambda: d.copy_(h, non_blocking=True))
    t_d2h = timed(lambda: h.copy_(d, non_blocking=True))

    def both():
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)
    t_both = timed(both)
    return {"h2d_gbs": round(nbytes / t_h2d / 1e9, 1), "d2h_gbs": round(nbytes / t_d2h / 1e9, 1),
            "both_directions_gbs": round(2 * nbytes / t_both / 1e9, 1),
            "bytes_per_copy": nbytes, "how": "torch copy_ of pinned uint8 buffers, wall clock "
                                             "over 5 copies after one untimed"}


def kernel_of(st, label: str, path: str = "auto") -> str:
    if label.startswith("topk"):
        return "topk_rows_kernel"
    w = workloads.WORKLOADS[label]
    code = st.OS_F32 if w.dtype == "f32" else st.OS_BF16
    p = st.plan((w.rows, w.cols), code, path=path)
    fam = {st.OS_PATH_WARP: "warp_rows_kernel", st.OS_PATH_ONCHIP: "onchip_rows_kernel",
           st.OS_PATH_STREAM: "stream_rows_kernel",
           st.OS_PATH_STREAM_POLY: "stream_rows_kernel[fma-pipe exp]"}[p["path"]]
    if p["path"] == st.OS_PATH_ONCHIP and p["stages"] > 0:
        fam = "tma_rows_kernel"
    return f"{fam}<{w.dtype},{w.dtype},threads={p['threads']},cluster={p['cluster']}>"


def run_e2e(st, dev, args):
    """Same step through the public API from pinned host buffers: every
    input copied host->device and every result device->host inside the timed
    region, pipelined over row blocks and, through two device buffer sets,
    across consecutive steps."""
    host_in, host_out = [], []
    h2d = d2h = 0
    for n in SOFTMAX_STEP:
        w = workloads.WORKLOADS[n]
        x = workloads.make(w, device=dev).cpu().pin_memory()
        host_in.append(x)
        host_out.append(torch.empty_like(x).pin_memory())
        h2d += x.numel() * x.element_size()
        d2h += x.numel() * x.element_size()
    w = workloads.WORKLOADS[TOPK_NAME]
    xt = workloads.make(w, device=dev).cpu().pin_memory()
    h2d += xt.numel() * 4
    topk_out = []
    for K in TOPK_KS:
        topk_out.append((torch.empty(w.rows, K).pin_memory(),
                         torch.empty(w.rows, K, dtype=torch.int32).pin_memory()))
        d2h += w.rows * K * 8
    # Two device buffer sets, alternating by step: the copy-in of a step's
    # first blocks overlaps the copy-out of the previous step's last ones.  A
    # set is refilled only after the step that used it two steps before has
    # copied its results out (an event on the copy-out stream).
    sets = []
    for _ in range(2):
        sets.append({"in": [torch.empty_like(h, device=dev) for h in host_in],
                     "out": [torch.empty_like(h, device=dev) for h in host_in],
                     "xt": torch.empty_like(xt, device=dev),
                     "topk": [(torch.empty(w.rows, K, device=dev),
                               torch.empty(w.rows, K, dtype=torch.int32, device=dev))
                              for K in TOPK_KS]})

    # Pipelined over row blocks on three streams: copy-in of a block overlaps
    # the kernel on the block before and the copy-out of the one before that
    # (host->device and device->host copies run on separate copy engines).
    # The TopK block (51 MB in, a few KB out) goes first and the softmax rows
    # follow in blocks of about 130 MB, so the link's two directions are busy
    # together for as much of the step as possible.
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    main = torch.cuda.current_stream(dev)

    def pieces_of(bufs):
        out = [("topk", xt, bufs["xt"], bufs["topk"], topk_out)]
        for h, d, o, ho in zip(host_in, bufs["in"], bufs["out"], host_out):
            blocks = max(1, -(-h.numel() * h.element_size() // (136 << 20)))
            step = -(-h.shape[0] // blocks)
            for r0 in range(0, h.shape[0], step):
                r1 = min(h.shape[0], r0 + step)
                out.append(("softmax", h[r0:r1], d[r0:r1], o[r0:r1], ho[r0:r1]))
        return out
    set_pieces = [pieces_of(b) for b in sets]
    freed = [None, None]  # copy-out of the last step that used each set

    def one_step(i):
        k = i % 2
        if freed[k] is not None:
            s_in.wait_event(freed[k])
        for kind, h, d, o, ho in set_pieces[k]:
            with torch.cuda.stream(s_in):
                d.copy_(h, non_blocking=True)
            s_comp.wait_stream(s_in)
            with torch.cuda.stream(s_comp):
                if kind == "softmax":
                    st.softmax(d, out=o)
                else:
                    for K, (v, ix) in zip(TOPK_KS, o):
                        st.softmax_topk(d, K, vals=v, idx=ix)
            s_out.wait_stream(s_comp)
            with torch.cuda.stream(s_out):
                if kind == "softmax":
                    ho.copy_(o, non_blocking=True)
                else:
                    for (v, ix), (hv, hi) in zip(o, ho):
                        hv.copy_(v, non_blocking=True)
                        hi.copy_(ix, non_blocking=True)
        freed[k] = torch.cuda.Event()
        freed[k].record(s_out)

    steps = max(3, min(args.steps, 20))
    for s_ in (s_in, s_comp, s_out):
        s_.wait_stream(main)
    for i in range(2):
        one_step(i)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for s_ in (s_in, s_comp, s_out):
        s_.wait_stream(main)
    for i in range(steps):
        one_step(i)
    main.wait_stream(s_out)
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / steps
    step_bytes = sum(u[1] for u in step_units())
    del host_in, host_out, sets, set_pieces, xt, topk_out
    link = link_rates(dev)
    # the host link alone, at the rates measured above, with both directions
    # overlapped as the pipeline overlaps them: the bound of this leg
    link_ms = max((h2d + d2h) / (link["both_directions_gbs"] * 1e9),
                  h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9)) * 1e3
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "link": link, "link_bound_ms_per_step": round(link_ms, 4),
            "frac_of_link_bound": round(link_ms / ms, 4)}


def run_extra(st, dev, args):
    """The other workloads (parity cases), timed the same way, for reference."""
    out = {}
    peak, _ = measured_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.current_stream(dev)
    for n in EXTRA:
        w = workloads.WORKLOADS[n]
        x = workloads.make(w, device=dev)
        copies = max(1, -(-3 * l2 // (x.numel() * x.element_size())) + 1)
        xs = [x] + [x.clone() for _ in range(copies - 1)] if x.numel() * 4 < 3 * l2 else [x]
        y = torch.empty_like(x)
        for i in range(3):
            st.softmax(xs[i % len(xs)], out=y)
        steps = max(10, args.steps)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        for i in range(steps):
            st.softmax(xs[i % len(xs)], out=y)
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b) / steps
        gbs = softmax_bytes(w) / (ms * 1e-3) / 1e9
        out[n] = {"ms": round(ms, 5), "gbs": round(gbs, 1), "rows_per_s": round(w.rows / ms * 1e3),
                  "frac_of_measured_hbm": round(gbs / peak, 4), "input_copies": len(xs)}
        del xs, x, y
    return out


def _time_ms(fn, dev, steps, warmup: int = 3):
    stream = torch.cuda.current_stream(dev)
    for i in range(max(3, warmup)):
        fn(i)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for i in range(steps):
        fn(i)
    b.record(stream)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / steps


def run_baselines(st, dev, args):
    """The unfused pipelines the online normalizer and the fused TopK replace
    ("Online normalizer calculation for softmax", sections 2 and 4): the
    three-pass safe softmax against the two-pass online kernel, and softmax
    followed by TopK of the probabilities against the fused kernel, on the
    step's workloads.  Times per call (CUDA events), inputs larger than L2 or
    rotated like the step's."""
    out = {}
    steps = max(20, min(args.steps, 200))
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    for n in SOFTMAX_STEP:
        w = workloads.WORKLOADS[n]
        x = workloads.make(w, device=dev)
        y = torch.empty_like(x)
        t_online = _time_ms(lambda i: st.softmax(x, out=y), dev, steps)
        t_safe = _time_ms(lambda i: st.softmax(x, out=y, path="safe"), dev, steps)
        out[n] = {"online_ms": round(t_online, 5), "safe_three_pass_ms": round(t_safe, 5),
                  "safe_over_online": round(t_safe / t_online, 3)}
        del x, y
    w = workloads.WORKLOADS[TOPK_NAME]
    x = workloads.make(w, device=dev)
    copies = max(1, -(-3 * l2 // (x.numel() * 4)) + 1)
    xs = [x] + [x.clone() for _ in range(copies - 1)]
    y = torch.empty_like(x)
    for K in TOPK_KS:
        vals = torch.empty(w.rows, K, device=dev)
        idx = torch.empty(w.rows, K, dtype=torch.int32, device=dev)
        t_fused = _time_ms(lambda i: st.softmax_topk(xs[i % copies], K, vals=vals, idx=idx), dev, steps)

        def unfused(i, path):
            st.softmax(xs[i % copies], out=y, path=path)
            st.topk(y, K, vals=vals, idx=idx)
        t_online = _time_ms(lambda i: unfused(i, "auto"), dev, steps)
        t_safe = _time_ms(lambda i: unfused(i, "safe"), dev, steps)
        u = torch.rand(w.rows, device=dev)
        draws = torch.empty(w.rows, dtype=torch.int32, device=dev)
        t_sample = _time_ms(lambda i: st.topk_sample(vals, idx, u, out=draws), dev, steps)
        out[f"{TOPK_NAME}_K{K}"] = {
            "fused_ms": round(t_fused, 5), "sample_after_fused_ms": round(t_sample, 5),
            "online_softmax_then_topk_ms": round(t_online, 5),
            "safe_softmax_then_topk_ms": round(t_safe, 5),
            "unfused_online_over_fused": round(t_online / t_fused, 3),
            "unfused_safe_over_fused": round(t_safe / t_fused, 3)}
    return out


def run_stats_and_causal(st, dev, args):
    """Row statistics (one read per element, 12 bytes out per row) on the
    step's softmax workloads, and the causal workload with the mask applied in
    the kernel (masked columns never read) against reading the planted -inf."""
    out = {}
    steps = max(20, min(args.steps, 200))
    peak, _ = measured_peaks()
    for n in SOFTMAX_STEP:
        w = workloads.WORKLOADS[n]
        x = workloads.make(w, device=dev)
        ms = _time_ms(lambda i: st.softmax_stats(x), dev, steps)
        b = x.numel() * x.element_size() + w.rows * 12
        out[f"stats_{n}"] = {"ms": round(ms, 5), "gbs": round(b / ms / 1e6, 1),
                             "frac_of_measured_hbm": round(b / ms / 1e6 / peak, 4)}
        del x
    w = workloads.WORKLOADS["causal_1048576x128_f32"]
    x = workloads.make(w, device=dev)
    dense = torch.where(torch.isinf(x), torch.zeros_like(x), x)
    y = torch.empty_like(x)
    t_read = _time_ms(lambda i: st.softmax(x, out=y), dev, steps)
    t_mask = _time_ms(lambda i: st.softmax_causal(dense, 128, 0, out=y), dev, steps)
    # compulsory bytes with the mask in the kernel: the kept entries read, every entry written
    kept = sum(min(w.cols, r % 128 + 1) for r in range(128)) * (w.rows // 128)
    b_mask = kept * 4 + w.rows * w.cols * 4
    out["causal_1048576x128_f32"] = {
        "read_minus_inf_ms": round(t_read, 5), "in_kernel_mask_ms": round(t_mask, 5),
        "read_over_mask": round(t_read / t_mask, 3),
        "in_kernel_mask_gbs": round(b_mask / t_mask / 1e6, 1),
        "in_kernel_mask_frac_of_measured_hbm": round(b_mask / t_mask / 1e6 / peak, 4)}
    return out


def attention_flops(w, causal: bool, head_dim: int | None = None) -> int:
    """Algorithmic FLOPs of one attention forward: 2 for each multiply-add of
    Q K^T and of P V over the (query, key) pairs the mask keeps."""
    d = head_dim or w.head_dim
    pairs = w.seq_len * (w.seq_len + 1) // 2 if causal else w.seq_len ** 2
    return 4 * w.bh * pairs * d


def attention_oracle_rate(w, causal: bool, target_seconds: float) -> dict:
    """The float64 oracle on a bounded sample of query rows of the attention
    workload: FLOP/s over the same algorithmic count per row."""
    import oracle
    q, k, v = workloads.make_attention(w, device="cpu")
    k64, v64 = k.double().numpy(), v.double().numpy()
    qf = q.double().numpy()
    rng = np.random.default_rng(7)
    n_rows, done_rows, flops, t_total = 16, 0, 0, 0.0
    while t_total < target_seconds and done_rows < 65536:
        sl = rng.integers(0, w.bh, n_rows)
        rw = rng.integers(0, w.seq_len, n_rows)
        t0 = time.perf_counter()
        oracle.attention_rows(qf[sl, rw], k64, v64, sl, rw, None, causal)
        t_total += time.perf_counter() - t0
        done_rows += n_rows
        flops += int(sum(4 * w.head_dim * ((r + 1) if causal else w.seq_len) for r in rw))
        n_rows = min(n_rows * 2, 512)
    return {"value": round(flops / t_total / 1e9, 3), "unit": "GFLOP/s", "kind": "oracle",
            "cores": oracle.num_threads(),
            "sample": f"{done_rows} random query rows of {w.name}, causal={causal}"}


def run_attention(st, dev, args, with_cpu: bool) -> dict:
    """Attention forward on the tensor cores: the 4 x 16 x 4096 x 128 workload
    (and its first 64 head dimensions) with and without the causal mask; FLOP/s
    against the measured dense bf16 peak (burst, and sustained for context)."""
    w = workloads.ATTENTION_WORKLOADS["attention_4x16x4096x128_bf16"]
    q, k, v = workloads.make_attention(w, device=dev)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pj = json.load(f)
        peaks = {"burst": pj.get("bf16_tflops"), "sustained": pj.get("bf16_tflops_sustained")}
    except (OSError, ValueError):
        peaks = {"burst": 1900.0, "sustained": 1700.0, "source": "fallback"}
    steps = max(20, min(args.steps, 200))
    out = {"workload": w.name, "layout": "[batch*heads][seq][head_dim] bf16, O bf16, L fp32",
           "inputs": "Q, K, V = 192 MiB, larger than L2", "peaks_tflops": peaks, "cases": {}}
    for d in (128, 64):
        qd, kd, vd = (t if d == 128 else t[..., :64].contiguous() for t in (q, k, v))
        o = torch.empty_like(qd)
        lse = torch.empty(qd.shape[:-1], dtype=torch.float32, device=dev)
        for causal in (False, True):
            ms = _time_ms(lambda i: st.attention(qd, kd, vd, causal=causal, out=o, lse=lse), dev,
                          steps)
            fl = attention_flops(w, causal, d)
            tf = fl / ms / 1e9
            case = {"ms": round(ms, 5), "tflops": round(tf, 1),
                    "frac_of_measured_bf16_burst": round(tf / peaks["burst"], 4),
                    "frac_of_measured_bf16_sustained": round(tf / peaks["sustained"], 4),
                    "algorithmic_flops": fl}
            out["cases"][f"d{d}_{'causal' if causal else 'full'}"] = case
        del qd, kd, vd, o, lse
    if with_cpu:
        out["cpu_baseline"] = attention_oracle_rate(w, False, args.cpu_seconds / 3)
    return out


# ------------------------------------------------------------------ oracle (CPU) legs
def oracle_sample_run(rows_fraction: float, seed_offset: int = 0, target_seconds: float = 0.0):
    """Run the float64 oracle on the first rows of every step workload, the
    inputs drawn once and the whole sample repeated (up to 20 times) until
    target_seconds of oracle time are reached.  Returns (seconds, compulsory
    bytes processed, description)."""
    import oracle
    oracle.build()
    inputs, parts = [], []
    for n in SOFTMAX_STEP + [TOPK_NAME]:
        w = workloads.WORKLOADS[n]
        rows = max(1, int(round(w.rows * rows_fraction)))
        ws = w.scaled(rows=rows)
        inputs.append((ws, workloads.make(ws, device="cpu", seed=w.seed + seed_offset).double().numpy()))
        parts.append(f"{rows} rows of {n}")
    t_total, b_total, passes = 0.0, 0, 0
    while passes == 0 or (t_total < target_seconds and passes < 20):
        for ws, x in inputs:
            if ws.op == "softmax":
                t = time.perf_counter()
                oracle.softmax(x)
                t_total += time.perf_counter() - t
                b_total += softmax_bytes(ws)
            else:
                for K in TOPK_KS:
                    t = time.perf_counter()
                    oracle.topk(x, K)
                    t_total += time.perf_counter() - t
                    b_total += topk_bytes(ws, K)
        passes += 1
    return t_total, b_total, "; ".join(parts) + f"; {passes} pass(es)"


def cpu_baseline(target_seconds: float) -> dict:
    import oracle
    frac = 1.0 / 256
    t, b, desc = oracle_sample_run(frac)
    if t < target_seconds / 4:  # grow the sample toward the target CPU time
        frac = min(1.0, frac * target_seconds / max(t, 1e-3) / 2)
        t, b, desc = oracle_sample_run(frac, target_seconds=target_seconds / 2)
    out = {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
           "kind": "oracle", "seconds": round(t, 2),
           "sample": f"{desc} (fraction {frac:.5f} of each step workload's rows)"}
    # the same oracle on one host thread, on a smaller sample of the same rows
    cores = oracle.num_threads()
    frac1 = frac / max(1, cores)
    oracle.set_num_threads(1)
    try:
        t1, b1, desc1 = oracle_sample_run(frac1, target_seconds=target_seconds / 4)
    finally:
        oracle.set_num_threads(cores)
    out["single_thread"] = {"value": round(b1 / t1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                            "seconds": round(t1, 2),
                            "sample": f"{desc1} (fraction {frac1:.6f} of each step workload's rows)"}
    return out


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    frac = 1.0 / 1024
    secs = []
    for i in range(args.warmup + args.steps):
        t, b, desc = oracle_sample_run(frac, seed_offset=i)
        if i >= args.warmup:
            secs.append(t)
    t = sum(secs) / len(secs)
    value = b / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "softmax 4096x32000 f32 + softmax 8192x128256 bf16 + TopK "
                                   "256x50257 f32 K=8,64",
                       "sample": f"each step: {desc}"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle",
                             "cores": oracle.num_threads(), "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_only(args):
    """One workload, optionally on fewer rows: a small, self-contained case for
    profilers (prints a short JSON line; not a benchmark result)."""
    import softmax_topk_gb300 as st
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.only in workloads.ATTENTION_WORKLOADS:
        return run_only_attention(st, dev, args)
    w = workloads.WORKLOADS[args.only]
    if args.rows:
        w = w.scaled(rows=args.rows)
    x = workloads.make(w, device=dev)
    stream = torch.cuda.current_stream(dev)
    if w.op == "softmax":
        y = torch.empty_like(x)
        fn = lambda: st.softmax(x, out=y, path=args.path)  # noqa: E731
        nbytes = softmax_bytes(w)
    else:
        vals = torch.empty(w.rows, args.K, device=dev)
        idx = torch.empty(w.rows, args.K, dtype=torch.int32, device=dev)
        fn = lambda: st.softmax_topk(x, args.K, vals=vals, idx=idx)  # noqa: E731
        nbytes = topk_bytes(w, args.K)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / args.steps
    out = {"only": w.name, "rows": w.rows, "cols": w.cols, "path": args.path,
           "K": args.K if w.op == "topk" else None, "ms": round(ms, 5),
           "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
           "note": "inputs not rotated: L2-resident when small"}
    if args.graph:  # the same launches replayed from a CUDA graph: no host time between them
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for _ in range(args.steps):
                    fn()
        torch.cuda.synchronize(dev)
        g.replay()
        torch.cuda.synchronize(dev)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        gms = a.elapsed_time(b) / args.steps
        out["graph_ms"] = round(gms, 5)
        out["graph_gbs"] = round(nbytes / (gms * 1e-3) / 1e9, 1)
    print(json.dumps(out), flush=True)


def run_only_attention(st, dev, args):
    """One attention case for profilers: --only <attention workload>
    [--batch-heads B] [--causal]; prints a short JSON line."""
    w = workloads.ATTENTION_WORKLOADS[args.only]
    if args.rows:  # batch x heads slices
        w = w.scaled(batch=1, heads=args.rows)
    q, k, v = workloads.make_attention(w, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    fn = lambda i: st.attention(q, k, v, causal=args.causal, out=o, lse=lse)  # noqa: E731
    for i in range(args.warmup):
        fn(i)
    ms = _time_ms(fn, dev, args.steps)
    fl = attention_flops(w, args.causal)
    print(json.dumps({"only": w.name, "bh": w.bh, "causal": args.causal, "ms": round(ms, 5),
                      "tflops": round(fl / ms / 1e9, 1)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--extra", action="store_true", help="also time the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--only", default=None, help="time one workload by name (profiling case)")
    ap.add_argument("--rows", type=int, default=0, help="with --only: number of rows")
    ap.add_argument("--K", type=int, default=64, help="with --only on the TopK workload")
    ap.add_argument("--path", default="auto", help="with --only: softmax kernel family")
    ap.add_argument("--graph", action="store_true", help="with --only: also time a CUDA graph replay")
    ap.add_argument("--causal", action="store_true", help="with --only on an attention workload")
    ap.add_argument("--attention", action="store_true",
                    help="time only the attention forward leg (one JSON line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.only:
        run_only(args)
    elif args.attention:
        import softmax_topk_gb300 as st
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps({"attention": run_attention(st, dev, args, not args.no_cpu_baseline)}),
              flush=True)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

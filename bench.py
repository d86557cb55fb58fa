#!/usr/bin/env python
"""Benchmark of the Prof-K top-k engine on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one full selection (sample -> threshold -> filter -> fallback check
-> exact refine and sort) over one synthetic input resident in HBM.  The
default workload is the single huge row: N = 2^28 fp32 Pareto(1.5) values with
random sign, k = 1024, eps = 1e-6.  Inputs are larger than L2 (1 GiB), so no
flush is needed between steps.  Prints one JSON line (rank 0).

With N > 1 GPUs (torchrun) every rank runs an independent replica of the same
selection; there is no data-path collective.  `--impl reference` times the CPU
oracle (plain nth_element + sort, one host core) on the same workload, or on a
prefix of it when the full one would not finish within a few minutes.
"""
from __future__ import annotations

import argparse
import ctypes
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "single_row_2p28_pareto15_k1024"
SECONDARY_WORKLOAD = "batchtopk_4096x65536_relu_bf16_k131072"
SECONDARY_MIN_STEPS = 1000
NOMINAL_READ_GBS = 8000.0  # GB300 HBM3e nominal rate: the one-read roofline the fractions use
CLOCK_SOAK_S = 1.5
ORACLE_SAMPLE_ELEMS = 1 << 25
RELAXED_RECALL = 0.95
REFERENCE_BUDGET_S = 240.0   # the reference arm's whole run: full workload when it fits, else a prefix
CONFIG_MISS_CALLS = 10000


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true", help="skip the BatchTopK side measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-miss-rate", action="store_true", help="skip the measured miss rate against eps")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the side measurements (forced miss, unsorted, relaxed recall, autotune); for profiling")
    ap.add_argument("--miss-calls", type=int, default=CONFIG_MISS_CALLS,
                    help="seeded calls per workload and rule for the miss rate on the tied rows and BatchTopK")
    ap.add_argument("--scale-down", type=int, default=0,
                    help="divide the workload by 2^s (row length, or rows for global mode); for profiling")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--sweep", action="store_true",
                    help="the paper's N x K sweep: Prof-K against torch.topk on the same GPU (one JSON line)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms, device, world):
    """The slowest rank's time: every rank runs its own replica, so the job
    takes as long as its slowest one (all-reduce MAX; no-op with one rank)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gelems(n_elems_per_rank, world, ms_step):
    """Elements selected by all ranks per second (G elem/s), at the slowest rank's step time."""
    return n_elems_per_rank * world / (ms_step * 1e-3) / 1e9


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    return 6800.0, "fallback (6.8 TB/s)"


def workload(name, scale_down=0):
    from top_selection_prof_gb300 import workloads
    if name not in workloads.WORKLOADS:
        raise SystemExit("unknown workload %r; choose from %s" % (name, sorted(workloads.WORKLOADS)))
    cfg = dict(workloads.WORKLOADS[name])
    if scale_down:
        if cfg["mode"] == "global" or cfg["rows"] > 1:
            cfg["rows"] = max(1, cfg["rows"] >> scale_down)
        else:
            cfg["n"] = max(cfg["k"] * 4, cfg["n"] >> scale_down)
        cfg["k"] = min(cfg["k"], cfg["n"] * (cfg["rows"] if cfg["mode"] == "global" else 1))
    return cfg


def make_input(cfg, seed):
    from top_selection_prof_gb300 import workloads
    return workloads.make(cfg["kind"], cfg["rows"], cfg["n"], seed)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
            self.t0 = time.time()
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as fh:
            lines = fh.readlines()
        os.unlink(self.file.name)
        return summarize_clocks(lines)


def summarize_clocks(lines):
    """Median SM clock, the largest max clock and power, and every throttle reason seen Active, from the
    nvidia-smi CSV rows of ClockSampler.FIELDS (noheader, nounits); rows that do not parse are skipped."""
    sm, smax, power, reasons = [], [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        r = ln.strip().split(", ")
        if len(r) < 9:
            continue
        try:
            sm.append(float(r[1]))
            smax.append(float(r[2]))
            power.append(float(r[3]))
        except ValueError:
            continue
        for nm, val in zip(names, r[5:9]):
            if val.strip().lower() == "active":
                reasons.add(nm)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# ncu traffic record for the dominant kernel (stale once the kernel changes)
# ---------------------------------------------------------------------------
def filter_source_sha():
    h = hashlib.sha256()
    for f in ("kernels_filter.cu", "filter_core.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "top_selection_prof_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name, n_elems):
    """dram bytes per filter launch from the committed ncu summary, scaled to this workload."""
    path = os.path.join(ROOT, "profiles", "filter_ring_kernel_ncu.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    if not sha or sha.group(1) != filter_source_sha():
        return None
    m = re.search(r"dram_bytes_per_element\[%s\]:\s*([0-9.eE+-]+)" % re.escape(workload_name), text)
    if not m:
        return None
    return float(m.group(1)) * n_elems


# ---------------------------------------------------------------------------
# the CPU oracle, as it stands (baseline and reference arm)
# ---------------------------------------------------------------------------
def cpu_model():
    """The host CPU's model name (lscpu), else what the platform module reports."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_prefix(cfg, x):
    """A bounded sample of the workload for the CPU oracle: a prefix of the selection."""
    if cfg["mode"] == "global":
        flat = x.reshape(-1)[:ORACLE_SAMPLE_ELEMS]
        return flat[None, :], True, "first %d of the %d flattened elements, global k=%d" % (
            flat.size, x.size, min(cfg["k"], flat.size))
    if cfg["rows"] == 1:
        row = x[:, :ORACLE_SAMPLE_ELEMS]
        return row, False, "first %d of %d elements of the row, k=%d" % (row.shape[1], x.shape[1], cfg["k"])
    rows = max(1, ORACLE_SAMPLE_ELEMS // cfg["n"])
    return x[:rows], False, "%d of %d rows of %d, k=%d per row" % (rows, cfg["rows"], cfg["n"], cfg["k"])


def time_oracle(cfg, x, steps, warmup, budget_s=None, parallel=False):
    """The CPU oracle timed on the host cores (single thread as it stands, or
    the all-cores variant), on the full workload -- or on a prefix of it when
    `steps` calls of the full one would exceed `budget_s` seconds."""
    from oracle import plain
    glob = cfg["mode"] == "global"
    fn = plain.topk_parallel if parallel else plain.topk
    threads = os.cpu_count() or 1
    sample, desc = x, "the full workload (%s, k=%d%s)" % (
        "x".join(str(d) for d in x.shape), cfg["k"], ", global" if glob else " per row")
    t0 = time.perf_counter()
    fn(sample, cfg["k"], global_=glob)
    first = time.perf_counter() - t0
    same = True
    if budget_s is not None and first * (steps + warmup) > budget_s:
        sample, glob, desc = oracle_prefix(cfg, x)
        same = False
    k = min(cfg["k"], sample.size if glob else sample.shape[1])
    for _ in range(warmup if not same else max(0, warmup - 1)):
        fn(sample, k, global_=glob)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        fn(sample, k, global_=glob)
        times.append(time.perf_counter() - t0)
    per_step = statistics.mean(times)
    return {"value": sample.size / per_step / 1e9, "unit": "G elem/s", "cores": threads if parallel else 1,
            "kind": "oracle_parallel" if parallel else "oracle", "sample": desc, "same_config": same,
            "cpu_model": cpu_model(), "host_cores": threads, "seconds_per_step": per_step}


# ---------------------------------------------------------------------------
# our engine
# ---------------------------------------------------------------------------


def tk_plan(cfg):
    """The exact tail bound P[R < k] + P[R > M] of the workload's own plan."""
    import top_selection_prof_gb300 as tk
    n = cfg["n"] * (cfg["rows"] if cfg.get("mode") == "global" else 1)
    pl = tk.plan(n, cfg["k"], cfg["eps"])
    return {"S": int(pl["S"]), "t": int(pl["t"]), "M": int(pl["M"]),
            "p_recall_fail": float(pl["p_recall_fail"]), "p_overflow": float(pl["p_overflow"])}


def binomial_ci95(x, n):
    """Clopper-Pearson 95 % interval for x successes in n trials."""
    from scipy import stats
    lo = 0.0 if x == 0 else float(stats.beta.ppf(0.025, x, n - x + 1))
    hi = 1.0 if x == n else float(stats.beta.ppf(0.975, x + 1, n - x))
    return [lo, hi]


def measure_miss_rate(runs=300):
    """Measured fallback frequency against the exact tail bound of the (S, t, M)
    in use: a 2^20 uniform row, k = 100, eps = 0.2, S = 2048 draws, so that
    misses are frequent enough to count (the same case as the stage tests)."""
    import torch
    import top_selection_prof_gb300 as tk
    from top_selection_prof_gb300 import workloads
    n, k, eps, S = 1 << 20, 100, 0.2, 2048
    xd = torch.from_numpy(workloads.make("uniform", 1, n, 5)).cuda()
    misses = 0
    for c in range(runs):
        _, _, st = tk.select_ex(xd, k, eps=eps, counter=c, s_min=S, s_max=S)
        misses += int(st["misses"])
    pl = tk.plan(n, k, eps, s_min=S, s_max=S)
    bound = float(pl["p_recall_fail"] + pl["p_overflow"])
    return {"n": n, "k": k, "eps": eps, "S": int(pl["S"]), "t": int(pl["t"]), "M": int(pl["M"]), "calls": runs,
            "misses": misses, "measured": round(misses / runs, 4), "exact_tail_bound": round(bound, 4),
            "ci95": [round(v, 4) for v in binomial_ci95(misses, runs)]}


MISS_RATE_WORKLOADS = ["single_row_2p26_ties1000_k10000", "single_row_2p26_ties1000_sorted_k10000",
                       "batchtopk_4096x65536_relu_bf16_k131072"]


def measure_config_miss_rates(calls, seed=0):
    """Theorem 3 on the workloads themselves: `calls` seeded calls (Philox
    counter = call number) per workload and parameter rule, each reporting
    whether its selection took the fallback; the count, a binomial 95 %
    interval and the exact tail bound P[R < k] + P[R > M] of the plan."""
    import numpy as np
    import torch
    import top_selection_prof_gb300 as tk
    out = []
    for name in MISS_RATE_WORKLOADS:
        cfg = workload(name)
        x = make_input(cfg, seed)
        bf16 = x.dtype == np.uint16
        xd = torch.from_numpy(x.view(np.int16) if bf16 else x).cuda()
        if bf16:
            xd = xd.view(torch.bfloat16)
        del x
        glob = cfg["mode"] == "global"
        n_sel = cfg["n"] * (cfg["rows"] if glob else 1)
        for rule_name, rule in (("exact", tk.TOPK_RULE_EXACT), ("alg1", tk.TOPK_RULE_ALG1)):
            pl = tk.plan(n_sel, cfg["k"], cfg["eps"], rule=rule)
            misses = 0
            t0 = time.time()
            for c in range(calls):
                _, _, st = tk.select_ex(xd, cfg["k"], eps=cfg["eps"], global_=glob, counter=c, rule=rule)
                misses += int(st["misses"])
            bound = float(pl["p_recall_fail"] + pl["p_overflow"])
            out.append({"workload": name, "rule": rule_name, "eps": cfg["eps"], "S": int(pl["S"]),
                        "t": int(pl["t"]), "M": int(pl["M"]), "calls": calls, "misses": misses,
                        "rate": misses / calls, "ci95": binomial_ci95(misses, calls),
                        "exact_tail_bound": bound, "seconds": round(time.time() - t0, 1)})
        del xd
        torch.cuda.empty_cache()
    return out


def run_ours(cfg, name, x_host, steps, warmup, world, rank, with_clocks=True, with_e2e=True, extras=True):
    import numpy as np
    import torch
    import torch.distributed as dist
    import top_selection_prof_gb300 as tk
    from top_selection_prof_gb300 import _lib

    dev = torch.device("cuda", torch.cuda.current_device())
    bf16 = x_host.dtype == np.uint16
    x_cpu = torch.from_numpy(x_host.view(np.int16) if bf16 else x_host)
    x_pin = x_cpu.pin_memory()
    xd = x_pin.to(dev, non_blocking=True)
    if bf16:
        xd = xd.view(torch.bfloat16)
        x_pin_t = x_pin.view(torch.bfloat16)
    else:
        x_pin_t = x_pin
    torch.cuda.synchronize()
    rows, n, k, eps = cfg["rows"], cfg["n"], cfg["k"], cfg["eps"]
    glob = cfg["mode"] == "global"
    n_elems = rows * n
    bytes_per_elem = 2 if bf16 else 4
    out_shape = (k,) if glob else (rows, k)
    vals = torch.empty(out_shape, dtype=xd.dtype, device=dev)
    idx = torch.empty(out_shape, dtype=torch.int64, device=dev)

    # one call with stats: path, (S, t, M), R
    _, _, st = tk.select_ex(xd, k, eps=eps, global_=glob)
    path = st["path_name"]

    lib = _lib.get()
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    code = _lib.TOPK_BF16 if bf16 else _lib.TOPK_F32
    opt = tk.options()

    def call(events=None):
        for j in range(6):
            opt.events[j] = events[j] if events is not None else None
        rc = lib.topk_select_ex(xd.data_ptr(), code, rows, n, k, 1, eps, vals.data_ptr(), idx.data_ptr(), sp,
                                int(glob), ctypes.byref(opt), None)
        if rc != 0:
            raise RuntimeError("topk_select_ex failed: %d" % rc)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device()) if with_clocks else None
    if clocks:
        clocks.start()
        t_end = time.time() + CLOCK_SOAK_S          # untimed soak so the clock record covers load
        while time.time() < t_end:
            for _ in range(20):
                call()
            torch.cuda.synchronize()

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        call()
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_total = start.elapsed_time(end)
    clock_info = clocks.stop() if clocks else None

    # Profiled pass: the same K steps again with CUDA events recorded on the
    # launching stream at every stage boundary (recording events between the
    # kernels stops them from overlapping their launches, so this pass is kept
    # out of the throughput number above).
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    for evs in stage_ev:
        for e in evs:
            e.record(stream)
    handles = [[ctypes.c_void_p(e.cuda_event).value for e in evs] for evs in stage_ev]
    torch.cuda.synchronize()
    for s_ in range(steps):
        call(handles[s_] if path == "profk" else None)
    torch.cuda.synchronize()

    # The miss path: calls whose every selection takes the fallback (a miss
    # is injected on the host), timed alone.
    forced_miss_ms = None
    if path == "profk" and extras:
        opt.force_miss = 1
        call()
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(3):
            call()
        f1.record(stream)
        torch.cuda.synchronize()
        forced_miss_ms = round(f0.elapsed_time(f1) / 3, 4)
        opt.force_miss = 0

    # BatchTopK needs only the set of winners: the same selection with the
    # sort left out (the unsorted option), timed alone
    unsorted_ms = None
    if glob and path == "profk" and k >= 8192 and extras:
        opt.unsorted = 1
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        u0.record(stream)
        for _ in range(steps):
            call()
        u1.record(stream)
        torch.cuda.synchronize()
        unsorted_ms = round(u0.elapsed_time(u1) / steps, 4)
        opt.unsorted = 0

    def time_steps(nsteps):
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(nsteps):
            call()
        a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / nsteps

    # Relaxed recall (the paper's accuracy-speed trade-off): the same
    # selection with a recall target of 0.95, and the recall it returned
    relaxed = None
    if path == "profk" and world == 1 and extras:
        opt.recall = RELAXED_RECALL
        r_ms = time_steps(steps)
        _, i_r, st_r = tk.select_ex(xd, k, eps=eps, global_=glob, recall=RELAXED_RECALL)
        real = int((i_r >= 0).sum().item())
        relaxed = {"recall_target": RELAXED_RECALL, "ms_per_step": round(r_ms, 4), "S_t_M": [st_r["S"], st_r["t"], st_r["M"]],
                   "R": st_r["R"], "returned_fraction_of_k": round(real / i_r.numel(), 6)}
        opt.recall = 0.0

    # The cost model measured on this device (topk_autotune) and the same
    # selection with the sample size it gives (cost_ratio = 0)
    autotuned = None
    if path == "profk" and world == 1 and extras:
        tn = _lib.TopkTuning()
        rc = lib.topk_autotune(0, sp, ctypes.byref(tn))
        if rc == 0:
            opt.cost_ratio = 0.0
            a_ms = time_steps(steps)
            _, _, st_a = tk.select_ex(xd, k, eps=eps, global_=glob, cost_ratio=0.0)
            autotuned = {"tau_a_ns": tn.tau_a_ns, "tau_b_ns": tn.tau_b_ns, "cost_ratio": tn.cost_ratio,
                         "crossover_n_at_k1024": tn.crossover_n, "ms_per_step": round(a_ms, 4),
                         "S_t_M": [st_a["S"], st_a["t"], st_a["M"]], "path": st_a["path_name"]}
            opt.cost_ratio = 1.0

    ms_total = max_over_ranks(ms_total, dev, world)
    ms_step = ms_total / steps
    value = whole_job_gelems(n_elems, world, ms_step)

    stages = None
    filt_ms = None
    if path == "profk":
        names = ["sample", "threshold", "filter", "fallback_check", "refine_sort"]
        # stage boundaries come from the profiled pass
        per = {nm: [] for nm in names}
        for evs in stage_ev:
            for j, nm in enumerate(names):
                per[nm].append(evs[j].elapsed_time(evs[j + 1]))
        stages = {nm + "_us": round(1e3 * statistics.mean(v), 2) for nm, v in per.items()}
        filt_ms = statistics.mean(per["filter"])

    peak, peak_src = load_peaks()
    roofline = None
    if filt_ms:
        alg_bytes = n_elems * bytes_per_elem + st["R"] * 8
        achieved = alg_bytes / (filt_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "traffic": recorded_traffic(name, n_elems),
                    # (one selection over 16-byte aligned data: the TMA-ring filter)
                    "kernel": "filter_ring_kernel" if (glob or rows == 1) else "filter_kernel",
                    "algorithmic_bytes_per_launch": alg_bytes,
                    "peak_source": peak_src}

    e2e = None
    if with_e2e:
        e2e_steps = max(3, min(steps, 10))
        vals_h = torch.empty(out_shape, dtype=xd.dtype).pin_memory()
        idx_h = torch.empty(out_shape, dtype=torch.int64).pin_memory()
        for _ in range(2):
            xd.copy_(x_pin_t, non_blocking=True)
            call()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        e0.record(stream)
        for _ in range(e2e_steps):
            xd.copy_(x_pin_t, non_blocking=True)
            v2, i2 = (tk.select_global(xd, k, eps=eps) if glob else tk.select(xd, k, eps=eps))
            vals_h.copy_(v2, non_blocking=True)
            idx_h.copy_(i2, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev, world)
        e2e = {"value": round(whole_job_gelems(n_elems, world, ms_e2e), 3), "unit": "G elem/s",
               "h2d_bytes_per_step": n_elems * bytes_per_elem,
               "d2h_bytes_per_step": (k if glob else rows * k) * (bytes_per_elem + 8),
               "ms_per_step": round(ms_e2e, 4), "steps": e2e_steps}

    return {
        "value": value, "ms_per_step": ms_step, "path": path, "stats": st, "stages": stages,
        "roofline": roofline, "e2e": e2e, "clocks": clock_info, "forced_miss_ms_per_step": forced_miss_ms,
        "unsorted_ms_per_step": unsorted_ms, "relaxed_recall": relaxed, "autotuned": autotuned,
        # the library reports the kernels each call launched (sample and
        # threshold, filter, fallback when it runs as its own grid, refinement,
        # bin sort for large k; the direct path's one kernel)
        "gpu_launches": int(st["launches"]) * steps,
        "hbm_gbs_whole_step": n_elems * bytes_per_elem / (ms_step * 1e-3) / 1e9,
    }


# ---------------------------------------------------------------------------
# the paper's sweep (section 5, Figure 2): N x K x distribution, against
# torch.topk timed on the same GPU (context; torch.topk is not on our path)
# ---------------------------------------------------------------------------
SWEEP_NS = [1 << p for p in (22, 24, 26, 28, 30)]
SWEEP_KS = [32, 1024, 32768, 131072]
SWEEP_DISTS = ["uniform", "normal", "pareto15"]
L2_BYTES = 126 << 20


def sweep_input(dist, n, gen, dev):
    import torch
    if dist == "uniform":
        return torch.rand(n, generator=gen, device=dev)
    if dist == "normal":
        return torch.randn(n, generator=gen, device=dev)
    # Pareto(1.5), x_m = 1, random sign: +-U^(-2/3), U in (0, 1]
    u = 1.0 - torch.rand(n, generator=gen, device=dev)
    sign = torch.where(torch.rand(n, generator=gen, device=dev) < 0.5, -1.0, 1.0)
    return sign * u.pow(-2.0 / 3.0)


def time_call(fn, reps, flush):
    """Median device time of one call (CUDA events on the current stream), L2 flushed first when given."""
    import torch
    for _ in range(2):
        fn()
    times = []
    for _ in range(reps):
        if flush is not None:
            flush.add_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(times)


SWEEP_ORACLE_MAX_N = 1 << 24


def run_sweep(args):
    import numpy
    import torch
    import top_selection_prof_gb300 as tk
    torch.cuda.set_device(0)
    tk._lib.get()   # fails loudly if the engine is not built
    dev = torch.device("cuda", 0)
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed)
    reps = max(3, min(args.steps, 20))
    points = []
    for n in SWEEP_NS:
        for dist in SWEEP_DISTS:
            x = sweep_input(dist, n, gen, dev)
            fl = flush if n * 4 < 2 * L2_BYTES else None
            for k in SWEEP_KS:
                if k > n // 8:
                    continue
                ours_us = time_call(lambda: tk.select(x, k, eps=1e-3), reps, fl)
                torch_us = time_call(lambda: torch.topk(x, k, sorted=True), reps, fl)
                v, i = tk.select(x, k, eps=1e-3)
                tv, _ = torch.topk(x, k, sorted=True)
                _, _, st = tk.select_ex(x, k, eps=1e-3)
                point = {"n": n, "k": k, "dist": dist, "path": st["path_name"],
                         "ours_us": round(ours_us, 1), "torch_topk_us": round(torch_us, 1),
                         "speedup": round(torch_us / ours_us, 2),
                         "ours_gbs": round(n * 4 / (ours_us * 1e-6) / 1e9, 1),
                         "values_equal_torch": bool(torch.equal(v, tv)),
                         # (torch.topk does not fix the order of equal values: indices are
                         # checked by what they point at, and against the oracle where it is cheap)
                         "indices_hold_values": bool(torch.equal(x[i], v))}
                if n <= SWEEP_ORACLE_MAX_N:
                    from oracle import plain
                    xh = x.cpu().numpy()
                    ov, oi = plain.topk(xh[None, :], k)
                    point["oracle_exact"] = bool(numpy.array_equal(i.cpu().numpy(), oi[0]) and
                                                 numpy.array_equal(v.cpu().numpy().view(numpy.uint32),
                                                                   ov[0].view(numpy.uint32)))
                points.append(point)
            del x
    sp = [p["speedup"] for p in points]
    geo = float(math.exp(sum(math.log(v) for v in sp) / len(sp)))
    line = {"sweep": "Prof-K (topk_select, eps=1e-3, f32, one row) vs torch.topk(sorted=True), same GPU",
            "gpu": torch.cuda.get_device_name(0), "torch": torch.__version__, "reps": reps,
            "l2": "flushed before each call when the input is below 2x L2", "data": "synthetic (torch generator)",
            "points": points,
            "summary": {"speedup_min": min(sp), "speedup_max": max(sp), "speedup_geomean": round(geo, 2),
                        "all_values_equal": all(p["values_equal_torch"] for p in points),
                        "all_indices_hold_values": all(p["indices_hold_values"] for p in points),
                        "oracle_points": sum("oracle_exact" in p for p in points),
                        "all_oracle_exact": all(p.get("oracle_exact", True) for p in points)}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    world, rank, local = dist_env()
    cfg = workload(args.workload, args.scale_down)
    if args.sweep:
        return run_sweep(args) if rank == 0 else 0

    if args.impl == "reference":
        if rank != 0:
            return 0
        x = make_input(cfg, args.seed)
        r = time_oracle(cfg, x, args.steps, args.warmup, budget_s=REFERENCE_BUDGET_S)
        line = {"metric": "top-k G elem/s and achieved HBM GB/s vs ~8 TB/s peak, 1xGB300", "impl": "reference",
                "value": round(r["value"], 4), "unit": "G elem/s", "n_gpus": 0, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(r["seconds_per_step"] * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype":
                    "bf16" if cfg["kind"].endswith("_bf16") else "f32",
                "data": "synthetic (seeded numpy)",
                "config": {"workload": args.workload, "rows": cfg["rows"], "n": cfg["n"], "k": cfg["k"],
                           "eps": cfg["eps"], "mode": cfg["mode"]},
                "cpu_baseline": {k2: r[k2] for k2 in ("value", "unit", "cores", "kind", "sample", "same_config",
                                                      "cpu_model", "host_cores")},
                "e2e": {"value": round(r["value"], 4), "unit": "G elem/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import top_selection_prof_gb300 as tk
    tk._lib.get()   # fails loudly if the engine is not built

    x = make_input(cfg, args.seed + rank)
    res = run_ours(cfg, args.workload, x, args.steps, args.warmup, world, rank,
                   with_clocks=not args.no_clocks, with_e2e=not args.no_e2e, extras=not args.no_extras)

    secondary = None
    if not args.no_secondary and args.workload != SECONDARY_WORKLOAD:
        c2 = workload(SECONDARY_WORKLOAD, args.scale_down)
        del x
        x2 = make_input(c2, args.seed + rank)
        # (at least 1000 steps: a miss, about one call in 1/eps = 1000, costs
        # ~1.3 ms, so a short window that happens to hold one overstates the
        # expected cost of eps x 1.3 ms per call many times over)
        r2 = run_ours(c2, SECONDARY_WORKLOAD, x2, max(args.steps, SECONDARY_MIN_STEPS), args.warmup, world, rank,
                      with_clocks=False, with_e2e=False, extras=not args.no_extras)
        secondary = {"workload": SECONDARY_WORKLOAD, "value": round(r2["value"], 3), "unit": "G elem/s",
                     "ms_per_step": round(r2["ms_per_step"], 4), "path": r2["path"],
                     "hbm_gbs_whole_step": round(r2["hbm_gbs_whole_step"], 1),
                     "frac_of_8tbs_whole_step": round(r2["hbm_gbs_whole_step"] / NOMINAL_READ_GBS, 4),
                     "roofline": r2["roofline"], "stages": r2["stages"], "R": r2["stats"]["R"],
                     "forced_miss_ms_per_step": r2["forced_miss_ms_per_step"],
                     "unsorted_ms_per_step": r2["unsorted_ms_per_step"],
                     "relaxed_recall": r2["relaxed_recall"], "autotuned": r2["autotuned"],
                     "steps": max(args.steps, SECONDARY_MIN_STEPS),
                     "S_t_M": [r2["stats"]["S"], r2["stats"]["t"], r2["stats"]["M"]]}
        x = None

    cpu = cpu_par = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        xb = make_input(cfg, args.seed) if x is None else x
        keys = ("value", "unit", "cores", "kind", "sample", "same_config", "cpu_model", "host_cores")
        cb = time_oracle(cfg, xb, steps=2, warmup=0, budget_s=40.0)
        cpu = {k2: cb[k2] for k2 in keys}
        cp = time_oracle(cfg, xb, steps=3, warmup=1, budget_s=40.0, parallel=True)
        cpu_par = {k2: cp[k2] for k2 in keys}
        del xb

    if rank == 0:
        st = res["stats"]
        line = {
            "metric": "top-k G elem/s and achieved HBM GB/s vs ~8 TB/s peak, 1xGB300",
            "value": round(res["value"], 3), "unit": "G elem/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if cfg["kind"].endswith("_bf16") else "f32",
            "data": "synthetic (seeded numpy: %s)" % cfg["kind"],
            "config": {"workload": args.workload + ("/2^%d" % args.scale_down if args.scale_down else ""),
                       "rows": cfg["rows"], "n": cfg["n"], "k": cfg["k"],
                       "eps": cfg["eps"], "mode": cfg["mode"], "path": res["path"],
                       "S": st["S"], "t": st["t"], "M": st["M"], "R": st["R"],
                       "l2": "inputs larger than L2 (no flush)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "hbm_gbs_whole_step": round(res["hbm_gbs_whole_step"], 1),
            "frac_of_8tbs_whole_step": round(res["hbm_gbs_whole_step"] / NOMINAL_READ_GBS, 4),
            "roofline": res["roofline"], "stages": res["stages"], "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_par, "e2e": res["e2e"],
            "gpu_launches": res["gpu_launches"], "clocks": res["clocks"], "secondary": secondary,
            "forced_miss_ms_per_step": res["forced_miss_ms_per_step"],
            "relaxed_recall": res["relaxed_recall"], "autotuned": res["autotuned"],
        }
        if cfg.get("eps", 0) > 0 and not args.no_miss_rate:
            # the workload's own bound, and a measured rate where misses are countable
            pl = tk_plan(cfg)
            line["miss_rate"] = {"workload_bound": pl, "measured_case": measure_miss_rate()}
            if world == 1 and args.miss_calls > 0:
                line["miss_rate"]["configs"] = measure_config_miss_rates(args.miss_calls)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

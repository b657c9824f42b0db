#!/usr/bin/env python3
"""Benchmark: routed MoE EP dispatch + combine on one GB300 (W ranks in HBM).

One step = one dispatch (routing/slot kernel + fused a1->batched row mover)
and one combine (weighted gather-reduce) over the whole batch of all W
simulated ranks, with identity experts (expert_out = b_a1). Prints one JSON
line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 3] [--impl ours|reference]

With N > 1 (under torch.distributed.run) every rank runs an independent
replica of the workload: the path has no data exchange between GPUs here, so
nothing is sharded and no collective touches the data; the ranks only meet at
the barriers around the timed region and in the max-over-ranks of its time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from combine_ep_route_gb300 import workloads as wl  # noqa: E402

METRIC = "dispatch+combine tokens/s and effective HBM GB/s (fraction of peak), 1 GB300"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="fused", choices=["fused", "sendbuf"])
    ap.add_argument("--combine", default="fused", choices=["fused", "two_stage"],
                    help="two_stage: the page's own finalize rounding (comparison only)")
    ap.add_argument("--tokens-per-rank", type=int, default=None,
                    help="override T of the workload (a smaller case for profiling)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E of the workload (a smaller case for profiling)")
    ap.add_argument("--hidden", type=int, default=None,
                    help="override h of the workload (a smaller case for profiling)")
    ap.add_argument("--eager", dest="graph", action="store_false",
                    help="launch every kernel from the host each step instead of replaying one "
                         "captured CUDA graph of dispatch + combine (the default)")
    ap.add_argument("--route", default="a2a", choices=["a2a", "agrs"],
                    help="agrs: time the all-gather / reduce-scatter route instead (auxiliary line)")
    ap.add_argument("--top-k", type=int, default=None, help="override top_k of the workload")
    ap.add_argument("--x-dtype", default="bf16", choices=["bf16", "fp8", "fp4x2"],
                    help="dispatched rows as opaque fp8 (h bytes) or packed fp4 (h/2 bytes) with "
                         "their scales as an extra payload (fp32 per 128 values, or one byte per "
                         "16 values); the combine reduces a separate bf16 expert-output buffer")
    ap.add_argument("--weight-on-input", action="store_true",
                    help="apply_router_weight_on_input (needs --top-k 1)")
    ap.add_argument("--ragged", action="store_true",
                    help="tokens per rank drawn uniformly in [T/2, T] (seeded)")
    ap.add_argument("--zero-pad", action="store_true",
                    help="also zero every batched-expert row past the expert's count, as the page does")
    ap.add_argument("--out-dtype", default="bf16", choices=["bf16", "f32"],
                    help="combine output type (f32: the fp32-output variant; an auxiliary line)")
    ap.add_argument("--hot", action="store_true",
                    help="no L2 flush between timed steps: the L2-resident figure of a small "
                         "workload, reported beside the flushed one, never as the headline")
    ap.add_argument("--probe", default=None, choices=["ceilings"],
                    help="ceilings: auxiliary line with the device's read-only, write-only and copy "
                         "bandwidth (1 GiB buffers, torch's own kernels) and the host link's copy "
                         "rates (pinned 118 MiB buffers); changes no GPU setting")
    ap.add_argument("--option", action="append", default=[], metavar="NAME=VALUE",
                    help="set a library option (EP_OPT_<NAME>) on the context before timing, "
                         "e.g. --option PDL=1; named in the line's config")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def workload_counts(x: wl.Workload):
    """Exact counts of the algorithmic byte formula from the drawn inputs."""
    ids = x.topk_ids
    W, T, K = ids.shape
    live = np.arange(T)[None, :] < x.num_tokens[:, None]
    kept = (ids >= 0) & live[:, :, None]
    n_pairs = int(kept.sum())
    n_tok_routed = int(kept.any(axis=2).sum())
    n_tok = int(x.num_tokens.sum())
    return n_pairs, n_tok_routed, n_tok


def algorithmic_bytes(x: wl.Workload, out_bytes_per_elem: int = 2, x_row_bytes: int = 0,
                      extra_bytes: int = -1):
    """(dispatch bytes, combine bytes): each routed token row (+ extras) read
    once and written once per pair; each pair row read once and each output row
    written once. Metadata (ids, weights, maps; < 1 %) is not counted. The
    dispatched row may be narrower than the bf16 expert output (quantised rows)."""
    s = x.spec
    n_pairs, n_tok_routed, n_tok = workload_counts(x)
    bx = x_row_bytes or 2 * s.h
    bp = sum(x.extra_row_bytes) if extra_bytes < 0 else extra_bytes
    disp = (bx + bp) * (n_tok_routed + n_pairs)
    comb = 2 * s.h * n_pairs + out_bytes_per_elem * s.h * n_tok
    return disp, comb


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# translation unit of each timed kernel; its hash also covers every shared header
# and api.cu, which sets the kernel's launch shape
KERNEL_TU = {"dispatch_fused": "move.cu", "dispatch_small": "dispatch_small.cu",
             "move_fused": "move.cu", "pack": "move.cu",
             "exchange": "move.cu", "deliver": "move.cu", "route": "route.cu",
             "combine": "combine.cu", "combine_two_stage": "combine.cu", "zero_pad": "combine.cu",
             "agrs_gather": "agrs.cu", "agrs_experts": "agrs.cu", "agrs_reduce": "agrs.cu"}


def code_tokens(src: str) -> str:
    """C/C++/CUDA source with comments removed and whitespace runs collapsed to
    one space (string and character literals kept as written), so that edits
    to comments or layout leave the kernel's hash unchanged."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code (not the comments) of a kernel's translation unit, the
    shared headers and api.cu: the key of the committed DRAM figures."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "combine_ep_route_gb300", "csrc")
    names = sorted(n for n in os.listdir(csrc)
                   if n.endswith(".cuh") or n in (KERNEL_TU[kernel], "api.cu"))
    for n in names:
        with open(os.path.join(csrc, n), encoding="utf-8") as f:
            h.update(n.encode() + b"\0" + code_tokens(f.read()).encode() + b"\0")
    return h.hexdigest()[:16]


def traffic_config(args, s, variant=None):
    """The workload key of the committed DRAM figures: the named workload's
    number when this run measures that workload unchanged, else None (an
    override or a variant moves other bytes than the captured ones)."""
    if variant or s.name != wl.spec(args.config).name:
        return None
    return args.config


def traffic_for(kernel: str, cfg):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources and the same workload (else None)."""
    if cfg is None or not os.path.exists(TRAFFIC_FILE):
        return None
    src = kernel_source_hash(kernel)
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
            if (parts.get("kernel") == kernel and parts.get("config") == str(cfg)
                    and parts.get("source") == src and "bytes_per_launch" in parts):
                return float(parts["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = f"/tmp/ep_clocks_{os.getpid()}.csv"

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return self
        # start the timed region only once the sampler is producing lines
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                c = [v.strip() for v in line.split(",")]
                if len(c) < 9:
                    continue
                try:
                    sm.append(float(c[1]))
                    mx = float(c[2])
                except ValueError:
                    continue
                for n, v in zip(names, c[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


class NvmlSampler:
    """SM clock, power and clock-event (throttle) reasons read through NVML's
    read-only queries every ~0.5 ms on a background thread, so that even a timed
    region of a few milliseconds holds several samples. ``mark()`` opens and
    closes named windows (the timed passes); ``summary(name)`` describes the
    samples inside one. Nothing here changes any GPU setting. Falls back to
    None when the NVML library cannot be loaded."""
    # clock-event reason bits of NVML's public API
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int, interval_s: float = 0.0005):
        import ctypes
        import threading
        self.ok = False
        self.samples = []          # (t, sm_mhz, reasons_mask, power_mw)
        self.windows = {}
        self.interval = interval_s
        self._stop = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            idx = cuda_index
            parts = [p.strip() for p in vis.split(",") if p.strip()]
            if parts and all(p.isdigit() for p in parts) and cuda_index < len(parts):
                idx = int(parts[cuda_index])
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) != 0:
                return
            self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx))   # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
            self._lib, self._h, self._ct = lib, h, ctypes
            self.ok = True
        except Exception:
            return
        self._thread = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        ct, lib, h = self._ct, self._lib, self._h
        clk, rs, pw = ct.c_uint(), ct.c_ulonglong(), ct.c_uint()
        while not self._stop.is_set():
            t = time.perf_counter()
            a = lib.nvmlDeviceGetClockInfo(h, ct.c_int(1), ct.byref(clk))
            b = self._reasons_fn(h, ct.byref(rs))
            c = lib.nvmlDeviceGetPowerUsage(h, ct.byref(pw))
            if a == 0:
                self.samples.append((t, float(clk.value), int(rs.value) if b == 0 else None,
                                     int(pw.value) if c == 0 else None))
            time.sleep(self.interval)

    def __enter__(self):
        if self.ok:
            self._thread.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 2.0:
                time.sleep(0.001)
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._thread.join(timeout=2)

    def mark(self, name: str, start: bool):
        w = self.windows.setdefault(name, [None, None])
        w[0 if start else 1] = time.perf_counter()

    def summary(self, name: str):
        if not self.ok:
            return None
        t0, t1 = self.windows.get(name, (None, None))
        sel = [x for x in list(self.samples) if t0 is not None and t1 is not None and t0 <= x[0] <= t1]
        reasons = set()
        for _, _, m, _ in sel:
            for bit, n in self.REASONS.items():
                if m is not None and m & bit:
                    reasons.add(n)
        pw = [x[3] / 1000.0 for x in sel if x[3] is not None]
        sm = [x[1] for x in sel]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sel),
                "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": max(pw) if pw else None,
                "window_ms": (t1 - t0) * 1e3 if t0 is not None and t1 is not None else None,
                "source": "NVML read-only queries every ~0.5 ms on a host thread"}


def replica_aggregate(ms_local: float, tokens_local: int, dist=None, device=None):
    """Whole-job figures of N independent replicas: the step time is the max over
    ranks, the tokens are summed over ranks. Returns (ms, tokens, tokens/s)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms_local, tokens_local, tokens_local / (ms_local * 1e-3)
    import torch
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    n = torch.tensor([tokens_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    ms, tok = float(t.item()), int(n.item())
    return ms, tok, tok / (ms * 1e-3)


def workload_spec(args):
    over = {}
    if args.tokens_per_rank:
        over["T"] = args.tokens_per_rank
    if args.experts:
        over["E"] = args.experts
    if args.hidden:
        over["h"] = args.hidden
    if getattr(args, "top_k", None):
        over["K"] = args.top_k
    s = wl.spec(args.config, **over)
    if over:
        s = wl.spec(args.config, name=f"{s.name}-override-T{s.T}-E{s.E}-K{s.K}-h{s.h}", **over)
    return s


def variant_of(args) -> dict:
    """The dispatch variant a run measures, empty for the headline path."""
    v = {}
    if args.x_dtype != "bf16":
        v["x_dtype"] = args.x_dtype
    if args.weight_on_input:
        v["weight_on_input"] = True
    if args.ragged:
        v["ragged"] = "num_tokens ~ U[T/2, T] per rank, seed 7"
    if args.zero_pad:
        v["zero_pad"] = True
    if getattr(args, "out_dtype", "bf16") != "bf16":
        v["out_dtype"] = args.out_dtype
    if getattr(args, "option", None):
        v["options"] = sorted(args.option)
    return v


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------ CPU oracle legs

def oracle_step(x: wl.Workload):
    from oracle import ref
    s = x.spec
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights, x.num_tokens)
    rows = ref.dispatch_rows(m, x.a1)
    ref.combine(m, x.topk_weights, rows)
    return int(x.num_tokens.sum())


def cpu_baseline(cfg: int, budget_s: float = 12.0):
    """The oracle as it stands (one host thread) on the full workload, repeated
    until about budget_s of CPU work (at most 64 steps)."""
    x = wl.make(cfg)
    toks, t_all, reps = 0, 0.0, 0
    while t_all < budget_s and reps < 64:
        t0 = time.perf_counter()
        toks += oracle_step(x)
        t_all += time.perf_counter() - t0
        reps += 1
    return {"value": toks / t_all, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{reps} full step(s) of {x.spec.name} ({toks} tokens) on one host thread, "
                      f"{t_all:.1f} s"}


def _host_memory_bytes() -> int:
    """Memory free for new processes: free pages, capped by a cgroup limit if any."""
    free = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    for lim, use in (("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory.current"),
                     ("/sys/fs/cgroup/memory/memory.limit_in_bytes",
                      "/sys/fs/cgroup/memory/memory.usage_in_bytes")):
        try:
            with open(lim) as f:
                v = f.read().strip()
            with open(use) as f:
                u = int(f.read().strip())
        except (OSError, ValueError):
            continue
        if v.isdigit():
            free = min(free, int(v) - u)
    return max(0, free)


def _oracle_replica(cfg: int, budget_s: float, start, out):
    try:
        x = wl.make(cfg)
        oracle_step(x)                 # untimed: pages the buffers in
    except BaseException:
        start.abort()                  # release the others at once
        raise
    start.wait(timeout=300)
    toks, reps, t0 = 0, 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s and reps < 64:
        toks += oracle_step(x)
        reps += 1
    out.put((toks, reps, time.perf_counter() - t0))


def cpu_baseline_all_cores(cfg: int, budget_s: float = 8.0, bytes_per_replica: int = 4 << 30):
    """The same oracle, unchanged, as independent replicas: one spawned process per
    host core (fewer if memory is short; each holds about 2.5 GB at the prefill
    size), each running full steps for about budget_s after a common start.
    Throughput = all replicas' tokens / the slowest replica's time."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    n = max(1, min(cores, _host_memory_bytes() // 2 // bytes_per_replica))
    ctx = mp.get_context("spawn")
    start, out = ctx.Barrier(n), ctx.Queue()
    procs = [ctx.Process(target=_oracle_replica, args=(cfg, budget_s, start, out)) for _ in range(n)]
    for pr in procs:
        pr.start()
    import queue
    res, deadline = [], time.monotonic() + budget_s + 300
    while len(res) < n and time.monotonic() < deadline:
        try:
            res.append(out.get(timeout=1.0))
        except queue.Empty:
            if all(pr.exitcode is not None for pr in procs):
                while True:            # every replica has ended: take what is left
                    try:
                        res.append(out.get(timeout=1.0))
                    except queue.Empty:
                        break
                break
    ok = len(res) == n
    for pr in procs:
        pr.join(timeout=30)
        if pr.is_alive():
            pr.terminate()
            pr.join()
    if not ok:
        return None
    toks = sum(r[0] for r in res)
    el = max(r[2] for r in res)
    return {"value": toks / el, "unit": UNIT, "cores": n,
            "sample": f"{n} spawned replicas of the one-thread oracle, each full steps of "
                      f"{wl.spec(cfg).name} for ~{budget_s:.0f} s from a common start "
                      f"({sum(r[1] for r in res)} steps, {toks} tokens in {el:.1f} s)"}


def _oracle_omp_child(cfg: int, budget_s: float, threads: int, out):
    os.environ["OMP_NUM_THREADS"] = str(threads)
    try:
        from oracle import ref
        ref.use_openmp(True)
        x = wl.make(cfg)
        oracle_step(x)                 # untimed: builds/loads the library, pages buffers in
        toks, reps, t0 = 0, 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s and reps < 64:
            toks += oracle_step(x)
            reps += 1
        out.put((toks, reps, time.perf_counter() - t0))
    except BaseException as e:         # report, never hang the parent
        out.put(("error", repr(e)))


def cpu_baseline_openmp(cfg: int, budget_s: float = 8.0):
    """The oracle's OpenMP build (same source, same results) on all host cores:
    one full step at a time, its row copies and combine split over the cores,
    its routing on one thread, repeated for about budget_s. Throughput = tokens
    over wall time, so one step's latency is ms_per_step."""
    import multiprocessing as mp
    import queue
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    pr = ctx.Process(target=_oracle_omp_child, args=(cfg, budget_s, cores, out))
    pr.start()
    r, deadline = None, time.monotonic() + budget_s + 600
    while r is None and time.monotonic() < deadline:
        try:
            r = out.get(timeout=1.0)
        except queue.Empty:
            if pr.exitcode is not None:     # ended without a result
                try:
                    r = out.get(timeout=1.0)
                except queue.Empty:
                    pass
                break
    pr.join(timeout=30)
    if pr.is_alive():
        pr.terminate()
        pr.join()
    if not r or r[0] == "error":
        return None
    toks, reps, el = r
    return {"value": toks / el, "unit": UNIT, "cores": cores, "ms_per_step": el / reps * 1e3,
            "kind": "oracle, OpenMP build (copies and combine over all cores, routing on one)",
            "sample": f"{reps} full step(s) of {wl.spec(cfg).name} ({toks} tokens) in {el:.1f} s, "
                      f"one step at a time on {cores} threads"}


_REF_X = {}


def _ref_step(arg):
    cfg, T = arg
    if (cfg, T) not in _REF_X:
        _REF_X.clear()
        _REF_X[(cfg, T)] = wl.make(wl.spec(cfg, T=T))
    return oracle_step(_REF_X[(cfg, T)])


def run_reference(args, budget_s: float = 200.0):
    """The oracle, unchanged, on the host cores: one spawned replica per core
    (fewer if memory is short), each step every replica running one oracle step.
    Each replica runs the full workload when warm-up plus timed steps fit in
    about budget_s; otherwise a token sample of it, sized so the run ends in
    minutes, and the line's config names the sampled tokens per rank."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import multiprocessing as mp
    full = wl.spec(args.config)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    per_replica = 4 << 30              # ~2.5 GB at the full prefill step, far less per sample
    n = max(1, min(cores, _host_memory_bytes() // 2 // per_replica))
    n_steps = max(1, args.steps + args.warmup)
    with mp.get_context("spawn").Pool(n) as pool:
        def step(T):
            return sum(pool.map(_ref_step, [(args.config, T)] * n, chunksize=1))
        # one full step with every replica running (the first call also loads the
        # library and draws the inputs, so time a second one)
        step(full.T)
        t0 = time.perf_counter()
        step(full.T)
        dt_full = time.perf_counter() - t0
        T = full.T
        if dt_full * n_steps > budget_s:
            T = max(1, min(full.T, int(full.T * budget_s / n_steps / dt_full)))
            step(T)
        for _ in range(args.warmup):
            step(T)
        toks = 0
        t0 = time.perf_counter()
        for _ in range(args.steps):
            toks += step(T)
        el = time.perf_counter() - t0
    v = toks / el
    same = T == full.T
    sample = (f"each step: {n} spawned replicas of the one-thread oracle, one per host core, each "
              f"one step of {full.name} " + ("(the full workload)" if same else
                                            f"on a sample of {T} tokens per rank (same generators)"))
    cfg = {"workload": full.name if same else f"{full.name}-sample-T{T}", "W": full.W, "E": full.E,
           "top_k": full.K, "tokens_per_rank": T, "hidden": full.h, "path": "oracle"}
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": n, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    from combine_ep_route_gb300 import EpConfig, EpContext, _lib as L

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    variant = variant_of(args)
    spec = workload_spec(args)
    nt_draw = None
    if args.ragged:
        nt_draw = np.random.default_rng(7).integers(spec.T // 2, spec.T + 1, size=spec.W).astype(np.int32)
    x = wl.make(spec, num_tokens=nt_draw)
    s = x.spec
    quant = args.x_dtype != "bf16"
    extra_row_bytes = list(x.extra_row_bytes)
    if quant:
        # opaque quantised rows and their scales, sized as the pages' one-sided manager
        # assumes: fp8 with one fp32 scale per 128 values, packed fp4 with one byte per 16
        rng = np.random.default_rng(1000 + args.config)
        xb = s.h if args.x_dtype == "fp8" else s.h // 2
        sb = (s.h // 128) * 4 if args.x_dtype == "fp8" else s.h // 16
        sb = (sb + 15) // 16 * 16
        a1_host = rng.integers(0, 256, size=(s.W, s.T, xb), dtype=np.uint8)
        extra_host = [rng.integers(0, 256, size=(s.W, s.T, sb), dtype=np.uint8)] + list(x.extras)
        extra_row_bytes = [sb] + extra_row_bytes
    cfg = EpConfig(s.W, s.E, s.K, s.T, s.h, extra_row_bytes=tuple(extra_row_bytes),
                   sendbuf=args.path == "sendbuf" or args.combine == "two_stage",
                   x_dtype=args.x_dtype, weight_on_input=args.weight_on_input, zero_pad=args.zero_pad)
    ctx = EpContext(cfg, dev)
    for o in getattr(args, "option", None) or []:
        name, val = o.split("=", 1)
        ctx.set_option(getattr(L, "EP_OPT_" + name.strip().upper()), int(val))
    if quant:
        a1 = torch.from_numpy(a1_host).to(dev).view(cfg.x_torch_dtype)
        extras = [torch.from_numpy(e).to(dev) for e in extra_host]
    else:
        a1 = torch.from_numpy(x.a1.view(np.int16)).to(dev).view(torch.bfloat16)
        extras = [torch.from_numpy(e).to(dev) for e in x.extras]
    ids = torch.from_numpy(x.topk_ids).to(dev)
    w = torch.from_numpy(x.topk_weights).to(dev)
    nt = torch.from_numpy(x.num_tokens).to(dev)
    out = ctx.alloc_dispatch_outputs()
    # identity experts read the dispatched rows; quantised rows need a bf16 expert output
    expert_out = out.b_a1 if not quant else torch.zeros(
        (s.W, s.E // s.W, ctx.expert_cap, s.h), dtype=torch.bfloat16, device=dev)
    out_t = torch.float32 if args.out_dtype == "f32" else torch.bfloat16
    y = torch.empty((s.W, s.T, s.h), dtype=out_t, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    combine_fn = ctx.combine if args.combine == "fused" else ctx.combine_two_stage

    def combine(eo, out):
        return combine_fn(eo, out=out, out_dtype=out_t)

    def step():
        ctx.dispatch(a1, ids, w, num_tokens=nt, extras=extras, out=out, path=args.path)
        combine(expert_out, out=y)

    n_warm = max(3, args.warmup)
    for _ in range(n_warm):
        flush.zero_()
        step()
    ctx.check()
    per_step_launches = sum(v[0] for v in ctx.kernel_times().values()) // n_warm
    eager_step = step
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            eager_step()
        step = graph.replay
        for _ in range(3):
            flush.zero_()
            step()
        ctx.check()
        ctx.kernel_times()

    n = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]

    def timed_region():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for i in range(n):
            if not args.hot:
                flush.zero_()                # L2 flush between steps (outside the step's events)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        if world > 1:
            dist.barrier()
        st = ctx.status()
        if st != 0:
            raise SystemExit(f"device status {st} after the timed region")
        return [a.elapsed_time(b) for a, b in ev], t_wall

    # 1. the headline: K steps, nothing but the library's kernels between the step events
    nv = NvmlSampler(local)
    nv.__enter__()
    if nv.ok:
        nv.mark("headline", True)
        step_ms, t_wall = timed_region()
        nv.mark("headline", False)
        clocks = nv.summary("headline")
    else:
        with ClockSampler(local) as clk:
            step_ms, t_wall = timed_region()
        clocks = clk.summary()
    launches = int(sum(v[0] for v in ctx.kernel_times().values()))
    if args.graph:   # replays do not pass through the host API: count the captured kernels
        launches = n * per_step_launches
    step = eager_step
    # 2. per-kernel durations for the roofline: K more steps with CUDA events around
    #    every kernel launch, on the launching stream (after a few untimed eager steps
    #    with the events on, so the pass starts warm like the headline one)
    ctx.set_option(L.EP_OPT_KERNEL_TIMING, 1)
    for _ in range(max(3, args.warmup)):
        if not args.hot:
            flush.zero_()
        step()
    ctx.check()
    ctx.kernel_times()
    nv.mark("per_kernel", True)
    step_ms_ev, _ = timed_region()
    nv.mark("per_kernel", False)
    kt = ctx.kernel_times()
    ctx.set_option(L.EP_OPT_KERNEL_TIMING, 0)
    # 3. medians of dispatch and combine timed separately (events around each call,
    #    L2 flushed before every step), over a fixed 200 repetitions
    reps = 200
    evm = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    torch.cuda.synchronize()
    nv.mark("separate_calls", True)
    for i in range(reps):
        if not args.hot:
            flush.zero_()
        evm[i][0].record(stream)
        ctx.dispatch(a1, ids, w, num_tokens=nt, extras=extras, out=out, path=args.path)
        evm[i][1].record(stream)
        combine(expert_out, out=y)
        evm[i][2].record(stream)
    torch.cuda.synchronize()
    nv.mark("separate_calls", False)
    nv.__exit__()
    if nv.ok:
        clocks["other_passes"] = {k: nv.summary(k) for k in ("per_kernel", "separate_calls")}
    med_d = float(np.median([e[0].elapsed_time(e[1]) for e in evm]))
    med_c = float(np.median([e[1].elapsed_time(e[2]) for e in evm]))
    disp_b, comb_b = algorithmic_bytes(x, out_bytes_per_elem=4 if args.out_dtype == "f32" else 2,
                                       x_row_bytes=cfg.x_row_bytes, extra_bytes=sum(extra_row_bytes))
    n_pairs, n_tok_routed, n_tok = workload_counts(x)
    ms, _, value = replica_aggregate(sum(step_ms) / n, n_tok, dist if world > 1 else None, dev)
    peak, peak_src = measured_peaks()
    # per-kernel durations (CUDA events around every launch, on the launch stream)
    per = {}
    for name in ("route", "move_fused", "pack", "exchange", "deliver", "combine", "combine_two_stage",
                 "dispatch_fused", "dispatch_small"):
        _, tot, timed = kt[name]
        if timed:
            per[name] = tot / timed
    cands = [k for k in ("dispatch_fused", "dispatch_small", "move_fused", "pack", "exchange", "deliver",
                         "combine", "combine_two_stage") if k in per]
    dom = max(cands, key=lambda k: per[k])
    # algorithmic bytes of one launch of the dominant kernel (send-buffer steps and the
    # two-stage combine are charged the same algorithmic bytes as the fused step's)
    dom_bytes = disp_b if dom in ("dispatch_fused", "dispatch_small", "move_fused", "pack", "exchange",
                                  "deliver") else comb_b
    achieved = dom_bytes / (per[dom] * 1e-3) / 1e9
    traffic = traffic_for(dom, traffic_config(args, s, variant))

    e2e = None
    if not args.no_e2e and not variant:
        e2e = run_e2e(ctx, x, dev, out, n, stream, combine)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not variant:
        cpu = cpu_baseline(args.config)
        cpu["all_cores"] = cpu_baseline_openmp(args.config)
        cpu["replicas"] = cpu_baseline_all_cores(args.config)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": s.name, "W": s.W, "E": s.E, "top_k": s.K, "tokens_per_rank": s.T,
                   "hidden": s.h, "extra_row_bytes": list(extra_row_bytes), "path": args.path,
                   "combine": args.combine, "launch": "cuda graph replay" if args.graph else "stream",
                   "out_dtype": args.out_dtype, "accumulate": "f32",
                   "experts": ("identity (expert_out = b_a1)" if not quant else
                               "a bf16 expert-output buffer (the dispatched rows are quantised)"),
                   "l2": ("hot: no flush between steps" if args.hot else
                          "flushed: 256 MiB write before every step, outside the step's events"),
                   "replicas": world, **({"variant": variant} if variant else {})},
        "num_tokens": x.num_tokens.tolist() if args.ragged else None,
        "ms_per_step_median": float(np.median(step_ms)),
        "effective_gbs": (disp_b + comb_b) / (ms * 1e-3) / 1e9,
        "effective_frac_of_peak": (disp_b + comb_b) / (ms * 1e-3) / 1e9 / peak,
        "alg_bytes_per_step": {"dispatch": disp_b, "combine": comb_b},
        "counts": {"pairs": n_pairs, "tokens_routed": n_tok_routed, "tokens": n_tok},
        "pairs_per_s": world * n_pairs / (ms * 1e-3),
        "kernel_ms": {k: round(v, 5) for k, v in per.items()},
        "call_ms_median": {"dispatch": round(med_d, 5), "combine": round(med_c, 5),
                           "sum": round(med_d + med_c, 5),
                           "note": "200 eager steps, events around each call, L2 flushed per step"},
        "kernel_ms_note": "second pass of K steps with CUDA events around every launch "
                          f"(step {sum(step_ms_ev) / n:.4f} ms with those events)",
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic,
                     **({"traffic_source": "profiles/dram_traffic.txt (one-launch ncu capture; "
                                           "rows still dirty in L2 at the kernel's end are not "
                                           "counted)"} if traffic is not None else {})},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def agrs_bytes(x: wl.Workload):
    """Algorithmic bytes of one all-gather / reduce-scatter step with identity
    experts: the gather reads each valid token row (and its ids and weights)
    once and writes it to all W ranks; each rank reads a gathered row only when
    one of its experts is among the token's kept pairs, reads every gathered
    id/weight row, and writes one expert-output row per gathered token; the
    reduce-scatter reads the W expert-output rows of each valid token and
    writes every output row."""
    s = x.spec
    ids = x.topk_ids
    live = np.arange(s.T)[None, :] < x.num_tokens[:, None]
    n_tok = int(live.sum())
    kept = (ids >= 0) & live[:, :, None]          # the drawn ids are distinct and < E
    dest = np.where(kept, ids // s.e_local, -1).reshape(-1, s.K)
    n_local_rows = sum(len(set(r[r >= 0].tolist())) for r in dest)
    bx, bm = 2 * s.h, 8 * s.K
    gather = (bx + bm) * n_tok * (1 + s.W)
    experts = s.W * n_tok * bm + n_local_rows * bx + s.W * n_tok * bx
    reduce = s.W * n_tok * bx + s.W * s.T * bx
    return {"gather": gather, "experts": experts, "reduce_scatter": reduce}, n_local_rows


def run_agrs(args):
    import torch

    from combine_ep_route_gb300 import EpConfig, agrs, alloc_agrs_buffers

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x = wl.make(workload_spec(args))
    s = x.spec
    cfg = EpConfig(s.W, s.E, s.K, s.T, s.h)
    a1 = torch.from_numpy(x.a1.view(np.int16)).to(dev).view(torch.bfloat16)
    ids = torch.from_numpy(x.topk_ids).to(dev)
    w = torch.from_numpy(x.topk_weights).to(dev)
    nt = torch.from_numpy(x.num_tokens).to(dev)
    buf = alloc_agrs_buffers(cfg, dev)
    y = torch.empty((s.W, s.T, s.h), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        agrs(cfg, a1, ids, w, num_tokens=nt, buffers=buf, out=y)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if int(buf.status.item()) != 0:
        raise SystemExit(f"device status {int(buf.status.item())}")
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        step = graph.replay
        for _ in range(3):
            flush.zero_()
            step()
    n = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    def timed():
        torch.cuda.synchronize()
        for i in range(n):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()

    nv = NvmlSampler(local)
    if nv.ok:
        with nv:
            nv.mark("timed", True)
            timed()
            nv.mark("timed", False)
        clocks = nv.summary("timed")
    else:
        with ClockSampler(local) as clk:
            timed()
        clocks = clk.summary()
    if int(buf.status.item()) != 0:
        raise SystemExit(f"device status {int(buf.status.item())} after the timed region")
    ms = sum(a.elapsed_time(b) for a, b in ev) / n
    parts, n_local_rows = agrs_bytes(x)
    total = sum(parts.values())
    peak, peak_src = measured_peaks()
    n_tok = int(x.num_tokens.sum())
    achieved = total / (ms * 1e-3) / 1e9
    key = traffic_config(args, s)
    tr = [traffic_for(k, key) for k in ("agrs_gather", "agrs_experts", "agrs_reduce")]
    traffic = sum(tr) if all(t is not None for t in tr) else None
    line = {
        "metric": METRIC, "value": n_tok / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": n,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "route": "agrs",
        "config": {"workload": s.name, "W": s.W, "E": s.E, "top_k": s.K, "tokens_per_rank": s.T,
                   "hidden": s.h, "route": "all-gather / experts / reduce-scatter",
                   "launch": "cuda graph replay" if args.graph else "stream", "out_dtype": "bf16",
                   "experts": "identity", "l2": "flushed: 256 MiB write before every step"},
        "alg_bytes_per_step": parts,
        "counts": {"tokens": n_tok, "rank_rows_with_local_experts": n_local_rows},
        "roofline": {"kernel": "agrs step (gather + experts + reduce-scatter)", "bound": "hbm",
                     "achieved": achieved, "peak": peak, "peak_source": f"{peak_src} hbm_gbs",
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic},
        "gpu_launches": 3 * n,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(ctx, x, dev, out, n, stream, combine=None):
    """Same metric through the public API from pinned host buffers. Every step
    copies its own inputs host->device, dispatches, combines and copies its
    output back, all inside the timed region. Uploads and downloads run on
    their own streams with double-buffered device copies, so step i+1's upload
    and step i-1's download overlap step i's kernels, as a serving loop would."""
    import torch
    s = x.spec
    h_a1 = torch.from_numpy(x.a1.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_ids = torch.from_numpy(x.topk_ids).pin_memory()
    h_w = torch.from_numpy(x.topk_weights).pin_memory()
    h_ex = [torch.from_numpy(e).pin_memory() for e in x.extras]
    h_y = torch.empty((s.W, s.T, s.h), dtype=torch.bfloat16).pin_memory()
    h_in = [h_a1, h_ids, h_w, *h_ex]
    d_in = [[torch.empty_like(t, device=dev) for t in h_in] for _ in range(2)]
    d_y = [torch.empty((s.W, s.T, s.h), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_y.numel() * h_y.element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in comp_done + out_done:
        e.record(stream)

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(comp_done[b])          # step i-2 finished reading these inputs
            for d, h in zip(d_in[b], h_in):
                d.copy_(h, non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_done[b])              # step i-2's output has been read back
        a1, ids, w, *ex = d_in[b]
        ctx.dispatch(a1, ids, w, extras=ex, out=out)
        (combine or ctx.combine)(out.b_a1, out=d_y[b])
        comp_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            h_y.copy_(d_y[b], non_blocking=True)
            out_done[b].record(s_out)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    m = 200   # a fixed pipeline length, so that its fill and drain weigh the same at any K
    a = torch.cuda.Event(enable_timing=True)
    b_ = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(m):
        step(i)
    b_.record(s_out)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b_) / m
    ctx.check()
    ctx.kernel_times()
    tokens = int(x.num_tokens.sum())
    return {"value": tokens / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": m,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "EpContext.dispatch/combine; pinned host inputs copied in and the output "
                   "copied back every step on separate streams (double-buffered)"}


def run_ceilings(args):
    """Reference points for the roofline discussion, not the roofline's denominator
    (that is the measured copy peak): how fast plain read-only, write-only
    and copy kernels move 1 GiB on this GPU, and how fast the host link copies.
    CUDA events on the stream that launches each op; best and median of 10."""
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    n = 1 << 30
    a = torch.ones(n // 4, dtype=torch.int32, device=dev)
    b = torch.empty(n // 4, dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()

    def timed(fn, nbytes, reps=10, streams=None):
        ms = []
        for i in range(reps + 2):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(st)
            fn()
            for s2 in streams or ():
                st.wait_stream(s2)
            e1.record(st)
            torch.cuda.synchronize()
            if i >= 2:
                ms.append(e0.elapsed_time(e1))
        return {"best_gbs": nbytes / (min(ms) * 1e-3) / 1e9,
                "median_gbs": nbytes / (float(np.median(ms)) * 1e-3) / 1e9, "bytes": nbytes}

    reads = {"int32 max": timed(lambda: a.max(), n),
             "int32 sum": timed(lambda: a.sum(), n),
             "count_nonzero": timed(lambda: torch.count_nonzero(a), n),
             "int64 view max": timed(lambda: a.view(torch.int64).max(), n)}
    best = max(reads, key=lambda k: reads[k]["best_gbs"])
    out = {"probe": "ceilings", "device": torch.cuda.get_device_name(dev),
           "read_only": dict(reads[best], op=best), "read_only_ops": reads,
           "write_only": timed(lambda: b.zero_(), n),
           "copy": timed(lambda: b.copy_(a), 2 * n)}
    del a, b
    # the fixed cost a timed step carries: a replayed graph of one or two minimal
    # kernels between the step's events, after the 256 MiB L2-flushing write
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    tiny = [torch.zeros(16, dtype=torch.int32, device=dev) for _ in range(2)]
    floor = {}
    for n_k in (1, 2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for k in range(n_k):
                tiny[k].zero_()
        us = []
        for i in range(220):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            g.replay()
            e1.record(st)
            e1.synchronize()
            if i >= 20:
                us.append(e0.elapsed_time(e1) * 1e3)
        floor[f"{n_k}_kernel_graph_us"] = {"median": float(np.median(us)), "min": float(min(us))}
    out["launch_floor"] = floor
    del flush
    m = 118 << 20
    h_src = torch.ones(m, dtype=torch.uint8).pin_memory()
    h_dst = torch.empty(m, dtype=torch.uint8).pin_memory()
    d_src = torch.ones(m, dtype=torch.uint8, device=dev)
    d_dst = torch.empty(m, dtype=torch.uint8, device=dev)
    s_up, s_dn = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def both():
        s_up.wait_stream(st)
        s_dn.wait_stream(st)
        with torch.cuda.stream(s_up):
            d_dst.copy_(h_src, non_blocking=True)
        with torch.cuda.stream(s_dn):
            h_dst.copy_(d_src, non_blocking=True)

    out["host_to_device"] = timed(lambda: d_dst.copy_(h_src, non_blocking=True), m)
    out["device_to_host"] = timed(lambda: h_dst.copy_(d_src, non_blocking=True), m)
    out["both_directions"] = timed(both, 2 * m, streams=(s_up, s_dn))
    out["note"] = ("read_only: the fastest of four torch reductions over 1 GiB (a lower bound on "
                   "the read ceiling); write_only: zero_ of 1 GiB; copy: copy_ of "
                   "1 GiB (read + write bytes); host link: cudaMemcpyAsync through torch on "
                   "pinned 118 MiB buffers, both directions on two streams at once; launch_floor: "
                   "a replayed CUDA graph of one or two 64-byte zero_ kernels between CUDA events, "
                   "after the L2 flush, as the timed steps are (200 repetitions)")
    if rank == 0:
        print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.probe == "ceilings":
        run_ceilings(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.route == "agrs":
        run_agrs(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the stable co-rank merge on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload: int32 merge of two sorted uniform full-range arrays,
m = n = 2^28 (2^29 outputs, 2 GiB read + 2 GiB written per merge).  One step
= one om_merge_i32 call (one tile-merge launch whose CTAs find their own
range boundaries) on inputs already resident in HBM.  Prints ONE JSON line on
rank 0.

  value      merged elements/s over the K timed steps (CUDA events on the
             launching stream; max over ranks for N > 1, times N replicas)
  roofline   the tile-merge kernel: algorithmic bytes per launch
             ((m+n) * (4 read + 4 written)) / its mean launch time (the
             library's launch trace: events around each launch, recorded in a
             second pass over the same K steps, so that the call times above
             carry no trace events), against the measured HBM copy peak
  e2e        the same metric with the host<->device copies inside the timed
             region: pinned host A, B -> device, merge, device C -> pinned host
  cpu_baseline  the CPU oracle (single thread) on the same workload
  clocks     nvidia-smi samples taken during the timed region
  other_configs  the evens/odds, heavy-tie pairs, skewed and sort workloads,
             each timed the same way in the same run with fewer steps

--impl reference times the CPU oracle alone on a bounded sample per step.
N > 1 runs independent replicas (the merge needs no exchange across GPUs in
this configuration), one process per GPU under torchrun.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "merged elements/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "elements/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal

WORKLOADS = {
    "uniform": "int32 merge at bandwidth scale: A, B = 2^28 sorted uniform full-range int32 each",
    "evens_odds": "int32 merge, A = evens (2^21+611), B = odds (2^21)",
    "skewed": "int32 merge, A = 2^28 sorted full-range, B = 2^10 sorted in [-2^20, 2^20]",
    "pairs_ties": "uint32 key+value merge, m = n = 2^24, keys in [0,16)",
    "sort": "stable merge sort of 2^26 uint32 keys with index payload",
    "f64": "float64 merge: A, B = 2^27 sorted float64 each (int32 draws x 2^-20)",
    "i64_desc": "int64 merge, descending: A, B = 2^27 full-range int64 each, sorted nonincreasing",
    "sort_f32_desc": "stable descending merge sort of 2^26 float32 keys with index payload",
    "sort_f64": "stable merge sort of 2^26 float64 keys, keys only",
}
SORTS = ("sort", "sort_f32_desc", "sort_f64")

# Source files whose change invalidates a recorded ncu traffic figure (the
# tile-merge and one-pass merge kernels).
KERNEL_SOURCES = [
    "ordered_merge_gb300/csrc/merge_kernels.cuh",
    "ordered_merge_gb300/csrc/one_pass_merge.cuh",
    "ordered_merge_gb300/csrc/sort_kernels.cuh",
    "ordered_merge_gb300/csrc/om_ptx.cuh",
    "ordered_merge_gb300/csrc/api_internal.cuh",
    "ordered_merge_gb300/csrc/api.cu",
    "ordered_merge_gb300/csrc/typed_merge.cu",
]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "tile_merge_traffic.json")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, units_per_launch: int):
    """Per-launch DRAM bytes (read + write) of the tile-merge kernel on this
    workload from the committed ncu summary, or None when there is none, the
    kernel sources changed since it was taken, or it was taken at another
    size (a scaled run)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_hash") != kernel_source_hash():
        return None
    wl = rec.get("workloads", {}).get(workload)
    if not wl or wl.get("units_per_launch") != units_per_launch:
        return None
    return wl.get("traffic_bytes_per_launch")


def load_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------ distributed --

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_init(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of x over ranks (identity for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist

        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="om_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", str(self.period_ms)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        # samples under load: power above the midpoint of the observed range
        if power:
            thr = (min(power) + max(power)) / 2
            loaded = [num(r[1]) for r in rows if num(r[3]) is not None and num(r[3]) >= thr and num(r[1])]
        else:
            loaded = sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {
            "sm_mhz": statistics.median(loaded or sm) if (loaded or sm) else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": reasons,
            "samples": len(rows),
            "power_w_max": max(power) if power else None,
        }


# --------------------------------------------------------------- L2 flush --

class L2Flusher:
    """Evicts L2 by writing a buffer twice its size on the current stream,
    twice: about 80 us of GPU work, longer than the host takes to enqueue the
    timed step after it, so the step's events hold GPU work only and no wait
    for the host."""

    @staticmethod
    def l2_bytes(device) -> int:
        import torch

        return int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 128 << 20))

    def __init__(self, device):
        import torch

        self.buf = torch.empty(2 * self.l2_bytes(device), dtype=torch.uint8, device=device)
        self.val = 0

    def __call__(self):
        for _ in range(2):
            self.val = (self.val + 1) & 0xFF
            self.buf.fill_(self.val)


# ------------------------------------------------------------ CPU oracle --

def oracle_call(wl: str, h: dict):
    """(callable, units): one run of the CPU oracle on host arrays `h` of
    workload `wl` (a merge, or a sort from the unsorted keys), and the
    elements it produces."""
    import oracle
    import synth

    lib = oracle.load()
    if wl in ("uniform", "evens_odds", "skewed"):
        return (lambda: oracle.merge_i32(h["A"], h["B"], lib=lib)), h["A"].size + h["B"].size
    if wl == "pairs_ties":
        return ((lambda: oracle.merge_pairs_u32(h["keysA"], h["valsA"], h["keysB"], h["valsB"], lib=lib)),
                h["keysA"].size + h["keysB"].size)
    if wl == "sort":
        return (lambda: oracle.merge_sort_pairs_u32(h["keys"], h["vals"], lib=lib)), h["keys"].size
    kt, desc = synth.TYPED[wl]
    if "A" in h:
        return (lambda: oracle.merge_keys(h["A"], h["B"], descending=desc, lib=lib)), h["A"].size + h["B"].size
    return (lambda: oracle.merge_sort_keys(h["keys"], h.get("vals"), descending=desc, lib=lib)), h["keys"].size


def oracle_rate(wl: str, h: dict, budget_s: float = 12.0, max_reps: int = 5):
    """Elements/s of the single-thread oracle on host arrays of workload wl."""
    fn, units = oracle_call(wl, h)
    times = []
    t_start = time.perf_counter()
    while len(times) < max_reps:
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s:
            break
    best = statistics.median(times)
    return units / best, len(times), best, units


# ------------------------------------------------------------- our arm --

def measure(wl: str, args, device, world: int, steps: int, warmup: int, keep: bool = False):
    """Times `steps` calls of workload `wl` after `warmup` untimed ones (CUDA
    events on the launching stream; L2 flushed before every timed call when
    the bytes a call moves fit twice in L2) and returns the figures of one
    bench line: time, rate, the tile-merge kernel's roofline and the clocks
    sampled meanwhile.  keep: also return the device tensors (end-to-end leg)."""
    import torch

    import ordered_merge_gb300 as om
    import synth

    d = synth.make_device(wl, device, scale_log2=args.scale_log2)
    stream = torch.cuda.current_stream(device)
    tensors = {}

    if wl in ("uniform", "evens_odds", "skewed"):
        A, B = d["A"], d["B"]
        m, n = A.numel(), B.numel()
        total = m + n
        bytes_per_elem = 8
        C = torch.empty(total, dtype=torch.int32, device=device)
        step = lambda: om.merge_i32(A, B, C)
        tensors = {"A": A, "B": B, "C": C}
    elif wl in ("f64", "i64_desc"):
        kt, desc = synth.TYPED[wl]
        A, B = d["A"], d["B"]
        m, n = A.numel(), B.numel()
        total = m + n
        bytes_per_elem = 2 * A.element_size()
        C = torch.empty(total, dtype=A.dtype, device=device)
        step = lambda: om.merge_keys(A, B, C, key_type=kt, descending=desc)
    elif wl == "pairs_ties":
        ka, va, kb, vb = d["keysA"], d["valsA"], d["keysB"], d["valsB"]
        m, n = ka.numel(), kb.numel()
        total = m + n
        bytes_per_elem = 16
        kc = torch.empty(total, dtype=torch.int32, device=device)
        vc = torch.empty_like(kc)
        step = lambda: om.merge_pairs_u32(ka, va, kb, vb, kc, vc)
    else:  # sorts: restore the unsorted input before each step (outside the timed events)
        keys0, vals0 = d["keys"], d.get("vals")
        m, n = keys0.numel(), 0
        total = m
        # per element of one late pass: key read + written, value read + written
        bytes_per_elem = 2 * keys0.element_size() + (8 if vals0 is not None else 0)
        keys = keys0.clone()
        vals = vals0.clone() if vals0 is not None else None
        kt, desc = synth.TYPED.get(wl, ("u32", False))
        step = None

        def sort_once():
            keys.copy_(keys0)
            if vals is not None:
                vals.copy_(vals0)

        def sort_call():
            if wl == "sort":
                om.merge_sort_u32(keys, vals)
            else:
                om.merge_sort_keys(keys, vals, key_type=kt, descending=desc)

    units_per_step = total
    # ---- warm-up, then K timed steps.  A workload whose bytes moved per step
    # fit twice in L2 gets L2 flushed before every step (a write larger than
    # L2, outside the timed events); larger ones stream back to back.
    flush = L2Flusher(device) if total * bytes_per_elem < 2 * L2Flusher.l2_bytes(device) else None
    per_step = []  # per-call times where each call is timed alone (flushed merges, sorts)
    if step is not None:
        for _ in range(warmup):
            step()
        torch.cuda.synchronize(device)
        if om.device_error() != 0:
            raise RuntimeError("device error during warm-up")

        def timed_loop(count):
            if flush is None:
                ev0 = torch.cuda.Event(enable_timing=True)
                ev1 = torch.cuda.Event(enable_timing=True)
                ev0.record(stream)
                for _ in range(count):
                    step()
                ev1.record(stream)
                torch.cuda.synchronize(device)
                return ev0.elapsed_time(ev1)
            pairs = []
            for _ in range(count):
                flush()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                step()
                e1.record(stream)
                pairs.append((e0, e1))
            torch.cuda.synchronize(device)
            per_step.extend(a.elapsed_time(b) for a, b in pairs)
            return sum(a.elapsed_time(b) for a, b in pairs)
    else:
        for _ in range(warmup):
            sort_once()
            sort_call()
        torch.cuda.synchronize(device)

        def timed_loop(count):
            total_ms = 0.0
            for _ in range(count):
                sort_once()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                sort_call()
                e1.record(stream)
                e1.synchronize()
                per_step.append(e0.elapsed_time(e1))
                total_ms += per_step[-1]
            return total_ms

    barrier(world, device)
    torch.cuda.synchronize(device)
    with ClockSampler(device.index) as clk:
        # the calls as a user makes them (the library's launch trace off) ...
        launches0 = om.om_launch_count()
        ms = timed_loop(steps)
        launches = om.om_launch_count() - launches0
        call_ms = sorted(per_step)
        # ... then the same loop once more with the launch trace on, for the
        # kernels' own durations (its events sit around every launch, so the
        # call time is not taken from this loop)
        om.om_trace_reset()
        om.om_trace_enable(True)
        timed_loop(steps)
        om.om_trace_enable(False)
    if om.device_error() != 0:
        raise RuntimeError("device error during the timed region")
    clocks = clk.summary()

    ms_max = reduce_max(ms, world, device)
    tm_launches, tm_ms = om.om_trace_read(om.KIND_TILE_MERGE)
    op_launches, op_ms = om.om_trace_read(om.KIND_ONE_PASS)
    bs_launches, bs_ms = om.om_trace_read(om.KIND_BLOCK_SORT)
    merge_kernel = "tile_merge_kernel"
    if op_launches and not tm_launches:  # a merge small enough for the one-pass kernel
        tm_launches, tm_ms, merge_kernel = op_launches, op_ms, "one_pass_merge_kernel"
    peak, peak_src = load_peak()
    # merges: one launch moves every element once (read + written); sorts: the
    # dominant kernel is the late-pass tile merge, one pass of n elements per
    # launch.  Either way total * bytes_per_elem per launch.
    alg_bytes = total * bytes_per_elem
    tm_avg_ms = tm_ms / tm_launches if tm_launches else float("nan")
    achieved = alg_bytes / (tm_avg_ms / 1e3) / 1e9 if tm_launches else None
    roofline = {
        "kernel": merge_kernel,
        "bound": "hbm",
        "achieved": round(achieved, 1) if achieved else None,
        "peak": peak,
        "peak_source": peak_src,
        "unit": "GB/s",
        "frac": round(achieved / peak, 4) if achieved else None,
        "traffic": recorded_traffic(wl, total),
        "alg_bytes_per_launch": alg_bytes,
        "mean_launch_ms": round(tm_avg_ms, 5),
        "launches": tm_launches,
    }
    out = {
        "wl": wl, "m": m, "n": n, "total": total, "bytes_per_elem": bytes_per_elem,
        "steps": steps, "ms": ms, "ms_max": ms_max, "ms_per_step": ms_max / steps,
        "value": world * units_per_step * steps / (ms_max / 1e3),
        "achieved_gbs": (round(units_per_step * bytes_per_elem * steps / (ms / 1e3) / 1e9, 1)
                         if wl not in SORTS else None),
        "flushed": flush is not None, "roofline": roofline, "launches": launches, "clocks": clocks,
        "ms_per_step_median": round(statistics.median(call_ms), 5) if call_ms else None,
        "ms_per_step_min": round(call_ms[0], 5) if call_ms else None,
        "kernel_time_ms": {"tile_merge_ms": round(tm_ms, 4), "block_sort_ms": round(bs_ms, 4),
                           "block_sort_launches": bs_launches},
        "peak": peak,
    }
    if keep:
        out["tensors"] = tensors
    return out


# configs measured beside the headline one in the same run, with fewer steps
OTHER_CONFIGS = ("evens_odds", "pairs_ties", "skewed", "sort")


def other_config_line(r: dict) -> dict:
    """The short record of one extra config in the bench line."""
    rec = {
        "workload": WORKLOADS[r["wl"]],
        "m": r["m"],
        "n": r["n"],
        "steps": r["steps"],
        "ms_per_step": round(r["ms_per_step"], 5),
        "value": r["value"],
        "unit": UNIT,
        "achieved_gbs": r["achieved_gbs"],
        "merge_kernel": r["roofline"]["kernel"],
        "merge_kernel_frac_of_peak": r["roofline"]["frac"],
        "merge_kernel_mean_launch_ms": r["roofline"]["mean_launch_ms"],
        "l2": "flushed before every timed step" if r["flushed"] else "inputs larger than L2 (no flush)",
        "clocks": {k: r["clocks"].get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "gpu_launches": r["launches"],
    }
    if r["ms_per_step_median"] is not None:  # each call timed alone: its median and fastest call too
        rec["ms_per_step_median"] = r["ms_per_step_median"]
        rec["ms_per_step_min"] = r["ms_per_step_min"]
    if r["wl"] in SORTS:
        # all passes: one block pass and the late passes, each moving every pair once
        passes = 1 + r["roofline"]["launches"] // max(1, r["steps"])
        rec["passes"] = passes
        rec["pass_bytes_gbs"] = round(passes * r["total"] * r["bytes_per_elem"] / (r["ms_per_step"] / 1e3) / 1e9, 1)
        rec["block_sort_mean_launch_ms"] = round(r["kernel_time_ms"]["block_sort_ms"]
                                                 / max(1, r["kernel_time_ms"]["block_sort_launches"]), 5)
    elif r["achieved_gbs"] is not None:
        rec["pct_of_hbm_peak"] = round(100.0 * r["achieved_gbs"] / r["peak"], 2)
    return rec


def bench_ours(args):
    import torch

    import ordered_merge_gb300 as om
    import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")

    wl = args.workload
    r = measure(wl, args, device, world, args.steps, args.warmup, keep=True)
    m, n, total = r["m"], r["n"], r["total"]
    ms, ms_per_step, value = r["ms"], r["ms_per_step"], r["value"]
    roofline, kernel_share, launches, clocks, peak = (r["roofline"], r["kernel_time_ms"], r["launches"],
                                                      r["clocks"], r["peak"])
    flush = r["flushed"] or None
    units_per_step, bytes_per_elem = total, r["bytes_per_elem"]
    stream = torch.cuda.current_stream(device)
    if wl in ("uniform", "evens_odds", "skewed"):
        A, B, C = r["tensors"]["A"], r["tensors"]["B"], r["tensors"]["C"]
    r.pop("tensors", None)

    # ---- end to end through the C-ABI call with host buffers
    # Every step copies its inputs from pinned host memory, merges and copies
    # the result back to pinned host memory.  A pipeline of three streams --
    # host-to-device copies, merges, device-to-host copies -- chained by
    # events over two buffer sets: each direction's copies run one at a time
    # on their own stream (no two copies split one direction's bandwidth) and
    # overlap the other direction's and the merges, as a caller streaming
    # merges would run them.
    e2e = None
    if wl in ("uniform", "evens_odds", "skewed") and args.e2e_steps > 0:
        nbuf = 2
        hA = torch.empty(m, dtype=torch.int32, pin_memory=True)
        hB = torch.empty(n, dtype=torch.int32, pin_memory=True)
        hA.copy_(A)
        hB.copy_(B)
        hC = [torch.empty(total, dtype=torch.int32, pin_memory=True) for _ in range(nbuf)]
        dA = [torch.empty_like(A) for _ in range(nbuf)]
        dB = [torch.empty_like(B) for _ in range(nbuf)]
        dC = [C] + [torch.empty_like(C) for _ in range(nbuf - 1)]
        s_in, s_merge, s_out = (torch.cuda.Stream(device) for _ in range(3))
        loaded = [torch.cuda.Event() for _ in range(nbuf)]
        merged = [torch.cuda.Event() for _ in range(nbuf)]
        drained = [torch.cuda.Event() for _ in range(nbuf)]
        for b in range(nbuf):  # every buffer starts free
            merged[b].record(s_merge)
            drained[b].record(s_out)

        def e2e_step(i):
            b = i % nbuf
            with torch.cuda.stream(s_in):
                s_in.wait_event(merged[b])  # the merge two steps back has read dA/dB[b]
                dA[b].copy_(hA, non_blocking=True)
                dB[b].copy_(hB, non_blocking=True)
                loaded[b].record(s_in)
            with torch.cuda.stream(s_merge):
                s_merge.wait_event(loaded[b])
                s_merge.wait_event(drained[b])  # the copy-out two steps back has read dC[b]
                om.merge_i32(dA[b], dB[b], dC[b])
                merged[b].record(s_merge)
            with torch.cuda.stream(s_out):
                s_out.wait_event(merged[b])
                hC[b].copy_(dC[b], non_blocking=True)
                drained[b].record(s_out)
        streams = (s_in, s_merge, s_out)

        def copy_gbs(dst, src):
            """One copy's rate: best of 3 after a warm-up copy (the first
            copy from new pinned pages pays one-off mapping costs)."""
            dst.copy_(src, non_blocking=True)
            best = 0.0
            for _ in range(3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dst.copy_(src, non_blocking=True)
                e1.record(stream)
                torch.cuda.synchronize(device)
                best = max(best, dst.numel() * 4 / (e0.elapsed_time(e1) / 1e3) / 1e9)
            return best

        h2d_gbs = copy_gbs(dA[0], hA)
        d2h_gbs = copy_gbs(hC[0], dC[0])
        for i in range(nbuf):
            e2e_step(i)
        torch.cuda.synchronize(device)
        # Three timed runs of e2e_steps pipelined calls; the median run is
        # reported (the host link and host memory are shared with the
        # machine's other jobs, so single runs vary).
        run_ms = []
        for _ in range(3):
            barrier(world, device)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for st in streams:
                st.wait_event(e0)
            for i in range(args.e2e_steps):
                e2e_step(i)
            for st in streams:
                stream.wait_stream(st)
            e1.record(stream)
            torch.cuda.synchronize(device)
            run_ms.append(reduce_max(e0.elapsed_time(e1), world, device))
            if not torch.equal(hC[(args.e2e_steps - 1) % nbuf].to(device), C if nbuf == 1 else dC[0]):
                raise RuntimeError("end-to-end result differs from the device-resident merge")
        e_ms = sorted(run_ms)[1]
        e2e = {
            "value": world * total * args.e2e_steps / (e_ms / 1e3),
            "unit": UNIT,
            "h2d_bytes_per_step": (m + n) * 4,
            "d2h_bytes_per_step": total * 4,
            "steps": args.e2e_steps,
            "ms_per_step": e_ms / args.e2e_steps,
            "ms_per_step_runs": [round(x / args.e2e_steps, 3) for x in run_ms],
            "timing": "median of 3 timed runs of `steps` pipelined calls",
            "streams": "3 (copy in, merge, copy out), 2 buffer sets",
            "h2d_gbs_single_copy": round(h2d_gbs, 1),
            "d2h_gbs_single_copy": round(d2h_gbs, 1),
        }
        del dA, dB, dC, hC

    # ---- the other configs, measured the same way in the same process
    others = None
    if not args.no_other_configs and args.scale_log2 == 0:
        A = B = C = None
        torch.cuda.empty_cache()
        others = {}
        for ow in OTHER_CONFIGS:
            if ow == wl:
                continue
            k = max(5, min(args.steps, 20 if ow in SORTS else 100))
            others[ow] = other_config_line(measure(ow, args, device, world, k, args.warmup))
            torch.cuda.empty_cache()

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle (test infrastructure: the baseline leg only) on the same
        # seeded workload, built on the host
        h = synth.make_host(wl, scale_log2=args.scale_log2)
        rate, reps, best, units = oracle_rate(wl, h)
        cpu = {
            "value": rate,
            "unit": UNIT,
            "cores": 1,
            "kind": "oracle",
            "sample": f"the full workload ({units} outputs), median of {reps} single-thread oracle runs "
                      f"({best:.2f} s each)",
            "host_threads_available": os.cpu_count(),
        }

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value,
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": {"f64": "f64", "i64_desc": "int64", "sort_f32_desc": "f32", "sort_f64": "f64"}.get(
                wl, "int32" if wl in ("uniform", "evens_odds", "skewed") else "u32"),
            "data": "synthetic (seeded SplitMix64, sorted on device)",
            "config": {
                "workload": WORKLOADS[wl],
                "name": wl,
                "scale_log2": args.scale_log2,
                "m": m,
                "n": n,
                "l2": "inputs larger than L2 (no flush)" if flush is None else
                      "L2 flushed before every timed step (two writes of 2x L2, outside the timed events)",
                "parallelism": "replicas" if world > 1 else "single GPU",
            },
            "achieved_gbs": r["achieved_gbs"],
            "roofline": roofline,
            "kernel_time_ms": kernel_share,
            "other_configs": others,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": launches,
            "clocks": clocks,
        }
        if r["ms_per_step_median"] is not None:  # each call timed alone (flushed merges, sorts)
            line["ms_per_step_median"] = r["ms_per_step_median"]
            line["ms_per_step_min"] = r["ms_per_step_min"]
        if line["achieved_gbs"] is not None:
            line["pct_of_hbm_peak"] = round(100.0 * line["achieved_gbs"] / peak, 2)
            # the same against the nominal HBM3e bandwidth of one GB300 (context)
            line["pct_of_nominal_hbm"] = round(100.0 * line["achieved_gbs"] / NOMINAL_HBM_GBS, 2)
        print(json.dumps(line), flush=True)
    barrier(world, device)


# ------------------------------------------------- comparison merges --

def bench_baselines(args):
    """The unstaged merges the pages measure (one device thread; one thread
    per slice of 1, 4, 16, 64, 256 outputs with a co-rank search each, no
    shared memory) beside om_merge_i32, on an int32 merge workload (default
    of this mode: evens_odds, the pages' own input).  Each row: 3 warm-ups,
    then --steps timed calls, L2 flushed before each when the workload fits
    in L2; every row's output is compared with om_merge_i32's first.  Prints
    one JSON line."""
    import torch

    import ordered_merge_gb300 as om
    import synth

    rank, world, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    wl = args.workload
    if wl not in ("uniform", "evens_odds", "skewed"):
        raise SystemExit("--baselines needs an int32 merge workload (evens_odds, uniform, skewed)")
    d = synth.make_device(wl, device, scale_log2=args.scale_log2)
    A, B = d["A"], d["B"]
    total = A.numel() + B.numel()
    stream = torch.cuda.current_stream(device)
    flush = L2Flusher(device) if total * 8 < 2 * L2Flusher.l2_bytes(device) else None
    want = om.merge_i32(A, B)
    C = torch.empty_like(want)

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        if not torch.equal(C, want):
            raise RuntimeError("a comparison merge gave a different result")
        times = []
        for _ in range(reps):
            if flush is not None:
                flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times), min(times)

    rows = []
    reps = max(3, min(args.steps, 20))
    if total <= (1 << 23):
        med, best = timed(lambda: om.merge_i32_one_thread(A, B, C), max(3, reps // 4))
        rows.append({"kernel": "one device thread", "per_thread": total, "threads": 1, "ms_median": med,
                     "ms_min": best})
    for s_ in (1, 4, 16, 64, 256):
        med, best = timed(lambda: om.merge_i32_slices(A, B, C, per_thread=s_), reps)
        rows.append({"kernel": "one thread per slice, co-rank in global memory, no shared memory",
                     "per_thread": s_, "threads": (total + s_ - 1) // s_, "ms_median": med, "ms_min": best})
    med, best = timed(lambda: om.merge_i32(A, B, C), reps)
    rows.append({"kernel": "om_merge_i32 (range search + circular-buffer tile merge)", "per_thread": None,
                 "threads": None, "ms_median": med, "ms_min": best})
    one = rows[0]["ms_median"] if rows[0]["threads"] == 1 else None
    for r in rows:
        r["gbs"] = round(total * 8 / (r["ms_median"] / 1e3) / 1e9, 2)
        r["vs_one_thread"] = round(one / r["ms_median"], 2) if one else None
        r["ms_median"] = round(r["ms_median"], 5)
        r["ms_min"] = round(r["ms_min"], 5)
    line = {"metric": "comparison of merge kernels on one workload", "unit": "ms per call (median)",
            "workload": WORKLOADS[wl], "name": wl, "m": A.numel(), "n": B.numel(), "reps": reps,
            "l2": "flushed before every timed call" if flush is not None else "inputs larger than L2",
            "gbs_counts": "(m+n) x (4 B read + 4 B written); co-rank reads excluded", "rows": rows}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- reference arm --

def bench_reference(args):
    """The CPU oracle as it stands, timed on the host cores, on a bounded
    sample of the same workload per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import synth

    wl = args.workload
    # per-step sample: same recipe, scaled so all K + W steps take about
    # --ref-budget-s seconds on one core (a sort costs about log2(n) merges)
    budget_s = float(args.ref_budget_s)
    full = sum(synth.sizes(wl, 0))
    rate_guess = 2.5e8 / (max(1, full.bit_length() - 12) if wl in SORTS else 1)
    per_step = budget_s * rate_guess / max(1, args.steps + args.warmup)
    scale = 0
    while full >> scale > per_step and scale < 20:
        scale += 1
    d = synth.make_host(wl, scale_log2=scale)
    fn, total = oracle_call(wl, d)
    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    dt = time.perf_counter() - t0
    value = total * args.steps / dt
    m, n = synth.sizes(wl, scale)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"f64": "f64", "i64_desc": "int64", "sort_f32_desc": "f32", "sort_f64": "f64"}.get(
            wl, "int32" if wl in ("uniform", "evens_odds", "skewed") else "u32"),
        "data": "synthetic (seeded SplitMix64)",
        "config": {"workload": WORKLOADS[wl], "name": wl, "m": int(m), "n": int(n),
                   "sample_scale_log2": scale, "parallelism": "host CPU, 1 thread"},
        "cpu_baseline": {
            "value": value,
            "unit": UNIT,
            "cores": 1,
            "kind": "oracle",
            "sample": f"{wl} recipe scaled by 2^-{scale}: {total} outputs per step",
        },
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default="uniform", choices=sorted(WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--e2e-steps", type=int, default=16)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-other-configs", action="store_true",
                   help="skip the other configs the line records beside the headline one")
    p.add_argument("--ref-budget-s", type=float, default=60.0,
                   help="reference arm: CPU seconds the K + W oracle steps should take in total")
    p.add_argument("--scale-log2", type=int, default=0,
                   help="shrink the workload by 2^-s (profiling small cases; 0 = the named size)")
    p.add_argument("--baselines", action="store_true",
                   help="time the unstaged comparison merges beside om_merge_i32 (one JSON line)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.baselines:
        bench_baselines(args)
    elif args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()

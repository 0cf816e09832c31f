"""Benchmark: all-reduce algorithm bandwidth of the ring all-reduce engines.

One step = one in-place all-reduce of the workload (p rank buffers of N
elements) by the engine under test.  The headline workload is p = 8 virtual
ranks, N = 2^30 bf16 elements per rank (16 GiB in total, far above the
129 MB L2, so no flush is needed between steps), op = sum.

    python bench.py [--steps K] [--warmup W] [--engine fused|ring|ring_bidir|tree|all]
    python bench.py --impl reference      # the CPU oracle on the host cores
    python bench.py --sweep [--pair 0|1|2] # p = 16, N = 4^5 ... 4^13, every engine
    python bench.py --configs             # every workload on every engine
    python bench.py --hops                # smallest buffers, p = 2 ... 64
    python bench.py --next                # the widened rows on the 16 GiB shape

Metric: algBW = p * N * element bytes / time per step (GB/s), summed over
GPUs when run under torchrun (independent replicas, weak scaling).  Also
reported: each engine's fraction of the HBM roofline, with the roofline
bytes 2 p N e (fused) and 5 (p - 1) N e (ring and tree executors), against
the measured copy bandwidth in MEASURED_PEAKS.json.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as w  # noqa: E402

METRIC = "allreduce algBW GB/s (p·N·bytes/s) and % of GB300 HBM roofline, per engine"
DTYPE_SHORT = {"bfloat16": "bf16", "float32": "f32", "int32": "i32", "float16": "f16"}
FALLBACK_HBM_GBS = 6800.0


def roofline_bytes(engine: str, p: int, n: int, e: int) -> int:
    """Minimum HBM bytes of one all-reduce: fused reads and writes every rank
    once; the ring moves 3 elements per reduce-scatter hop and 2 per
    all-gather hop over (p - 1) steps of n elements in total each."""
    if engine in ("fused", "fused_tree"):
        return 2 * p * n * e
    return 5 * (p - 1) * n * e


def dram_floor_bytes(p: int, n: int, e: int) -> int:
    """DRAM bytes no in-place all-reduce can go below: every rank's input
    read once and its result written once, whatever the engine."""
    return 2 * p * n * e


def roofline_object(engine: str, p: int, n: int, e: int, ms_per_launch: float, peak: float, peak_kind: str,
                    traffic, l2_bytes=None):
    """The bench line's roofline object for one engine.

    frac: the engine's algorithmic bytes (roofline_bytes) per launch time
    over the HBM peak.  For the fused engine these are the DRAM floor, so
    frac is a true fraction of HBM bandwidth.  For the executors they count
    the schedule's element moves, 5 (p - 1) n e, most of which L2 serves:
    that frac is not bounded by HBM peak.  dram_frac (measured DRAM bytes,
    `traffic`) and floor_frac (the 2 p n e floor) are the bounded ones."""
    R = roofline_bytes(engine, p, n, e)
    F = dram_floor_bytes(p, n, e)
    sec = ms_per_launch * 1e-3
    achieved = R / sec / 1e9
    obj = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
           "frac": round(achieved / peak, 4), "traffic": traffic, "algorithmic_bytes": R,
           "peak_kind": f"of {peak_kind}",
           "frac_kind": ("DRAM floor bytes (inputs read once, results written once) per launch time"
                         if R == F else
                         "algorithmic element moves 5(p-1)Ne per launch time; L2 serves part of them, "
                         "so this is not bounded by HBM peak (see dram_frac, floor_frac)"),
           "floor_bytes": F, "floor_frac": round(F / sec / 1e9 / peak, 4)}
    if traffic:
        obj["dram_frac"] = round(traffic / sec / 1e9 / peak, 4)
        obj["l2_served"] = round(1.0 - traffic / R, 4)
        obj["traffic_over_floor"] = round(traffic / F, 4)
    else:
        obj["dram_frac"] = None
        obj["l2_served"] = None
        obj["traffic_over_floor"] = None
    if l2_bytes:
        # bytes through L2 (lts__t_bytes) per launch time: beside ncu's own
        # L2 throughput percentage, the load the schedule puts on L2
        obj["l2_bytes"] = l2_bytes
        obj["l2_gbs"] = round(l2_bytes / sec / 1e9, 1)
    return obj


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources that make each timed kernel and its launch configuration.
ENGINE_SOURCES = {
    "fused": ("rar_internal.h", "elem_ops.cuh", "fused_impl.cuh", "fused.cu", "fused_stream.cu", "rar_api.cu"),
    "ring": ("rar_internal.h", "elem_ops.cuh", "flag_sync.cuh", "ring.cu", "rar_api.cu"),
    "tree": ("rar_internal.h", "elem_ops.cuh", "flag_sync.cuh", "tree_plan.h", "tree.cu", "rar_api.cu"),
}
ENGINE_SOURCES["ring_bidir"] = ENGINE_SOURCES["ring"]


def _code_only(text: str) -> str:
    """C/C++ source without comments and blank lines (string literals in
    these sources hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(engine: str) -> str:
    """Hash of the code (comments dropped) of the CUDA sources behind one
    engine's kernel, to tell whether stored ncu counters still describe the
    kernel being timed."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ring_all_reduce_rar_gb300", "csrc")
    for name in ENGINE_SOURCES[engine]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def stored_counters(engine: str, workload: str):
    """The committed ncu counters of one engine's launch on a workload
    (profiles/traffic.json), or None if the kernel changed since the
    capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    ent = d.get(workload, {}).get(engine)
    if not ent or engine not in ENGINE_SOURCES or ent.get("kernel_source_hash") != kernel_source_hash(engine):
        return None
    return ent


def stored_traffic(engine: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel changed since the capture."""
    ent = stored_counters(engine, workload)
    return ent.get("dram_bytes_per_launch") if ent else None


class ClockSampler:
    """nvidia-smi samples (every 200 ms) around the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not getattr(self, "lines", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unparsed"], "samples": 0}
        load = [s for s, pw in zip(sm, power) if pw > 200.0] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# ------------------------------------------------------------------ our arm

def time_engine(rar, engine, rows, op, steps, warmup, dist_ctx):
    """Warm up, then time exactly `steps` all-reduces with CUDA events on the
    stream the kernels are launched on."""
    stream = torch.cuda.current_stream()
    with rar.Handle(torch.cuda.current_device(), skip_pointer_check=True, **VARIANTS[engine]) as h:
        for _ in range(warmup):
            h.allreduce(rows, op=op, stream=stream)
        h.check()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dist_ctx.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(steps):
            h.allreduce(rows, op=op, stream=stream)
        end.record(stream)
        torch.cuda.synchronize()
        dist_ctx.barrier()
        rc = h.status()
        if rc != 0:
            raise RuntimeError(f"engine {engine}: device status {rc}: {rar.rar_last_error(h.h)}")
        ms = start.elapsed_time(end)
    return dist_ctx.max(ms)


def time_e2e(rar, engine, host_rows, op, steps, warmup, dist_ctx):
    """End to end through the public host-buffer call on pinned host rank
    buffers: every step the GPU reads all p inputs from host memory and
    writes all p results back (rar_allreduce_host's zero-copy form)."""
    stream = torch.cuda.current_stream()
    with rar.Handle(torch.cuda.current_device(), skip_pointer_check=True, **VARIANTS[engine]) as h:
        def step():
            h.allreduce_host(host_rows, None, op=op, stream=stream)
        for _ in range(warmup):
            step()
        h.check()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dist_ctx.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        dist_ctx.barrier()
        ms = start.elapsed_time(end)
    return dist_ctx.max(ms)


def host_link_copy_gbs(dev_buf, nbytes: int = 1 << 30, reps: int = 3):
    """Copy rate of the host link with both directions busy: a pinned-host to
    device copy and a device to pinned-host copy of `nbytes` each, on two
    streams at once (bytes both ways over the time), best of `reps`.  The
    yardstick for the host-buffer call, which reads its inputs from and
    writes its results to host memory at the same time."""
    try:
        flat = dev_buf.view(-1).view(torch.uint8)
        nbytes = min(nbytes, flat.numel() // 2)
        h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        d_in, d_out = flat[:nbytes], flat[nbytes:2 * nbytes]
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            with torch.cuda.stream(s1):
                d_in.copy_(h_in, non_blocking=True)
            with torch.cuda.stream(s2):
                h_out.copy_(d_out, non_blocking=True)
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        del h_in, h_out
        return round(2 * nbytes / best / 1e9, 1)
    except RuntimeError:
        return None


class DistCtx:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.dist = dist

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, v: float) -> float:
        if self.world == 1:
            return v
        t = torch.tensor([v], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            self.dist.destroy_process_group()


def cpu_baseline(cfg, op):
    """The oracle as it stands, single-threaded on a host core, on a bounded
    sample of the workload (same p and dtype, N = 2^25 per rank)."""
    import numpy as np
    import oracle
    p, dtype = cfg["p"], cfg["dtype"]
    n = 1 << 25 if cfg["n"] > (1 << 25) else cfg["n"]
    _, rows = w.make_inputs(p, n, dtype, cfg["dist"], w.seed_of(cfg["index"]))
    base = [w.to_storage_numpy(t).copy() for t in rows]
    times = []
    for _ in range(2):
        bufs = [b.copy() for b in base]
        t0 = time.perf_counter()
        oracle.simulate(bufs, dtype, op)
        times.append(time.perf_counter() - t0)
    e = torch.tensor([], dtype=w.TORCH_DTYPES[dtype]).element_size()
    t = min(times)
    return {"value": round(p * n * e / t / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"schedule simulator, p={p}, N={n} {dtype} per rank (of N={cfg['n']}), op={op}, "
                      f"best of {len(times)}, single thread"}


def run_ours(args):
    import ring_all_reduce_rar_gb300 as rar
    rar.load_library()
    ctx = DistCtx()
    torch.cuda.set_device(ctx.local_rank)
    dev = torch.device("cuda", ctx.local_rank)
    cfg = dict(w.WORKLOADS[args.workload])
    if args.n:
        cfg["n"] = args.n
    p, n, dtype, op = cfg["p"], cfg["n"], cfg["dtype"], args.op or cfg["ops"][0]
    e = torch.tensor([], dtype=w.TORCH_DTYPES[dtype]).element_size()
    # each GPU holds its own replica of the workload (distinct seed per GPU)
    seed = w.seed_of(cfg["index"]) + 1000 * ctx.rank
    big, rows = w.make_inputs(p, n, dtype, cfg["dist"], seed, device=dev)
    torch.cuda.synchronize()
    engines = ["fused", "ring", "ring_bidir", "tree"] if args.engine == "all" else [args.engine]
    peak, peak_kind = hbm_peak()
    results = {}
    with ClockSampler(ctx.local_rank) as clk:
        for eng in engines:
            ms = time_engine(rar, eng, rows, op, args.steps, args.warmup, ctx)
            per_step = ms / args.steps
            results[eng] = {
                "value": round(ctx.world * p * n * e / (per_step * 1e-3) / 1e9, 2),
                "ms_per_step": round(per_step, 4),
                "roofline": roofline_object(eng, p, n, e, per_step, peak, peak_kind,
                                            stored_traffic(eng, args.workload),
                                            (stored_counters(eng, args.workload) or {}).get("lts_bytes_per_launch")),
            }
    clocks = clk.summary()
    head = engines[0]
    e2e = None
    if not args.no_e2e:
        e2e_engine = head
        host_rows = None
        try:
            host_big = torch.empty(big.shape, dtype=big.dtype, pin_memory=True)
            host_big.copy_(big)
            host_rows = [host_big[r, :n] for r in range(p)]
        except RuntimeError as ex:
            e2e = {"value": None, "unit": "GB/s", "unavailable": f"pinned host buffers: {ex}"[:200]}
        if host_rows is not None:
            k = args.steps
            ms = time_e2e(rar, e2e_engine, host_rows, op, k, args.warmup, ctx)
            link = host_link_copy_gbs(big)
            host_gbs = 2 * p * n * e / (ms / k * 1e-3) / 1e9
            e2e = {"value": round(ctx.world * p * n * e / (ms / k * 1e-3) / 1e9, 2), "unit": "GB/s",
                   "h2d_bytes_per_step": p * n * e, "d2h_bytes_per_step": p * n * e,
                   "engine": e2e_engine, "steps": k, "warmup": args.warmup, "ms_per_step": round(ms / k, 3),
                   "mode": "rar_allreduce_host on pinned host buffers: the kernel reads the inputs from and "
                           "writes the results to host memory over the host link (no staging copies)",
                   "bound": "host link: every step moves 2 p N e bytes across it (inputs in, results out)",
                   "host_link_gbs": round(host_gbs, 1),
                   "host_link_copy_gbs": link,
                   "host_link_frac": round(host_gbs / link, 4) if link else None}
            del host_big, host_rows
    cpu = None
    if ctx.rank == 0 and ctx.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, op)
    if ctx.rank == 0:
        line = {
            "metric": METRIC,
            "value": results[head]["value"],
            "unit": "GB/s",
            "n_gpus": ctx.world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": results[head]["ms_per_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": DTYPE_SHORT[dtype],
            "data": "synthetic (seeded splitmix64 inputs, N(0, 1e-2) in bf16)",
            "config": {"workload": args.workload, "p": p, "n": n, "op": op, "engine": head,
                       "l2": f"inputs ({p * n * e / 2**30:.3g} GiB) vs L2 (129 MB): "
                             + ("larger, no flush needed" if p * n * e > 4 * 129e6 else "NOT larger"),
                       "parallelism": "independent replica per GPU"},
            "roofline": results[head]["roofline"],
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clocks,
            "engines": results,
        }
        print(json.dumps(line), flush=True)
    ctx.close()


# ------------------------------------------------------------------ size sweep

# Engine variants of the sweeps: "ring" and "tree" pick their hand-off by
# size (rar_options.protocol auto); the "_simple" / "_ll" variants force one.
VARIANTS = {"fused": dict(engine="fused"), "ring": dict(engine="ring"),
            "ring_simple": dict(engine="ring", protocol="simple"), "ring_ll": dict(engine="ring", protocol="ll"),
            "ring_bidir": dict(engine="ring_bidir"), "fused_tree": dict(engine="fused_tree"), "tree": dict(engine="tree"),
            "tree_simple": dict(engine="tree", protocol="simple"), "tree_ll": dict(engine="tree", protocol="ll")}


def run_sweep(args):
    """Device time per call across message sizes (the p = 16 sweep workload),
    one JSON line per (engine, size).  The GPU is first held by a short sleep
    kernel so that the host can queue K calls ahead; CUDA events around the K
    calls then time back-to-back device execution, not host call overhead."""
    import ring_all_reduce_rar_gb300 as rar
    rar.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dtype, op, dist = w.SWEEP_PAIRS[args.pair]
    p = w.SWEEP_P
    e = torch.tensor([], dtype=w.TORCH_DTYPES[dtype]).element_size()
    engines = (["fused", "ring", "ring_simple", "ring_ll", "ring_bidir", "tree", "tree_simple", "tree_ll"]
               if args.engine == "all" else [args.engine])
    for n in w.SWEEP_SIZES:
        _, rows = w.make_inputs(p, n, dtype, dist, w.seed_of(w.SWEEP_INDEX), device=dev)
        k = 200 if n <= 4 ** 9 else 20
        for eng in engines:
            try:
                us = device_us_per_call(rar, VARIANTS[eng], rows, op, k)
            except rar.RarError as ex:
                if ex.code != 2:  # RAR_EUNSUPPORTED: e.g. too large for the low-latency mailbox
                    raise
                continue
            rb = (2 * p * n * e) if eng == "fused" else 5 * (p - 1) * n * e
            print(json.dumps({"sweep": f"p{p}_{dtype}_{op}", "engine": eng, "n": n, "us_per_call": round(us, 2),
                              "algbw_gbs": round(p * n * e / us / 1e3, 2),
                              "roofline_frac": round(rb / us / 1e3 / hbm_peak()[0], 4)}), flush=True)
        del rows
        torch.cuda.empty_cache()


def run_hops(args):
    """Per-call time of the smallest buffers (N = 64 p fp32 elements per
    rank) for p = 2 ... 64: with the data negligible, the time is the fixed
    cost of a call plus the schedule's steps (2 (p - 1) ring hops,
    2 ceil(log2 p) tree steps), for each hand-off.  One JSON line per p."""
    import ring_all_reduce_rar_gb300 as rar
    rar.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for p in [2, 4, 8, 16, 32, 64]:
        n = 64 * p
        _, rows = w.make_inputs(p, n, "float32", ("normal", 1.0), w.seed_of(w.SWEEP_INDEX), device=dev)
        line = {"hops": f"p{p}_n{n}_float32", "p": p, "n": n, "ring_steps": 2 * (p - 1),
                "tree_steps": 2 * max(1, (p - 1).bit_length())}
        for eng in ["fused", "ring_simple", "ring_ll", "tree_simple", "tree_ll"]:
            line[eng + "_us"] = round(device_us_per_call(rar, VARIANTS[eng], rows, "sum", 200), 2)
        print(json.dumps(line), flush=True)


def run_next(args):
    """The widened rows on the 16 GiB workload shape (p = 8, N = 2^30), device
    time per call and the fraction of each one's minimum-traffic roofline, one
    JSON line each: reduce-scatter and all-gather alone, the hierarchical
    schedule, and fp16 with the post- and pre-divided average."""
    import ring_all_reduce_rar_gb300 as rar
    rar.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak = hbm_peak()[0]
    cfg = w.WORKLOADS["p8_n1073741824_bf16"]
    p, n, e = cfg["p"], cfg["n"], 2

    def emit(row, engine, us, bytes_):
        print(json.dumps({"row": row, "engine": engine, "p": p, "n": n, "us_per_call": round(us, 2),
                          "algbw_gbs": round(p * n * e / us / 1e3, 2), "roofline_bytes": bytes_,
                          "roofline_frac": round(bytes_ / us / 1e3 / peak, 4)}), flush=True)

    big, rows = w.make_inputs(p, n, "bfloat16", cfg["dist"], w.seed_of(cfg["index"]), device=dev)
    # reduce-scatter and all-gather alone ("Ring All-Reduce, in depth",
    # "Trade-offs").  Minimum bytes: the fused reduce-scatter reads every rank
    # and writes the owner's chunk, (p + 1) N e; its all-gather reads the owner
    # and writes the p - 1 others, p N e; the ring's halves move 3 (p - 1) N e
    # and 2 (p - 1) N e.
    for eng, rs_bytes, ag_bytes in [("fused", (p + 1) * n * e, p * n * e),
                                    ("ring", 3 * (p - 1) * n * e, 2 * (p - 1) * n * e)]:
        for fn, b in [("reduce_scatter", rs_bytes), ("all_gather", ag_bytes)]:
            emit(fn, eng, device_us_per_call_fn(rar, VARIANTS[eng], rows, fn, 10), b)
    # hierarchical 2D schedule ("Ring All-Reduce, in depth", "Hierarchy"):
    # the same minimum bytes as the flat engines
    for g in (2, 4):
        for eng in ("fused", "ring"):
            opts = dict(VARIANTS[eng], hier_group=g)
            if eng == "fused":
                opts["fused_path"] = "registers"  # the hierarchical order runs on the per-thread path
            emit(f"hierarchical g={g}", eng, device_us_per_call(rar, opts, rows, "sum", 10),
                 2 * p * n * e if eng == "fused" else 5 * (p - 1) * n * e)
    del big, rows
    torch.cuda.empty_cache()
    # fp16 with the post- and pre-divided average ("Ring All-Reduce, in
    # depth", "Failure modes")
    big, rows = w.make_inputs(p, n, "float16", cfg["dist"], w.seed_of(cfg["index"]), device=dev)
    for op in ("sum", "avg", "avg_prediv"):
        for eng in ("fused", "ring"):
            emit(f"fp16 {op}", eng, device_us_per_call(rar, VARIANTS[eng], rows, op, 10),
                 2 * p * n * e if eng == "fused" else 5 * (p - 1) * n * e)
    del big, rows
    torch.cuda.empty_cache()


def device_us_per_call_fn(rar, opts, rows, fn, k):
    """As device_us_per_call, for the handle method `fn` (reduce_scatter,
    all_gather) on the rank buffers."""
    with rar.Handle(0, skip_pointer_check=True, **opts) as h:
        call = getattr(h, fn)
        for _ in range(3):
            call(rows)
        h.check()
        torch.cuda.synchronize()
        torch.cuda._sleep(200_000_000)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(k):
            call(rows)
        end.record()
        torch.cuda.synchronize()
        if h.status() != 0:
            raise RuntimeError(rar.rar_last_error(h.h))
        return start.elapsed_time(end) * 1e3 / k


def device_us_per_call(rar, opts, rows, op, k):
    """Device time per call: the GPU is held by a short sleep kernel while
    the host queues k calls, so events time back-to-back execution only."""
    with rar.Handle(0, skip_pointer_check=True, **opts) as h:
        for _ in range(3):
            h.allreduce(rows, op=op)
        h.check()
        torch.cuda.synchronize()
        torch.cuda._sleep(200_000_000)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for _ in range(k):
            h.allreduce(rows, op=op)
        end.record()
        torch.cuda.synchronize()
        if h.status() != 0:
            raise RuntimeError(rar.rar_last_error(h.h))
        return start.elapsed_time(end) * 1e3 / k


def run_configs(args):
    """Every workload (p = 4 ... 64) on every engine: device time per call and
    the fraction of the engine's HBM roofline; one JSON line each."""
    import ring_all_reduce_rar_gb300 as rar
    rar.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak = hbm_peak()[0]
    engines = [(e, VARIANTS[e]) for e in ("fused", "ring", "ring_simple", "ring_ll", "ring_bidir", "tree")]
    for name, cfg in w.WORKLOADS.items():
        p, n, dtype = cfg["p"], cfg["n"], cfg["dtype"]
        e = torch.tensor([], dtype=w.TORCH_DTYPES[dtype]).element_size()
        big, rows = w.make_inputs(p, n, dtype, cfg["dist"], w.seed_of(cfg["index"]), device=dev)
        for op in cfg["ops"]:
            for eng, opts in engines:
                k = 10 if p * n * e > 1e9 else (50 if p * n * e > 1e7 else 200)
                try:
                    us = device_us_per_call(rar, opts, rows, op, k)
                except rar.RarError as ex:
                    if ex.code != 2:  # RAR_EUNSUPPORTED: too large for the low-latency mailbox
                        raise
                    continue
                rb = 2 * p * n * e if eng == "fused" else 5 * (p - 1) * n * e
                print(json.dumps({"workload": name, "op": op, "engine": eng, "us_per_call": round(us, 2),
                                  "algbw_gbs": round(p * n * e / us / 1e3, 2),
                                  "roofline_frac": round(rb / us / 1e3 / peak, 4)}), flush=True)
        del big, rows
        torch.cuda.empty_cache()


MID_SHAPES = [(8, 500_000, "bfloat16"), (8, 1_000_000, "bfloat16"), (8, 2_000_000, "bfloat16"),
              (8, 1_000_000, "float32"), (8, 2_400_000, "float32"), (4, 1_000_000, "float32"),
              (4, 2_000_000, "float32"), (16, 500_000, "bfloat16"), (16, 524_288, "bfloat16"),
              (24, 500_000, "bfloat16"), (32, 500_000, "bfloat16"), (32, 524_288, "bfloat16"),
              (32, 500_000, "float32"), (40, 1_048_576, "bfloat16"), (64, 250_000, "bfloat16"),
              (64, 262_144, "bfloat16")]


def run_mid(args):
    """The fused engine on mid-size buffers (1-16 MB per rank, p = 4 ... 64,
    chunk starts aligned to 16 bytes or not): device time per call and the
    fraction of the 2 p N e roofline, one JSON line per shape.  Values N(0,
    1e-2) (fp32 N(0, 1e-3)), sum."""
    import ring_all_reduce_rar_gb300 as rar
    rar.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak = hbm_peak()[0]
    for p, n, dtype in MID_SHAPES:
        e = torch.tensor([], dtype=w.TORCH_DTYPES[dtype]).element_size()
        dist = ("normal", 1e-3 if dtype == "float32" else 1e-2)
        big, rows = w.make_inputs(p, n, dtype, dist, 5, device=dev)
        us = device_us_per_call(rar, VARIANTS["fused"], rows, "sum", 50)
        chunk = n // p
        print(json.dumps({"p": p, "n": n, "dtype": dtype, "chunk_starts_aligned": all(
            ((c * chunk + min(c, n % p)) * e) % 16 == 0 for c in range(1, p)),
            "us_per_call": round(us, 2), "algbw_gbs": round(p * n * e / us / 1e3, 2),
            "roofline_frac": round(2 * p * n * e / us / 1e3 / peak, 4)}), flush=True)
        del big, rows
        torch.cuda.empty_cache()


def run_trace(args):
    """The executors' step trace (rar_options.trace) on one workload: per
    engine, the share of time the first warp of each CTA spent waiting for its
    neighbour, and per schedule step the mean over ranks of the wait and work
    time summed over the rank's CTAs; one JSON line per engine.  A traced call
    runs the traced kernel instantiation, so its times are not bench times."""
    import ring_all_reduce_rar_gb300 as rar
    rar.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cfg = w.WORKLOADS[args.workload]
    p, dtype, op = cfg["p"], cfg["dtype"], args.op or cfg["ops"][0]
    n = args.n or cfg["n"]
    big, rows = w.make_inputs(p, n, dtype, cfg["dist"], w.seed_of(cfg["index"]), device=dev)
    for eng in ("ring", "ring_bidir", "tree"):
        opts = dict(engine=eng, trace=True, **({} if eng == "ring_bidir" else dict(protocol="simple")))
        with rar.Handle(0, skip_pointer_check=True, **opts) as h:
            for _ in range(args.warmup):
                h.allreduce(rows, op=op)
            torch.cuda.synchronize()
            h.check()
            work, wait = h.trace(p)
        steps = len(work[0])
        tw, tt = sum(map(sum, work)), sum(map(sum, wait))
        print(json.dumps({
            "workload": args.workload, "n": n, "op": op, "engine": eng, "steps": steps,
            "wait_share": round(tt / max(1, tw + tt), 4),
            "wait_us_per_step": [round(sum(wait[r][s] for r in range(p)) / p / 1e3, 1) for s in range(steps)],
            "work_us_per_step": [round(sum(work[r][s] for r in range(p)) / p / 1e3, 1) for s in range(steps)],
        }), flush=True)
    del big, rows
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The oracle (plain C simulator of the pages' schedule) on the host
    cores, same metric and workload, one bounded sample per step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    cfg = w.WORKLOADS[args.workload]
    p, dtype, op = cfg["p"], cfg["dtype"], args.op or cfg["ops"][0]
    n = min(cfg["n"], 1 << 22)
    e = torch.tensor([], dtype=w.TORCH_DTYPES[dtype]).element_size()
    _, rows = w.make_inputs(p, n, dtype, cfg["dist"], w.seed_of(cfg["index"]))
    base = [w.to_storage_numpy(t).copy() for t in rows]
    for _ in range(args.warmup):
        oracle.simulate([b.copy() for b in base], dtype, op)
    total = 0.0
    for _ in range(args.steps):
        bufs = [b.copy() for b in base]
        t0 = time.perf_counter()
        oracle.simulate(bufs, dtype, op)
        total += time.perf_counter() - t0
    per = total / args.steps
    value = round(p * n * e / per / 1e9, 4)
    sample = f"schedule simulator, p={p}, N={n} {dtype} per rank (of N={cfg['n']}), op={op}, single thread"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_SHORT[dtype],
        "data": "synthetic", "config": {"workload": args.workload, "p": p, "n": cfg["n"], "op": op,
                                        "engine": "oracle"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--engine", choices=["fused", "ring", "ring_simple", "ring_ll", "ring_bidir", "fused_tree", "tree",
                                         "tree_simple", "tree_ll", "all"], default="all")
    ap.add_argument("--sweep", action="store_true",
                    help="device time per call over the p = 16 message-size sweep (not the benchmark line)")
    ap.add_argument("--pair", type=int, default=0, help="--sweep: dtype/op pair of the sweep workload (0..2)")
    ap.add_argument("--next", action="store_true",
                    help="reduce-scatter / all-gather alone, the hierarchical schedule, fp16 averages (16 GiB shape)")
    ap.add_argument("--hops", action="store_true",
                    help="per-call time of the smallest buffers for p = 2 ... 64 (fixed cost + step latency)")
    ap.add_argument("--configs", action="store_true",
                    help="device time per call of every workload on every engine (not the benchmark line)")
    ap.add_argument("--mid", action="store_true",
                    help="the fused engine on mid-size buffers, p = 4 ... 64 (not the benchmark line)")
    ap.add_argument("--trace", action="store_true",
                    help="step trace of the ring, bidirectional ring and tree executors on --workload")
    ap.add_argument("--workload", choices=sorted(w.WORKLOADS), default="p8_n1073741824_bf16")
    ap.add_argument("--op", choices=["sum", "avg", "max"], default=None)
    ap.add_argument("--n", type=int, default=None,
                    help="elements per rank instead of the workload's N (small cases for ncu captures)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.sweep:
        run_sweep(args)
    elif args.hops:
        run_hops(args)
    elif args.next:
        run_next(args)
    elif args.configs:
        run_configs(args)
    elif args.trace:
        run_trace(args)
    elif args.mid:
        run_mid(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

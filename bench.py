#!/usr/bin/env python3
"""Benchmark of one decode step of the paged read: append + read (+ reduce).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Prints ONE JSON line.  ``value`` is KV GB/s: the K and V bytes of every row's
history (sum_r c_r * 2 * kv_heads * head_dim * elem_size) read by one step,
divided by the device time of the step (CUDA events, K steps between a
barrier + synchronize on both sides, max over ranks), aggregated over ranks.
Inputs are resident in HBM before timing.  ``e2e`` is the same metric when
every step also copies its per-step inputs (q, new K/V, slot mapping, block
tables, context lengths) from pinned host memory and reads the output back.
``--impl reference`` times the CPU oracle instead, on a bounded sample.

Multi-GPU (torchrun): rows are independent, so each rank runs its own
replica of the workload (its own pool and batch) with no collective on the
data path ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math

import numpy as np
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as wl  # noqa: E402

DEFAULT_WORKLOAD = "bf16-long"
REF_TOTAL_S = 150.0  # oracle work of the whole --impl reference run, about
METRIC = "paged decode read: KV GB/s and % of GB300 HBM peak; µs per decode step"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2**20


# ------------------------------------------------------------ accounting ---
def algorithmic_bytes(w: wl.Workload, md: wl.Metadata) -> dict:
    """Bytes one step must move at minimum, by kernel.

    decode: every history token's K and V rows once, q once, out once, the
    table entries the walk needs once, the context lengths once (the split
    partials are not algorithmic: they are this implementation's overhead),
    plus the fused append: the new tokens' K/V read once and written once and
    their slots.
    """
    cl = md.context_lens.to(torch.int64)
    es = w.elem_size
    qn = w.query_len
    kv = int(cl.sum()) * 2 * w.kv_heads * w.head_dim * es
    qo = 2 * w.rows * qn * w.q_heads * w.head_dim * es
    tab = int(((cl + w.block_size - 1) // w.block_size).sum()) * 4 + 4 * w.rows
    app = 2 * 2 * w.rows * qn * w.kv_heads * w.head_dim * es + 8 * w.rows * qn
    return {"kv": kv, "decode": kv + qo + tab + app, "append": app}


def l2_plan(kv_bytes_per_step: int, pool_bytes: int) -> int:
    """How the timed steps keep K/V out of L2: the number of pool copies the
    steps rotate among, or 0 for an L2 flush between steps.

    K/V of at least 4x L2 per step needs nothing (1 copy).  A smaller pool of
    at least L2/16 is rotated: copies of it, more than 3x L2 in all, are read
    in turn, so no step finds its K/V in L2 and steps still run back to back.
    A tinier pool gets a 2x L2 buffer written between timed steps (outside
    the timed region).
    """
    if kv_bytes_per_step >= 4 * L2_BYTES:
        return 1
    n = math.ceil(3 * L2_BYTES / pool_bytes) + 1
    return n if n <= 48 else 0


def measured_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sources_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_np_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str) -> float | None:
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", f"decode_{workload}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"kernel_sources_sha256:\s*([0-9a-f]+)", txt)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m or not t or m.group(1) != kernel_sources_hash():
        return None
    return float(t.group(1))


# ---------------------------------------------------------------- clocks ---
class _Nvml:
    """Read-only NVML queries through ctypes (the library ships with the
    driver): SM clock, its maximum and the active clock-event reasons."""
    SM = 1  # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id: str):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(),
                                                     ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for " + pci_bus_id)
        try:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        c = self.c
        sm, mx, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        if (self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, c.byref(sm)) != 0 or
                self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, c.byref(mx)) != 0):
            return None
        if self.reasons_fn(self.h, c.byref(rs)) != 0:
            return None
        return (float(sm.value), float(mx.value),
                [n for b, n in self.REASONS.items() if rs.value & b])

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clocks and clock-event reasons sampled while the timed steps run:
    NVML polled every 2 ms where it loads (a timed region of a few ms still
    gets samples), else ``nvidia-smi -lms 200``."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device: torch.device):
        self.gpu = None
        try:  # NVML and nvidia-smi want the PCI bus id of the device torch is using
            pr = torch.cuda.get_device_properties(device)
            self.gpu = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        except Exception:
            pass
        self.proc = None
        self.nvml = None
        self.stop = threading.Event()
        self.t = None
        self.samples: list[tuple[float, float, float, list]] = []  # (time, sm, max, reasons)
        self.window = None
        self.source = None

    def __enter__(self):
        if self.gpu is not None:
            try:
                self.nvml = _Nvml(self.gpu)
                if self.nvml.sample() is None:
                    raise OSError("NVML query failed")
                self.source = "nvml, 2 ms"
                self.t = threading.Thread(target=self._poll, daemon=True)
                self.t.start()
                time.sleep(0.05)
                return self
            except (OSError, AttributeError):
                self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *([f"--id={self.gpu}"] if self.gpu else []),
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi, 200 ms"
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _poll(self):
        while not self.stop.is_set():
            x = self.nvml.sample()
            if x is not None:
                self.samples.append((time.time(), *x))
            self.stop.wait(0.002)

    def _read(self):
        for ln in self.proc.stdout:
            parts = [p.strip() for p in ln.strip().split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            rs = [n for n, v in zip(self.NAMES, parts[5:9]) if v.lower().startswith("active")]
            self.samples.append((time.time(), sm, mx, rs))

    def mark(self, start: float, end: float) -> None:
        """The host wall-clock window of the timed region."""
        self.window = (start, end)

    def __exit__(self, *exc):
        if self.nvml is not None:
            time.sleep(0.01)
            self.stop.set()
            self.t.join(timeout=5)
            self.nvml.close()
        elif self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self) -> dict:
        samples = self.samples
        inside = []
        if self.window is not None:  # samples taken while the timed steps ran
            inside = [x for x in samples
                      if self.window[0] <= x[0] <= self.window[1] + 0.005]
        use = inside or samples
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = sorted({r for x in use for r in x[3]})
        return {"sm_mhz": statistics.median(x[1] for x in use),
                "sm_max_mhz": max(x[2] for x in use), "reasons": reasons,
                "samples": len(use), "in_timed_region": bool(inside), "source": self.source}


# ------------------------------------------------------------ distributed --
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle ---
def oracle_sample(inp: wl.Inputs, budget_s: float, seed: int = 0, threads: int = 1,
                  token_cap: int | None = None, hosts: dict | None = None) -> dict:
    """Time the oracle (the C oracle as it stands) on randomly chosen rows of
    the step until ``budget_s`` seconds of wall time are done.  ``threads``
    rows run at once, each in its own host thread (the C calls release the
    interpreter lock); each batch's host copies are made before its clock
    starts, or taken from ``hosts`` (row -> copy) when given -- the oracle's
    append writes the same token again, so a copy serves many steps.
    ``token_cap`` reads at most that many history tokens of a row (a prefix:
    the same work per token, for short samples)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    w = inp.w
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(w.rows, generator=g).tolist()
    done_rows, kv_bytes, elapsed = [], 0, 0.0
    per_token = 2 * w.kv_heads * w.head_dim * w.elem_size

    def one(host):
        kp, vp = host["k_pool"], host["v_pool"]
        oracle.kv_append(kp, vp, host["k_new"], host["v_new"], host["slot_mapping"])
        oracle.paged_decode(host["q"], kp, vp, host["block_tables"], host["context_lens"],
                            w.softmax_scale)

    def copy_of(r):
        if hosts is not None and r in hosts:
            return hosts[r]
        h = wl.row_subproblem(inp, [r], max_tokens=token_cap)
        if hosts is not None:
            hosts[r] = h
        return h

    with ThreadPoolExecutor(max_workers=threads) as ex:
        for i in range(0, len(order), threads):
            batch = order[i:i + threads]
            hs = [copy_of(r) for r in batch]
            t0 = time.perf_counter()
            list(ex.map(one, hs))
            elapsed += time.perf_counter() - t0
            done_rows += batch
            kv_bytes += sum(int(h["context_lens"][0]) for h in hs) * per_token
            if elapsed >= budget_s:
                break
    return {"rows": done_rows, "kv_bytes": kv_bytes, "seconds": elapsed, "threads": threads,
            "gbs": kv_bytes / elapsed / 1e9 if elapsed > 0 else None}


def host_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def cpu_model() -> str:
    """The host CPU's model name as lscpu reports it (else the machine type)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() in ("Model name", "Model Name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine() or "unknown"


# ---------------------------------------------------------------- arms ----
def run_reference(args, w: wl.Workload, dist, rank):
    """The oracle arm: each step is the oracle on a bounded sample of rows."""
    if rank != 0:
        return None
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = wl.make_inputs(w, device=dev, poison=False)
    nt = host_threads()
    # the whole arm within a few minutes: about REF_TOTAL_S of oracle work in
    # all; rows are cut to a prefix when one batch of whole rows would exceed
    # a step's share (the per-token rate comes from a one-row calibration)
    step_budget = min(args.ref_step_seconds, REF_TOTAL_S / max(1, args.steps + args.warmup))
    cal = oracle_sample(inp, 0.0, seed=999, threads=1, token_cap=2048)
    tok_s = (cal["kv_bytes"] / (2 * w.kv_heads * w.head_dim * w.elem_size)) / max(
        cal["seconds"], 1e-6)
    token_cap = max(w.block_size, int(tok_s * step_budget))
    cap = token_cap if token_cap < int(inp.md.context_lens.max()) else None
    hosts: dict = {}  # host copies made once, reused by every step
    for i in range(args.warmup):
        oracle_sample(inp, step_budget, seed=1000 + i, threads=nt, token_cap=cap, hosts=hosts)
    times, kvb, rows = [], 0, []
    for i in range(args.steps):
        s = oracle_sample(inp, step_budget, seed=i, threads=nt, token_cap=cap, hosts=hosts)
        times.append(s["seconds"])
        kvb += s["kv_bytes"]
        rows.append(len(s["rows"]))
    total = sum(times)
    value = kvb / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nt, "kind": "oracle",
                         "cpu_model": cpu_model(), "hardware_threads": os.cpu_count(),
                         "sample": f"each step: the C oracle (fp64) on randomly chosen rows "
                                   f"of the {w.name} step, {nt} rows at a time in {nt} host "
                                   f"threads, until {step_budget:.3g} s of wall time "
                                   f"({statistics.mean(rows):.1f} rows per step on average"
                                   + (f", each row's first {cap} history tokens)" if cap
                                      else ")")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def run_ours(args, w: wl.Workload, dist, rank, world, local):
    import paged_kv_decode_np_gb300 as npg

    npg.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = wl.make_inputs(w, device=dev, poison=False)
    md = inp.md
    bt, cl, sm = (t.to(dev) for t in (md.block_tables, md.context_lens, md.slot_mapping))
    S = args.splits if args.splits is not None else npg.np_paged_decode_plan(w.rows, w.q_heads, w.kv_heads, w.head_dim,
                                                w.block_size, bt.shape[1], w.torch_dtype)
    ws = npg.workspace(w.rows, w.q_heads, w.head_dim, S, device=dev, query_len=w.query_len)
    out = torch.empty_like(inp.q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    nbytes = algorithmic_bytes(w, md)
    pools = [(inp.k_pool, inp.v_pool)]
    flush = None
    pool_bytes = 2 * inp.k_pool.numel() * inp.k_pool.element_size()
    n_pools = l2_plan(nbytes["kv"], pool_bytes)
    if n_pools == 0:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    else:
        pools += [(inp.k_pool.clone(), inp.v_pool.clone()) for _ in range(n_pools - 1)]

    def step(i=0, s=stream):
        # append fused into the read's launch, then the merge (balanced read)
        # or the split reduce; returns the kernels launched
        kp, vp = pools[i % len(pools)]
        npg.np_paged_append_decode(out if S <= 1 else None, inp.q, inp.k_new, inp.v_new, sm,
                                   kp, vp, bt, cl, w.softmax_scale, S, ws, err, s)
        if S > 1:
            npg.np_paged_decode_reduce(out, ws, S, s)
        return 2 if S == 0 or S > 1 else 1

    # CPU baseline first (host copies of the sampled rows before any kernel)
    cpu = cpu1 = None
    if rank == 0 and world == 1:
        cpu = oracle_sample(inp, args.cpu_seconds, threads=host_threads())
        cpu1 = oracle_sample(inp, args.cpu_seconds / 4, seed=1)

    for i in range(max(args.warmup, len(pools))):  # every pool copy touched once
        step(i)
        if flush is not None:
            flush.zero_()
    torch.cuda.synchronize()
    direct_out = out.clone()  # pool copy 0's step, launched directly

    # The K timed steps are captured once, back to back, as one CUDA graph
    # (step i on pool copy i mod the copies) and replayed: the same append,
    # read and merge launches with the same arguments as direct calls, without
    # the host's per-call cost between them (a 30 us step is shorter than one
    # Python call plus its event records), as a decode graph over a model's
    # layers would run them.  With an L2 flush between steps, one step is
    # captured and replayed per step.
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    n_cap = args.steps if flush is None else 1
    with torch.cuda.graph(graph, stream=cap):
        for i in range(n_cap):
            step_launches = step(i, cap)
    torch.cuda.synchronize()
    graph.replay()  # warm-up: the first launch uploads the graph
    torch.cuda.synchronize()
    if not torch.equal(out, direct_out):
        raise RuntimeError("graph replay of the steps differs from the direct call")

    st_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps if flush is not None else 0)]
    launches = 0
    with ClockSampler(dev) as clk:
        barrier(dist)
        torch.cuda.synchronize()
        wall0 = time.time()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        if flush is None:
            graph.replay()
            launches = step_launches * args.steps
        else:
            for i in range(args.steps):
                flush.zero_()
                st_ev[i][0].record(stream)
                graph.replay()
                st_ev[i][1].record(stream)
                launches += step_launches
        t_end.record(stream)
        torch.cuda.synchronize()
        clk.mark(wall0, time.time())
        barrier(dist)
    if flush is None:
        elapsed_ms = t_start.elapsed_time(t_end)
    else:  # exclude the L2 flushes between steps
        elapsed_ms = sum(a.elapsed_time(b) for a, b in st_ev)

    # the per-step distribution (median, p10, p90), from a separate pass:
    # one-step graphs (one per pool copy) replayed with an event pair around
    # each, so each sample is one step's device time; with the L2 flush, the
    # timed pass's own per-step pairs
    if flush is None:
        one = []
        for i in range(len(pools)):
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1, stream=cap):
                step(i, cap)
            one.append(g1)
        torch.cuda.synchronize()
        n_dist = min(args.steps, 200)
        d_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n_dist)]
        for i in range(n_dist):
            d_ev[i][0].record(stream)
            one[i % len(one)].replay()
            d_ev[i][1].record(stream)
        torch.cuda.synchronize()
        step_us = sorted(1e3 * a.elapsed_time(b) for a, b in d_ev)
    else:
        step_us = sorted(1e3 * a.elapsed_time(b) for a, b in st_ev)
    # a step is the library's launches and nothing else
    decode_ms = ([a.elapsed_time(b) for a, b in st_ev] if flush is not None
                 else [elapsed_ms / args.steps])
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flags {int(err.item()):#x}")

    # end-to-end through the C ABI with host buffers: the step's inputs sit
    # in one pinned staging buffer (256-byte aligned sections), copied to the
    # device in one transfer per step; the result comes back the same way.
    # Two measurements: serial (each step's upload, kernels and download in
    # turn on one stream) and pipelined two deep, as a serving loop runs it
    # (step i+1's upload on an upload stream while step i computes, step i's
    # download on a download stream while step i+1 computes; two staging
    # buffers and two outputs alternate, events order each buffer's reuse).
    # Every step still uploads all its inputs and downloads its whole result.
    srcs = dict(q=inp.q, k_new=inp.k_new, v_new=inp.v_new, sm=sm, bt=bt, cl=cl)
    offs, total_b = {}, 0
    for k, t in srcs.items():
        offs[k] = total_b
        total_b += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_h = torch.empty(total_b, dtype=torch.uint8).pin_memory()
    stage_d = [torch.empty(total_b, dtype=torch.uint8, device=dev) for _ in range(2)]

    def section(buf, k):
        t = srcs[k]
        nb = t.numel() * t.element_size()
        return buf[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)

    for k, t in srcs.items():
        section(stage_h, k).copy_(t.to("cpu"))
    dbufs = [{k: section(sd, k) for k in srcs} for sd in stage_d]
    outs = [out, torch.empty_like(out)]
    out_hosts = [torch.empty_like(out, device="cpu").pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in srcs.values())
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_h2d, ev_kern, ev_d2h = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    used = [False, False]

    # each (pool copy, staging slot) step prepared once: the loop then pays
    # the binding's checks and argument conversion once, not per step
    prepared = {}
    for pi, (kp, vp) in enumerate(pools):
        for k in range(2):
            db = dbufs[k]
            prepared[pi, k] = npg.PreparedStep(outs[k], db["q"], db["k_new"], db["v_new"],
                                               db["sm"], kp, vp, db["bt"], db["cl"],
                                               w.softmax_scale, S, ws, err, stream)

    def launch(i, k):
        prepared[i % len(pools), k].launch()

    def e2e_serial(i):
        stage_d[0].copy_(stage_h, non_blocking=True)
        launch(i, 0)
        out_hosts[0].copy_(outs[0], non_blocking=True)

    def e2e_pipelined(i):
        k = i & 1
        if used[k]:
            up.wait_event(ev_kern[k])  # step i-2 has read this staging buffer
        with torch.cuda.stream(up):
            stage_d[k].copy_(stage_h, non_blocking=True)
        ev_h2d[k].record(up)
        stream.wait_event(ev_h2d[k])
        if used[k]:
            stream.wait_event(ev_d2h[k])  # step i-2's result has left outs[k]
        launch(i, k)
        ev_kern[k].record(stream)
        down.wait_event(ev_kern[k])
        with torch.cuda.stream(down):
            out_hosts[k].copy_(outs[k], non_blocking=True)
        ev_d2h[k].record(down)
        used[k] = True

    for i in range(max(args.warmup, len(pools))):
        e2e_serial(i)
        e2e_pipelined(i)
    torch.cuda.synchronize()
    # serial: per-step event pairs (the L2 flush, where there is one, between
    # them and outside the sum)
    e_st = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        e_st[i][0].record(stream)
        e2e_serial(i)
        e_st[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    e2e_serial_ms = sum(a.elapsed_time(b) for a, b in e_st)
    e2e_ms = e2e_serial_ms
    if flush is None:  # pipelined: one event pair around all K steps
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        p0.record(stream)
        up.wait_event(p0)
        down.wait_event(p0)
        for i in range(args.steps):
            e2e_pipelined(i)
        p1.record(down)  # after the last download, itself after the last kernels
        torch.cuda.synchronize()
        barrier(dist)
        e2e_ms = p0.elapsed_time(p1)
    if not torch.equal(out_hosts[0].to(dev), direct_out):
        raise RuntimeError("end-to-end result differs from the device-resident step's")

    # aggregate over ranks: max time, summed bytes
    elapsed_ms = max_over_ranks(dist, elapsed_ms)
    e2e_ms = max_over_ranks(dist, e2e_ms)
    e2e_serial_ms = max_over_ranks(dist, e2e_serial_ms)
    kv_total = sum_over_ranks(dist, float(nbytes["kv"])) * args.steps
    if rank != 0:
        return None
    value = kv_total / (elapsed_ms / 1e3) / 1e9
    e2e_pipe = kv_total / (e2e_ms / 1e3) / 1e9
    e2e_serial = kv_total / (e2e_serial_ms / 1e3) / 1e9
    # the faster schedule is the loop's (a step shorter than the host's
    # per-step work runs faster serial: the pipelined loop's extra stream
    # and event calls then lengthen the host's share)
    pipelined = flush is None and e2e_pipe >= e2e_serial
    e2e_value = e2e_pipe if pipelined else e2e_serial
    peak, peak_kind = measured_peak()
    dec_avg_ms = statistics.mean(decode_ms)
    achieved = nbytes["decode"] / (dec_avg_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "us_per_step": 1e3 * elapsed_ms / args.steps,
        "frac_of_hbm_peak": value / world / peak,
        "frac_of_nominal_8tbs": value / world / 8000.0,
        "step_us": {"median": statistics.median(step_us), "p10": step_us[len(step_us) // 10],
                    "p90": step_us[(9 * len(step_us)) // 10], "samples": len(step_us),
                    "how": "one-step graph replays, an event pair around each (each sample "
                           "includes the graph's launch latency, which back-to-back steps "
                           "hide)" if flush is None else "the timed steps' event pairs"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) q/K/V, shuffled free-list block tables)",
        "config": {
            "workload": w.name, "description": w.description, "rows": w.rows,
            "q_heads": w.q_heads, "kv_heads": w.kv_heads, "head_dim": w.head_dim,
            "query_len": w.query_len,
            "block_size": w.block_size, "max_blocks_per_row": bt.shape[1],
            "num_blocks": md.num_blocks, "num_splits": S,
            "schedule": "balanced stream (one CTA per SM, equal chunk shares)" if S == 0
            else f"split-K x{S}",
            "split_len": npg.np_paged_decode_split_len(w.block_size, bt.shape[1], S) if S > 0
            else None,
            "mean_context": float(md.context_lens.double().mean()),
            "kv_bytes_per_step": nbytes["kv"],
            "l2": ("L2 flushed (2x L2 buffer written) between timed steps, flush excluded"
                   if flush is not None else
                   "inputs larger than L2: %.2f GB of K/V read per step vs 129 MB L2"
                   % (nbytes["kv"] / 1e9) if len(pools) == 1 else
                   "steps rotate among %d copies of the %.1f MB K/V pool (%.2f GB in all, "
                   "over 3x the 129 MB L2), back to back, no flush"
                   % (len(pools), pool_bytes / 1e6, len(pools) * pool_bytes / 1e9)),
            "parallelism": f"replicas x{world} (rows independent, no collective)",
            "launch": ("the K steps captured back to back as one CUDA graph and replayed"
                       if flush is None else "one step captured as a CUDA graph, replayed "
                       "once per step between L2 flushes")
                      + "; output checked equal to a direct call's",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": ("paged_decode_stream_kernel + its merge launch (timed together)"
                       if S == 0 else ("paged_decode_mma_kernel" if w.dtype == "bf16"
                                       else "paged_decode_kernel")
                       + (" + lse_reduce_kernel (timed together)" if S > 1 else "")),
            "achieved": achieved,
            "peak": peak, "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s",
            "unit": "GB/s", "frac": achieved / peak,
            "traffic": profiled_traffic(w.name),
            "algorithmic_bytes_per_launch": nbytes["decode"],
            "avg_launch_ms": dec_avg_ms,
        },
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "mode": ("steps pipelined two deep (uploads and downloads on their own "
                         "streams, overlapping the neighbouring steps' kernels)" if pipelined
                         else "serial (upload, kernels, download in turn on one stream"
                         + ("; L2 flushed between steps)" if flush is not None else
                            "; faster than the pipelined loop here, which is host-bound)")),
                "serial_value": e2e_serial,
                "pipelined_value": e2e_pipe if flush is None else None},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if cpu is not None:
        line["cpu_baseline"] = {
            "value": cpu["gbs"], "unit": UNIT, "cores": cpu["threads"], "kind": "oracle",
            "cpu_model": cpu_model(), "hardware_threads": os.cpu_count(),
            "sample": f"rows {cpu['rows']} of this step ({cpu['kv_bytes'] / 1e9:.3f} GB of K/V,"
                      f" {cpu['seconds']:.1f} s wall), the C oracle in fp64, append + read, "
                      f"{cpu['threads']} rows at a time in {cpu['threads']} host threads",
            "single_thread": {"value": cpu1["gbs"], "cores": 1,
                              "sample": f"rows {cpu1['rows']} ({cpu1['seconds']:.1f} s)"}}
    return line


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=2.0)
    ap.add_argument("--splits", type=int, default=None,
                    help="override the library's split plan (profiling)")
    ap.add_argument("--rows", type=int, default=None,
                    help="keep only the first N rows of the workload (small profiling cases)")
    args = ap.parse_args(argv)
    if args.impl == "ours" and args.warmup < 3:
        args.warmup = 3  # timing rule: at least 3 untimed warm-up steps
    w = wl.WORKLOADS[args.workload]
    if args.rows is not None and args.rows < w.rows:
        w = wl.truncated(w, args.rows)
    dist, rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, w, dist, rank)
    else:
        line = run_ours(args, w, dist, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

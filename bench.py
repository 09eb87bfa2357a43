"""Throughput of the RESOLVE step on one GB300 (or N, one process each).

A step is one decode step of the whole hot path: every sparse layer's
resolve (hash build, hit probe, victim choice, host fetch of the misses,
metadata update, publication) for every request of the batch.  Default
workload (the headline): the largest one, tight_prefetch -- 64 requests, 8
sparse layers in two anchor groups, L_ctx = 100352, k = B = 2048,
1152-byte records (576 bf16), a 59.2 GB pinned host pool -- with its seeded
128-step selection trace (steps past the end wrap around); then the
dsa_mla workload (8 requests x 4 layers, B = 4096) beside it (`--also`).

Passes over the headline, each on a freshly reset pool (warm-up steps
first, then timed ones):
  graph  -- each step is a CUDA graph of the per-layer hs_resolve launches;
            the L2 is flushed (a 256 MiB write, then a 256 MiB read so
            that no dirty line is left to write back) before every step and
            the step itself is timed with CUDA events: ``value``, and,
            divided by the launches of a step, the resolve kernel's average
            launch duration inside the graph (``roofline``).
  prefetch -- the same steps with exact layer-wise prefetch by anchor-plan
            replay (``prefetch_on``).
  copy-only -- the same steps' miss records moved by the copy-only kernel
            alone (``copy_only``; ``roofline.frac_of_copy_only``).
  measure -- the resolve without its fetch (``no_fetch``: the metadata
            roofline) and with stage timestamps (``stages``).
  continuous -- blocks of 16 consecutive steps captured as one graph, the
            L2 flushed before each block only (``continuous``).
  kernel -- the same steps launched one call at a time with events around
            every launch (``roofline.avg_launch_us_eager``, for context).
  e2e    -- the user's loop through the public API with host buffers: each
            step a graph of the pinned host -> device copy of its
            selections, the resolves and the device -> host copy of the
            published slots, replayed and synchronised, all inside the timed
            region (``e2e``).
The headline's pool is allocated first: on the GB300 machines measured, host
reads of pinned pools allocated after other large pinned pools had been
freed ran slower and sped up again over seconds, so the other workloads
are timed after it, in the same process (``other_workloads``).  The
host-link ceiling is measured in the same run (pinned H2D memcpy and a
scattered-record GPU-load probe, best of 10).  The CPU oracle is timed on
the host's cores over a stated sample (``cpu_baseline``).

``--impl reference`` times the CPU oracle alone as the reference arm.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("resolves/sec and miss-fetch GB/s (fraction of measured pinned H2D BW) "
          "at 1 GB300")
L2_FLUSH_BYTES = 256 << 20
HOST_ALLOC = {"auto": 0, "pinned": 1, "vmm": 2, "thp": 3}
OVERLAP = {"auto": 0, "on": 1, "off": 2}
CONT_STEPS, CONT_BLOCKS = 16, 3
PREROLL_STEPS = 32  # untimed steps before the diagnostic passes of --prefetch-overlap

# Counters of one steady-state resolve launch from an ncu capture
# (profiles/resolve_kernel_tight_prefetch_full.md: tight_prefetch at full
# size, one layer of 64 resolves), valid only for that workload and for the
# kernel sources they were taken on: reported as null otherwise.
PROFILED_WORKLOAD = "tight_prefetch"
PROFILED_SOURCES = {"resolve.cu": "04d298886bf806c7", "hs_internal.cuh": "48a56b6be5e1ce3e"}
PROFILED_LAUNCH = {"dram_bytes": 8_592_896 + 97_024, "link_bytes": 22_635_648,
                   "algorithmic_link_bytes": 22_635_648}


def profiled_counters(workload_name: str):
    import hashlib
    if workload_name != PROFILED_WORKLOAD:
        return None
    csrc = os.path.join(ROOT, "hierarchical_kv_cache_resolve_gb300", "csrc")
    for name, digest in PROFILED_SOURCES.items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != digest:
                return None
    return PROFILED_LAUNCH


# ---------------------------------------------------------------- helpers ---

class L2Flush:
    """Empties the L2 between timed iterations: a 256 MiB write (about twice
    the L2), then a 256 MiB read of a second buffer, so that the L2 holds
    only clean lines and the timed work pays no write-back of the flush."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.sink = None

    def __call__(self, i):
        self.w.fill_(i)
        self.sink = self.r.max()


class nvtx:
    """An NVTX range around a bench pass (seen by ncu --nvtx and nsys)."""

    def __init__(self, name: str):
        self.name = name

    def __enter__(self):
        import torch
        torch.cuda.nvtx.range_push(self.name)
        return self

    def __exit__(self, *exc):
        import torch
        torch.cuda.nvtx.range_pop()


def workload_name(w) -> str:
    return (f"{w.name}: batch {w.n_requests}, {w.n_layers} sparse layers, "
            f"L_ctx={w.n_positions}, k={w.k}, B={w.slots}, W={w.record_bytes} B/record, "
            f"{w.steps}-step seeded trace")


def hbm_bytes_per_resolve(k: int, B: int, m: float, W: int) -> float:
    """Algorithmic HBM bytes of one resolve with m misses (all victims
    occupied, the steady state): reads selections 4k, slot map 4B, LRU order
    2B; writes published slots 4k, stamps 4k (every selected slot), slot map
    4m, page table 8m (new entry + evicted entry), LRU order 2B, records m*W."""
    return 4 * k + 4 * B + 2 * B + 4 * k + 4 * k + 4 * m + 8 * m + 2 * B + m * W


def hbm_sector_bytes_per_resolve(k: int, B: int, m: float, W: int) -> float:
    """The same resolve counted in 32-byte sectors, as the memory system
    moves it: the contiguous arrays as above; every scattered 4-byte access
    a whole sector (the page-table reads of the k selected positions with
    which the data-moving CTAs predict the misses, the 8m page-table and 4m
    slot-map writes); the stamp writes the sectors of the stamp array that
    the k selected slots fall in (8 slots a sector, selected slots spread
    over the B)."""
    stamp_sectors = (B / 8.0) * (1.0 - (1.0 - min(k, B) / B) ** 8)
    reads = 4 * k + 4 * B + 2 * B + 32 * k
    writes = 4 * k + 32 * stamp_sectors + 32 * m + 64 * m + 2 * B + m * W
    return reads + writes


def host_pages(addr: int, nbytes: int) -> dict:
    """How the host pool's pages are backed, from /proc/self/smaps: the
    mappings overlapping [addr, addr + nbytes) summed (kB), their page
    sizes, and the system's transparent-huge-page settings.  The GPU's
    scattered reads of pinned host memory depend on the pages behind it."""
    res = {"mappings": 0, "size_kb": 0, "rss_kb": 0, "anon_huge_kb": 0,
           "kernel_page_kb": set(), "mmu_page_kb": set()}
    lo, hi = addr, addr + nbytes
    try:
        with open("/proc/self/smaps") as f:
            cur = False
            for line in f:
                head = line.split()
                if not head:
                    continue
                if "-" in head[0] and len(head) >= 5 and ":" not in head[0]:
                    a, b = (int(x, 16) for x in head[0].split("-"))
                    cur = a < hi and b > lo
                    if cur:
                        res["mappings"] += 1
                    continue
                if not cur:
                    continue
                key = head[0].rstrip(":")
                if key == "Size":
                    res["size_kb"] += int(head[1])
                elif key == "Rss":
                    res["rss_kb"] += int(head[1])
                elif key == "AnonHugePages":
                    res["anon_huge_kb"] += int(head[1])
                elif key == "KernelPageSize":
                    res["kernel_page_kb"].add(int(head[1]))
                elif key == "MMUPageSize":
                    res["mmu_page_kb"].add(int(head[1]))
    except OSError as e:
        res["error"] = str(e)
    res["kernel_page_kb"] = sorted(res["kernel_page_kb"])
    res["mmu_page_kb"] = sorted(res["mmu_page_kb"])
    thp = {}
    for name in ("enabled", "defrag", "hpage_pmd_size"):
        try:
            with open(f"/sys/kernel/mm/transparent_hugepage/{name}") as f:
                thp[name] = f.read().strip()
        except OSError:
            pass
    res["thp"] = thp
    return res


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return None


def reduce_max(value: float, dist_on: bool, device=None) -> float:
    """Maximum of a float over all ranks (identity without torch.distributed)."""
    if not dist_on:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, dist_on: bool, device=None) -> float:
    if not dist_on:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_workload(w, rank: int):
    """Weak scaling: every rank owns its own batch of requests, with its own
    seeded trace and records (seed offset by the rank)."""
    return w.with_(seed=w.seed + rank)


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read-only).

    NVML is initialised once per process and device (`shared`), before any
    timed work: its initialisation keeps the host busy for a while, and a
    GPU left idle that long before a timed pass reads a large host pool
    slowly for its first steps.  `start` and `stop` bracket each timed
    region; `start` clears the previous region's samples."""

    _by_pci = {}
    PERIOD_S = 0.002

    @classmethod
    def shared(cls, pci_bus_id: str) -> "ClockSampler":
        if pci_bus_id not in cls._by_pci:
            cls._by_pci[pci_bus_id] = cls(pci_bus_id)
        return cls._by_pci[pci_bus_id]

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, pci_bus_id: str):
        self.samples = []
        self.max_mhz = None
        self.err = None
        self._stop = threading.Event()
        self._thr = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(),
                                                          ctypes.byref(self.h)) != 0:
                raise OSError(f"no NVML handle for {pci_bus_id}")
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
        except OSError as e:
            self.err = str(e)
            self.nvml = None

    def _read(self):
        clk = ctypes.c_uint()
        rsn = ctypes.c_ulonglong()
        self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk))
        self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rsn))
        return clk.value, rsn.value

    def _run(self):
        while not self._stop.is_set():
            self.samples.append(self._read())
            time.sleep(self.PERIOD_S)

    def start(self):
        self.samples = []
        self._stop.clear()
        if self.nvml is not None:
            self._thr = threading.Thread(target=self._run, daemon=True)
            self._thr.start()

    def stop(self):
        self._stop.set()
        if self._thr is not None:
            self._thr.join()
            self._thr = None

    def summary(self):
        if self.nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": f"unavailable: {self.err}"}
        busy = [s for s in self.samples if not (s[1] & 0x1)] or self.samples
        reasons = set()
        for _, r in busy:
            for bit, name in self.REASONS.items():
                if r & bit and bit != 0x1:
                    reasons.add(name)
        return {"sm_mhz": statistics.median([c for c, _ in busy]) if busy else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples), "samples_not_idle": len(busy), "source": "nvml"}


# ----------------------------------------------------------- CPU oracle ----

def time_oracle(w, n_pairs: int, steps: int, threads: int):
    """The CPU oracle as it stands, with host records and a cache mirror
    (so it also copies every missed record), on the first n_pairs
    (request, layer) pairs for `steps` steps of the trace, spread over
    `threads` threads (one pair per task).  Returns (resolves/s, wall s,
    resolves, miss bytes)."""
    from concurrent.futures import ThreadPoolExecutor

    from oracle.oracle import OK, Pair
    from workloads import records, traces

    pairs = [(r, l) for r in range(w.n_requests) for l in range(w.n_layers)][:n_pairs]
    sel = traces.generate(w, requests=sorted({r for r, _ in pairs}))
    rid = {r: i for i, r in enumerate(sorted({r for r, _ in pairs}))}
    states = []
    for r, l in pairs:
        host = np.empty((w.n_positions, w.record_bytes), np.uint8)
        records.fill(host.ctypes.data, w, r, l)
        states.append(((r, l), Pair(w.slots, w.n_positions, w.record_bytes, host=host,
                                    mirror=True)))
    T = sel.shape[0]
    idx = [s % T for s in range(steps)]

    def run(item):
        (r, l), p = item
        ss = np.ascontiguousarray(sel[idx, rid[r], l, :])
        rc, _, _ = p.run(ss, out_base=r * w.slots)
        assert rc == OK
        return p.fetched_bytes

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        fetched = sum(ex.map(run, states))
    wall = time.perf_counter() - t0
    n = len(pairs) * steps
    return n / wall, wall, n, fetched


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    machine type)."""
    import platform
    import subprocess
    try:
        outp = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in outp.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


CPU_SAMPLE_PAIRS = 32


def cpu_baseline(w, threads: int, epochs: int = 4):
    """The oracle on a bounded sample of the workload: the first
    CPU_SAMPLE_PAIRS (request, layer) pairs (all of them for the smaller
    workloads), each replayed over its whole trace `epochs` times back to
    back (steps past the end wrap around, as in the GPU passes), one thread
    per pair; and one pair on one thread.  About ten seconds of CPU work."""
    pairs = min(w.n_requests * w.n_layers, CPU_SAMPLE_PAIRS)
    steps = epochs * w.steps
    value, wall, n, fetched = time_oracle(w, pairs, steps, threads)
    one, one_wall, one_n, _ = time_oracle(w, 1, steps, 1)
    return {"value": value, "unit": "resolves/s", "cores": min(threads, pairs), "kind": "oracle",
            "cpu_model": cpu_model(),
            "single_thread": {"value": one, "unit": "resolves/s",
                              "sample": f"one (request, layer) pair x {steps} steps, one thread",
                              "wall_s": one_wall},
            "sample": (f"{pairs} of the {w.n_requests * w.n_layers} (request, layer) pairs x "
                       f"{steps} steps ({epochs} passes over the {w.name} trace; {n} resolves, "
                       f"{fetched / 1e9:.2f} GB of misses copied), one thread per pair, "
                       f"{min(threads, pairs)} threads"),
            "wall_s": wall, "cpu_s": wall * min(threads, pairs),
            "miss_fetch_gbs": fetched / wall / 1e9}


# -------------------------------------------------------------- GPU arm ----

def run_gpu(args, w, rank, world, dist_on, lite=False):
    """All GPU passes on workload `w`; `lite`: the graph pass (`value`) and
    its roofline only (a second workload reported beside the headline)."""
    import torch

    from hierarchical_kv_cache_resolve_gb300 import hs
    from workloads import records, traces

    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    pci = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    sampler = ClockSampler.shared(pci)   # NVML initialised before the pool exists
    R, NL, k, B, W, T = w.n_requests, w.n_layers, w.k, w.slots, w.record_bytes, w.steps

    kind = HOST_ALLOC[args.host_alloc]
    sel = traces.generate(w)
    dsel = torch.from_numpy(np.ascontiguousarray(sel.transpose(0, 2, 1, 3))).to(dev)
    # the pool first: a process's first large pinned allocation is the one
    # the host's memory serves best (see host_pages and the docstring)
    t_fill = time.perf_counter()
    pool = hs.Pool.for_workload(w, host_alloc=kind, launch_overlap=OVERLAP[args.launch_overlap])
    pool_info = pool.info()
    for r in range(R):
        for l in range(NL):
            records.fill(pool.host_records(r, l).ctypes.data, w, r, l)
    pool_info["create_and_fill_s"] = time.perf_counter() - t_fill
    h2d_gbs, gather_gbs = hs.hs_link_probe(1 << 30, 10, W, kind)
    base_addr = pool.host_records(0, 0).ctypes.data
    pool_info["pages"] = host_pages(base_addr, w.host_bytes)
    pool_info["host_address"] = hex(base_addr)
    pool_info["host_address_mod_2mib"] = base_addr % (2 << 20)
    pool_info["host_address_mod_512mib"] = base_addr % (512 << 20)
    out = torch.empty((NL, R, k), dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    main = torch.cuda.current_stream()
    Wm, K = args.warmup, args.steps
    launches_per_step = NL * hs.hs_kernels_per_call()

    def step_eager(t, stream=None):
        for l in range(NL):
            hs.hs_resolve(pool.handle, l, R, None, dsel[t, l], k, out[l], None, stream)

    def barrier():
        torch.cuda.synchronize()
        if dist_on:
            import torch.distributed as dist
            dist.barrier()

    # ---- graph pass -------------------------------------------------------
    pool.reset()
    cap = torch.cuda.Stream()
    graphs = []
    for t in range(T):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for l in range(NL):
                hs.hs_resolve(pool.handle, l, R, None, dsel[t, l], k, out[l], None, cap)
        graphs.append(g)
    # the records are written and the graphs captured: read the records once
    # from the device and resolve synthetic steps, then reset (hs_warm_pool;
    # outside every timed region, right before the steps)
    pool.warm()
    pool_info["warmup_us"] = pool.info()["warmup_us"]
    # step 0 from an empty cache (every selection misses), timed on its own;
    # it is the first of the warm-up steps
    flush(0)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(main)
    graphs[0].replay()
    c1.record(main)
    torch.cuda.synchronize()
    cold_ms = c0.elapsed_time(c1)
    st_cold = pool.stats()
    for s in range(1, Wm):
        flush(s)
        graphs[s % T].replay()
    st0 = pool.stats()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    barrier()
    sampler.start()
    wall0 = time.perf_counter()
    torch.cuda.nvtx.range_push("timed steps")
    for i in range(K):
        flush(i)
        ev[i][0].record(main)
        graphs[(Wm + i) % T].replay()
        ev[i][1].record(main)
    torch.cuda.nvtx.range_pop()
    barrier()
    wall_graph = time.perf_counter() - wall0
    sampler.stop()
    st1 = pool.stats()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dev_s = sum(step_ms) / 1e3
    dev_s_max = reduce_max(dev_s, dist_on, dev)
    fetched = st1["fetched_bytes"] - st0["fetched_bytes"]
    misses = st1["misses"] - st0["misses"]
    resolves = st1["resolves"] - st0["resolves"]
    assert resolves == K * R * NL, (resolves, K * R * NL)
    total_resolves = reduce_sum(resolves, dist_on, dev)
    total_fetched = reduce_sum(fetched, dist_on, dev)
    del graphs

    # the dominant kernel's average launch duration: the graph-timed steps
    # hold nothing but resolve launches, so a step's events divided by its
    # launches is the per-launch time inside the decode graph
    avg_launch_s = dev_s / (K * launches_per_step)
    link_bytes_per_launch = fetched / (K * launches_per_step)
    m_per_resolve = misses / resolves
    hbm_per_launch = R * hbm_bytes_per_resolve(k, B, m_per_resolve, W)
    hbm_sectors_per_launch = R * hbm_sector_bytes_per_resolve(k, B, m_per_resolve, W)

    if lite:
        pool.close()
        return {
            "workload": workload_name(w), "resolves_per_s": total_resolves / dev_s_max,
            "ms_per_step": dev_s_max / K * 1e3, "steps": K, "warmup": Wm,
            "miss_rate": misses / (resolves * k),
            "miss_fetch_gbs": total_fetched / dev_s_max / 1e9,
            "roofline": {"kernel": "resolve_kernel", "bound": "link",
                         "achieved": link_bytes_per_launch / avg_launch_s / 1e9,
                         "peak": h2d_gbs, "unit": "GB/s",
                         "frac": link_bytes_per_launch / avg_launch_s / 1e9 / h2d_gbs,
                         "algorithmic_bytes_per_launch": link_bytes_per_launch,
                         "avg_launch_us": avg_launch_s * 1e6},
            "repeats": [len(g) * R * NL / (sum(g) / 1e3)
                        for g in np.array_split(np.array(step_ms), 3) if len(g)],
            "step_ms": step_time_summary(step_ms, R * NL),
            "cold_step_ms": cold_ms, "host_pool": pool_info,
            "l2": "flushed before every timed step"}

    # ---- exact prefetch in the pure resolve step, and the copy-only rate of
    # the same miss records (both beside `value`) ----------------------------
    with nvtx("prefetch pass"):
        prefetch_on = run_prefetch_pass(pool, w, dsel, flush, main, cap, K, Wm, h2d_gbs)
    with nvtx("copy-only pass"):
        copy_only = run_copy_only(pool, w, dsel, flush, main, cap, K, Wm, h2d_gbs)

    # ---- continuous pass (diagnostic, not `value`) --------------------------
    # blocks of CONT_STEPS consecutive steps captured as one graph, L2
    # flushed before each block only: the per-launch time of decode steps
    # that follow each other with nothing in between
    blocks = []
    for b in range(CONT_BLOCKS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for j in range(CONT_STEPS):
                t = (Wm + b * CONT_STEPS + j) % T
                for l in range(NL):
                    hs.hs_resolve(pool.handle, l, R, None, dsel[t, l], k, out[l], None, cap)
        blocks.append(g)
    pool.reset()
    for s in range(Wm):
        flush(s)
        step_eager(s % T, main)
    cont_ms, cont_bytes = [], 0
    for g in blocks:
        flush(0)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sb = pool.stats()
        c0.record(main)
        g.replay()
        c1.record(main)
        torch.cuda.synchronize()
        cont_ms.append(c0.elapsed_time(c1))
        cont_bytes += pool.stats()["fetched_bytes"] - sb["fetched_bytes"]
    del blocks
    cont_launches = CONT_BLOCKS * CONT_STEPS * launches_per_step
    cont_s = sum(cont_ms) / 1e3
    continuous = {
        "what": f"{CONT_BLOCKS} blocks of {CONT_STEPS} consecutive steps, each block one graph "
                "replay, L2 flushed before each block only; a diagnostic, not `value`",
        "us_per_launch": cont_s / cont_launches * 1e6,
        "resolves_per_s": CONT_BLOCKS * CONT_STEPS * R * NL / cont_s,
        "miss_fetch_gbs": cont_bytes / cont_s / 1e9,
        "frac_of_h2d": cont_bytes / cont_s / 1e9 / h2d_gbs,
    }

    # ---- measurement passes: no fetch, stage stamps (diagnostics) ------------
    with nvtx("measurement passes"):
        measure = run_measure_passes(pool, w, dsel, flush, main, cap, K, Wm)

    # ---- kernel pass (per-launch events, eager launches) ---------------------
    pool.reset()
    for s in range(Wm):
        flush(s)
        step_eager(s % T, main)
    kev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(NL)] for _ in range(K)]
    barrier()
    for i in range(K):
        flush(i)
        t = (Wm + i) % T
        for l in range(NL):
            kev[i][l][0].record(main)
            hs.hs_resolve(pool.handle, l, R, None, dsel[t, l], k, out[l], None, main)
            kev[i][l][1].record(main)
    barrier()
    launch_ms = [a.elapsed_time(b) for row in kev for a, b in row]
    avg_launch_eager_s = sum(launch_ms) / len(launch_ms) / 1e3

    # ---- e2e pass (public API, host buffers) ----------------------------------
    # each step, captured once as a graph like a decode step: pinned host ->
    # device copy of its selections, the resolves, device -> pinned host copy
    # of the published slots; every replay is followed by a synchronisation
    host_sel = torch.from_numpy(np.ascontiguousarray(sel.transpose(0, 2, 1, 3))).pin_memory()
    host_out = torch.empty((NL, R, k), dtype=torch.int32).pin_memory()
    stage = torch.empty((NL, R, k), dtype=torch.int32, device=dev)
    # the steps this pass replays only: capturing is host time, and after
    # the GPU has paused for half a second or more the first steps over a
    # large huge-page pool read slowly
    e2e_graphs = {}
    for t in sorted({s % T for s in range(Wm + K)}):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            stage.copy_(host_sel[t], non_blocking=True)
            for l in range(NL):
                hs.hs_resolve(pool.handle, l, R, None, stage[l], k, out[l], None, cap)
            host_out.copy_(out, non_blocking=True)
        e2e_graphs[t] = g

    def e2e_step(t):
        e2e_graphs[t].replay()
        main.synchronize()

    # every step's selections, written by the CPU into one pinned buffer, are
    # read once from the device before timing (the device's first read of
    # host memory the CPU has written is slow on these machines; a serving
    # loop reuses its pinned buffers), and the output buffer written once
    pool.reset()
    for t in range(T):
        stage.copy_(host_sel[t], non_blocking=True)
    host_out.copy_(out, non_blocking=True)
    main.synchronize()

    for s in range(Wm):
        e2e_step(s % T)
    barrier()
    e0 = time.perf_counter()
    for i in range(K):
        e2e_step((Wm + i) % T)
    barrier()
    e2e_s = reduce_max(time.perf_counter() - e0, dist_on, dev)
    del e2e_graphs
    pool.close()

    peaks = load_peaks()
    prof = profiled_counters(w.name)
    hbm_peak = peaks.get("hbm_gbs") if peaks else None
    miss_gbs = total_fetched / dev_s_max / 1e9
    link_achieved = link_bytes_per_launch / avg_launch_s / 1e9
    hbm_achieved = hbm_per_launch / avg_launch_s / 1e9
    res = {
        "metric": METRIC,
        "value": total_resolves / dev_s_max,
        "unit": "resolves/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": dev_s_max / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int32",
        "data": "synthetic",
        "config": {
            "workload": workload_name(w),
            "global_batch": R * world,
            "resolves_per_step": R * NL * world,
            "parallelism": f"requests sharded, {world} independent pool(s), no collective",
            "launch": (f"per-step CUDA graph of {NL} hs_resolve launches, launch overlap "
                       f"{'on' if pool_info['launch_overlap'] == 1 else 'off'}"),
            "l2": "flushed before every timed step (256 MiB write + 256 MiB read, outside the events)",
            "record_values": "bf16 N(0,1)" if w.value_format else "fp16 U(-1,1)",
        },
        "miss_fetch": {
            "gbs": miss_gbs,
            "unit": "GB/s",
            "over": "device time of the timed steps",
            "bytes": total_fetched,
            "misses": misses,
            "miss_rate": misses / (resolves * k),
            "link_h2d_ceiling_gbs": h2d_gbs,
            "frac_of_h2d": miss_gbs / h2d_gbs,
            "in_kernel_gbs": link_achieved,
            "in_kernel_frac_of_h2d": link_achieved / h2d_gbs,
            "gather_probe_gbs": gather_gbs,
        },
        "roofline": {
            "kernel": "resolve_kernel",
            "bound": "link",
            "achieved": link_achieved,
            "peak": h2d_gbs,
            "unit": "GB/s",
            "frac": link_achieved / h2d_gbs,
            # ncu counters of one captured launch: DRAM read+write bytes (the
            # spec's traffic) and the host-link (sysmem) read bytes, beside
            # that launch's own algorithmic link bytes
            "traffic": prof["dram_bytes"] if prof else None,
            "link_traffic": prof["link_bytes"] if prof else None,
            "traffic_launch_algorithmic_link_bytes": prof["algorithmic_link_bytes"] if prof else None,
            "peak_source": "pinned cudaMemcpyAsync H2D, 1 GiB, best of 10, this run",
            "algorithmic_bytes_per_launch": link_bytes_per_launch,
            "avg_launch_us": avg_launch_s * 1e6,
            "avg_launch_from": "graph-timed steps / launches per step",
            "avg_launch_us_eager": avg_launch_eager_s * 1e6,
            "frac_of_copy_only": link_achieved / copy_only["link_gbs"] if copy_only else None,
        },
        "roofline_hbm": {
            "kernel": "resolve_kernel",
            "bound": "hbm",
            "achieved": hbm_achieved,
            "peak": hbm_peak,
            "unit": "GB/s",
            "frac": (hbm_achieved / hbm_peak) if hbm_peak else None,
            "traffic": prof["dram_bytes"] if prof else None,
            "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if hbm_peak else None,
            "algorithmic_bytes_per_launch": hbm_per_launch,
            "sector_bytes_per_launch": hbm_sectors_per_launch,
        },
        "e2e": {
            "value": total_resolves / e2e_s,
            "unit": "resolves/s",
            "h2d_bytes_per_step": NL * R * k * 4,
            "d2h_bytes_per_step": NL * R * k * 4,
            "what": "per step one graph replay (pinned H2D of the step's selections, "
                    "hs_resolve per layer, D2H of the published slots) and a stream "
                    "synchronize; wall clock",
        },
        "prefetch_on": prefetch_on,
        "copy_only": copy_only,
        "continuous": continuous,
        "no_fetch": measure["no_fetch"],
        "stages": measure["stages"],
        "repeats": {
            "what": "the timed steps in three consecutive groups, each as resolves/s "
                    "(rank 0's device time)",
            "resolves_per_s": [len(g) * R * NL / (sum(g) / 1e3)
                               for g in np.array_split(np.array(step_ms), 3) if len(g)],
        },
        "step_ms": step_time_summary(step_ms, R * NL),
        "cold_step": {
            "what": "step 0 from an empty cache (every selection misses), one graph replay, "
                    "L2 flushed; not in `value`",
            "resolves_per_s_with_timed_steps": R * NL * (K + 1) / (cold_ms / 1e3 + dev_s),
            "ms": cold_ms, "resolves_per_s": R * NL / (cold_ms / 1e3),
            "misses": st_cold["misses"],
            "miss_fetch_gbs": st_cold["fetched_bytes"] / (cold_ms / 1e3) / 1e9,
        },
        "gpu_launches": K * launches_per_step,
        "host_pool": pool_info,
        "clocks": sampler.summary(),
        "graph_wall_s": wall_graph,
    }
    return res


def step_time_summary(step_ms, resolves_per_step):
    """Distribution of the timed steps' device times (rank 0), beside the
    mean that `value` is: the median step is the steady rate, the upper
    ones show steps slowed by the host (stalls after a pool is created or
    the GPU has idled).  Not a replacement for `value`."""
    a = np.sort(np.asarray(step_ms, dtype=np.float64))
    if a.size == 0:
        return None
    med = float(np.median(a))
    return {"what": "device time of each timed step (rank 0), ms; `value` is the mean rate",
            "min": float(a[0]), "median": med, "p90": float(np.percentile(a, 90)),
            "max": float(a[-1]),
            "resolves_per_s_at_median": resolves_per_step / (med / 1e3) if med > 0 else None}


def _timed_graph_steps(graphs, flush, main):
    """Replays the per-step graphs, L2 flushed before each, events on the
    launching stream around each replay; returns the steps' milliseconds."""
    import torch
    ms = []
    for i, g in enumerate(graphs):
        flush(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        g.replay()
        e1.record(main)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    return ms


def run_prefetch_pass(pool, w, dsel, flush, main, cap, K, Wm, h2d_gbs):
    """The timed steps with exact layer-wise prefetch by anchor-plan replay.

    Per step, in layer order: an anchor's resolve (hs_resolve_anchor) writes
    its miss plan; a side stream, forked after it, replays the plan into
    each layer sharing the anchor's selection (hs_prefetch_copy); each such
    layer's resolve waits for its copy and consumes the plan (it commits
    the metadata and fetches only what does not match).  One graph per
    step, L2 flushed before every step.  Without compute between the
    layers the copies can only overlap other resolves, so this measures
    what the replay costs or saves in a pure resolve step."""
    import torch

    from hierarchical_kv_cache_resolve_gb300 import hs
    R, NL, k, T = w.n_requests, w.n_layers, w.k, w.steps
    shared = [l for l in range(NL) if w.anchors[l] != l]
    if not shared:
        return None
    anchors = sorted({w.anchors[l] for l in shared})
    plans = {a: torch.empty(hs.hs_plan_bytes(R, k), dtype=torch.uint8, device=dsel.device)
             for a in anchors}
    out = torch.empty((NL, R, k), dtype=torch.int32, device=dsel.device)
    side = torch.cuda.Stream()

    def step(t, stream):
        evs = {}
        for l in range(NL):
            if l in plans:
                pool.resolve_anchor(l, dsel[t, l], out[l], plans[l], stream=stream)
                fork = torch.cuda.Event()
                fork.record(stream)
                side.wait_event(fork)
                for l2 in shared:
                    if w.anchors[l2] == l:
                        pool.prefetch_copy(l2, R, k, plans[l], stream=side)
                        evs[l2] = torch.cuda.Event()
                        evs[l2].record(side)
            elif l in evs:
                stream.wait_event(evs[l])
                pool.resolve(l, dsel[t, l], out[l], plan=plans[w.anchors[l]], stream=stream)
            else:
                pool.resolve(l, dsel[t, l], out[l], stream=stream)

    # graphs first: capturing keeps only the host busy, and the warm-up
    # steps run right before the timed ones
    graphs = []
    for i in range(K):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step((Wm + i) % T, cap)
        graphs.append(g)
    pool.reset()
    for s in range(Wm):
        step(s % T, main)
    st0 = pool.stats(check=False)
    ms = _timed_graph_steps(graphs, flush, main)
    st1 = pool.stats(check=False)
    del graphs
    d = {x: st1[x] - st0[x] for x in ("resolves", "misses", "fetched_bytes", "prefetched_bytes",
                                      "plan_hits", "plan_mismatches")}
    sec = sum(ms) / 1e3
    link = (d["fetched_bytes"] + d["prefetched_bytes"]) / sec / 1e9
    pool.reset()
    return {"what": "exact prefetch by anchor-plan replay in the pure resolve step "
                    "(hs_resolve_anchor, hs_prefetch_copy on a side stream, plan-consuming "
                    "hs_resolve); per-step graphs, L2 flushed before every step",
            "resolves_per_s": d["resolves"] / sec, "ms_per_step": sum(ms) / K,
            "counters": d, "status": st1["status"],
            "link_gbs": link, "frac_of_h2d": link / h2d_gbs,
            "kernels_per_step": NL + len(shared),
            "repeats": [len(g) * R * NL / (sum(g) / 1e3)
                        for g in np.array_split(np.array(ms), 3) if len(g)]}


def run_copy_only(pool, w, dsel, flush, main, cap, K, Wm, h2d_gbs):
    """The copy-only rate of exactly the records the timed steps miss.

    The timed steps are resolved once with every layer writing its miss
    plan (hs_resolve_anchor); then, after a reset, the copy-only kernel
    (hs_prefetch_copy, a full-GPU grid of 16-byte loads and nothing else)
    moves each step's planned records into their slots, one graph per step
    and the L2 flushed before each.  The resolve's own link rate divided by
    this one says how close the fused kernel comes to moving the same host
    records with no decision, metadata or staging around the loads; on a
    pool past the GPU's host translation reach both are bound by it."""
    import torch

    from hierarchical_kv_cache_resolve_gb300 import hs
    R, NL, k, T = w.n_requests, w.n_layers, w.k, w.steps
    nb = hs.hs_plan_bytes(R, k)
    plans = torch.empty((K, NL, nb), dtype=torch.uint8, device=dsel.device)
    out = torch.empty((NL, R, k), dtype=torch.int32, device=dsel.device)
    graphs = []
    for i in range(K):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for l in range(NL):
                pool.prefetch_copy(l, R, k, plans[i, l], stream=cap)
        graphs.append(g)
    pool.reset()
    for s in range(Wm):
        for l in range(NL):
            pool.resolve(l, dsel[s % T, l], out[l], stream=main)
    for i in range(K):
        for l in range(NL):
            pool.resolve_anchor(l, dsel[(Wm + i) % T, l], out[l], plans[i, l], stream=main)
    st0 = pool.stats(check=False)
    ms = _timed_graph_steps(graphs, flush, main)
    st1 = pool.stats(check=False)
    del graphs
    moved = st1["prefetched_bytes"] - st0["prefetched_bytes"]
    sec = sum(ms) / 1e3
    pool.reset()
    return {"what": "the timed steps' miss records moved by hs_prefetch_copy alone (plans "
                    "written by the resolves), per-step graphs of one copy per layer, L2 "
                    "flushed before every step",
            "bytes": moved, "link_gbs": moved / sec / 1e9,
            "frac_of_h2d": moved / sec / 1e9 / h2d_gbs, "ms_per_step": sum(ms) / K,
            "status": st1["status"]}


def metadata_bytes_per_resolve(k: int, B: int, m: float) -> float:
    """Algorithmic HBM bytes of one resolve without its records (the no-fetch
    variant): hbm_bytes_per_resolve less the m * W record bytes."""
    return hbm_bytes_per_resolve(k, B, m, 0)


STAGE_US = (
    # (name, what, later stamp, earlier stamp, CTA: leader / followers)
    ("leader_load", "selection, slot map, LRU order into shared memory", "LOADED", "ENTRY", "L"),
    ("leader_hash", "validate + hash build + membership bits", "HASHED", "LOADED", "L"),
    ("leader_probe", "probe every slot (mark hits)", "PROBED", "HASHED", "L"),
    ("leader_victims", "rank misses, choose LRU victims", "DECIDED", "PROBED", "L"),
    ("leader_wait_check", "previous grid complete, decision checked", "CHECKED", "DECIDED", "L"),
    ("leader_to_verdict", "cluster barrier publishing the decision", "VERDICT", "CHECKED", "L"),
    ("leader_commit", "page table, slot map, stamps, LRU order, counter", "COMMITTED", "VERDICT",
     "L"),
)


def summarise_stamps(a, C):
    """Stage durations of resolve launches from hs_resolve_measure stamps.

    `a` is [launches][R][8][16] u64 (ns).  Per launch, t0 = the earliest CTA
    entry; per request the leader's phases (STAGE_US) and the followers'
    fetch milestones relative to t0 (first staging copy issued, staged
    records landed, slot stores issued), then medians over requests and
    launches (microseconds).  `fetch` = last landing - first issue per
    request: the host-link transfer; `decision` = leader entry to decision."""
    from hierarchical_kv_cache_resolve_gb300 import hs
    S = hs.HS_STAMP
    a = a.astype(np.float64)
    rows = []
    for launch in a:
        t0 = launch[:, :C, S["ENTRY"]].min()
        span = launch[:, :C, S["EXIT"]].max() - t0
        for req in launch:
            ld = req[0]
            d = {name: (ld[S[hi]] - ld[S[lo]]) / 1e3 for name, _, hi, lo, _ in STAGE_US}
            d["leader_start"] = (ld[S["ENTRY"]] - t0) / 1e3
            d["decision_done"] = (ld[S["DECIDED"]] - t0) / 1e3
            d["commit_done"] = (ld[S["COMMITTED"]] - t0) / 1e3
            d["leader_share_fetched"] = ((ld[S["LEAD_FETCHED"]] - t0) / 1e3
                                         if ld[S["LEAD_FETCHED"]] > 0 else None)
            d["launch_span"] = span / 1e3
            d["attempts"] = ld[S["ATTEMPTS"]]
            if C > 1:
                f = req[1:C]
                d["first_host_load_issued"] = (f[:, S["F_ISSUE"]][f[:, S["F_ISSUE"]] > 0].min()
                                               - t0) / 1e3 if (f[:, S["F_ISSUE"]] > 0).any() else None
                d["staging_issued"] = (f[:, S["F_ISSUED"]].max() - t0) / 1e3
                d["staged_landed"] = (f[:, S["F_LANDED"]].max() - t0) / 1e3
                d["slots_stored"] = (f[:, S["F_STORED"]].max() - t0) / 1e3
            rows.append(d)
    out = {}
    for key in rows[0]:
        vals = [r[key] for r in rows if r.get(key) is not None]
        out[key] = float(np.median(vals)) if vals else None
    if out.get("staged_landed") is not None and out.get("first_host_load_issued") is not None:
        out["fetch"] = out["staged_landed"] - out["first_host_load_issued"]
    return out


def run_measure_passes(pool, w, dsel, flush, main, cap, K, Wm):
    """Two diagnostics beside `value` (same steps, per-step graphs, L2
    flushed before every step, pool reset first):

    no_fetch -- hs_resolve_measure(HS_MEASURE_NO_FETCH): the resolve with
       every metadata step and no host fetch; per-launch time and the
       metadata HBM roofline (the no-IO analogue of the pages' no-IO run);
    stages   -- the resolve with stage timestamps (%globaltimer): a
       miss-resolution breakdown per launch (summarise_stamps).
    """
    import torch

    from hierarchical_kv_cache_resolve_gb300 import hs
    R, NL, k, B, T = w.n_requests, w.n_layers, w.k, w.slots, w.steps
    out = torch.empty((NL, R, k), dtype=torch.int32, device=dsel.device)
    slots = hs.hs_measure_stamp_slots()
    res = {}
    for name, flags, stamped in (("no_fetch", hs.HS_MEASURE_NO_FETCH, False),
                                 ("stages", 0, True)):
        times = (torch.zeros((K, NL, R, slots), dtype=torch.int64, device=dsel.device)
                 if stamped else None)
        graphs = []
        for i in range(K):
            g = torch.cuda.CUDAGraph()
            t = (Wm + i) % T
            with torch.cuda.graph(g, stream=cap):
                for l in range(NL):
                    pool.resolve_measure(l, dsel[t, l], out[l], flags=flags,
                                         times=times[i, l] if stamped else None, stream=cap)
            graphs.append(g)
        pool.reset()
        for s in range(Wm):
            for l in range(NL):
                pool.resolve_measure(l, dsel[s % T, l], out[l], flags=flags, stream=main)
        st0 = pool.stats(check=False)
        ms = 0.0
        for i in range(K):
            flush(i)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(main)
            graphs[i].replay()
            e1.record(main)
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
        st1 = pool.stats(check=False)
        del graphs
        launches = K * NL
        us = ms * 1e3 / launches
        m = (st1["misses"] - st0["misses"]) / max(1, st1["resolves"] - st0["resolves"])
        entry = {"what": ("hs_resolve_measure without the fetch, per-step graphs, L2 flushed "
                          "before every step" if not stamped else
                          "hs_resolve_measure with %globaltimer stage stamps, per-step graphs, "
                          "L2 flushed before every step; medians over requests and launches, "
                          "microseconds from the launch's first CTA entry"),
                 "us_per_launch": us, "resolves_per_s": launches * R / (ms / 1e3),
                 "misses_per_resolve": m, "status": st1["status"]}
        if not stamped:
            peaks = load_peaks()
            hbm = peaks.get("hbm_gbs") if peaks else None
            meta = R * metadata_bytes_per_resolve(k, B, m)
            achieved = meta / (us * 1e-6) / 1e9
            entry["roofline_hbm_metadata"] = {
                "kernel": "resolve_kernel (no fetch)", "bound": "hbm", "achieved": achieved,
                "peak": hbm, "unit": "GB/s", "frac": achieved / hbm if hbm else None,
                "algorithmic_bytes_per_launch": meta,
                "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if hbm else None}
        else:
            a = times.cpu().numpy().reshape(K, NL, R, 8, 16)
            C = 1
            while C < 8 and a[:, :, :, C, hs.HS_STAMP["ENTRY"]].any():
                C += 1
            entry["cluster_ctas"] = C
            entry["median_us"] = summarise_stamps(a.reshape(K * NL, R, 8, 16), C)
            # the first launch of a step has no launch ahead of it to overlap
            entry["first_launch_of_step_median_us"] = summarise_stamps(a[:, 0], C)
            if NL > 1:
                entry["later_launches_median_us"] = summarise_stamps(
                    a[:, 1:].reshape(K * (NL - 1), R, 8, 16), C)
            entry["stage_legend"] = {name: what for name, what, _, _, _ in STAGE_US}
        res[name] = entry
    pool.reset()
    return res


# ------------------------------------------------ exact prefetch overlap ----

def run_prefetch_overlap(args, w):
    """Resolves against compute, with and without exact layer-wise prefetch.

    Each layer of a decode step is its resolve, the sparse attention
    consumer over the slots it published (`--attn-heads` query heads per
    request), and a bf16 GEMM that stands in for the layer's MLP
    (`--compute-us` long).  For a layer that shares its anchor's selection,
    prefetch ON plans its misses and copies them on a side stream as soon as
    the anchor's selection is known (ahead of the anchor's resolve), so plan
    and copy overlap the layers in between; the main stream waits for the
    copy before the GEMM ahead of the layer's resolve, which then consumes
    the plan.  After PREROLL_STEPS untimed steps and a reset, four timings
    of the same steps (CUDA events, L2 flushed before each step): the
    resolves alone, the compute alone, both without prefetch, both with
    prefetch.
    The share of the resolves' own time hidden behind the compute is
    1 - (both - compute) / alone, with and without prefetch; `prefetch_gain`
    is what prefetch adds over resolves that already start under the
    preceding kernel (programmatic launch).
    """
    import torch

    from hierarchical_kv_cache_resolve_gb300 import hs
    from workloads import records, traces

    dev = torch.device("cuda", torch.cuda.current_device())
    R, NL, k, T = w.n_requests, w.n_layers, w.k, w.steps
    sel = traces.generate(w)
    dsel = torch.from_numpy(np.ascontiguousarray(sel.transpose(0, 2, 1, 3))).to(dev)
    pool = hs.Pool.for_workload(w, host_alloc=HOST_ALLOC[args.host_alloc],
                                launch_overlap=OVERLAP[args.launch_overlap])
    for r in range(R):
        for l in range(NL):
            records.fill(pool.host_records(r, l).ctypes.data, w, r, l)
    pool.warm()
    # published slots; before the first resolve, k distinct rows per request
    B = w.slots
    out = (torch.arange(R, dtype=torch.int32, device=dev)[:, None] * B
           + torch.arange(k, dtype=torch.int32, device=dev)[None, :]).repeat(NL, 1, 1)
    replay = args.prefetch_source == "replay"
    shared = [l for l in range(NL) if w.anchors[l] != l]
    # replay: one plan per anchor, written by its resolve; plan: one per
    # shared layer, written by hs_prefetch_plan
    plans = {l: torch.empty(hs.hs_plan_bytes(R, k), dtype=torch.uint8, device=dev)
             for l in range(NL) if (w.anchors[l] != l) != replay}
    flush = L2Flush(dev)
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()

    heads = args.attn_heads
    attn = w.record_bytes == 1152 and heads > 0
    if attn:
        q = torch.randn((R, heads, 576), device=dev).to(torch.bfloat16)
        o = torch.empty((R, heads, 512), dtype=torch.float32, device=dev)
        caches = [pool.views(l)["cache"] for l in range(NL)]
        scale = 1.0 / math.sqrt(576.0)

    def attention(l):
        if attn:
            hs.hs_sparse_attention(q, caches[l], R * B, out[l], R, k, heads, scale, o,
                                   stream=main)

    # MLP stand-in: [4096 x 4096] x [4096 x n] bf16, n chosen for the target time
    a = torch.randn(4096, 4096, device=dev, dtype=torch.bfloat16)
    b = torch.randn(4096, 4096, device=dev, dtype=torch.bfloat16)
    for _ in range(3):
        a @ b
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        a @ b
    e1.record()
    torch.cuda.synchronize()
    us_full = e0.elapsed_time(e1) * 100.0
    n = max(64, min(4096, int(4096 * args.compute_us / us_full) // 64 * 64))
    bb = b[:, :n].contiguous()

    def compute():
        return a @ bb

    def step(t, mode):
        evs = {}
        for l in range(NL):
            anc = w.anchors[l]
            if mode != "compute":
                if l == anc:
                    if mode == "on" and replay and l in plans:
                        # the anchor's resolve writes its miss plan
                        pool.resolve_anchor(l, dsel[t, l], out[l], plans[l], stream=main)
                    if mode == "on":
                        # The anchor's selection is known and the shared
                        # layers' previous resolves and attention calls are
                        # behind this point of the main stream (with replay,
                        # the anchor's plan too): copy the shared layers'
                        # misses on the side stream from here on.
                        ready = torch.cuda.Event()
                        ready.record(main)
                        side.wait_event(ready)
                        for l2 in shared:
                            if w.anchors[l2] != l:
                                continue
                            if not replay:
                                pool.prefetch_plan(l, l2, dsel[t, l2], plans[l2], stream=side)
                            pool.prefetch_copy(l2, R, k, plans[l if replay else l2], stream=side)
                            evs[l2] = torch.cuda.Event()
                            evs[l2].record(side)
                    if not (mode == "on" and replay and l in plans):
                        pool.resolve(l, dsel[t, l], out[l], stream=main)
                elif mode == "on":
                    pool.resolve(l, dsel[t, l], out[l], plan=plans[anc if replay else l],
                                 stream=main)
                else:
                    pool.resolve(l, dsel[t, l], out[l], stream=main)
            if mode != "resolve":
                attention(l)
                if mode == "on" and l + 1 in evs:
                    # the next layer's copy completes before the GEMM ahead
                    # of its resolve starts
                    main.wait_event(evs[l + 1])
                compute()

    # untimed pre-roll: on a freshly created huge-page pool the first tens of
    # steps can stall, and the mode timed first would carry them
    pool.reset()
    for s in range(PREROLL_STEPS):
        step(s % T, "off")
    torch.cuda.synchronize()
    results = {}
    for mode in ("resolve", "compute", "off", "on"):
        pool.reset()
        for s in range(args.warmup):
            step(s % T, mode)
        torch.cuda.synchronize()
        total = 0.0
        for i in range(args.steps):
            flush(i)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(main)
            step((args.warmup + i) % T, mode)
            e1.record(main)
            torch.cuda.synchronize()
            total += e0.elapsed_time(e1)
        results[mode] = total / args.steps
        if mode in ("off", "on"):
            st = pool.stats(check=False)
            results[mode + "_stats"] = {x: st[x] for x in ("misses", "fetched_bytes",
                                                          "prefetched_bytes", "plan_hits",
                                                          "plan_mismatches", "status")}
    attn_res = time_attention(lambda: attention(0), flush, main, R, k, heads,
                              args.steps) if attn else None
    kern = time_prefetch_kernels(pool, w, dsel, out, plans, flush, main, args, replay)
    pool_launch_overlap = pool.info()["launch_overlap"]
    pool.close()
    alone = results["resolve"]
    hidden_off = 1.0 - (results["off"] - results["compute"]) / alone
    hidden_on = 1.0 - (results["on"] - results["compute"]) / alone
    return {
        "metric": "resolve time hidden behind compute: step time with and without resolves",
        "value": hidden_on, "unit": "fraction of the resolves' own time hidden (prefetch on)",
        "hidden_without_prefetch": hidden_off,
        "prefetch_gain": 1.0 - (results["on"] - results["compute"]) /
                         (results["off"] - results["compute"]),
        "higher_is_better": True,
        "config": {"workload": workload_name(w), "shared_layers_per_step": len(shared),
                   "launch_overlap": "on" if pool_launch_overlap == hs.HS_OVERLAP_ON else "off",
                   "prefetch_source": ("the anchor's miss plan written by its resolve "
                                       "(hs_resolve_anchor)" if replay else
                                       "hs_prefetch_plan per shared layer"),
                   "attention": (f"hs_sparse_attention over the published slots, {heads} "
                                 f"heads per request" if attn else "none"),
                   "mlp_stand_in": f"bf16 GEMM 4096x4096x{n} after every layer",
                   "l2": "flushed before every timed step"},
        "ms_per_step": {"resolves_alone": alone, "compute_only": results["compute"],
                        "prefetch_off": results["off"], "prefetch_on": results["on"]},
        "counters": {"off": results["off_stats"], "on": results["on_stats"]},
        "attention": attn_res,
        "prefetch_kernels": kern,
        "steps": args.steps, "warmup": args.warmup,
        "preroll_steps": PREROLL_STEPS,
    }


def time_prefetch_kernels(pool, w, dsel, out, plans, flush, stream, args, replay=False):
    """The plan and copy kernels of exact prefetch, each timed alone.

    The same decode steps as prefetch ON, all on one stream and without the
    compute: the anchor's resolve, then for each layer sharing its selection
    the plan and the copy (each bracketed by CUDA events), then the shared
    layers' resolves consuming the plans, so that the pool evolves exactly as
    it does with prefetch.  L2 is flushed before every timed step.  The copy
    moves m records of W bytes per request over the host link (roofline
    against the pinned H2D ceiling measured here); the plan reads the
    selection, slot map and LRU order of each request and writes its plan
    entry (HBM roofline; its phases run one after another, so it is
    latency-bound at these sizes).
    """
    import torch

    from hierarchical_kv_cache_resolve_gb300 import hs

    R, NL, k, B, W, T = w.n_requests, w.n_layers, w.k, w.slots, w.record_bytes, w.steps
    h2d_gbs, _ = hs.hs_link_probe(1 << 30, 10, W)

    shared = [l for l in range(NL) if w.anchors[l] != l]

    def step(t, pending):
        for l in range(NL):
            if w.anchors[l] == l:
                if replay and l in plans:
                    pool.resolve_anchor(l, dsel[t, l], out[l], plans[l], stream=stream)
                else:
                    pool.resolve(l, dsel[t, l], out[l], stream=stream)
                for l2 in shared:
                    if w.anchors[l2] != l:
                        continue
                    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                    ev[0].record(stream)
                    if not replay:
                        pool.prefetch_plan(l, l2, dsel[t, l2], plans[l2], stream=stream)
                    ev[1].record(stream)
                    pool.prefetch_copy(l2, R, k, plans[l if replay else l2], stream=stream)
                    ev[2].record(stream)
                    pending.append(ev)
            else:
                pool.resolve(l, dsel[t, l], out[l], plan=plans[w.anchors[l] if replay else l],
                             stream=stream)

    pool.reset()
    for s in range(args.warmup):
        step(s % T, [])
    torch.cuda.synchronize()
    before = pool.stats(check=False)
    plan_ms = copy_ms = 0.0
    calls = 0
    for i in range(args.steps):
        flush(i)
        pending = []
        step((args.warmup + i) % T, pending)
        torch.cuda.synchronize()
        for e in pending:
            plan_ms += e[0].elapsed_time(e[1])
            copy_ms += e[1].elapsed_time(e[2])
        calls += len(pending)
    after = pool.stats(check=False)
    if calls == 0:
        return None
    moved = after["prefetched_bytes"] - before["prefetched_bytes"]
    planned = moved // W
    plan_bytes = calls * (R * (4 * k + 6 * B + 16) + 16) + 8 * planned
    peaks = load_peaks()
    hbm = peaks.get("hbm_gbs") if peaks else None
    plan_gbs = plan_bytes / (plan_ms / 1e3) / 1e9 if not replay and plan_ms > 0 else None
    copy_gbs = moved / (copy_ms / 1e3) / 1e9
    return {
        "calls": calls,
        "requests_per_call": R,
        "records_per_call": planned / calls,
        "plan": None if replay else {"us_per_call": plan_ms * 1e3 / calls, "kernels_per_call": 1,
                 "algorithmic_bytes_per_call": plan_bytes / calls,
                 "roofline": {"bound": "hbm", "achieved": plan_gbs, "peak": hbm,
                              "unit": "GB/s", "frac": plan_gbs / hbm if hbm else None,
                              "peak_source": ("MEASURED_PEAKS.json hbm_gbs (of measured)"
                                              if hbm else None)}},
        "copy": {"us_per_call": copy_ms * 1e3 / calls, "kernels_per_call": 1,
                 "link_bytes_per_call": moved / calls,
                 "roofline": {"bound": "link", "achieved": copy_gbs, "peak": h2d_gbs,
                              "unit": "GB/s", "frac": copy_gbs / h2d_gbs,
                              "peak_source": "pinned cudaMemcpyAsync H2D, 1 GiB, "
                                             "best of 10, this run"}},
        "l2": "flushed before every timed step",
    }


def attention_bytes(R: int, k: int, heads: int) -> int:
    """Algorithmic HBM bytes of one sparse attention call: the k gathered
    576-element bf16 records and k int32 slot indices per request, the bf16
    queries, the fp32 outputs (the split results merge on chip)."""
    return R * k * (1152 + 4) + R * heads * (1152 + 512 * 4)


def attention_heads_bytes(R: int, k: int, heads: int) -> int:
    """Algorithmic HBM bytes of one per-head attention call: the k gathered
    records of heads * 512 bytes and k int32 slot indices per request, the
    bf16 queries (128 per head) and the fp32 outputs (128 per head)."""
    return R * k * (heads * 512 + 4) + R * heads * (128 * 2 + 128 * 4)


def time_attention(call, flush, stream, R, k, heads, steps, nbytes=None):
    """CUDA-event time of one sparse attention call (one kernel) on
    `stream`, L2 flushed before every timed call; HBM roofline against the
    measured copy bandwidth."""
    import torch
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    total = 0.0
    for i in range(steps):
        flush(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    s = total / steps / 1e3
    if nbytes is None:
        nbytes = attention_bytes(R, k, heads)
    peaks = load_peaks()
    peak = peaks.get("hbm_gbs") if peaks else None
    achieved = nbytes / s / 1e9
    return {"us_per_call": s * 1e6, "kernels_per_call": 1,
            "algorithmic_bytes_per_call": nbytes,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak if peak else None,
                         "peak_source": ("MEASURED_PEAKS.json hbm_gbs (of measured)"
                                         if peak else None)}}


# ------------------------------------------------ attention consumer alone ----

def run_attention(args, w):
    """The sparse attention consumer alone on a workload's shape: a layer
    cache of R*B random bf16 records in HBM, k distinct published rows per
    request inside its own B slots (as a resolve publishes them), `--attn-heads`
    query heads per request; L2 flushed before every timed call."""
    import torch

    from hierarchical_kv_cache_resolve_gb300 import hs
    per_head = w.record_bytes != 1152
    if per_head and (w.record_bytes % 512 or not 1 <= w.record_bytes // 512 <= 8):
        raise SystemExit("bench.py --attention: the consumers read 576-element MLA records "
                         "or token records of 1 to 8 heads of 128 (keys, then values)")
    dev = torch.device("cuda", torch.cuda.current_device())
    R, k, B = w.n_requests, w.k, w.slots
    heads = w.record_bytes // 512 if per_head else args.attn_heads
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    cache = torch.randn((R * B, w.record_bytes // 2), device=dev,
                        generator=g).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(B, device=dev, generator=g)[:k] + r * B
                       for r in range(R)]).to(torch.int32)
    flush = L2Flush(dev)
    main = torch.cuda.current_stream()
    if per_head:
        q = torch.randn((R, heads, 128), device=dev, generator=g).to(torch.bfloat16)
        o = torch.empty((R, heads, 128), dtype=torch.float32, device=dev)
        scale = 1.0 / math.sqrt(128.0)

        def call():
            hs.hs_sparse_attention_heads(q, cache, R * B, idx, R, k, heads, scale, o,
                                         stream=main)
    else:
        q = torch.randn((R, heads, 576), device=dev, generator=g).to(torch.bfloat16)
        o = torch.empty((R, heads, 512), dtype=torch.float32, device=dev)
        scale = 1.0 / math.sqrt(576.0)

        def call():
            hs.hs_sparse_attention(q, cache, R * B, idx, R, k, heads, scale, o, stream=main)

    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler.shared(f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:"
                                  f"{props.pci_device_id:02x}.0")
    sampler.start()
    res = time_attention(call, flush, main, R, k, heads, args.steps,
                         nbytes=attention_heads_bytes(R, k, heads) if per_head else None)
    sampler.stop()
    status = hs.hs_attention_status()
    return {"metric": "sparse attention over published slots: gathered HBM GB/s",
            "value": res["roofline"]["achieved"], "unit": "GB/s", "higher_is_better": True,
            "config": {"workload": workload_name(w), "heads": heads,
                       "consumer": ("hs_sparse_attention_heads (per-head token records)"
                                    if per_head else "hs_sparse_attention (MLA records)"),
                       "l2": "flushed before every timed call"},
            "attention": res, "status": status, "clocks": sampler.summary(),
            "steps": args.steps, "warmup": 3}


# ------------------------------------------------------------------ main ----

def link_sweep(sizes_gib, record_bytes: int) -> dict:
    """hs_link_probe over host buffers of each size, for each allocation
    kind: the pinned H2D copy rate (1 GiB from the buffer's start) and the
    rate of gathering 1 GiB of `record_bytes` records from indices spread
    uniformly over the whole buffer -- where scattered GPU-thread reads of a
    pool of that size stand against the link (best of 3 each)."""
    from hierarchical_kv_cache_resolve_gb300 import hs
    rows = []
    for gib in sizes_gib:
        for name in ("pinned", "vmm", "thp"):
            t0 = time.perf_counter()
            try:
                h2d, gather = hs.hs_link_probe(gib << 30, 3, record_bytes, HOST_ALLOC[name])
                rows.append({"gib": gib, "host_alloc": name, "h2d_gbs": h2d,
                             "gather_gbs": gather, "s": time.perf_counter() - t0})
            except hs.HsError as e:
                rows.append({"gib": gib, "host_alloc": name, "error": str(e)})
    return {"what": "hs_link_probe per host allocation kind and buffer size", "unit": "GB/s",
            "record_bytes": record_bytes, "rows": rows}


def spawn_ranks(n: int, argv) -> int:
    """`bench.py --gpus N` started as one process: re-run it under
    torch.distributed.run with one rank per GPU on this node (rendezvous on
    127.0.0.1), and return the launcher's exit status.  Rank 0 prints the
    JSON line."""
    import socket
    import subprocess
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def bind_to_device_numa(device: int):
    """Runs this process on the CPUs of the host NUMA node closest to
    `device` (cudaDevAttrHostNumaId), so the records it generates are
    written by local cores; returns (node, cpus) or (None, None) when the
    system reports no node for the device.  The pool's pinned pages are
    placed on that node by the library itself (hs_create_pool)."""
    from hierarchical_kv_cache_resolve_gb300 import hs
    node = hs.hs_device_host_numa(device)
    if node < 0:
        return None, None
    try:
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            cpus = parse_cpulist(f.read())
        cpus &= os.sched_getaffinity(0) or cpus
        if cpus:
            os.sched_setaffinity(0, cpus)
        return node, len(cpus)
    except OSError:
        return node, None


def host_memory_available():
    """MemAvailable of /proc/meminfo in bytes (None if unknown)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return None


def parse_cpulist(text: str) -> set:
    """'0-3,8,10-11' -> {0, 1, 2, 3, 8, 10, 11}"""
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        else:
            cpus.add(int(part))
    return cpus


def reference_arm(args, w, threads: int) -> dict:
    """The reference arm: the CPU oracle as it stands on a bounded sample of
    the workload (the first CPU_SAMPLE_PAIRS (request, layer) pairs, each
    over warm-up + timed steps of its trace, one thread per pair)."""
    pairs = min(w.n_requests * w.n_layers, CPU_SAMPLE_PAIRS)
    steps = args.warmup + args.steps
    value, wall, n, fetched = time_oracle(w, pairs, steps, threads)
    sample = (f"the CPU oracle on {pairs} of the {w.n_requests * w.n_layers} (request, layer) "
              f"pairs x {steps} steps (warm-up included), one thread per pair, "
              f"{min(threads, pairs)} threads")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "resolves/s",
            "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wall / steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int32", "data": "synthetic",
            "config": {"workload": workload_name(w), "global_batch": w.n_requests,
                       "sample": sample},
            "cpu_baseline": {"value": value, "unit": "resolves/s", "cores": min(threads, pairs),
                             "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "resolves/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "miss_fetch": {"gbs": fetched / wall / 1e9, "unit": "GB/s"}}


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="tight_prefetch",
                    help="the headline workload (default: the largest, tight_prefetch)")
    ap.add_argument("--also", default="dsa_mla",
                    help="comma-separated workloads timed after the headline (graph pass "
                         "only) and reported beside it; 'none' for none")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--host-alloc", choices=sorted(HOST_ALLOC), default="auto",
                    help="how the pinned host pool is allocated (hs_pool_desc.host_alloc)")
    ap.add_argument("--launch-overlap", choices=sorted(OVERLAP), default="auto",
                    help="whether consecutive resolves may overlap (hs_pool_desc.launch_overlap)")
    ap.add_argument("--cpu-threads", type=int, default=0)
    ap.add_argument("--l-ctx", type=int, default=0,
                    help="profiling captures only: shrink L_ctx (same k, B, W, batch), so "
                         "that the pinned pool and page tables stay small")
    ap.add_argument("--requests", type=int, default=0,
                    help="override the workload's batch (requests per launch)")
    ap.add_argument("--prefetch-overlap", action="store_true",
                    help="measure exact layer-wise prefetch against stand-in compute "
                         "(a workload with shared layers, e.g. tight_prefetch)")
    ap.add_argument("--prefetch-source", choices=["replay", "plan"], default="replay",
                    help="--prefetch-overlap: the anchor's own miss plan (hs_resolve_anchor) "
                         "or one hs_prefetch_plan launch per shared layer")
    ap.add_argument("--compute-us", type=float, default=60.0,
                    help="MLP stand-in compute per layer for --prefetch-overlap")
    ap.add_argument("--attention", action="store_true",
                    help="time the sparse attention consumer alone on the workload's shape")
    ap.add_argument("--link-sweep", default="",
                    help="comma-separated GiB sizes: time hs_link_probe (pinned H2D copy and "
                         "scattered record gather over the whole buffer) for each host "
                         "allocation kind and size, print one JSON line, and exit")
    ap.add_argument("--attn-heads", type=int, default=16,
                    help="query heads per request of the sparse attention consumer in "
                         "--prefetch-overlap (a multiple of 16; 0: no attention)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return spawn_ranks(args.gpus, argv)

    from workloads import configs

    def shaped(name):
        w = configs.BY_NAME[name]
        if args.l_ctx:
            w = w.with_(n_positions=args.l_ctx, local_window=min(w.local_window, args.l_ctx // 8))
        if args.requests:
            w = w.with_(n_requests=args.requests)
        return w

    base = shaped(args.workload)
    also = [] if args.also in ("", "none") else [x for x in args.also.split(",")
                                                  if x and x != args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    threads = args.cpu_threads or len(os.sched_getaffinity(0))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args, base, threads)))
        return 0

    import torch
    dist_on = world > 1
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the resolve path has no CPU fallback)")
    need = max([base.host_bytes] + [shaped(n).host_bytes for n in also]) * world
    avail = host_memory_available()
    if avail is not None and need > avail:
        raise SystemExit(f"bench.py: {world} rank(s) need {need / 1e9:.1f} GB of pinned host "
                         f"memory for their pools, {avail / 1e9:.1f} GB is available")
    torch.cuda.set_device(local)
    numa, numa_cpus = bind_to_device_numa(local)
    if dist_on:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.link_sweep:
        if rank == 0:
            print(json.dumps(link_sweep([int(x) for x in args.link_sweep.split(",") if x],
                                        base.record_bytes)))
        return 0
    w = rank_workload(base, rank)
    if args.prefetch_overlap or args.attention:
        if rank == 0:
            run = run_prefetch_overlap if args.prefetch_overlap else run_attention
            print(json.dumps(run(args, w)))
        return 0
    # the headline first: its pool is the process's first large pinned
    # allocation; the other workloads follow
    res = run_gpu(args, w, rank, world, dist_on)
    res["config"]["host_numa_node"] = numa
    res["config"]["process_cpus"] = numa_cpus
    others = {}
    for name in also:
        lite = run_gpu(args, rank_workload(shaped(name), rank), rank, world, dist_on, lite=True)
        lite["timed_after"] = "the headline workload, in the same process"
        others[name] = lite
    if others:
        res["other_workloads"] = others
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(base, threads)
        print(json.dumps(res))
    if dist_on:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python
"""Benchmark of the paged KV-cache transfer on GB300.

One step = the whole hot path over one batch: the all-layer D2H backup of the
workload's pages, then the per-layer H2D load-back burst of those pages into
fresh device pages with one layer-done event per layer.  The headline metric
is KV transfer GB/s (payload bytes of both operations / device time) and its
fraction of the host-link peak measured in the same run with pinned
cudaMemcpyAsync copies (D2H and H2D, 1 GiB, best of 5).

Default workload: the 78-layer MLA model with two host pools (latent KV of
576 bf16 per token plus the DSA indexer-K of 132 bytes per token, page_size
64): an all-layer backup of 1024 pages (6.56 GB) and a load-back burst of 1024
pages with 78 layer events (80.25 MiB per layer).  The pools hold 13.1 GB on
each side, far larger than L2, so no flush is needed between steps.  After the
timed region, a consumer kernel gated by each layer event reads that layer on
another stream, to report how much of the consumers' work the burst hides.

Multi-GPU: every pair is independent and each GPU holds its own pool replica,
so N ranks run N independent replicas (weak scaling, no collective on the data
path); rank 0 prints the aggregate.

``--impl reference`` times the CPU oracle (plain C loops) on a bounded sample
of the same workload, the only baseline that exists for this path.
"""
from __future__ import annotations

import argparse
import contextlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

REPO = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, REPO)

METRIC = "KV transfer GB/s (D2H backup, H2D per-layer load) & % of measured host-link peak"
UNIT = "GB/s"
GB = 1e9
# layers of at least this many bytes give the burst's first layer a launch of
# its own (the library's rule); smaller bursts are one signalling launch
SPLIT_FIRST_LAYER_BYTES = 16 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3, help="at least 3 (untimed)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mla78_dsa")
    ap.add_argument("--path", choices=["auto", "zero_copy", "staged"], default="auto")
    ap.add_argument("--staging-mib", type=int, default=256)
    ap.add_argument("--max-ctas", type=int, default=0)
    ap.add_argument("--burst", choices=["per_layer", "single_launch"], default="single_launch",
                    help="load burst as one kernel launch per layer, or one launch for all layers")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--duplex", action="store_true",
                    help="also measure backup and load-back running concurrently (full duplex)")
    ap.add_argument("--no-consumer", action="store_true",
                    help="skip the consumer kernels gated by each layer event (run after the "
                         "timed region by default)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    ap.add_argument("--pages", type=int, default=0,
                    help="override the pages moved per op (smaller profiling cases)")
    ap.add_argument("--device-slots", type=int, default=0, help="override device slots per pool")
    ap.add_argument("--host-pages", type=int, default=0, help="override host pages per pool")
    ap.add_argument("--layout", choices=["page_first_direct", "page_first"], default=None,
                    help="override the host layout of every pool of the workload")
    ap.add_argument("--sweep", action="store_true",
                    help="run the row-size / page-size / length / fragmentation sweep instead")
    ap.add_argument("--sweep-rows", default="16,64,256,1152,2048")
    ap.add_argument("--sweep-pages", default="1,16,64,256")
    ap.add_argument("--sweep-tokens", default="1024,4096,16384,65536,262144")
    ap.add_argument("--sweep-layers", type=int, default=4)
    ap.add_argument("--dma-sweep", action="store_true",
                    help="measure the copy engine's cost per copy against the copy size instead")
    ap.add_argument("--latency", action="store_true",
                    help="measure per-op latency for small page counts instead")
    ap.add_argument("--latency-pages", default="1,4,16,64,256")
    ap.add_argument("--contention", action="store_true",
                    help="measure both paths beside a bf16 GEMM loop that occupies the SMs "
                         "(the regime the staged path is for) instead")
    ap.add_argument("--contention-reps", type=int, default=3)
    ap.add_argument("--contention-staged-ctas", default="0,4,8,16",
                    help="copy CTA caps of the staged path under --contention")
    ap.add_argument("--contention-alone-only", action="store_true",
                    help="time the transfers alone only (no GEMM loop beside them)")
    ap.add_argument("--contention-ctas", default="4,8,16,24,76,152",
                    help="copy CTA caps to measure under contention (0 = library default)")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Largest value of x over all ranks (NCCL on GPUs, gloo on CPU)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(world, steps, step_bytes, max_ms):
    """Whole-job GB/s of `world` replicas that each moved steps * step_bytes, timed by the slowest."""
    return world * steps * step_bytes / (max_ms * 1e-3) / GB


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------- host link peak

def measure_duplex_peak(nbytes=1 << 30, reps=3):
    """Pinned DMA in both directions at once (two streams), best of `reps`: GB/s of both."""
    import torch
    h1 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h2 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d1 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    best = 0.0
    for r in range(reps + 1):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(sa)
        sb.wait_event(e0)
        with torch.cuda.stream(sa):
            h1.copy_(d1, non_blocking=True)
        with torch.cuda.stream(sb):
            d2.copy_(h2, non_blocking=True)
        sa.wait_stream(sb)
        e1.record(sa)
        e1.synchronize()
        if r:
            best = max(best, 2 * nbytes / (e0.elapsed_time(e1) * 1e-3) / GB)
    del h1, h2, d1, d2
    torch.cuda.synchronize()
    return best


def run_duplex(hk, pools, wl, idx_b, L, opts_b, opts_l, n, reps=10):
    """Backup on one stream and a load burst of other host pages on another, concurrently.

    Write-back of newly computed KV and load-back of cache hits are independent
    in a serving system; the host link is full duplex.  The load reads host
    pages the backup does not write and fills device slots the backup does not
    read.
    """
    import torch
    from hierarchical_kv_cache_gb300 import workloads as W
    s0 = wl.pools[0]
    P = s0.page_size
    dev_pages = min(s.device_slots for s in wl.pools) // P
    host_pages = min(s.host_pages for s in wl.pools)
    d_b = idx_b[0].cpu().numpy()
    h_b = idx_b[1].cpu().numpy()
    g = W.rng(wl.seed + 77)
    hp = W.sample_pages(g, host_pages, wl.move_pages, exclude=np.unique(h_b // P))
    dp = W.sample_pages(g, dev_pages, wl.move_pages, exclude=np.unique(d_b // P))
    h_l = torch.as_tensor(W.expand_pages(hp, P)).cuda()
    d_l = torch.as_tensor(W.expand_pages(dp, P)).cuda()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    evs = [torch.cuda.Event() for _ in range(L)]
    bytes_backup, bytes_layer = payload_bytes(wl, n)
    peak = measure_duplex_peak()
    times = []
    for r in range(reps + 2):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(sa)
        sb.wait_event(e0)
        hk.hicache_backup_all_layers(pools, idx_b[0], idx_b[1], opts=opts_b, stream=sa)
        hk.hicache_load_burst(pools, 0, L, h_l, d_l, opts=opts_l, stream=sb, layer_done=evs)
        sa.wait_stream(sb)
        e1.record(sa)
        e1.synchronize()
        if r >= 2:
            times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    gbs = (bytes_backup + bytes_layer * L) / (ms * 1e-3) / GB
    return {"what": "all-layer backup and a load-back burst of other host pages, concurrently "
                    "on two streams",
            "gbs": round(gbs, 2), "ms": round(ms, 4), "duplex_dma_peak_gbs": round(peak, 2),
            "frac_of_duplex_dma_peak": round(gbs / peak, 4), "reps": reps}


def measure_link_peak(nbytes=1 << 30, reps=5):
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    h.fill_(1)
    d.fill_(2)
    s = torch.cuda.Stream()
    out = {}
    for name, dst, src in (("d2h", h, d), ("h2d", d, h)):
        best = 0.0
        with torch.cuda.stream(s):
            for r in range(reps + 1):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(s)
                dst.copy_(src, non_blocking=True)
                e1.record(s)
                e1.synchronize()
                if r:
                    best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / GB)
        out[name] = best
    del h, d
    torch.cuda.synchronize()
    return out


def hbm_peak():
    """Measured HBM copy bandwidth of the GB300s, else the recipe's fallback."""
    try:
        with open(os.path.join(REPO, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        return 6800.0


def traffic_per_launch(workload, which, algorithmic_bytes):
    """DRAM bytes (read + write) per launch from the committed ncu record of this workload,
    scaled to this launch's algorithmic bytes; None when the record has no such launch or
    the kernel source changed since the capture."""
    import hashlib
    try:
        with open(os.path.join(REPO, "profiles", "row_copy_kernel_traffic.json")) as f:
            rec = json.load(f)
        src = open(os.path.join(REPO, rec["source_file"]), "rb").read()
    except (OSError, ValueError, KeyError):
        return None
    if hashlib.sha256(src).hexdigest()[:16] != rec.get("source_sha256_16"):
        return None
    c = rec.get("workloads", {}).get(workload, {}).get("launches", {}).get(which)
    if c is None:
        return None
    per_byte = (c["dram_read_bytes"] + c["dram_write_bytes"]) / c["algorithmic_bytes"]
    return int(per_byte * algorithmic_bytes)


# ---------------------------------------------------------------- host placement

def _read(path):
    try:
        with open(path) as f:
            return f.read().strip()
    except OSError:
        return None


def _cpulist(text):
    """'0-3,8' -> {0, 1, 2, 3, 8}."""
    cpus = set()
    for part in (text or "").split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part.strip():
            cpus.add(int(part))
    return cpus


@contextlib.contextmanager
def pinned_allocation_near_gpu(dev):
    """Binds the process to the GPU's local CPUs while the pinned pools are first
    touched, so that their pages land on the NUMA node attached to the GPU, and
    restores the previous affinity afterwards (the CPU baseline keeps every core).
    Yields what the system reports: the GPU's PCI address, NUMA node and local
    CPUs, the nodes online, and whether the affinity had to change."""
    import torch
    info = {"nodes_online": _read("/sys/devices/system/node/online")}
    prop = torch.cuda.get_device_properties(dev)
    try:
        addr = "%04x:%02x:%02x.0" % (prop.pci_domain_id, prop.pci_bus_id, prop.pci_device_id)
    except AttributeError:
        addr = None
    if addr:
        base = f"/sys/bus/pci/devices/{addr}"
        info.update(pci=addr, gpu_numa_node=_read(base + "/numa_node"),
                    gpu_local_cpus=_read(base + "/local_cpulist"))
    old = os.sched_getaffinity(0)
    near = _cpulist(info.get("gpu_local_cpus")) & old
    bound = bool(near) and near != old
    info["bound_for_allocation"] = bound
    if bound:
        os.sched_setaffinity(0, near)
    try:
        yield info
    finally:
        if bound:
            os.sched_setaffinity(0, old)


# ---------------------------------------------------------------- workload

def build_workload(name, seed_offset=0, args=None):
    import dataclasses

    from hierarchical_kv_cache_gb300 import workloads as W
    wl = W.WORKLOADS[name]()
    if args is not None and args.layout:
        wl = dataclasses.replace(wl, pools=tuple(dataclasses.replace(s, layout=args.layout)
                                                 for s in wl.pools),
                                 name=wl.name + f" [host layout {args.layout}]")
    if args is not None and (args.pages or args.device_slots or args.host_pages):
        pools = tuple(dataclasses.replace(
            s, device_slots=args.device_slots or s.device_slots,
            host_pages=args.host_pages or s.host_pages) for s in wl.pools)
        wl = dataclasses.replace(wl, pools=pools, move_pages=args.pages or wl.move_pages,
                                 name=wl.name + " [resized for profiling]")
    s0 = wl.pools[0]
    P = s0.page_size
    dev_pages = min(s.device_slots for s in wl.pools) // P
    host_pages = min(s.host_pages for s in wl.pools)
    d, h, dp, _ = W.page_pairs(wl.seed + seed_offset, wl.move_pages, dev_pages, host_pages, P)
    d2, _, _, _ = W.page_pairs(wl.seed + seed_offset + 1, wl.move_pages, dev_pages, host_pages, P,
                               exclude_device_pages=dp)
    return wl, d, h, d2


def payload_bytes(wl, n):
    backup = sum(n * s.num_layers * s.num_tensors * s.row_bytes for s in wl.pools)
    per_layer = sum(n * s.num_tensors * s.row_bytes for s in wl.pools)
    return backup, per_layer


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world):
    import torch
    import hierarchical_kv_cache_gb300 as hk
    from hierarchical_kv_cache_gb300 import pools as hpools
    from hierarchical_kv_cache_gb300.build import build

    build()
    wl, d, h, d2 = build_workload(args.workload, args=args)
    L = wl.pools[0].num_layers
    n = d.size
    t_alloc = time.time()
    pools = []
    with pinned_allocation_near_gpu(torch.cuda.current_device()) as placement:
        for i, s in enumerate(wl.pools):
            p = hpools.allocate_pool(s)
            hpools.fill_device_random_(p, wl.seed + i, s.value_kind)
            for ht in p.host_tensors:
                ht.zero_()
            pools.append(p)
        torch.cuda.synchronize()
    t_alloc = time.time() - t_alloc

    path = {"auto": hk.HICACHE_PATH_AUTO, "zero_copy": hk.HICACHE_PATH_ZERO_COPY,
            "staged": hk.HICACHE_PATH_STAGED}[args.path]
    staged = args.path == "staged"
    staging = None
    if args.path != "zero_copy":
        staging = [torch.empty(args.staging_mib << 20, dtype=torch.uint8, device="cuda")
                   for _ in range(2)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    words = (torch.zeros(4 * L, dtype=torch.int32, device="cuda")
             if args.burst == "single_launch" else None)

    # device-resident indices for the device-timed value
    dt = torch.as_tensor(d).cuda()
    ht_dev = torch.as_tensor(h).cuda()
    d2t = torch.as_tensor(d2).cuda()
    # pinned host indices for the end-to-end leg and the staged path
    dt_h = torch.as_tensor(d).pin_memory()
    ht_h = torch.as_tensor(h).pin_memory()
    d2t_h = torch.as_tensor(d2).pin_memory()
    if args.path == "staged":
        # the staged path plans its DMAs on the CPU: pinned host indices, which
        # the library copies into HBM (opts.index_staging) for its kernels
        idx_b, idx_l = (dt_h, ht_h), (ht_h, d2t_h)
        opts = hk.Opts(path=path, index_location=hk.HICACHE_INDEX_HOST, staging=staging,
                       max_ctas=args.max_ctas, device_error=err, burst_words=words,
                       index_staging=torch.empty(hk.index_staging_bytes(n, 64),
                                                 dtype=torch.uint8, device="cuda"))
    else:
        idx_b, idx_l = (dt, ht_dev), (ht_dev, d2t)
        opts = hk.Opts(path=path, index_location=hk.HICACHE_INDEX_DEVICE, staging=staging,
                       max_ctas=args.max_ctas, device_error=err, burst_words=words)

    link = measure_link_peak()
    bytes_backup, bytes_layer = payload_bytes(wl, n)
    bytes_load = bytes_layer * L
    step_bytes = bytes_backup + bytes_load

    # warm-up; each warm-up burst is also enqueued on an idle stream to time the
    # host cost of one burst (in the timed loop the host runs ahead and can block
    # on a full launch queue, which would inflate it)
    warm_events = [torch.cuda.Event(enable_timing=True) for _ in range(L)]
    enq_idle = []
    for _ in range(args.warmup):
        hk.hicache_backup_all_layers(pools, idx_b[0], idx_b[1], opts=opts, stream=stream)
        stream.synchronize()
        t0 = time.perf_counter()
        hk.hicache_load_burst(pools, 0, L, idx_l[0], idx_l[1], opts=opts, stream=stream,
                              layer_done=warm_events)
        enq_idle.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    host_s0 = measure_host_costs(hk, pools, d, h, dt_h, ht_h, d2t_h, L, opts, stream, n)

    K = args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_m = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_layers = [[torch.cuda.Event(enable_timing=True) for _ in range(L)] for _ in range(K)]
    enq = []
    launches0 = hk.kernel_launches()
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    wall0 = time.perf_counter()
    for k in range(K):
        ev_s[k].record(stream)
        hk.hicache_backup_all_layers(pools, idx_b[0], idx_b[1], opts=opts, stream=stream)
        ev_m[k].record(stream)
        t0 = time.perf_counter()
        hk.hicache_load_burst(pools, 0, L, idx_l[0], idx_l[1], opts=opts, stream=stream,
                              layer_done=ev_layers[k])
        enq.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clk = clocks.stop() if clocks else None
    launches = hk.kernel_launches() - launches0
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())}")

    total_ms = ev_s[0].elapsed_time(ev_layers[-1][-1])
    t_backup = [ev_s[k].elapsed_time(ev_m[k]) for k in range(K)]
    t_load = [ev_m[k].elapsed_time(ev_layers[k][-1]) for k in range(K)]
    t_first = [ev_m[k].elapsed_time(ev_layers[k][0]) for k in range(K)]
    # layers 1..L-1 of a single-launch burst are one launch: first event to last event
    t_rest = [ev_layers[k][0].elapsed_time(ev_layers[k][-1]) for k in range(K)]
    t_step = [ev_s[k].elapsed_time(ev_layers[k][-1]) for k in range(K)]
    k_med = sorted(range(K), key=lambda k: t_load[k])[K // 2]  # step with the median burst
    per_layer = [ev_layers[k][l - 1].elapsed_time(ev_layers[k][l]) for k in range(K)
                 for l in range(1, L)]
    total_ms = max_over_ranks(total_ms, world)
    value = aggregate_gbs(world, K, step_bytes, total_ms)

    mb, ml = statistics.mean(t_backup), statistics.mean(t_load)
    # the committed DRAM-traffic record is per workload, in its default host layout
    traffic_key = args.workload + (f":{args.layout}" if args.layout else "")
    backup_gbs = bytes_backup / (mb * 1e-3) / GB
    load_gbs = bytes_load / (ml * 1e-3) / GB
    layer_gbs = bytes_layer / (statistics.median(per_layer) * 1e-3) / GB if per_layer else None
    if staged:
        layer_gbs = None  # the staged load lands layers in groups: only the burst has a rate
    first_us = statistics.mean(t_first) * 1e3
    bound_us = ml * 1e3 / L + 20.0
    # time-weighted link peak of the step's mix of directions
    peak_mix = step_bytes / (bytes_backup / link["d2h"] + bytes_load / link["h2d"])
    achieved = step_bytes / ((mb + ml) * 1e-3) / GB

    duplex = None
    if args.duplex and args.path != "staged":
        words2 = (torch.zeros(4 * L, dtype=torch.int32, device="cuda")
                  if args.burst == "single_launch" else None)
        opts_l = hk.Opts(path=path, index_location=hk.HICACHE_INDEX_DEVICE,
                         max_ctas=args.max_ctas, device_error=err, burst_words=words2)
        duplex = run_duplex(hk, pools, wl, idx_b, L, opts, opts_l, n)

    consumer = None
    if not args.no_consumer:
        consumer = run_consumer_overlap(hk, pools, idx_l, opts, L, stream, bytes_layer)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(hk, pools, wl, dt_h, ht_h, d2t_h, L, staging, path, args, step_bytes, n,
                      words)

    res = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4), "higher_is_better": True,
        "first_layer_event_us": round(first_us, 1),
        "first_event_bound_us": round(bound_us, 1),
        "first_event_within_bound": first_us <= bound_us,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded bf16 ~N(0,1) pools, seeded random page lists)",
        "config": {
            "workload": wl.name, "description": wl.description,
            "values": "bf16 ~N(0,1) KV bytes (uint8 for indexer / SSM state), moved opaquely",
            "pages_per_op": wl.move_pages, "tokens_per_op": int(n), "layers": L,
            "step": "all-layer D2H backup + H2D per-layer load-back burst with layer events",
            "step_payload_bytes": int(step_bytes), "path": args.path, "burst": args.burst,
            "index_location": ("device (HBM)" if args.path != "staged" else
                               "host (pinned), copied by the call into opts.index_staging"),
            "l2": "inputs larger than L2 (pools of GiBs on each side), no flush",
            "parallelism": f"replicas x{world}",
            "host_alloc_s": round(t_alloc, 1),
            "host_placement": placement,
        },
        "ops": {
            "backup_d2h_gbs": round(backup_gbs, 2),
            "backup_frac_of_link_d2h": round(backup_gbs / link["d2h"], 4),
            "backup_ms": round(mb, 4),
            "load_h2d_gbs": round(load_gbs, 2),
            "load_frac_of_link_h2d": round(load_gbs / link["h2d"], 4),
            "load_burst_ms": round(ml, 4),
            "load_per_layer_median_gbs": round(layer_gbs, 2) if layer_gbs else None,
            "first_layer_event_us": round(first_us, 1),
            "first_event_bound_us": round(bound_us, 1),
            "first_event_within_bound": first_us <= bound_us,
            "step_ms_min_median_max": [round(min(t_step), 4), round(statistics.median(t_step), 4),
                                       round(max(t_step), 4)],
            "step_ms_each": [round(t, 3) for t in t_step],
            "backup_ms_p50": round(statistics.median(t_backup), 4),
            "load_burst_ms_p50": round(statistics.median(t_load), 4),
            "layer_event_us_median_step": [round(ev_m[k_med].elapsed_time(e) * 1e3, 1)
                                           for e in ev_layers[k_med]],
            "enqueue_us_per_layer": round(statistics.median(enq_idle) * 1e6 / L, 2),
            "enqueue_us_per_layer_queue_full": round(statistics.median(enq) * 1e6 / L, 2),
            "link_peak_gbs": {k: round(v, 2) for k, v in link.items()},
            "host_s0": host_s0,
        },
        "roofline": None,  # filled below with the launch that dominates the step
        "roofline_backup": {
            "bound": "host_link", "achieved": round(backup_gbs, 2), "peak": round(link["d2h"], 2),
            "unit": "GB/s", "frac": round(backup_gbs / link["d2h"], 4),
            "traffic": (None if staged else
                        traffic_per_launch(traffic_key, "backup_all_layers", bytes_backup)),
            "kernel": ("staged backup: gather kernels into two HBM staging buffers, then one "
                       "cudaMemcpyAsync per host-page run, whole operation"
                       if staged else
                       "row_copy_kernel<int64,512,static>: one all-layer backup launch")
                      + f" ({bytes_backup} algorithmic bytes = n x L x T x R)",
            "peak_source": "pinned cudaMemcpyAsync D2H measured in this run (of measured); "
                           "HBM is not the bound: the launch reads its payload once from HBM",
            "hbm_frac_of_measured": round(backup_gbs / hbm_peak(), 4),
            "ms_per_launch": round(mb, 4),
        },
        "roofline_load": ({
            "bound": "host_link", "achieved": round(load_gbs, 2), "peak": round(link["h2d"], 2),
            "unit": "GB/s", "frac": round(load_gbs / link["h2d"], 4), "traffic": None,
            "kernel": "staged load burst: one cudaMemcpy2DAsync per host-page run and layer "
                      "group into HBM staging, then one scatter launch per layer, whole burst "
                      f"({bytes_load} algorithmic bytes = n x L x T x R)",
            "ms_per_launch": round(ml, 4),
        } if staged else {
            "bound": "host_link", "achieved": round(layer_gbs, 2) if layer_gbs else None,
            "peak": round(link["h2d"], 2), "unit": "GB/s",
            "frac": round(layer_gbs / link["h2d"], 4) if layer_gbs else None,
            "traffic": traffic_per_launch(traffic_key, "load_one_layer"
                                          if args.burst == "per_layer"
                                          else "load_burst_signalling", bytes_layer),
            "kernel": ("row_copy_kernel<int64,16,8>: one per-layer load launch"
                       if args.burst == "per_layer" else
                       "row_copy_kernel<int64,16,512,signalling>: one layer of the "
                       "single-launch burst (event-to-event)")
                      + f" ({bytes_layer} algorithmic bytes = n x T x R), median of the burst",
            "ms_per_launch": round(bytes_layer / (layer_gbs * GB) * 1e3, 4) if layer_gbs else None,
        }),
        "roofline_step": {
            "bound": "host_link", "achieved": round(achieved, 2), "peak": round(peak_mix, 2),
            "unit": "GB/s", "frac": round(achieved / peak_mix, 4),
            "peak_source": "in-run D2H/H2D peaks weighted by the step's bytes per direction",
        },
        "gpu_launches": int(launches),
        "clocks": clk,
        "e2e": e2e,
        "consumer_overlap": consumer,
        "duplex": duplex,
        "wall_s_timed": round(wall, 3),
    }
    if args.burst == "single_launch" and args.path != "staged" and L > 1:
        mr = statistics.mean(t_rest)
        rest_bytes = bytes_layer * (L - 1)
        rest_gbs = rest_bytes / (mr * 1e-3) / GB
        res["roofline_burst"] = {
            "bound": "host_link", "achieved": round(rest_gbs, 2), "peak": round(link["h2d"], 2),
            "unit": "GB/s", "frac": round(rest_gbs / link["h2d"], 4),
            "traffic": traffic_per_launch(traffic_key, "load_burst_signalling", rest_bytes),
            "kernel": ("row_copy_kernel<int64,512,signalling>: the launch covering layers "
                       f"1..{L - 1} of the burst"
                       if bytes_layer >= SPLIT_FIRST_LAYER_BYTES else
                       "row_copy_kernel<int64,512,signalling>: layers "
                       f"1..{L - 1} of the one-launch burst, layer 0's event to the last")
                      + f" ({rest_bytes} algorithmic bytes = n x (L-1) x T x R)",
            "peak_source": "pinned cudaMemcpyAsync H2D measured in this run (of measured)",
            "hbm_frac_of_measured": round(rest_gbs / hbm_peak(), 4),
            "ms_per_launch": round(mr, 4),
        }
        dominant = "roofline_burst" if mr > mb else "roofline_backup"
    elif staged and ml > mb:
        dominant = "roofline_load"  # the staged load-back takes most of the step
    else:
        dominant = "roofline_backup"
    res["roofline"] = dict(res[dominant], which=dominant)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    return res


def measure_host_costs(hk, pools, d, h, dt_h, ht_h, d2t_h, L, opts, stream, n, reps=7):
    """Host time of run planning and of whole calls with pinned host-located indices.

    With host-located indices every call validates the pairs on the CPU (range,
    distinct destinations, whole pages where needed) before it enqueues
    anything.  Each call is issued on an idle stream, so the time is the call's
    own host work, not a wait for a full launch queue; medians of `reps`.
    """
    import ctypes
    import dataclasses

    import torch
    P = pools[0].page_size
    dd = np.ascontiguousarray(d, dtype=np.int64)
    hh = np.ascontiguousarray(h, dtype=np.int64)
    count = ctypes.c_int64(0)
    plan = []
    for _ in range(reps):  # the C planner alone: it walks every pair
        t0 = time.perf_counter()
        st = hk.lib().hicache_plan_runs(dd.ctypes.data, hh.ctypes.data, 64, dd.size, P, None, 0,
                                        ctypes.byref(count), None)
        plan.append(time.perf_counter() - t0)
        assert st == hk.HICACHE_OK
    idx_staging = torch.empty(hk.index_staging_bytes(n, 64), dtype=torch.uint8, device="cuda")
    o = dataclasses.replace(opts, index_location=hk.HICACHE_INDEX_HOST, index_staging=idx_staging)
    events = [torch.cuda.Event() for _ in range(L)]
    t_b, t_l = [], []
    for _ in range(reps):
        stream.synchronize()
        t0 = time.perf_counter()
        hk.hicache_backup_all_layers(pools, dt_h, ht_h, opts=o, stream=stream)
        t_b.append(time.perf_counter() - t0)
        stream.synchronize()
        t0 = time.perf_counter()
        hk.hicache_load_burst(pools, 0, L, ht_h, d2t_h, opts=o, stream=stream, layer_done=events)
        t_l.append(time.perf_counter() - t0)
    stream.synchronize()
    return {"pairs": int(n),
            "plan_runs_us": round(statistics.median(plan) * 1e6, 1),
            "runs": int(count.value),
            "backup_call_us_host_indices": round(statistics.median(t_b) * 1e6, 1),
            "burst_call_us_host_indices": round(statistics.median(t_l) * 1e6, 1),
            "note": "host wall time on an idle stream: the run planner over the op's pairs, "
                    "and whole calls with pinned host indices (CPU validation, index copy to "
                    "opts.index_staging, enqueue)"}


def run_consumer_overlap(hk, pools, idx_l, opts, L, stream, bytes_layer, reps=5):
    """Each layer's event gates a consumer kernel on another stream that reads that layer.

    The consumer is the library's checksum kernel over the loaded rows of the
    layer (every tensor of the first pool).  Reported: how long after its
    layer's event each consumer finishes, and how much of the consumers' work is
    hidden behind the burst (1.0 = all of it, 0.0 = none, as when every layer
    lands before the forward starts).
    """
    import torch
    cons = torch.cuda.Stream()
    sums = torch.zeros(L, dtype=torch.int64, device="cuda")
    pool0 = pools[0]
    dev_idx = idx_l[1] if idx_l[1].is_cuda else idx_l[1].cuda()
    hk.hicache_layer_checksum(pool0, 0, 0, dev_idx, sums[0:1], stream=cons)  # load the module
    torch.cuda.synchronize()
    lag, hidden, burst_ms, alone_ms, early = [], [], [], [], []
    for _ in range(reps):
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(L)]
        done = [torch.cuda.Event(enable_timing=True) for _ in range(L)]
        t0 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        cons.wait_stream(stream)
        hk.hicache_load_burst(pools, 0, L, idx_l[0], idx_l[1], opts=opts, stream=stream,
                              layer_done=evs)
        for l in range(L):
            cons.wait_event(evs[l])
            for t in range(pool0.num_tensors):
                hk.hicache_layer_checksum(pool0, t, l, dev_idx, sums[l:l + 1], stream=cons)
            done[l].record(cons)
        torch.cuda.synchronize()
        lag.append(statistics.mean(evs[l].elapsed_time(done[l]) for l in range(L)) * 1e3)
        # consumers that finished while the burst was still loading later layers
        early.append(sum(1 for l in range(L - 1) if done[l].elapsed_time(evs[-1]) > 0))
        burst = t0.elapsed_time(evs[-1])
        total = t0.elapsed_time(done[-1])
        # the consumers alone, back to back on loaded data
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(cons)
        for l in range(L):
            for t in range(pool0.num_tensors):
                hk.hicache_layer_checksum(pool0, t, l, dev_idx, sums[l:l + 1], stream=cons)
        a1.record(cons)
        torch.cuda.synchronize()
        alone = a0.elapsed_time(a1)
        burst_ms.append(burst)
        alone_ms.append(alone)
        hidden.append(max(0.0, min(1.0, (burst + alone - total) / alone)) if alone > 0 else None)
    return {"consumer": "checksum kernel over each loaded layer, gated by that layer's event",
            "mean_lag_after_event_us": round(statistics.median(lag), 1),
            "burst_ms": round(statistics.median(burst_ms), 4),
            "consumers_alone_ms": round(statistics.median(alone_ms), 4),
            "fraction_of_consumer_work_hidden": round(statistics.median(hidden), 4),
            "consumers_done_before_last_layer_event": int(statistics.median(early)),
            "layers": L,
            "reps": reps}


def run_e2e(hk, pools, wl, dt_h, ht_h, d2t_h, L, staging, path, args, step_bytes, n, words):
    """Public-API steps with pinned host indices (host validation included) and a D2H status read.

    Every step validates its host indices on the CPU, copies them to the device
    (opts.index_staging), runs the backup and the burst, and copies the device
    error word back to pinned host memory, where the host checks it.  Two loops
    are timed: a synchronous one (each step waits for its own status before the
    next is issued) and a pipelined one with one step in flight, as a serving
    loop would run it (step k+1 is validated and enqueued while step k moves
    data; step k's status is checked once its event has completed).
    """
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    err_h = [torch.zeros(1, dtype=torch.int32).pin_memory() for _ in range(2)]
    idx_staging = torch.empty(hk.index_staging_bytes(n, 64), dtype=torch.uint8, device="cuda")
    opts = hk.Opts(path=path, index_location=hk.HICACHE_INDEX_HOST, staging=staging,
                   max_ctas=args.max_ctas, device_error=err, burst_words=words,
                   index_staging=idx_staging)
    events = [torch.cuda.Event() for _ in range(L)]
    done = [torch.cuda.Event() for _ in range(2)]
    stream = torch.cuda.Stream()

    def issue(k):
        hk.hicache_backup_all_layers(pools, dt_h, ht_h, opts=opts, stream=stream)
        hk.hicache_load_burst(pools, 0, L, ht_h, d2t_h, opts=opts, stream=stream,
                              layer_done=events)
        with torch.cuda.stream(stream):
            err_h[k % 2].copy_(err, non_blocking=True)
        done[k % 2].record(stream)

    def check(k):
        done[k % 2].synchronize()
        if int(err_h[k % 2].item()) != 0:
            raise RuntimeError("device error in e2e step")

    def timed(K, depth):
        t0 = time.perf_counter()
        for k in range(K):
            issue(k)
            if k >= depth:
                check(k - depth)
        for k in range(max(0, K - depth), K):
            check(k)
        return (time.perf_counter() - t0) / K

    for depth in (0, 1):
        timed(2, depth)  # warm-up
    K = max(3, args.steps // 2)
    dt_sync = timed(K, 0)
    dt_pipe = timed(K, 1)
    idx_bytes = 3 * n * 8
    bytes_backup, bytes_layer = payload_bytes(wl, n)
    return {"value": round(step_bytes / dt_pipe / GB, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(bytes_layer * L + idx_bytes),
            "d2h_bytes_per_step": int(bytes_backup + 4),
            "sync_value": round(step_bytes / dt_sync / GB, 2),
            "steps": K,
            "note": "host wall clock per step over K steps; every step validates its pinned "
                    "host indices on the CPU, the library copies them into opts.index_staging, "
                    "and the step's device error word is read back to pinned host memory and "
                    "checked; value: one step in flight (the next step is validated and "
                    "enqueued while the current one moves data), sync_value: each step waits "
                    "for its own status first; payload crosses the host link by definition "
                    "of the op"}


# ---------------------------------------------------------------- CPU oracle

def oracle_step_sample(wl, d, h, d2, pages, dev_imgs, host_imgs):
    """One oracle pass over the first `pages` pages of the step: backup then load burst."""
    import oracle
    P = wl.pools[0].page_size
    m = pages * P
    nbytes = 0
    for s, dimg, himg in zip(wl.pools, dev_imgs, host_imgs):
        for t in range(s.num_tensors):
            oracle.backup_all_layers(dimg[t], himg[t], d[:m], h[:m], page_size=P,
                                     row_bytes=s.row_bytes)
            oracle.load_burst(dimg[t], himg[t], 0, s.num_layers, h[:m], d2[:m], page_size=P,
                              row_bytes=s.row_bytes)
            nbytes += 2 * m * s.num_layers * s.row_bytes
    return nbytes


def oracle_images(wl, device_slots=None, host_pages=None):
    """Host-memory images of the pools for the oracle, optionally resized."""
    dev, host = [], []
    for s in wl.pools:
        slots = device_slots or s.device_slots
        pages = host_pages or s.host_pages
        dev.append([[np.zeros(slots * s.row_bytes, dtype=np.uint8)
                     for _ in range(s.num_layers)] for _ in range(s.num_tensors)])
        host.append([np.zeros(pages * s.num_layers * s.page_size * s.row_bytes, dtype=np.uint8)
                     for _ in range(s.num_tensors)])
    return dev, host


def compact_sample(wl, rank, nworkers, pages_per_pass):
    """A worker's slice of the workload's pages, renumbered into compact pool images.

    The slice keeps whole pages and a seeded random page order, but the device
    and host images hold only the pages it names (2k device pages: sources and
    load destinations; k host pages), so parallel workers do not need the full
    pools in memory.  The oracle's loops and bytes per row are unchanged.
    """
    from hierarchical_kv_cache_gb300 import workloads as W
    P = wl.pools[0].page_size
    lo = (wl.move_pages * rank) // nworkers
    k = max(1, min(pages_per_pass, (wl.move_pages * (rank + 1)) // nworkers - lo))
    g = W.rng(wl.seed * 1000 + rank)
    dev_pages = g.permutation(2 * k)
    host_pages = g.permutation(k)
    d = W.expand_pages(dev_pages[:k], P)
    d2 = W.expand_pages(dev_pages[k:], P)
    h = W.expand_pages(host_pages, P)
    return d, h, d2, 2 * k * P, k


def _oracle_worker(args):
    """One process: the oracle on its own compact slice of the workload for `seconds`."""
    name, rank, nworkers, seconds, pages_per_pass = args
    sys.path.insert(0, REPO)
    wl, _, _, _ = build_workload(name)
    d, h, d2, slots, hpages = compact_sample(wl, rank, nworkers, pages_per_pass)
    k = hpages
    dev_imgs, host_imgs = oracle_images(wl, slots, hpages)
    oracle_step_sample(wl, d, h, d2, k, dev_imgs, host_imgs)  # first touch
    total, t0, reps = 0, time.perf_counter(), 0
    while time.perf_counter() - t0 < seconds:
        total += oracle_step_sample(wl, d, h, d2, k, dev_imgs, host_imgs)
        reps += 1
    return total, time.perf_counter() - t0, reps, k


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl_name, seconds, workers=None, pages_per_pass=32):
    """The oracle, unchanged, on one core and on every core of this host.

    Each worker process runs the plain C loops on its own slice of the pages;
    the processes are spawned (the parent has used the GPU already).
    """
    import multiprocessing as mproc
    workers = workers or host_cores()
    one = _oracle_worker((wl_name, 0, 1, seconds / 2, pages_per_pass))
    ctx = mproc.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(workers) as pool:
        res = pool.map(_oracle_worker, [(wl_name, r, workers, seconds, pages_per_pass)
                                        for r in range(workers)])
    wall = time.perf_counter() - t0
    total = sum(r[0] for r in res)
    span = max(r[1] for r in res)
    return {"value": round(total / span / GB, 3), "unit": UNIT, "cores": workers,
            "kind": "oracle",
            "single_core_value": round(one[0] / one[1] / GB, 3),
            "sample": f"{workers} processes, each running the oracle unchanged on its own "
                      f"{res[0][3]}-page slice of the workload (backup + load of all layers, "
                      f"compact pool images) for {seconds:.0f} s "
                      f"({sum(r[2] for r in res)} passes in all, {wall:.1f} s wall); one core "
                      f"alone: {one[2]} passes of {one[3]} pages in {one[1]:.1f} s"}


def _reference_worker(args):
    """One process of the reference arm: warm-up passes, then timed passes of the oracle."""
    name, rank, nworkers, steps, warmup, pages_per_pass = args
    sys.path.insert(0, REPO)
    wl, _, _, _ = build_workload(name)
    d, h, d2, slots, k = compact_sample(wl, rank, nworkers, pages_per_pass)
    dev_imgs, host_imgs = oracle_images(wl, slots, k)
    for _ in range(max(1, warmup)):
        oracle_step_sample(wl, d, h, d2, k, dev_imgs, host_imgs)
    total, t0 = 0, time.perf_counter()
    for _ in range(steps):
        total += oracle_step_sample(wl, d, h, d2, k, dev_imgs, host_imgs)
    return total, time.perf_counter() - t0, k


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import multiprocessing as mproc
    wl, _, _, _ = build_workload(args.workload, args=args)
    workers = host_cores()
    ctx = mproc.get_context("spawn")
    with ctx.Pool(workers) as pool:
        res = pool.map(_reference_worker, [(args.workload, r, workers, args.steps, args.warmup, 16)
                                           for r in range(workers)])
    total = sum(r[0] for r in res)
    dt = max(r[1] for r in res)
    pages = res[0][2]
    v = round(total / dt / GB, 3)
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic", "config": {"workload": wl.name, "path": "cpu oracle"},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": workers, "kind": "oracle",
                         "sample": f"{workers} processes, each {pages} of {wl.move_pages} pages "
                                   "per step, all layers, backup + load"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- sweep

def _time_op(fn, stream, min_ms=20.0, max_reps=200):
    """Mean device ms of fn() over enough repetitions to fill min_ms."""
    import torch
    fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    fn()
    e1.record(stream)
    e1.synchronize()
    one = max(e0.elapsed_time(e1), 1e-3)
    reps = int(max(3, min(max_reps, min_ms / one)))
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def run_sweep(args):
    """Config 5: bytes per row x page size x tokens x contiguity x direction x path."""
    import torch
    import hierarchical_kv_cache_gb300 as hk
    from hierarchical_kv_cache_gb300 import workloads as W
    from hierarchical_kv_cache_gb300._binding import Pool
    from hierarchical_kv_cache_gb300.build import build

    build()
    torch.cuda.set_device(0)
    rows = [int(x) for x in args.sweep_rows.split(",")]
    psizes = [int(x) for x in args.sweep_pages.split(",")]
    tokens = [int(x) for x in args.sweep_tokens.split(",")]
    L = args.sweep_layers
    link = measure_link_peak()
    stream = torch.cuda.Stream()
    staging = [torch.empty(args.staging_mib << 20, dtype=torch.uint8, device="cuda")
               for _ in range(2)]
    events = [torch.cuda.Event() for _ in range(L)]
    words = torch.zeros(4 * L, dtype=torch.int32, device="cuda")
    out = []
    nmax = max(tokens)
    for R in rows:
        slots = 2 * nmax
        dev = [[torch.empty(slots * R, dtype=torch.uint8, device="cuda") for _ in range(L)]]
        host = [torch.empty(slots * L * R, dtype=torch.uint8, pin_memory=True)]
        for buf in dev[0]:
            buf.random_(0, 256)
        for P in psizes:
            pool = Pool(device_layers=dev, host_tensors=host, num_layers=L, head_num=1,
                        head_dim=R // 2, dtype_size=2, page_size=P, device_slots=slots,
                        host_pages=slots // P,
                        layout=(hk.HICACHE_LAYOUT_PAGE_FIRST if args.layout == "page_first"
                                else hk.HICACHE_LAYOUT_PAGE_FIRST_DIRECT))
            for n in tokens:
                for frag in (False, True):
                    d, h = W.token_pairs(1000 + n + P, n, slots, slots, P, fragmented=frag)
                    runs, full = hk.hicache_plan_runs(d, h, P)
                    dt = torch.as_tensor(d).cuda()
                    htd = torch.as_tensor(h).cuda()
                    dth = torch.as_tensor(d).pin_memory()
                    hth = torch.as_tensor(h).pin_memory()
                    nbytes = n * L * R
                    for path in ("zero_copy", "staged"):
                        whole = (n % P == 0 and full == n // P) or P == 1
                        spans = len(runs) if frag else 1
                        if path == "staged" and (not whole or spans > 8192):
                            continue
                        if path == "zero_copy":
                            o = hk.Opts(path=hk.HICACHE_PATH_ZERO_COPY,
                                        index_location=hk.HICACHE_INDEX_DEVICE,
                                        burst_words=words if args.burst == "single_launch"
                                        else None)
                            ib, il = (dt, htd), (htd, dt)
                        else:
                            o = hk.Opts(path=hk.HICACHE_PATH_STAGED,
                                        index_location=hk.HICACHE_INDEX_HOST, staging=staging)
                            ib, il = (dth, hth), (hth, dth)
                        t_b = _time_op(lambda: hk.hicache_backup_all_layers(
                            pool, ib[0], ib[1], opts=o, stream=stream), stream)
                        t_l = _time_op(lambda: hk.hicache_load_burst(
                            pool, 0, L, il[0], il[1], opts=o, stream=stream,
                            layer_done=events), stream)
                        for direction, t, peak in (("d2h_backup", t_b, link["d2h"]),
                                                   ("h2d_burst", t_l, link["h2d"])):
                            gbs = nbytes / (t * 1e-3) / GB
                            rec = {"row_bytes": R, "page_size": P, "tokens": n,
                                   "fragmented": frag, "runs": int(len(runs)),
                                   "direction": direction, "path": path, "layers": L,
                                   "layout": args.layout or "page_first_direct",
                                   "burst": args.burst if path == "zero_copy" else "per_layer",
                                   "ms": round(t, 4), "gbs": round(gbs, 2),
                                   "frac_of_link": round(gbs / peak, 4)}
                            out.append(rec)
                            print(json.dumps(rec), flush=True)
        del dev, host
        torch.cuda.synchronize()
    if args.out:
        with open(args.out, "w") as f:
            for rec in out:
                f.write(json.dumps(rec) + "\n")
    print(json.dumps({"sweep_points": len(out), "link_peak_gbs": link}), flush=True)


def run_dma_sweep(args):
    """The copy engine's cost per copy, against the copy size.

    Copies of one size between random 4 MiB pages of a pinned host buffer and
    HBM, issued on 1 or 4 streams behind a sleep kernel, so that the timed
    region holds the copies only and not the host's enqueue.  This is what
    bounds the staged path: it issues one copy per host-page run (and layer
    group), and on GB300 a copy costs a few microseconds whatever its size.
    """
    import numpy as np
    import torch
    torch.cuda.set_device(0)
    page, pages = 4 << 20, 1024
    host = torch.empty(pages * page, dtype=torch.uint8, pin_memory=True)  # 4 GiB
    host.fill_(1)
    dev = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    pick = np.random.default_rng(1).permutation(pages)[:256]
    streams = [torch.cuda.Stream() for _ in range(4)]
    main_s = torch.cuda.Stream()
    out = []
    for direction in ("h2d", "d2h"):
        for block in (128 << 10, 256 << 10, 512 << 10, 1 << 20, 2 << 20, 4 << 20):
            ncopy = min(256, (64 << 20) // block)
            for nstreams in (1, 4):
                times, enq = [], []
                for rep in range(6):
                    torch.cuda.synchronize()
                    t0 = torch.cuda.Event(enable_timing=True)
                    t1 = torch.cuda.Event(enable_timing=True)
                    with torch.cuda.stream(main_s):
                        torch.cuda._sleep(100_000_000)  # ~50 ms: the copies queue up behind it
                        t0.record(main_s)
                    for st in streams[:nstreams]:
                        st.wait_stream(main_s)
                    w0 = time.perf_counter()
                    for k in range(ncopy):
                        st = streams[k % nstreams]
                        h = host[int(pick[k]) * page:int(pick[k]) * page + block]
                        d = dev[k * block:(k + 1) * block]
                        with torch.cuda.stream(st):
                            if direction == "h2d":
                                d.copy_(h, non_blocking=True)
                            else:
                                h.copy_(d, non_blocking=True)
                    enq.append(time.perf_counter() - w0)
                    for st in streams[:nstreams]:
                        main_s.wait_stream(st)
                    t1.record(main_s)
                    t1.synchronize()
                    if rep:
                        times.append(t0.elapsed_time(t1))
                ms = statistics.median(times)
                rec = {"direction": direction, "copy_bytes": block, "copies": ncopy,
                       "streams": nstreams, "ms": round(ms, 4),
                       "us_per_copy": round(ms * 1e3 / ncopy, 2),
                       "gbs": round(ncopy * block / (ms * 1e-3) / GB, 2),
                       "enqueue_hidden": max(enq) < 0.04}
                out.append(rec)
                print(json.dumps(rec), flush=True)
    if args.out:
        with open(args.out, "w") as f:
            for rec in out:
                f.write(json.dumps(rec) + "\n")


def run_latency(args, reps=30):
    """Latency of one op for small page counts.

    device: the op is enqueued behind a sleep kernel of about 0.2 ms on its
    stream, so that the timing events around it hold its GPU work only, not the
    host's enqueue (median of `reps`).  call-to-done: wall time from the call on
    an idle stream to the end of a synchronize, what a caller waiting for the
    op sees.  host enqueue: the Python call's host time; library host: the same
    call through the C ABI with its arguments built beforehand.  Ops: the all-layer
    backup, one layer's load, and the whole load-back burst (single-launch, one
    event per layer), with device-located indices, on the first k pages of the
    workload's lists.
    """
    import ctypes

    import torch
    import hierarchical_kv_cache_gb300 as hk
    from hierarchical_kv_cache_gb300 import _binding as B
    from hierarchical_kv_cache_gb300 import pools as hpools
    from hierarchical_kv_cache_gb300.build import build

    build()
    torch.cuda.set_device(0)
    wl, d, h, d2 = build_workload(args.workload, args=args)
    L = wl.pools[0].num_layers
    P = wl.pools[0].page_size
    pools = []
    for i, sh in enumerate(wl.pools):
        p = hpools.allocate_pool(sh)
        hpools.fill_device_random_(p, wl.seed + i, sh.value_kind)
        pools.append(p)
    stream = torch.cuda.Stream()
    words = torch.zeros(4 * L, dtype=torch.int32, device="cuda")
    opts = hk.Opts(path=hk.HICACHE_PATH_ZERO_COPY, index_location=hk.HICACHE_INDEX_DEVICE,
                   burst_words=words, max_ctas=args.max_ctas)
    evs = [torch.cuda.Event() for _ in range(L)]
    out = []
    for k in [int(x) for x in args.latency_pages.split(",")]:
        m = min(k, wl.move_pages) * P
        dt = torch.as_tensor(d[:m]).cuda()
        ht = torch.as_tensor(h[:m]).cuda()
        d2t = torch.as_tensor(d2[:m]).cuda()
        bytes_backup, bytes_layer = payload_bytes(wl, m)
        ops = {"backup_all_layers": (bytes_backup, lambda: hk.hicache_backup_all_layers(
                   pools, dt, ht, opts=opts, stream=stream)),
               "load_one_layer": (bytes_layer, lambda: hk.hicache_load_layer(
                   pools, 0, ht, d2t, opts=opts, stream=stream, layer_done=evs[0])),
               "load_burst": (bytes_layer * L, lambda: hk.hicache_load_burst(
                   pools, 0, L, ht, d2t, opts=opts, stream=stream, layer_done=evs))}
        # the same calls through the C ABI with every argument built beforehand:
        # the library's own host time, without the Python binding's marshalling
        lib = hk.lib()
        arr, npools, _keep = B._pools_arg(pools)  # _keep: pointer arrays arr points into
        co = B._opts_arg(opts, dt, ht)
        sh = stream.cuda_stream
        ev_h = (ctypes.c_void_p * L)(*[B._event_handle(e, sh) for e in evs])
        raw = {"backup_all_layers": lambda: lib.hicache_backup_all_layers(
                   arr, npools, dt.data_ptr(), ht.data_ptr(), 64, m, ctypes.byref(co), sh),
               "load_one_layer": lambda: lib.hicache_load_layer(
                   arr, npools, 0, ht.data_ptr(), d2t.data_ptr(), 64, m, ctypes.byref(co), sh,
                   ev_h[0]),
               "load_burst": lambda: lib.hicache_load_burst(
                   arr, npools, 0, L, ht.data_ptr(), d2t.data_ptr(), 64, m, ctypes.byref(co), sh,
                   ev_h)}
        for name, (nbytes, fn) in ops.items():
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            dev_us, wall_us, enq_us, lib_us = [], [], [], []
            for _ in range(reps):
                stream.synchronize()
                w0 = time.perf_counter()
                assert raw[name]() == hk.HICACHE_OK
                lib_us.append((time.perf_counter() - w0) * 1e6)
                t0 = torch.cuda.Event(enable_timing=True)
                t1 = torch.cuda.Event(enable_timing=True)
                stream.synchronize()
                with torch.cuda.stream(stream):
                    torch.cuda._sleep(400_000)  # the op queues up behind it
                t0.record(stream)
                fn()
                t1.record(stream)
                t1.synchronize()
                dev_us.append(t0.elapsed_time(t1) * 1e3)
                stream.synchronize()
                w0 = time.perf_counter()
                fn()
                w1 = time.perf_counter()
                stream.synchronize()
                wall_us.append((time.perf_counter() - w0) * 1e6)
                enq_us.append((w1 - w0) * 1e6)
            med = statistics.median(dev_us)
            rec = {"workload": args.workload, "pages": m // P, "op": name, "bytes": int(nbytes),
                   "device_us_p50": round(med, 2), "device_us_min": round(min(dev_us), 2),
                   "call_to_done_us_p50": round(statistics.median(wall_us), 2),
                   "host_enqueue_us_p50": round(statistics.median(enq_us), 2),
                   "library_host_us_p50": round(statistics.median(lib_us), 2),
                   "gbs": round(nbytes / (med * 1e-6) / GB, 2)}
            out.append(rec)
            print(json.dumps(rec), flush=True)
    if args.out:
        with open(args.out, "a") as f:
            for rec in out:
                f.write(json.dumps(rec) + "\n")


def run_contention(args):
    """Both paths beside compute that occupies the SMs (path choice, S5).

    A bf16 GEMM loop (cuBLAS, 8192^3 per matmul) runs on its own stream for
    the whole measurement.  For each path and copy CTA cap, the backup and the
    load-back burst of the workload are timed alone and beside the GEMM loop,
    and the GEMM throughput is timed alone and beside each transfer.  The
    staged path moves its bytes with the copy engine and holds the SMs only for
    its gather and scatter kernels; the zero-copy path holds them for the whole
    transfer.
    """
    import torch
    import hierarchical_kv_cache_gb300 as hk
    from hierarchical_kv_cache_gb300 import pools as hpools
    from hierarchical_kv_cache_gb300.build import build

    build()
    torch.cuda.set_device(0)
    wl, d, h, d2 = build_workload(args.workload, args=args)
    L = wl.pools[0].num_layers
    n = d.size
    pools = []
    for i, sh in enumerate(wl.pools):
        p = hpools.allocate_pool(sh)
        hpools.fill_device_random_(p, wl.seed + i, sh.value_kind)
        pools.append(p)
    staging = [torch.empty(args.staging_mib << 20, dtype=torch.uint8, device="cuda")
               for _ in range(2)]
    idx_staging = torch.empty(hk.index_staging_bytes(n, 64), dtype=torch.uint8, device="cuda")
    dt_h = torch.as_tensor(d).pin_memory()
    ht_h = torch.as_tensor(h).pin_memory()
    d2t_h = torch.as_tensor(d2).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    words = torch.zeros(4 * L, dtype=torch.int32, device="cuda")
    bytes_backup, bytes_layer = payload_bytes(wl, n)
    bytes_load = bytes_layer * L
    link = measure_link_peak()
    xfer_s = torch.cuda.Stream()
    gemm_s = torch.cuda.Stream()
    N = 8192
    a = torch.randn(N, N, device="cuda", dtype=torch.bfloat16)
    b = torch.randn(N, N, device="cuda", dtype=torch.bfloat16)
    c = torch.empty(N, N, device="cuda", dtype=torch.bfloat16)
    flops = 2.0 * N ** 3

    def gemms(k):
        with torch.cuda.stream(gemm_s):
            for _ in range(k):
                torch.matmul(a, b, out=c)

    def timed_gemm(k):
        """k GEMMs on gemm_s with an event before the first and after each."""
        e0 = torch.cuda.Event(enable_timing=True)
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
        e0.record(gemm_s)
        with torch.cuda.stream(gemm_s):
            for e in ends:
                torch.matmul(a, b, out=c)
                e.record(gemm_s)
        return e0, ends

    gemms(3)
    torch.cuda.synchronize()
    e0, ends = timed_gemm(20)
    torch.cuda.synchronize()
    gemm_ms = e0.elapsed_time(ends[-1]) / 20
    gemm_alone = flops / (gemm_ms * 1e-3) / 1e12
    def point(fn, nbytes, peak):
        """One transfer op, alone and beside the GEMM loop."""
        fn()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(xfer_s)
        for _ in range(3):
            fn()
        t1.record(xfer_s)
        torch.cuda.synchronize()
        alone_ms = t0.elapsed_time(t1) / 3
        alone = nbytes / (alone_ms * 1e-3) / GB
        if args.contention_alone_only:
            return {"alone_gbs": round(alone, 2), "alone_frac_of_link": round(alone / peak, 4)}
        # beside the GEMM loop: enough GEMMs to outlast the transfers even if
        # they slow down fourfold
        k = int(4 * 3 * alone_ms / gemm_ms) + 8
        g0, ends = timed_gemm(k)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        xfer_s.wait_event(g0)
        t0.record(xfer_s)
        for _ in range(3):
            fn()
        t1.record(xfer_s)
        torch.cuda.synchronize()
        window = t0.elapsed_time(t1)
        busy_ms = window / 3
        # GEMM throughput during the transfers: the GEMMs that ended inside
        # the window, over the window
        done = sum(1 for e in ends if 0.0 < t0.elapsed_time(e) <= window)
        if int(err.item()) != 0:
            raise RuntimeError(f"device error word {int(err.item())}")
        beside = nbytes / (busy_ms * 1e-3) / GB
        return {"alone_gbs": round(alone, 2), "beside_gemm_gbs": round(beside, 2),
                "alone_frac_of_link": round(alone / peak, 4),
                "beside_gemm_frac_of_link": round(beside / peak, 4),
                "gemm_tflops_alone": round(gemm_alone, 1),
                "gemm_tflops_during_transfers": round(done * flops / (window * 1e-3) / 1e12, 1),
                "gemm_outlasted_transfers": bool(t0.elapsed_time(ends[-1]) > window),
                "transfers_ms": round(window, 2)}

    out = []
    evs = [torch.cuda.Event() for _ in range(L)]
    caps = [int(x) for x in args.contention_ctas.split(",")]
    for path in ("zero_copy", "staged"):
        for cap in (caps if path == "zero_copy"
                    else [int(x) for x in args.contention_staged_ctas.split(",")]):
            o = hk.Opts(path=hk.HICACHE_PATH_ZERO_COPY if path == "zero_copy"
                        else hk.HICACHE_PATH_STAGED,
                        index_location=hk.HICACHE_INDEX_HOST, staging=staging, max_ctas=cap,
                        device_error=err, burst_words=words, index_staging=idx_staging)
            ops = {"backup": (bytes_backup, link["d2h"],
                              lambda: hk.hicache_backup_all_layers(pools, dt_h, ht_h, opts=o,
                                                                   stream=xfer_s)),
                   "burst": (bytes_load, link["h2d"],
                             lambda: hk.hicache_load_burst(pools, 0, L, ht_h, d2t_h, opts=o,
                                                           stream=xfer_s, layer_done=evs))}
            for name, (nbytes, peak, fn) in ops.items():
                for rep in range(args.contention_reps):
                    rec = {"path": path, "max_ctas": cap, "op": name, "rep": rep,
                           **point(fn, nbytes, peak)}
                    out.append(rec)
                    print(json.dumps(rec), flush=True)
    if args.out:
        with open(args.out, "w") as f:
            for rec in out:
                f.write(json.dumps(rec) + "\n")
    print(json.dumps({"contention_points": len(out), "workload": wl.name,
                      "link_peak_gbs": link, "gemm_tflops_alone": round(gemm_alone, 1)}),
          flush=True)


def main():
    args = parse_args()
    if args.contention:
        run_contention(args)
        return
    if args.latency:
        run_latency(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.dma_sweep:
        run_dma_sweep(args)
        return
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        res = run_reference(args, rank, world)
    else:
        rank, world = dist_setup(args.gpus)
        res = run_ours(args, rank, world)
    if res is not None and rank == 0:
        line = json.dumps(res)
        print(line, flush=True)
        if args.out:
            with open(args.out, "a") as f:
                f.write(line + "\n")
    if args.impl != "reference" and world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Benchmark of the expert slot cache decode step on one GB300 (or N replicas).

One step = restore the prepared cache state, then ensure_experts -> copy_missing ->
expert FFN for one synthetic batch, as the cache-copy benchmark of the FreeToken
benchmark guide (section 4: prepared state where the driven layer misses, CUDA-event
timing, time_ms of ensure + copy, copy_MiB = misses * bytes per expert,
bw_GBps = copied bytes / time, tok_ms = time_ms * L). The headline line reports:
  value      copy GB/s of ensure + copy (bytes copied / summed event time);
  roofline   the copy kernel against the host-to-device link peak measured in this
             run (max of a 1 GiB pinned->device cudaMemcpyAsync and an SM zero-copy
             read of 1 GiB);
  roofline_ffn  the FFN kernels against the measured HBM copy bandwidth;
  e2e        the same metric with the step's inputs copied from pinned host memory
             and the output read back inside the timed region;
  cpu_baseline  the CPU oracle timed on a bounded sample of the same workload.
``--impl reference`` times the CPU oracle itself on the same workload (host cores).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_CFG = "c3"   # the largest single-GPU workload: nvfp4 layer, E 256, H 7168, I 2048
DEFAULT_BS = 32
DEFAULT_MR = 1.0
# the other workloads measured in the same run (the `configs` block); the tiny bf16 layer
# is a parity case only (GPU tests and smoke()), the decode trace has its own summary
DEFAULT_OTHERS = "c2,c4,c6,c7,c5"
METRIC = "per-layer expert copy GB/s & tok_ms vs bs/miss_rate; expert FFN us/layer"
LINK_PROBE_BYTES = 1 << 30


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ftmoe", choices=["ftmoe", "reference"])
    ap.add_argument("--config", default=DEFAULT_CFG)
    ap.add_argument("--bs", type=int, default=DEFAULT_BS)
    ap.add_argument("--miss-rate", type=float, default=DEFAULT_MR)
    ap.add_argument("--repeat", type=int, default=25, help="repeats per sweep point (median)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--configs", default=DEFAULT_OTHERS,
                    help="comma list of other workloads swept in the same run ('none' to skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-hybrid", action="store_true", help="skip the hybrid-path measurements")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill-pipeline measurements")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay measurement")
    ap.add_argument("--copy-mode", default="fused", choices=["fused", "per_bank", "engine"])
    ap.add_argument("--ffn-kernels", default="auto", choices=["auto", "rows", "mma", "tc05"],
                    help="FFN kernel family of bf16 layers (auto: chosen per call)")
    ap.add_argument("--experts", type=int, default=0, help="override E (smaller profiling cases)")
    ap.add_argument("--slots", type=int, default=0, help="override S (smaller profiling cases)")
    return ap.parse_args()


# ------------------------------------------------------------------------------ dist


def dist_setup(n):
    import torch

    if n <= 1 or "RANK" not in os.environ:
        return 0, 1, None
    import torch.distributed as dist

    rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
    dist.init_process_group("nccl")
    return rank, world, dist


def aggregate(dist, total_bytes: float, seconds: float, device=None):
    """Whole-job throughput of independent replicas: bytes summed, time = max over ranks."""
    import torch

    if dist is None:
        return total_bytes, seconds
    t = torch.tensor([total_bytes, seconds], dtype=torch.float64, device=device)
    b = t[:1].clone()
    s = t[1:].clone()
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    dist.all_reduce(s, op=dist.ReduceOp.MAX)
    return float(b.item()), float(s.item())


# ------------------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while a region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int = 0):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([v.strip() for v in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            if len(r) >= 9:
                for n, v in zip(names, r[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ helpers


def install_hits(cache, r):
    """The prepared state's resident experts (slots 0..h-1) get their bytes."""
    for i, e in enumerate(sorted(int(v) for v in r.hits)):
        for b in range(cache.nb):
            cache.slots[b][i].copy_(cache.host[b][0][e])


# Kernel sources whose DRAM traffic is recorded under profiles/ (one ncu capture of the
# workload); a recorded figure is reported only while these sources are unchanged.
TRAFFIC_SOURCES = {
    "copy": ["copy.cu", "internal.cuh"],
    "ffn_rows": ["ffn_tma.cu", "ffn_common.cuh", "internal.cuh"],      # CUDA-core pipelines
    "ffn_mma": ["ffn_rows_mma.cu", "pipeline.cuh", "ffn_common.cuh", "internal.cuh"],  # tensor-core
    "ffn_mx": ["ffn_mx_tma.cu", "ffn_common.cuh", "internal.cuh"],     # mxfp4 tensor maps
    "ffn_fp8": ["ffn_rows_mma.cu", "pipeline.cuh", "ffn_common.cuh", "internal.cuh"],  # block FP8
    "ffn_tc05": ["ffn_tc05.cu", "pipeline.cuh", "ffn_common.cuh", "internal.cuh"],  # bf16 tcgen05
}


def source_hash(kind: str) -> str:
    """First 16 hex digits of the sha256 over the kernel sources of `kind`."""
    import hashlib
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "expert_slot_cache_device_gb300", "csrc")
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES[kind]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kind: str, units: int = 0):
    """DRAM bytes (read + write) per launch of `kind` on `workload` ("<name>/bs<bs>/mr<mr>")
    from the lines of profiles/traffic_*.md, or None if none matches the current sources.

    `traffic: <workload> <kind> <hash> <read> <write>` is a capture of that exact point;
    `traffic-per-unit: <name> <kind> <hash> <read> <write> <units>` is a capture of a smaller
    case of the same layer (fewer experts) whose traffic grows in proportion to the units one
    launch processes (missed experts for the copy, distinct experts for the FFN): it is scaled
    by `units` / <units>; `traffic-affine: <name> <kind> <hash> <bytes per unit> <offset>` is
    fitted to two such captures when traffic grows by a fixed amount per unit plus a constant
    (the copy kernel: its last written lines are still dirty in L2 when it ends)."""
    pdir = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles")
    if not os.path.isdir(pdir):
        return None
    cur = source_hash(kind)
    name = workload.split("/")[0]
    scaled = None
    for fn in sorted(os.listdir(pdir)):
        if not (fn.startswith("traffic_") and fn.endswith(".md")):
            continue
        with open(os.path.join(pdir, fn)) as f:
            for ln in f:
                parts = ln.split()
                if len(parts) == 6 and parts[0] == "traffic:" and parts[1] == workload and parts[2] == kind \
                        and parts[3] == cur:
                    return int(parts[4]) + int(parts[5])
                if len(parts) == 7 and parts[0] == "traffic-per-unit:" and parts[1] == name and parts[2] == kind \
                        and parts[3] == cur and units > 0:
                    scaled = int(round((int(parts[4]) + int(parts[5])) * units / int(parts[6])))
                if len(parts) == 6 and parts[0] == "traffic-affine:" and parts[1] == name and parts[2] == kind \
                        and parts[3] == cur and units > 0:
                    scaled = int(round(float(parts[4]) * units + float(parts[5])))
    return scaled


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy burst)"
    return 6800.0, "fallback 6.8 TB/s"


def link_peak(torch, F, stream):
    """Host-to-device link ceiling in this run (ftmoe_measure_link): best of 5 for a 1 GiB
    pinned->device cudaMemcpyAsync and for the SM zero-copy read kernel."""
    src = torch.empty(LINK_PROBE_BYTES, dtype=torch.uint8, pin_memory=True)
    src.fill_(7)
    dst = torch.empty(LINK_PROBE_BYTES, dtype=torch.uint8, device="cuda")
    mc, sm = F.ftmoe_measure_link(src.data_ptr(), dst.data_ptr(), LINK_PROBE_BYTES, 5, stream.cuda_stream)
    del src, dst
    return {"memcpy": mc, "sm_read": sm}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(cfg, r, host_banks_np, threads, ffn_tokens=4, reps=None, budget_s=12.0, slot_bufs=None):
    """Time the CPU oracle on a bounded sample of one step: ensure + copy of the whole
    step (the copy into a host-side slot buffer, allocated once and touched before timing),
    and the FFN for `ffn_tokens` tokens. Returns dict(copy GB/s, ensure+copy seconds per
    step, ffn seconds per token)."""
    import oracle

    schema_bytes = [b.shape[1] for b in host_banks_np]
    if slot_bufs is None:
        slot_bufs = host_slot_buffers(cfg, schema_bytes)
    t_ec = []
    t0 = time.perf_counter()
    m = 0
    while True:
        orc = oracle.Cache(cfg.E, cfg.L, cfg.S, r.owner, r.stamp, r.clock)
        a = time.perf_counter()
        rc, slots, mids, msl = orc.ensure(0, r.topk_ids)
        oracle.copy_missing(schema_bytes, host_banks_np, slot_bufs, cfg.E, mids, msl)
        t_ec.append(time.perf_counter() - a)
        m = mids.size
        if (reps is not None and len(t_ec) >= reps) or (reps is None and time.perf_counter() - t0 > budget_s / 2):
            break
    B = sum(schema_bytes)
    toks = list(range(min(ffn_tokens, r.topk_ids.shape[0])))
    pairs = [[hb.ctypes.data + int(e) * hb.shape[1] for hb in host_banks_np] for e in r.topk_ids[toks].reshape(-1)]
    a = time.perf_counter()
    oracle.expert_ffn(cfg.fmt, cfg.H, cfg.I, pairs, r.x[toks], r.weights[toks], threads=threads)
    t_ffn = (time.perf_counter() - a) / max(1, len(toks))
    ec = statistics.median(t_ec)
    return {"copy_gbps": m * B / ec / 1e9, "ensure_copy_s": ec, "ffn_s_per_token": t_ffn, "reps": len(t_ec),
            "misses": m, "ffn_tokens": len(toks)}


def host_slot_buffers(cfg, schema_bytes):
    """Host-side slot banks of the oracle's copy, pages touched up front so that the timed
    copies do not pay first-touch page faults."""
    bufs = [np.empty((cfg.S, n), np.uint8) for n in schema_bytes]
    for b in bufs:
        b.fill(0)
    return bufs


# ------------------------------------------------------------------------------ reference arm


def reference_banks(cfg, wl):
    """Host banks of layer 0 for the oracle (seeded; drawn on the GPU when there is one,
    which only generates inputs)."""
    import torch

    out = []
    for b, g in enumerate(wl.bank_schema(cfg)):
        if torch.cuda.is_available():
            t = torch.empty((cfg.E, g.bytes), dtype=torch.uint8)
            wl.fill_bank_device(cfg, b, t)
            out.append(t.numpy())
        else:
            a = np.empty((cfg.E, g.bytes), np.uint8)
            wl.fill_bank(cfg, b, a)
            out.append(a)
    return out



def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from expert_slot_cache_device_gb300 import workload as wl

    oracle.build()
    cfg = wl.CONFIGS[args.config]
    r = wl.make_route(cfg, args.bs, args.miss_rate)
    banks = reference_banks(cfg, wl)
    cores = cpu_cores()
    times = []
    bufs = host_slot_buffers(cfg, [b.shape[1] for b in banks])
    for i in range(args.warmup + args.steps):
        res = oracle_sample(cfg, r, banks, cores, ffn_tokens=1, reps=1, slot_bufs=bufs)
        if i >= args.warmup:
            times.append(res)
    ec = sum(t["ensure_copy_s"] for t in times)
    B = cfg.bytes_per_expert
    value = r.misses * B * len(times) / ec / 1e9
    ffn_s = statistics.median(t["ffn_s_per_token"] for t in times) * args.bs
    step_s = ec / len(times) + ffn_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_OF[cfg.fmt], "data": "synthetic",
        "config": {"workload": f"{cfg.name} bs={args.bs} miss_rate={args.miss_rate}", "bs": args.bs,
                   "miss_rate": args.miss_rate, "misses": r.misses, "parallelism": "host cores"},
        "time_ms": ec / len(times) * 1e3, "tok_ms": ec / len(times) * 1e3 * cfg.L,
        "ffn_us": ffn_s * 1e6,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: ensure + copy of the full step ({r.misses} experts, "
                                   f"{r.misses * B / 2**20:.0f} MiB memcpy into a host slot buffer, 1 thread); "
                                   f"FFN of 1 of {args.bs} tokens on {cores} threads, scaled to {args.bs}"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------ GPU arm


def run_gpu(args):
    import torch

    rank, world, dist = dist_setup(args.gpus)
    from expert_slot_cache_device_gb300 import build as B

    if rank == 0:
        B.build()
    if dist is not None:
        dist.barrier()
    from expert_slot_cache_device_gb300 import ftmoe as F
    from expert_slot_cache_device_gb300 import workload as wl
    from expert_slot_cache_device_gb300.synthetic import release_memory, synthetic_cache

    dev = torch.cuda.current_device()
    stream = torch.cuda.Stream()
    cfg = wl.CONFIGS[args.config]
    if args.experts or args.slots:
        cfg = wl.scaled(cfg, E=args.experts or cfg.E, S=args.slots or cfg.S)
    if cfg.steps > 0:  # the multi-step decode trace has its own measurement
        line = run_trace(cfg, stream, torch, F, wl, synthetic_cache)
        line.update({"n_gpus": world, "steps": args.steps, "warmup": args.warmup})
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0
    bs, mr = args.bs, args.miss_rate
    r = wl.make_route(cfg, bs, mr)
    B = cfg.bytes_per_expert
    # every layer's host source aliases layer 0's bank (allowed by the per-layer source
    # lists) so that the prefill probe can stream any layer
    cache = synthetic_cache(cfg, max(max(cfg.bs_list), bs, PREFILL_BS) * cfg.topk, alias_all=True, stream=stream)
    cache.set_copy_mode({"fused": F.COPY_FUSED, "per_bank": F.COPY_PER_BANK, "engine": F.COPY_ENGINE}[args.copy_mode])
    if args.ffn_kernels != "auto":
        cache.set_ffn_kernels({"rows": F.FFN_ROWS, "mma": F.FFN_MMA, "tc05": F.FFN_TC05}[args.ffn_kernels])
    ffn_kind = ffn_family(F, cache, cfg, bs)
    s = stream.cuda_stream
    d_ids = torch.from_numpy(r.topk_ids).cuda()
    d_slots = torch.empty_like(d_ids)
    d_w = torch.from_numpy(r.weights).cuda()
    d_x = torch.from_numpy(r.x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    d_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
    install_hits(cache, r)
    torch.cuda.synchronize()

    def step(ev):
        cache.set_state(r.owner, r.stamp, r.clock, stream=s)
        ev[0].record(stream)
        F.ftmoe_ensure_experts(cache.handle, 0, d_ids.data_ptr(), bs, cfg.topk, d_slots.data_ptr(), s)
        ev[1].record(stream)
        F.ftmoe_copy_missing(cache.handle, s)
        ev[2].record(stream)
        F.ftmoe_expert_ffn(cache.handle, d_x.data_ptr(), bs, d_slots.data_ptr(), d_w.data_ptr(), cfg.topk,
                           d_y.data_ptr(), s)
        ev[3].record(stream)

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for _ in range(args.warmup):
        step(mk())
    torch.cuda.synchronize()
    assert cache.status() == F.OK
    evs = [mk() for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev)
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    total_s = start.elapsed_time(end) / 1e3
    ens = [e[0].elapsed_time(e[1]) / 1e3 for e in evs]
    cpy = [e[1].elapsed_time(e[2]) / 1e3 for e in evs]
    ffn = [e[2].elapsed_time(e[3]) / 1e3 for e in evs]
    ec_sum = sum(a + b for a, b in zip(ens, cpy))
    bytes_total = r.misses * B * args.steps
    agg_bytes, agg_ec = aggregate(dist, bytes_total, ec_sum, device="cuda")
    _, agg_total = aggregate(dist, 0.0, total_s, device="cuda")
    value = agg_bytes / agg_ec / 1e9 if agg_ec > 0 else 0.0
    assert cache.status() == F.OK

    # end to end through the C-ABI with host buffers: inputs H2D, output D2H each step
    h_ids = torch.from_numpy(r.topk_ids).pin_memory()
    h_w = torch.from_numpy(r.weights).pin_memory()
    h_x = torch.from_numpy(r.x.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    h_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16).pin_memory()
    h2d = h_ids.numel() * 4 + h_w.numel() * 4 + h_x.numel() * 2
    d2h = h_y.numel() * 2
    e_ev = []
    for i in range(args.warmup + args.steps):
        cache.set_state(r.owner, r.stamp, r.clock, stream=s)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            d_ids.copy_(h_ids, non_blocking=True)
            d_w.copy_(h_w, non_blocking=True)
            d_x.copy_(h_x, non_blocking=True)
        F.ftmoe_ensure_experts(cache.handle, 0, d_ids.data_ptr(), bs, cfg.topk, d_slots.data_ptr(), s)
        F.ftmoe_copy_missing(cache.handle, s)
        F.ftmoe_expert_ffn(cache.handle, d_x.data_ptr(), bs, d_slots.data_ptr(), d_w.data_ptr(), cfg.topk,
                           d_y.data_ptr(), s)
        with torch.cuda.stream(stream):
            h_y.copy_(d_y, non_blocking=True)
        b.record(stream)
        if i >= args.warmup:
            e_ev.append((a, b))
    torch.cuda.synchronize()
    e2e_s = sum(a.elapsed_time(b) for a, b in e_ev) / 1e3
    agg_b2, agg_e2e = aggregate(dist, bytes_total, e2e_s, device="cuda")
    e2e_value = agg_b2 / agg_e2e / 1e9 if agg_e2e > 0 else 0.0

    line = None
    if rank == 0:
        hbm_peak, hbm_src = measured_peaks()
        links = link_peak(torch, F, stream)
        link = max(links.values())
        copy_s = statistics.median(cpy)
        ens_s = statistics.median(ens)
        ffn_s = statistics.median(ffn)
        time_ms = statistics.median([a + b for a, b in zip(ens, cpy)]) * 1e3
        copy_ach = r.misses * B / copy_s / 1e9 if r.misses else 0.0
        w_bytes = r.active * (cfg.bytes_per_expert) + 2 * bs * cfg.H * 2
        ffn_ach = w_bytes / ffn_s / 1e9
        launches_per_step = 2 + 1 + (1 if args.copy_mode == "fused" else (cache.nb if args.copy_mode == "per_bank" else 0)) \
            + ffn_launches(cfg, ffn_kind)
        workload = f"{cfg.name} bs={bs} miss_rate={mr}"
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": agg_total / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_OF[cfg.fmt], "data": "synthetic",
            "config": {"workload": workload, "format": cfg.fmt, "E": cfg.E, "topk": cfg.topk, "H": cfg.H,
                       "I": cfg.I, "L": cfg.L, "S": cfg.S, "bs": bs, "miss_rate": mr, "active": r.active,
                       "misses": r.misses, "copy_MiB": r.misses * B / 2 ** 20, "copy_mode": args.copy_mode,
                       "ffn_kernels": f"{args.ffn_kernels}: {FAMILY_NAMES[ffn_kind]}",
                       "l2": f"inputs larger than L2: {r.misses * B / 2**20:.0f} MiB copied and "
                             f"{r.active * B / 2**20:.0f} MiB of expert weights read per step",
                       "parallelism": f"replicas x{world}",
                       "step": "set_state (prepared state, 2 small kernels) + ensure + copy + FFN"},
            "time_ms": time_ms, "ensure_us": ens_s * 1e6, "copy_ms": copy_s * 1e3,
            "bw_GBps": r.misses * B / (time_ms / 1e3) / 1e9 if time_ms > 0 else 0.0,
            "tok_ms": time_ms * cfg.L, "ffn_us": ffn_s * 1e6,
            "roofline": {"bound": "host_link", "kernel": "copy_missing_kernel", "achieved": copy_ach, "peak": link,
                         "unit": "GB/s", "frac": copy_ach / link if link else None,
                         "traffic": recorded_traffic(f"{cfg.name}/bs{bs}/mr{mr}", "copy", units=r.misses),
                         "peak_source": f"measured in this run: max(1 GiB pinned->device cudaMemcpyAsync "
                                        f"{links['memcpy']:.1f}, SM zero-copy read {links['sm_read']:.1f}) GB/s"},
            "roofline_ffn": {"bound": "hbm", "kernel": "expert FFN (all kernels of one call)",
                             "achieved": ffn_ach, "peak": hbm_peak, "unit": "GB/s", "frac": ffn_ach / hbm_peak,
                             "traffic": recorded_traffic(f"{cfg.name}/bs{bs}/mr{mr}", ffn_kind, units=r.active),
                             "peak_source": hbm_src},
            "link_peak_GBps": links,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
        }
        configs = {}
        if not args.no_sweep:
            configs[cfg.name] = {"key": cfg.key, "format": cfg.fmt,
                                 "points": sweep(args, cfg, cache, stream, torch, F, wl, link, hbm_peak)}
        if not args.no_hybrid:
            line["hybrid"] = hybrid_probe(args, cfg, cache, stream, torch, F, wl, link, cpu_cores())
        if not args.no_prefill:
            line["prefill"] = prefill_probe(cfg, cache, torch, F)
        if not args.no_graph:
            line["graph"] = graph_probe(cfg, cache, torch, F, wl)
    if rank == 0 and not args.no_cpu_baseline:
        hb = [cache.host_tensor(b, 0).numpy() for b in range(cache.nb)]
        cores = cpu_cores()
        res = oracle_sample(cfg, r, hb, cores, ffn_tokens=2)
        line["cpu_baseline"] = {"value": res["copy_gbps"], "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": f"ensure + copy of the full step ({res['misses']} experts into a host slot "
                                          f"buffer, 1 thread, median of {res['reps']}); FFN of "
                                          f"{res['ffn_tokens']} of {bs} tokens on {cores} threads: "
                                          f"{res['ffn_s_per_token'] * 1e3:.1f} ms/token",
                                "ffn_us_per_layer_est": res["ffn_s_per_token"] * bs * 1e6}
        del hb
    cache.close(release=True)
    del cache, d_ids, d_slots, d_w, d_x, d_y, h_ids, h_w, h_x, h_y
    release_memory()
    if rank == 0:
        # every other workload of the metric, one after another (each one's banks freed before
        # the next is built): all (bs, miss_rate) points, or the decode trace's summary
        others = [] if args.configs in ("", "none") else [k for k in args.configs.split(",") if k != args.config]
        for key in others:
            ocfg = wl.CONFIGS[key]
            t0 = time.perf_counter()
            if ocfg.steps > 0:
                tr = run_trace(ocfg, stream, torch, F, wl, synthetic_cache)
                entry = {"key": key, "format": ocfg.fmt, "trace": tr["trace"], "trace_value_GBps": tr["value"],
                         "copy_frac_of_link": tr["value"] / link, "clocks": tr["clocks"]}
            else:
                entry = {"key": key, "format": ocfg.fmt,
                         "points": sweep_workload(args, ocfg, stream, torch, F, wl, synthetic_cache, link, hbm_peak)}
            entry["wall_s"] = time.perf_counter() - t0
            configs[ocfg.name] = entry
            release_memory()
        tiny = wl.CONFIGS["c1"]
        configs[tiny.name] = {"key": "c1", "format": tiny.fmt,
                              "parity_only": "checked against the oracle by the GPU tests and smoke(); 384 KiB of "
                                             "weights, too small to time"}
        line["configs"] = configs
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


# weight format the FFN computes from (the copy moves bytes); every format accumulates in fp32
DTYPE_OF = {"bf16": "bf16", "nvfp4": "nvfp4", "mxfp4": "mxfp4", "fp8": "e4m3", "q4_0": "q4_0", "raw": "u8"}
FAMILY_NAMES = {"ffn_rows": "CUDA-core bulk-copy pipeline", "ffn_mma": "tensor-core pipeline (mma.sync)",
                "ffn_tc05": "tcgen05 pipeline (TMEM accumulators)",
                "ffn_mx": "mxfp4 tensor-map pipeline (mma.sync)", "ffn_fp8": "block-FP8 tensor-map pipeline (mma.sync)"}


def ffn_family(F, cache, cfg, bs):
    """Kernel family one FFN call of `bs` tokens runs (keys of TRAFFIC_SOURCES)."""
    if cfg.fmt == "mxfp4":
        return "ffn_mx"
    if cfg.fmt == "fp8":
        return "ffn_fp8"
    if cfg.fmt == "bf16":
        kind = F.ftmoe_ffn_kernels_for(cache.handle, bs, cfg.topk)
        if kind == F.FFN_TC05:
            return "ffn_tc05"
        if kind == F.FFN_MMA:
            return "ffn_mma"
    return "ffn_rows"


def ffn_launches(cfg, kind):
    """Kernels one FFN call launches: routing, gate_up, down and the weighted combine."""
    return 4


def sweep_workload(args, cfg, stream, torch, F, wl, synthetic_cache, link, hbm_peak):
    """All (bs, miss_rate) points of one workload on a cache of its own (freed afterwards)."""
    cache = synthetic_cache(cfg, max(cfg.bs_list) * cfg.topk, alias_all=True, stream=stream)
    try:
        return sweep(args, cfg, cache, stream, torch, F, wl, link, hbm_peak)
    finally:
        cache.close(release=True)
        del cache


PREFILL_BS = 64      # tokens of the prefill batch of the pipeline probe
PREFILL_LAYERS = 6   # layers streamed by the probe


def graph_probe(cfg, cache, torch, F, wl, bs=1, calls=None, reps=20):
    """Decode calls at batch `bs` with every routed expert resident (the prepared state of
    miss rate 0), one call = ensure + copy_missing + FFN of one layer: `calls` calls issued
    one by one against the same calls captured once in a CUDA graph and replayed (what a
    serving loop does per token, rewriting the id / weight / activation buffers in place).
    Median over `reps` runs of the device time per call (CUDA events, warm L2: the resident
    experts' weights, bs * topk * B bytes, may partly stay in L2 between calls)."""
    calls = calls or cfg.L
    r = wl.make_route(cfg, bs, 0.0)
    d_ids = torch.from_numpy(r.topk_ids).cuda()
    d_w = torch.from_numpy(r.weights).cuda()
    d_x = torch.from_numpy(r.x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    d_slots = torch.empty_like(d_ids)
    d_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.Stream()

    def run():
        for _ in range(calls):
            cache.ensure(0, d_ids, d_slots, stream=st)
            cache.copy_missing(stream=st)
            cache.ffn(d_x, d_slots, d_w, d_y, stream=st)

    def timed(fn):
        out = []
        for _ in range(reps):
            cache.set_state(r.owner, r.stamp, r.clock, stream=st)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            with torch.cuda.stream(st):  # a graph replays on the current stream
                fn()
            b.record(st)
            b.synchronize()
            out.append(a.elapsed_time(b) * 1e3 / calls)
        return statistics.median(out)

    def run_ensure_copy():
        for _ in range(calls):
            cache.ensure(0, d_ids, d_slots, stream=st)
            cache.copy_missing(stream=st)

    def run_ffn():
        for _ in range(calls):
            cache.ffn(d_x, d_slots, d_w, d_y, stream=st)

    def replayed(fn):
        g = torch.cuda.CUDAGraph()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=st, capture_error_mode="thread_local"):
            fn()
        t = timed(g.replay)
        del g
        return t

    cache.set_state(r.owner, r.stamp, r.clock, stream=st)
    run()
    torch.cuda.synchronize()
    eager = timed(run)
    replay = replayed(run)
    # the parts of a call on their own (graph replays): ensure + copy (nothing to copy), FFN
    ensure_copy = replayed(run_ensure_copy)
    ffn_only = replayed(run_ffn)
    assert cache.status() == F.OK
    return {"bs": bs, "calls": calls, "misses_per_call": 0, "eager_us_per_call": eager,
            "graph_us_per_call": replay, "speedup": eager / replay if replay > 0 else None,
            "graph_ensure_copy_us_per_call": ensure_copy, "graph_ffn_us_per_call": ffn_only}


def prefill_probe(cfg, cache, torch, F):
    """Whole-layer double-buffered prefill (architecture deep-dive, section 五): a batch of
    PREFILL_BS tokens through PREFILL_LAYERS layers, every expert of each layer streamed in
    (prefetch) before its FFN. Times the same calls one after another on one stream (SM
    copy kernel) and the two-stream pipeline ftmoe_prefill_layers with the copy engines and
    with the SM copy kernel, plus the prefetch and the FFN alone for reference. Wall time
    around each run, the device synchronised on both sides; the cache starts empty."""
    if cfg.S < 2 * cfg.E:
        return {"skipped": f"needs S >= 2E (S={cfg.S}, E={cfg.E})"}
    rng = np.random.default_rng(20260)
    bs, k, L = PREFILL_BS, cfg.topk, PREFILL_LAYERS
    layers = [l % cfg.L for l in range(L)]
    ids = [torch.from_numpy(np.stack([rng.permutation(cfg.E)[:k] for _ in range(bs)]).astype(np.int32)).cuda()
           for _ in range(L)]
    w = [torch.full((bs, k), 1.0 / k, dtype=torch.float32, device="cuda") for _ in range(L)]
    x = [torch.from_numpy(wl_bits(rng.standard_normal((bs, cfg.H)).astype(np.float32))).view(torch.bfloat16).cuda()
         for _ in range(L)]
    y = [torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    d_slots = torch.empty((bs, k), dtype=torch.int32, device="cuda")
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    empty_owner = np.full(cfg.S, -1, np.int32)
    empty_stamp = np.zeros(cfg.S, np.uint32)
    B = cfg.bytes_per_expert

    def reset():
        cache.set_state(empty_owner, empty_stamp, 0, stream=compute)
        torch.cuda.synchronize()

    def timed(fn, reps=3):
        best = None
        for _ in range(reps):
            reset()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        return best * 1e3

    def sequential():
        for i, l in enumerate(layers):
            cache.prefetch_layer(l, compute)
            cache.ensure(l, ids[i], d_slots, compute)
            cache.ffn(x[i], d_slots, w[i], y[i], compute)

    def prefetch_only():
        for l in layers:
            cache.prefetch_layer(l, compute)

    def ffn_only():  # every layer's experts are resident after one prefetch of the same layer
        for i, l in enumerate(layers):
            cache.ensure(l, ids[i], d_slots, compute)
            cache.ffn(x[i], d_slots, w[i], y[i], compute)

    out = {"tokens": bs, "layers": L, "bytes_per_layer": cfg.E * B}
    cache.set_copy_mode(F.COPY_FUSED)
    out["sequential_ms"] = timed(sequential)
    out["prefetch_only_ms"] = timed(prefetch_only)
    reset()
    cache.prefetch_layer(layers[0], compute)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i, l in enumerate(layers[:1] * L):
        cache.ensure(l, ids[i], d_slots, compute)
        cache.ffn(x[i], d_slots, w[i], y[i], compute)
    torch.cuda.synchronize()
    out["ffn_only_ms"] = (time.perf_counter() - t0) * 1e3
    for mode, name in ((F.COPY_ENGINE, "pipelined_engine_ms"), (F.COPY_FUSED, "pipelined_sm_copy_ms")):
        cache.set_copy_mode(mode)
        out[name] = timed(lambda: cache.prefill_layers(layers, ids, x, w, y, compute, copy))
    cache.set_copy_mode(F.COPY_FUSED)
    best = min(out["pipelined_engine_ms"], out["pipelined_sm_copy_ms"])
    out["overlap_speedup"] = out["sequential_ms"] / best
    out["link_GBps_pipelined"] = L * cfg.E * B / (best / 1e3) / 1e9
    reset()
    return out


def wl_bits(a):
    from expert_slot_cache_device_gb300 import workload as wl
    return wl.f32_to_bf16_bits(a).view(np.int16)


def run_trace(cfg, stream, torch, F, wl, make_cache):
    """The multi-step decode trace: every (step, layer) call of cfg.steps steps x cfg.L
    layers at bs 1, from a cold cache, each call ensure + copy_missing + expert FFN on one
    stream. All inputs are generated and moved to the device before the timed region.
    CUDA events around every call give the ensure+copy and FFN times; the library's
    cumulative counters give calls, distinct ids and fetched misses."""
    k, n = cfg.topk, cfg.steps * cfg.L
    ids = np.empty((n, 1, k), np.int32)
    ws = np.empty((n, 1, k), np.float32)
    xs = np.empty((n, 1, cfg.H), np.uint16)
    for step in range(cfg.steps):
        for layer in range(cfg.L):
            i = step * cfg.L + layer
            ids[i], ws[i], xs[i] = wl.trace_call(cfg, step, layer)
    cache = make_cache(cfg, k, alias_all=True, stream=stream)
    d_ids = torch.from_numpy(ids).cuda()
    d_w = torch.from_numpy(ws).cuda()
    d_x = torch.from_numpy(xs.view(np.int16)).view(torch.bfloat16).cuda()
    d_slots = torch.empty((1, k), dtype=torch.int32, device="cuda")
    d_y = torch.empty((1, cfg.H), dtype=torch.bfloat16, device="cuda")
    s = stream.cuda_stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    torch.cuda.synchronize()
    cache.counters(reset=True)
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    for step in range(cfg.steps):
        for layer in range(cfg.L):
            i = step * cfg.L + layer
            ev[i][0].record(stream)
            cache.ensure(layer, d_ids[i], d_slots, stream=s)
            cache.copy_missing(stream=s)
            ev[i][1].record(stream)
            cache.ffn(d_x[i], d_slots, d_w[i], d_y, stream=s)
            ev[i][2].record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    calls, unique, misses = cache.counters()
    assert cache.status() == F.OK and calls == n
    fetch = np.array([ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]).reshape(cfg.steps, cfg.L)
    ffn = np.array([ev[i][1].elapsed_time(ev[i][2]) for i in range(n)]).reshape(cfg.steps, cfg.L)
    B = cfg.bytes_per_expert
    step_ms = fetch.sum(1)
    cache.close(release=True)
    del cache, d_ids, d_w, d_x
    hbm_peak, _ = measured_peaks()
    ffn_bytes_per_call = k * B + 2 * cfg.H * 2  # k distinct experts per call at bs 1, plus x and y
    return {
        "metric": METRIC, "value": misses * B / (fetch.sum() / 1e3) / 1e9, "unit": "GB/s",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{cfg.name} trace: {cfg.steps} steps x {cfg.L} layers, bs 1, zipf({cfg.zipf_a}) ids, "
                               f"cold start", "E": cfg.E, "topk": k, "H": cfg.H, "I": cfg.I, "L": cfg.L, "S": cfg.S,
                   "l2": "inputs larger than L2 (each miss copies 36 MiB)"},
        "trace": {"calls": calls, "distinct_ids": unique, "misses": misses, "hit_rate": 1.0 - misses / unique,
                  "copied_GB": misses * B / 1e9, "fetch_ms_total": float(fetch.sum()),
                  "ffn_ms_total": float(ffn.sum()),
                  "tok_ms": {"mean": float(step_ms.mean()), "p50": float(np.percentile(step_ms, 50)),
                             "p99": float(np.percentile(step_ms, 99)), "first_step": float(step_ms[0])},
                  "ffn_ms_per_token": float(ffn.sum(1).mean()),
                  "ffn_us_per_call_p50": float(np.percentile(ffn, 50) * 1e3),
                  "ffn_frac_of_hbm": ffn_bytes_per_call * n / (ffn.sum() / 1e3) / 1e9 / hbm_peak},
        "clocks": clocks,
    }


def hybrid_probe(args, cfg, cache, stream, torch, F, wl, link_gbps, cores):
    """Hybrid path measurements (benchmark guide, section 5.2 and 5.4): the CPU expert
    executor's weight bandwidth, the pages' decision rule (hybrid when the CPU MoE GB/s
    exceed 2x the link's), the fetch fraction pcie/cpu, and timed steps of the hybrid path
    (ensure_hybrid, then the copy overlapped with the CPU executor, then the GPU FFN with
    the CPU partial as addend) for the recommended fraction and for an even split."""
    import threading

    s = stream.cuda_stream
    B = cfg.bytes_per_expert
    bank_ptrs = [cache.host_ptrs[b][0] for b in range(cache.nb)]
    bank_bytes = [g.bytes for g in cache.schema]
    fmt = F.FORMATS[cfg.fmt]
    # CPU executor bandwidth (ftmoe_measure_cpu_moe) and the backend decision
    # (ftmoe_moe_backend_decision, default threshold 2x)
    k = cfg.topk
    cpu_gbps = F.ftmoe_measure_cpu_moe(fmt, cfg.H, cfg.I, cfg.E, bank_ptrs, bank_bytes, 2 * k, cores, 3)
    # STREAM-style read ceiling of the host memory the executor reads (the layer's largest bank)
    big = max(range(cache.nb), key=lambda b: bank_bytes[b])
    read_bytes = min(cfg.E * bank_bytes[big], 2 << 30)
    cpu_read = F.ftmoe_measure_cpu_read(bank_ptrs[big], read_bytes, cores, 3)
    backend, frac = F.ftmoe_moe_backend_decision(fmt, link_gbps, cpu_gbps, 0.0)
    out = {"cpu_moe_GBps": cpu_gbps, "cpu_read_ceiling_GBps": cpu_read,
           "cpu_moe_frac_of_read_ceiling": cpu_gbps / cpu_read if cpu_read > 0 else None,
           "link_GBps": link_gbps, "cores": cores,
           "decision": "hybrid" if backend == F.BACKEND_HYBRID else "offload",
           "fetch_fraction": F.ftmoe_hybrid_fetch_fraction(link_gbps, cpu_gbps)}

    r = wl.make_route(cfg, args.bs, args.miss_rate)
    install_hits(cache, r)
    d_ids = torch.from_numpy(r.topk_ids).cuda()
    d_slots = torch.empty_like(d_ids)
    d_counts = torch.zeros(2, dtype=torch.int32, device="cuda")
    d_w = torch.from_numpy(r.weights).cuda()
    d_x = torch.from_numpy(r.x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    d_y = torch.empty((args.bs, cfg.H), dtype=torch.bfloat16, device="cuda")
    d_add = torch.zeros((args.bs, cfg.H), dtype=torch.float32, device="cuda")
    h_add = torch.zeros((args.bs, cfg.H), dtype=torch.float32).pin_memory()

    def run(max_fetch, fraction, reps=5):
        best = None
        for _ in range(reps):
            cache.set_state(r.owner, r.stamp, r.clock, stream=s)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            F.ftmoe_ensure_experts_hybrid(cache.handle, 0, d_ids.data_ptr(), args.bs, cfg.topk, max_fetch, fraction,
                                          d_slots.data_ptr(), d_counts.data_ptr(), s)
            h_slots = d_slots.cpu().numpy()  # the host needs the CPU positions
            F.ftmoe_copy_missing(cache.handle, s)  # the link copy runs while the CPU computes
            F.ftmoe_cpu_expert_ffn(fmt, cfg.H, cfg.I, args.bs, cfg.topk, r.topk_ids.ctypes.data, h_slots.ctypes.data,
                                   bank_ptrs, bank_bytes, r.x.ctypes.data, r.weights.ctypes.data,
                                   h_add.data_ptr(), cores)
            with torch.cuda.stream(stream):
                d_add.copy_(h_add, non_blocking=True)
            F.ftmoe_expert_ffn_hybrid(cache.handle, d_x.data_ptr(), args.bs, d_slots.data_ptr(), d_w.data_ptr(),
                                      cfg.topk, d_add.data_ptr(), d_y.data_ptr(), s)
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            counts = d_counts.cpu().tolist()
            if best is None or dt < best[0]:
                best = (dt, counts)
        return {"step_ms": best[0] * 1e3, "fetched": best[1][0], "misses": best[1][1]}

    out["recommended"] = run(-1, frac)
    out["half_split"] = run(max(0, r.misses // 2), 0.0)
    out["offload"] = run(r.misses, 0.0)
    assert cache.status() == F.OK
    return out


def sweep(args, cfg, cache, stream, torch, F, wl, link=None, hbm_peak=None):
    """Every (bs, miss_rate) point of the workload: median of `repeat` ensure+copy times
    and FFN times (each repeat from the prepared state)."""
    out = []
    s = stream.cuda_stream
    B = cfg.bytes_per_expert
    for bs in cfg.bs_list:
        for mr in cfg.mr_list:
            r = wl.make_route(cfg, bs, mr)
            d_ids = torch.from_numpy(r.topk_ids).cuda()
            d_slots = torch.empty_like(d_ids)
            d_w = torch.from_numpy(r.weights).cuda()
            d_x = torch.from_numpy(r.x.view(np.int16).copy()).view(torch.bfloat16).cuda()
            d_y = torch.empty((bs, cfg.H), dtype=torch.bfloat16, device="cuda")
            install_hits(cache, r)
            tec, tf = [], []
            for i in range(args.repeat + 2):
                cache.set_state(r.owner, r.stamp, r.clock, stream=s)
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                ev[0].record(stream)
                F.ftmoe_ensure_experts(cache.handle, 0, d_ids.data_ptr(), bs, cfg.topk, d_slots.data_ptr(), s)
                F.ftmoe_copy_missing(cache.handle, s)
                ev[1].record(stream)
                F.ftmoe_expert_ffn(cache.handle, d_x.data_ptr(), bs, d_slots.data_ptr(), d_w.data_ptr(), cfg.topk,
                                   d_y.data_ptr(), s)
                ev[2].record(stream)
                ev[2].synchronize()
                if i >= 2:
                    tec.append(ev[0].elapsed_time(ev[1]))
                    tf.append(ev[1].elapsed_time(ev[2]))
            t = statistics.median(tec)
            f = statistics.median(tf)
            bw = r.misses * B / (t / 1e3) / 1e9
            fg = (r.active * B + 2 * bs * cfg.H * 2) / (f / 1e3) / 1e9
            out.append({"bs": bs, "active": r.active, "miss_rate": mr, "misses": r.misses, "time_ms": t,
                        "copy_MiB": r.misses * B / 2 ** 20, "bw_GBps": bw,
                        "copy_frac_of_link": bw / link if (link and r.misses) else None,
                        "tok_ms": t * cfg.L, "ffn_us": f * 1e3, "ffn_GBps": fg,
                        "ffn_frac_of_hbm": fg / hbm_peak if hbm_peak else None,
                        "ffn_kernels": ffn_family(F, cache, cfg, bs)})
    return out


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())

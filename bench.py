"""Paged-KV decode attention benchmark (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config gqa4k]
                    [--layout split|nhd] [--mode auto|v1|v2] [--impl ours|reference]

A step is one pa_decode call over one batch (partition kernel + log-sum-exp
reduce for v2, or the single v1 pass).  The metric is KV-read bandwidth:
bytes of K and V the method must read (sum_s seq_len_s * kv_heads * head_size
* 2 * elem_bytes) divided by the device time of a step.

Timing: inputs resident in HBM; several KV pools rotate so that the bytes
touched between two uses of a pool exceed 4x the L2 size; W warm-up steps, then
exactly K steps between CUDA events on the launching stream, bracketed by
barrier + synchronize; with N ranks every rank runs the same workload on its own
GPU (replicas: the path has no exchange step) and the time is the max over ranks.
Clocks are sampled with nvidia-smi while the steps run.  The main kernel's
launches are timed with CUDA events recorded around them inside the timed
region.  e2e repeats the measurement with host (pinned) buffers copied in and
the output copied out every step.  cpu_baseline times the fp64 CPU oracle on a
bounded sample of the same workload.  --impl reference times that oracle alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import workloads as W  # noqa: E402

METRIC = "paged-decode KV-read HBM GB/s (% of GB300 peak); µs per decode step"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers

def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """Hash of the device code of the kernels (host-side launch heuristics excluded)."""
    h = hashlib.sha256()
    csrc = ROOT / "paged_kv_attention_v2_gb300" / "csrc"
    for f in [csrc / "pa_kernels.cuh", csrc / "pa_ptx.cuh"] + sorted((ROOT / "include").glob("*.h")):
        h.update(f.name.encode())
        h.update(f.read_bytes())
    return h.hexdigest()[:16]


def recorded_traffic(config: str, layout: str, mode: str):
    """DRAM bytes per launch of the main kernel from a committed ncu summary,
    only if it was taken on the current kernel sources."""
    f = ROOT / "profiles" / "ncu_traffic.json"
    if not f.exists():
        return None
    d = json.loads(f.read_text())
    e = d.get(f"{config}/{layout}/{mode}")
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for t, line in self.lines:
            if not (t0 <= t <= t1):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "util": float(parts[4]),
                             "hw": parts[6], "hwt": parts[7], "swt": parts[8], "pcap": parts[9]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        load = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in load), "reasons": sorted(reasons),
                "samples": len(load)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over the ranks of the initialised process group
    (x itself without one): the whole job takes as long as its slowest replica."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank: int, world: int, ms_per_step: float) -> float:
    """Aggregate GB/s of `world` replicas that each move bytes_per_rank per step,
    timed by the slowest one (weak scaling: per-GPU work fixed)."""
    return bytes_per_rank * world / (ms_per_step * 1e-3) / 1e9


# ------------------------------------------------------------------ oracle timing

def time_oracle(w, budget_s: float, threads=None):
    """Time the fp64 oracle on the first n sequences of w, n sized to the
    budget; when the whole batch takes less than the budget, repeat it (up to
    20 passes) so the figure rests on about budget_s of CPU work."""
    import oracle
    threads = threads or oracle.default_threads()
    t = time.perf_counter()
    oracle.oracle_decode(w, seq_subset=[0], threads=threads)
    t1 = max(time.perf_counter() - t, 1e-4)
    lens = w.seq_lens.astype(np.int64)
    n = int(max(1, min(w.num_seqs, budget_s / t1)))
    subset = list(range(n))
    t = time.perf_counter()
    oracle.oracle_decode(w, seq_subset=subset, threads=threads)
    dt = time.perf_counter() - t
    passes = 1
    if n == w.num_seqs and dt < budget_s / 2:
        extra = int(min(19, budget_s / max(dt, 1e-4) - 1))
        t = time.perf_counter()
        for _ in range(extra):
            oracle.oracle_decode(w, seq_subset=subset, threads=threads)
        if extra > 0:
            dt = (dt + time.perf_counter() - t) / (extra + 1)
            passes += extra
    kv = int(lens[:n].sum()) * w.num_kv_heads * w.head_size * 2 * w.elem_bytes
    return {"seconds": dt, "kv_bytes": kv, "seqs": n, "threads": threads, "passes": passes}


# ------------------------------------------------------------------ GPU arm

SECONDARY = "long100k"  # the second target workload, timed in the same default run
MEDIAN_STEPS = 50       # steps timed one by one for the per-step median


def t_(a, dtype):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))  # fp32 / fp16, or raw fp8 bytes


class Setup:
    """Device buffers and prepared C argument structs of one workload: several
    KV pools that the steps rotate through, so the bytes touched between two
    uses of a pool exceed 4x the L2 size."""

    def __init__(self, w, mode_arg, dev, pa, counters=True, dynamic=True, metadata_ready=True):
        import torch
        self.w, self.dev = w, dev
        cdt = w.cache_dtype
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.pool_bytes = w.key_cache.nbytes + w.value_cache.nbytes
        self.copies = max(1, min(8, -(-4 * self.l2 // self.pool_bytes)))
        self.q = t_(w.query, w.dtype).to(dev)
        self.kcs = [t_(w.key_cache, cdt).to(dev) for _ in range(self.copies)]
        self.vcs = [t_(w.value_cache, cdt).to(dev) for _ in range(self.copies)]
        self.bt = torch.from_numpy(w.block_tables).to(dev)
        self.sl = torch.from_numpy(w.seq_lens).to(dev)
        self.al = None if w.alibi_slopes is None else torch.from_numpy(w.alibi_slopes).to(dev)
        self.out = torch.empty(self.q.shape, dtype=tdt, device=dev)
        self.qs = None if w.query_start is None else torch.from_numpy(w.query_start).to(dev)
        # v2 workspace with partition counters, so the library may merge the
        # partitions inside the partition kernel where its rule allows
        self.ws = pa.alloc_workspace(w.num_seqs, w.num_heads, w.head_size, w.max_seq_len, dev,
                                     num_kv_heads=w.num_kv_heads if counters else None,
                                     num_query_tokens=None if self.qs is None else w.num_query_tokens,
                                     tile_counters=dynamic)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        common = dict(num_kv_heads=w.num_kv_heads, scale=w.scale, max_seq_len=w.max_seq_len,
                      kv_dtype=w.kv_dtype, k_scale=w.k_scale, v_scale=w.v_scale,
                      alibi_slopes=self.al, softcap=w.softcap, layout=w.layout, mode=mode_arg,
                      dev_error=self.err, query_start=self.qs,
                      max_query_len=None if self.qs is None else w.max_query_len,
                      seq_lens_host=w.seq_lens,
                      # block tables and lengths are written once here, never by a
                      # kernel in the stream: the kernel may read them early
                      metadata_ready=metadata_ready, **self.ws)
        self.metadata_ready = metadata_ready
        self.cargs = [pa.make_args(self.out, self.q, self.kcs[i], self.vcs[i], self.bt, self.sl, **common)
                      for i in range(self.copies)]
        # what one call runs (mode, in-kernel merge, kernels per call), as the library plans it
        with torch.cuda.device(dev):
            self.plan = pa.plan(self.cargs[0])
        self.stream = torch.cuda.current_stream(dev)
        self.sh = self.stream.cuda_stream
        self.pa = pa

    def step(self, i, ev=None):
        a = self.cargs[i % self.copies]
        if ev is not None:
            a.event_main_begin, a.event_main_end = ev[0].cuda_event, ev[1].cuda_event
        else:
            a.event_main_begin = a.event_main_end = None
        st = self.pa.decode_args_call(a, self.sh)
        if st != 0:
            raise self.pa.PaDecodeError(st)


def measure(S, K, warmup, world, soak_s, sampler):
    """Time K back-to-back steps (the headline), then the same steps with
    events around the main kernel (roofline), MEDIAN_STEPS steps timed one by
    one (per-step median), and the warm-L2 steps on one pool."""
    import torch
    dev, stream = S.dev, S.stream

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    t_soak = time.time()
    i = 0
    while time.time() - t_soak < soak_s:  # clock soak (untimed)
        for _ in range(50):
            S.step(i)
            i += 1
        torch.cuda.synchronize(dev)
    for j in range(warmup):
        S.step(j)
    torch.cuda.synchronize(dev)

    def events(n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:  # torch creates events lazily: record once so the handles exist
            a.record(stream)
            b.record(stream)
        return ev

    kev = events(K)
    sev = events(max(K, MEDIAN_STEPS))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)

    # timed region: exactly K steps back to back
    t0 = time.time()
    barrier()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for j in range(K):
        S.step(j)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t1 = time.time()
    ms_total = e0.elapsed_time(e1)

    # the same K steps with CUDA events around the main kernel of every step
    # (roofline.achieved); the events split the programmatic overlap of the
    # kernels, so this pass is reported separately and not used for `value`
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for j in range(K):
        S.step(j, kev[j])
    e3.record(stream)
    torch.cuda.synchronize(dev)
    kernel_ms = [a.elapsed_time(b) for a, b in kev]
    ms_instrumented = e2.elapsed_time(e3) / K

    # every step between its own pair of events (each step then starts on an
    # idle stream): the per-step median the timing rule of the pages' context asks for
    for j, (a, b) in enumerate(sev):
        a.record(stream)
        S.step(j)
        b.record(stream)
    torch.cuda.synchronize(dev)
    step_ms = [a.elapsed_time(b) for a, b in sev]

    # warm: the same steps on one KV pool only (whatever of it L2 keeps between steps)
    e4, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        S.step(0)
    e4.record(stream)
    for _ in range(K):
        S.step(0)
    e5.record(stream)
    torch.cuda.synchronize(dev)
    ms_warm = e4.elapsed_time(e5) / K
    derr = int(S.err.item())
    if derr:
        raise SystemExit(f"device error bits {derr} during the bench ({S.w.name})")
    return {"ms_step": max_over_ranks(ms_total / K, dev), "kernel_ms": statistics.mean(kernel_ms),
            "ms_instrumented": ms_instrumented, "step_ms_median": statistics.median(step_ms),
            "step_ms_min": min(step_ms), "median_steps": len(step_ms), "ms_warm": ms_warm,
            "window": (t_soak, time.time()), "timed_window": (t0, t1)}


def total_bytes(w, S, mode):
    tb = (w.kv_bytes + w.query.nbytes + S.out.numel() * S.out.element_size() + w.block_tables.nbytes
          + w.seq_lens.nbytes)
    if mode == "v2":
        P = -(-w.seq_lens.astype(np.int64) // 512)
        qn = np.ones_like(P) if w.query_start is None else np.diff(w.query_start).astype(np.int64)
        tb += int((P * qn).sum()) * w.num_heads * (w.head_size + 2) * 4 * 2
    return int(tb)


def roofline(w, S, r, peak, peak_kind):
    kv = w.kv_bytes
    plan = S.plan
    return {"bound": "hbm", "achieved": round(kv / (r["kernel_ms"] * 1e-3) / 1e9, 2), "peak": peak,
            "unit": "GB/s", "frac": round(kv / (r["kernel_ms"] * 1e-3) / 1e9 / peak, 4),
            "peak_kind": peak_kind,
            "kernel": "pa_partition_kernel" + (" (v1)" if plan["mode"] == "v1" else ""),
            "kernel_ms": round(r["kernel_ms"], 6),
            "traffic": recorded_traffic(w.name, w.layout, plan["mode"]),
            "note": "achieved = algorithmic KV bytes / mean CUDA-event time of the partition kernel, "
                    "from a second pass of the same steps with events around that kernel (they split "
                    "its programmatic overlap with the next launch, so kernel_ms can exceed ms_per_step)"}


def config_record(w, S, r, args, world):
    plan = S.plan
    return {"workload": W.DESCRIPTIONS[w.name], "name": w.name, "layout": w.layout,
            "mode": plan["mode"],
            "merge": ("in the partition kernel" if plan["merge_in_kernel"] else "reduce kernel")
            if plan["mode"] == "v2" else "none (v1)",
            "partition_grid": plan["grid"], "ctas_per_sm": plan["ctas_per_sm"],
            "schedule": "dynamic" if plan["dynamic_schedule"] else "static",
            "metadata_ready": S.metadata_ready,
            "kv_bytes_per_step": w.kv_bytes, "total_bytes_per_step": total_bytes(w, S, plan["mode"]),
            "l2": f"rotate {S.copies} KV pools ({S.copies * S.pool_bytes} B >= 4x L2 {S.l2} B)"
            if S.copies * S.pool_bytes >= 4 * S.l2 else f"{S.copies} KV pools of {S.pool_bytes} B",
            "parallelism": f"replicas x{world}", "clock_soak_s": 0.0 if args.no_soak else 1.0,
            "ms_per_step_with_kernel_events": round(r["ms_instrumented"], 6),
            "per_step": {"median_ms": round(r["step_ms_median"], 6), "min_ms": round(r["step_ms_min"], 6),
                         "steps": r["median_steps"],
                         "note": "each step between its own events on an idle stream (no overlap "
                                 "with the previous step), median; the headline is the mean of K "
                                 "steps back to back"},
            "warm_l2": {"ms_per_step": round(r["ms_warm"], 6),
                        "value": round(whole_job_gbs(w.kv_bytes, 1, r["ms_warm"]), 3),
                        "note": "one KV pool reused step after step (rank-local)"}}


def run_ours(args, world, rank, local):
    import torch

    import paged_kv_attention_v2_gb300 as pa
    from paged_kv_attention_v2_gb300 import build as pabuild

    if pabuild.is_stale():
        raise SystemExit("libpa_decode.so is missing or stale: run __graft_entry__.build() first")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    soak = 0.0 if args.no_soak else 1.0
    peak, peak_kind = peaks()

    w = W.make_workload(args.config, args.layout)
    S = Setup(w, args.mode, dev, pa, counters=args.merge == "auto", dynamic=args.schedule == "dynamic",
              metadata_ready=args.metadata == "ready")
    r = measure(S, args.steps, args.warmup, world, soak, sampler)
    kv = w.kv_bytes
    value = whole_job_gbs(kv, world, r["ms_step"])

    # e2e: host buffers, copies inside the timed region, through the C ABI
    e2e = None
    if not args.no_e2e:
        cdt = w.cache_dtype
        hq = t_(w.query, w.dtype).pin_memory()
        hk = t_(w.key_cache, cdt).pin_memory()
        hv = t_(w.value_cache, cdt).pin_memory()
        hbt = torch.from_numpy(w.block_tables).pin_memory()
        hsl = torch.from_numpy(w.seq_lens).pin_memory()
        hal = None if w.alibi_slopes is None else torch.from_numpy(w.alibi_slopes).pin_memory()
        hqs = None if S.qs is None else torch.from_numpy(w.query_start).pin_memory()
        hout = torch.empty(S.out.shape, dtype=S.out.dtype).pin_memory()
        h2d = (hq.nbytes + hk.nbytes + hv.nbytes + hbt.nbytes + hsl.nbytes +
               (hal.nbytes if hal is not None else 0) + (hqs.nbytes if hqs is not None else 0))
        d2h = hout.nbytes
        Ke = max(3, min(args.steps, 50))

        def e2e_step():
            S.q.copy_(hq, non_blocking=True)
            S.kcs[0].copy_(hk, non_blocking=True)
            S.vcs[0].copy_(hv, non_blocking=True)
            S.bt.copy_(hbt, non_blocking=True)
            S.sl.copy_(hsl, non_blocking=True)
            if hal is not None:
                S.al.copy_(hal, non_blocking=True)
            if hqs is not None:
                S.qs.copy_(hqs, non_blocking=True)
            S.step(0)
            hout.copy_(S.out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(S.stream)
        for _ in range(Ke):
            e2e_step()
        f1.record(S.stream)
        torch.cuda.synchronize(dev)
        ms_e2e = max_over_ranks(f0.elapsed_time(f1) / Ke, dev)
        e2e = {"value": round(whole_job_gbs(kv, world, ms_e2e), 3), "unit": "GB/s",
               "ms_per_step": round(ms_e2e, 4), "steps": Ke,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}
    line_cfg = config_record(w, S, r, args, world)
    rl = roofline(w, S, r, peak, peak_kind)
    launches = args.steps * S.plan["kernels"]
    timed = r["timed_window"]
    del S
    torch.cuda.empty_cache()

    # the second target workload (100K-token context), same method, same run
    secondary = None
    if not args.no_secondary and args.config != SECONDARY:
        w2 = W.make_workload(SECONDARY, "split")
        S2 = Setup(w2, "auto", dev, pa, counters=args.merge == "auto", dynamic=args.schedule == "dynamic",
                   metadata_ready=args.metadata == "ready")
        r2 = measure(S2, args.steps, args.warmup, world, soak, sampler)
        v2 = whole_job_gbs(w2.kv_bytes, world, r2["ms_step"])
        secondary = {SECONDARY: {
            "value": round(v2, 3), "unit": "GB/s", "ms_per_step": round(r2["ms_step"], 6),
            "us_per_step": round(r2["ms_step"] * 1e3, 3), "frac_of_peak": round(v2 / world / peak, 4),
            "steps": args.steps, "warmup": args.warmup, "dtype": w2.dtype,
            "config": config_record(w2, S2, r2, args, world), "roofline": roofline(w2, S2, r2, peak, peak_kind),
            "clocks": sampler.summary(*r2["window"])}}
        del S2
        torch.cuda.empty_cache()
    time.sleep(0.15)
    sampler.stop()
    clocks = sampler.summary(*r["window"])

    cpu = None
    if rank == 0 and not args.no_cpu:
        c = time_oracle(w, args.cpu_budget)
        cpu = {"value": round(c["kv_bytes"] / c["seconds"] / 1e9, 6), "unit": "GB/s",
               "cores": c["threads"], "kind": "oracle",
               "seconds": round(c["seconds"], 3),
               "sample": f"first {c['seqs']} of {w.num_seqs} sequences (all heads, dense + "
                         f"partition statistics in fp64), {c['kv_bytes']} KV bytes, "
                         f"mean of {c['passes']} pass(es)"}

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms_step"], 6),
        "us_per_step": round(r["ms_step"] * 1e3, 3), "frac_of_peak": round(value / world / peak, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic: seeded N(0,1) inputs rounded to the storage dtype, shuffled block tables",
        "config": line_cfg,
        "roofline": rl,
        "secondary": secondary,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "timed_region_s": round(timed[1] - timed[0], 4),
    }


# ------------------------------------------------------------------ reference arm

def run_reference(args, world, rank):
    """The fp64 oracle on the host cores, on a bounded sample of the same
    workload per step.  With several ranks, rank 0 alone does the work."""
    own_pg = False
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("gloo")
            own_pg = True
        dist.barrier()  # every rank has joined
        print(f"bench: rank {rank} of {world} joined", file=sys.stderr, flush=True)
        if rank != 0:
            if own_pg:
                dist.destroy_process_group()
            return None
    elif rank != 0:
        return None
    import oracle
    w = W.make_workload(args.config, args.layout)
    threads = oracle.default_threads()
    per_step = max(0.5, min(20.0, args.ref_budget / max(1, args.steps + args.warmup)))
    t = time.perf_counter()
    oracle.oracle_decode(w, seq_subset=[0], threads=threads)
    t1 = max(time.perf_counter() - t, 1e-4)
    n = int(max(1, min(w.num_seqs, per_step / t1)))
    subset = list(range(n))
    for _ in range(args.warmup):
        oracle.oracle_decode(w, seq_subset=subset, threads=threads)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.oracle_decode(w, seq_subset=subset, threads=threads)
        times.append(time.perf_counter() - t)
    dt = sum(times) / len(times)
    kv = int(w.seq_lens[:n].astype(np.int64).sum()) * w.num_kv_heads * w.head_size * 2 * w.elem_bytes
    value = kv / dt / 1e9
    sample = (f"first {n} of {w.num_seqs} sequences per step (all heads, dense + partition "
              f"statistics in fp64), {kv} KV bytes")
    if own_pg:
        import torch.distributed as dist
        dist.destroy_process_group()
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded inputs)",
        "config": {"workload": W.DESCRIPTIONS[w.name], "name": w.name, "layout": w.layout},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ launcher

def _free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_ranks(n: int, argv) -> int:
    """Run this script as n ranks on this node (one per GPU) with torchrun's
    launcher over 127.0.0.1; returns its exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", str(Path(__file__).resolve()),
           *argv]
    return subprocess.call(cmd)


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="gqa4k", choices=sorted(W.SPECS))
    ap.add_argument("--layout", default="split", choices=W.LAYOUTS)
    ap.add_argument("--mode", default="auto", choices=("auto", "v1", "v2"))
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--merge", default="auto", choices=("auto", "reduce"),
                    help="auto: pass partition counters (the library may merge in the partition "
                         "kernel); reduce: no counters, v2 always launches the reduce kernel")
    ap.add_argument("--schedule", default="dynamic", choices=("dynamic", "static"),
                    help="dynamic: pass tile counters (tiles claimed by whichever CTA is free); "
                         "static: the round-robin schedule")
    ap.add_argument("--metadata", default="ready", choices=("ready", "late"),
                    help="ready: block tables and lengths are final when a step is enqueued (the "
                         "kernel reads them before waiting for the previous kernel); late: after")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help=f"skip the second target workload ({SECONDARY}) of the default run")
    ap.add_argument("--no-soak", action="store_true", help="skip the 1 s clock soak (profiling runs)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle wall time")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds for the reference arm")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.gpus < 1:
        raise SystemExit("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return launch_ranks(args.gpus, argv)
    world, rank, local = dist_setup()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {world}: launch one rank per GPU")
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())

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

    w = W.make_workload(args.config, args.layout)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]

    def t_(a, dtype=None):
        dtype = dtype or w.dtype
        if dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a))  # fp8 caches: raw bytes

    cdt = w.cache_dtype

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    pool_bytes = w.key_cache.nbytes + w.value_cache.nbytes
    copies = max(1, min(8, -(-4 * l2 // pool_bytes)))
    q = t_(w.query).to(dev)
    kcs = [t_(w.key_cache, cdt).to(dev) for _ in range(copies)]
    vcs = [t_(w.value_cache, cdt).to(dev) for _ in range(copies)]
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    al = None if w.alibi_slopes is None else torch.from_numpy(w.alibi_slopes).to(dev)
    out = torch.empty(q.shape, dtype=tdt, device=dev)
    qs = None if w.query_start is None else torch.from_numpy(w.query_start).to(dev)
    ws = pa.alloc_workspace(w.num_seqs, w.num_heads, w.head_size, w.max_seq_len, dev,
                            num_query_tokens=None if qs is None else w.num_query_tokens)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    # the library's AUTO choice with the host copy of the lengths a serving
    # loop has at hand (the same rule pa_decode applies to seq_lens_host)
    mode = args.mode if args.mode != "auto" else pa.choose_mode(w.num_seqs, w.num_kv_heads,
                                                                 w.max_seq_len, sm_count,
                                                                 w.seq_lens)
    fused = False  # no partition counters: v2 always launches the reduce kernel
    common = dict(num_kv_heads=w.num_kv_heads, scale=w.scale, max_seq_len=w.max_seq_len,
                  kv_dtype=w.kv_dtype, k_scale=w.k_scale, v_scale=w.v_scale,
                  alibi_slopes=al, softcap=w.softcap, layout=w.layout, mode=mode,
                  dev_error=err, query_start=qs,
                  max_query_len=None if qs is None else w.max_query_len, **ws)
    cargs = [pa.make_args(out, q, kcs[i], vcs[i], bt, sl, **common) for i in range(copies)]
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def step(i, ev=None):
        a = cargs[i % copies]
        if ev is not None:
            a.event_main_begin, a.event_main_end = ev[0].cuda_event, ev[1].cuda_event
        else:
            a.event_main_begin = a.event_main_end = None
        st = pa.decode_args_call(a, sh)
        if st != 0:
            raise pa.PaDecodeError(st)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # clock soak (untimed): run steps back to back for ~1 s while nvidia-smi samples start
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    t_soak = time.time()
    i = 0
    while not args.no_soak and time.time() - t_soak < 1.0:
        for _ in range(50):
            step(i)
            i += 1
        torch.cuda.synchronize(dev)

    for j in range(args.warmup):
        step(j)
    torch.cuda.synchronize(dev)

    K = args.steps
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for a, b in kev:  # torch creates events lazily: record once so the handles exist
        a.record(stream)
        b.record(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)

    # timed region: exactly K steps back to back (value, ms_per_step)
    barrier()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for j in range(K):
        step(j)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall1 = time.time()
    ms_total = e0.elapsed_time(e1)

    # the same K steps with CUDA events around the main kernel of every step
    # (roofline.achieved); the events split the programmatic overlap of the two
    # kernels, so this pass is reported separately and not used for `value`.
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for j in range(K):
        step(j, kev[j])
    e3.record(stream)
    torch.cuda.synchronize(dev)
    kernel_ms = [a.elapsed_time(b) for a, b in kev]
    ms_total_instrumented = e2.elapsed_time(e3)

    # warm: the same steps on one KV pool only (whatever of it L2 keeps between
    # steps is reused); reported beside the cold headline, not used for `value`
    e4, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        step(0)
    e4.record(stream)
    for _ in range(K):
        step(0)
    e5.record(stream)
    torch.cuda.synchronize(dev)
    ms_warm = e4.elapsed_time(e5) / K
    time.sleep(0.15)
    sampler.stop()
    clocks = sampler.summary(t_soak, time.time())

    derr = int(err.item())
    if derr:
        raise SystemExit(f"device error bits {derr} during the bench")

    ms_step = max_over_ranks(ms_total / K, dev)

    kv = w.kv_bytes
    value = whole_job_gbs(kv, world, ms_step)
    peak, peak_kind = peaks()
    k_ms = statistics.mean(kernel_ms)
    achieved = kv / (k_ms * 1e-3) / 1e9
    total_bytes = (kv + w.query.nbytes + out.numel() * out.element_size() + w.block_tables.nbytes
                   + w.seq_lens.nbytes)
    if mode == "v2":
        P = -(-w.seq_lens.astype(np.int64) // 512)
        qn = np.ones_like(P) if w.query_start is None else np.diff(w.query_start).astype(np.int64)
        total_bytes += int((P * qn).sum()) * w.num_heads * (w.head_size + 2) * 4 * 2

    # e2e: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        hq = t_(w.query).pin_memory()
        hk = t_(w.key_cache, cdt).pin_memory()
        hv = t_(w.value_cache, cdt).pin_memory()
        hbt = torch.from_numpy(w.block_tables).pin_memory()
        hsl = torch.from_numpy(w.seq_lens).pin_memory()
        hal = None if w.alibi_slopes is None else torch.from_numpy(w.alibi_slopes).pin_memory()
        hqs = None if qs is None else torch.from_numpy(w.query_start).pin_memory()
        hout = torch.empty(out.shape, dtype=tdt).pin_memory()
        h2d = (hq.nbytes + hk.nbytes + hv.nbytes + hbt.nbytes + hsl.nbytes +
               (hal.nbytes if hal is not None else 0) + (hqs.nbytes if hqs is not None else 0))
        d2h = hout.nbytes
        Ke = max(3, min(K, 50))

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            kcs[0].copy_(hk, non_blocking=True)
            vcs[0].copy_(hv, non_blocking=True)
            bt.copy_(hbt, non_blocking=True)
            sl.copy_(hsl, non_blocking=True)
            if hal is not None:
                al.copy_(hal, non_blocking=True)
            if hqs is not None:
                qs.copy_(hqs, non_blocking=True)
            step(0)
            hout.copy_(out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(Ke):
            e2e_step()
        f1.record(stream)
        torch.cuda.synchronize(dev)
        ms_e2e = max_over_ranks(f0.elapsed_time(f1) / Ke, dev)
        e2e = {"value": round(whole_job_gbs(kv, world, ms_e2e), 3), "unit": "GB/s",
               "ms_per_step": round(ms_e2e, 4), "steps": Ke,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    cpu = None
    if rank == 0 and not args.no_cpu:
        r = time_oracle(w, args.cpu_budget)
        cpu = {"value": round(r["kv_bytes"] / r["seconds"] / 1e9, 6), "unit": "GB/s",
               "cores": r["threads"], "kind": "oracle",
               "seconds": round(r["seconds"], 3),
               "sample": f"first {r['seqs']} of {w.num_seqs} sequences (all heads, dense + "
                         f"partition statistics in fp64), {r['kv_bytes']} KV bytes, "
                         f"mean of {r['passes']} pass(es)"}

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
        "us_per_step": round(ms_step * 1e3, 3), "frac_of_peak": round(value / world / peak, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic: seeded N(0,1) inputs rounded to the storage dtype, shuffled block tables",
        "config": {"workload": W.DESCRIPTIONS[w.name], "name": w.name, "layout": w.layout,
                   "mode": mode, "merge": ("in the partition kernel" if fused else "reduce kernel")
                   if mode == "v2" else "none (v1)", "kv_bytes_per_step": kv, "total_bytes_per_step": int(total_bytes),
                   "l2": f"rotate {copies} KV pools ({copies * pool_bytes} B >= 4x L2 {l2} B)"
                   if copies * pool_bytes >= 4 * l2 else f"{copies} KV pools of {pool_bytes} B",
                   "parallelism": f"replicas x{world}", "clock_soak_s": 0.0 if args.no_soak else 1.0,
                   "ms_per_step_with_kernel_events": round(ms_total_instrumented / K, 6),
                   "warm_l2": {"ms_per_step": round(ms_warm, 6),
                               "value": round(whole_job_gbs(kv, 1, ms_warm), 3),
                               "note": "one KV pool reused step after step (rank-local)"}},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "kernel": "pa_partition_kernel" if mode == "v2" else "pa_partition_kernel (v1)",
                     "kernel_ms": round(k_ms, 6),
                     "traffic": recorded_traffic(w.name, w.layout, mode)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * (2 if mode == "v2" and not fused else 1),
        "clocks": clocks,
    }
    return line


# ------------------------------------------------------------------ reference arm

def run_reference(args, world, rank):
    if rank != 0:
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


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="gqa4k", choices=sorted(W.SPECS))
    ap.add_argument("--layout", default="split", choices=W.LAYOUTS)
    ap.add_argument("--mode", default="auto", choices=("auto", "v1", "v2"))
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-soak", action="store_true", help="skip the 1 s clock soak (profiling runs)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle wall time")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds for the reference arm")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

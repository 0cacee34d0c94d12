"""Helpers for the GPU parity tests: move a workloads.Workload to the device, run
the CUDA path through the C ABI, and compare with the fp64 oracle element by
element.

Tolerances (stated for the method's inputs and fp32 accumulation):
  output and tmp_out, fp16/bf16 inputs:  |gpu - ref| <= 2e-3 + 1e-2 |ref|
  output and tmp_out, fp32 inputs:       |gpu - ref| <= 1e-5 + 1e-5 |ref|
  max_logits and exp_sums:               |gpu - ref| <= 1e-4 max(|ref|, 1)
  unused partitions:                     max_logits == -inf, exp_sums == 0 exactly
"""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_attention_v2_gb300 as pa

OUT_TOL = {"f32": (1e-5, 1e-5), "f16": (2e-3, 1e-2), "bf16": (2e-3, 1e-2)}
STAT_TOL = 1e-4


def torch_dtype(dtype: str):
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def to_torch(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype in ("e4m3", "e5m2"):
        return torch.from_numpy(np.ascontiguousarray(a))  # raw fp8 bytes
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


def to_device(w, device="cuda:0"):
    cdt = getattr(w, "kv_dtype", None) or w.dtype  # fp8 caches: raw uint8 tensors
    d = {
        "query": to_torch(w.query, w.dtype).to(device),
        "key_cache": to_torch(w.key_cache, cdt).to(device),
        "value_cache": to_torch(w.value_cache, cdt).to(device),
        "block_tables": torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(device),
        "seq_lens": torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(device),
        "alibi_slopes": None if w.alibi_slopes is None else torch.from_numpy(w.alibi_slopes).to(device),
        "query_start": (None if getattr(w, "query_start", None) is None
                        else torch.from_numpy(np.ascontiguousarray(w.query_start)).to(device)),
    }
    return d


def run_gpu(w, mode="auto", device="cuda:0", dev=None, max_seq_len=None, seq_lens=None,
            block_tables=None, poison_workspace=True, counters=None, calls=1, metadata_ready=False):
    """Run pa_decode on device; returns dict of float64 numpy arrays + dev_error.

    mode "v2f" is v2 with partition counters (the merge inside the partition
    kernel where the library's rule allows it); `counters` may pass an
    existing counter tensor, which must be all zero again after every call.
    metadata_ready lets the kernel read the block tables and lengths before it
    waits for the previous kernel in the stream.  The result holds the
    library's plan of the call ("plan")."""
    dev = dev or to_device(w, device)
    fused = mode == "v2f"
    if fused:
        mode = "v2"
        if counters is None:
            counters = torch.zeros((w.num_seqs, w.num_kv_heads), dtype=torch.int32, device=device)
    msl = w.max_seq_len if max_seq_len is None else max_seq_len
    S, H, d = w.num_seqs, w.num_heads, w.head_size
    multi = dev["query_start"] is not None
    R = w.num_query_tokens if multi else S  # rows of query / out / workspace
    out = torch.full((R, H, d), float("nan"), dtype=torch_dtype(w.dtype), device=device)
    # modes "auto" and "v2f" take the dynamic tile schedule, "v1" and "v2" the static one
    dynamic = mode == "auto" or fused
    ws = pa.alloc_workspace(S, H, d, msl, device, num_query_tokens=R if multi else None,
                            tile_counters=dynamic)
    tctr = ws.pop("tile_counters", None)
    mq = {"query_start": dev["query_start"], "max_query_len": w.max_query_len} if multi else {}
    if poison_workspace:
        for t in ws.values():
            t.fill_(float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=device)
    call = dict(num_kv_heads=w.num_kv_heads, scale=w.scale, max_seq_len=msl,
                alibi_slopes=dev["alibi_slopes"], softcap=w.softcap, layout=w.layout,
                mode=mode, dev_error=err, partition_counters=counters,
                seq_lens_host=w.seq_lens if mode == "auto" else None,
                window_left=getattr(w, "window_left", -1),
                kv_dtype=getattr(w, "kv_dtype", None), k_scale=getattr(w, "k_scale", 1.0),
                v_scale=getattr(w, "v_scale", 1.0), tile_counters=tctr,
                metadata_ready=metadata_ready, **mq, **ws)
    tensors = (out, dev["query"], dev["key_cache"], dev["value_cache"],
               dev["block_tables"] if block_tables is None else block_tables,
               dev["seq_lens"] if seq_lens is None else seq_lens)
    plan = pa.plan_for(*tensors, **call)
    for _ in range(calls):
        pa.pa_decode(*tensors, **call)
    torch.cuda.synchronize(device)
    if counters is not None:
        assert int(counters.abs().sum().item()) == 0, "partition counters not returned to zero"
    if tctr is not None:
        assert int(tctr.abs().sum().item()) == 0, "tile counters not returned to zero"
    return {
        "out": out.double().cpu().numpy(),
        "max_logits": ws["max_logits"].double().cpu().numpy(),
        "exp_sums": ws["exp_sums"].double().cpu().numpy(),
        "tmp_out": ws["tmp_out"].double().cpu().numpy(),
        "dev_error": int(err.item()),
        "plan": plan,
    }


def _violations(gpu, ref, atol, rtol):
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    bad = ~(np.abs(gpu - ref) <= atol + rtol * np.abs(ref))  # NaN counts as bad
    return bad


def tolerance_used(w, gpu_out, ref_out) -> float:
    """Largest |gpu - ref| / (atol + rtol |ref|) over the elements: the share of
    the tolerance the worst element uses (above 1 fails; NaN gives inf)."""
    atol, rtol = OUT_TOL[w.dtype]
    g, r = np.asarray(gpu_out), np.asarray(ref_out)
    q = np.abs(g - r) / (atol + rtol * np.abs(r))
    return float(np.inf) if np.isnan(q).any() else float(q.max(initial=0.0))


def check_out(w, gpu_out, ref_out, seqs=None, what="out"):
    """Element-by-element tolerance check; returns the share of the tolerance
    the worst element uses."""
    atol, rtol = OUT_TOL[w.dtype]
    sel = slice(None) if seqs is None else np.asarray(seqs)
    g, r = gpu_out[sel], ref_out[sel]
    bad = _violations(g, r, atol, rtol)
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        err = np.nanmax(np.abs(g - r) - rtol * np.abs(r))
        raise AssertionError(f"{w.name}/{w.layout} {what}: {int(bad.sum())} of {bad.size} "
                             f"elements out of tolerance; first at {idx}: gpu {g[idx]!r} "
                             f"ref {r[idx]!r}; worst excess {err:.3e}")
    return tolerance_used(w, g, r)


def stat_rows(w, s):
    """(row, keys visible) for each query token of sequence s: the single token
    sees the whole sequence; with query_start token i of qn sees seq_len - qn + 1 + i."""
    L = int(min(max(int(w.seq_lens[s]), 0), w.max_seq_len))
    qs = getattr(w, "query_start", None)
    if qs is None:
        return [(s, L)]
    q0, qn = int(qs[s]), int(qs[s + 1] - qs[s])
    return [(q0 + i, max(L - qn + 1 + i, 0)) for i in range(qn)]


def check_stats(w, gpu, ref, seqs=None):
    """max_logits / exp_sums / tmp_out of every used partition; padding exactly -inf / 0."""
    atol, rtol = OUT_TOL[w.dtype]
    seqs = range(w.num_seqs) if seqs is None else seqs
    for s, L in ((r, L) for q in seqs for r, L in stat_rows(w, q)):
        P = -(-L // 512)
        # partitions the oracle marks unused (before a sliding window): exactly -inf / 0
        unused = np.isneginf(ref["max_logits"][s, :, :P])
        assert np.all(np.isneginf(gpu["max_logits"][s, :, :P][unused])), f"{w.name} seq {s}"
        assert np.all(gpu["exp_sums"][s, :, :P][unused] == 0.0), f"{w.name} seq {s}"
        for key in ("max_logits", "exp_sums"):
            g = np.where(unused, 0.0, gpu[key][s, :, :P])
            r = np.where(unused, 0.0, ref[key][s, :, :P])
            bad = ~(np.abs(g - r) <= STAT_TOL * np.maximum(np.abs(r), 1.0))
            if bad.any():
                idx = tuple(np.argwhere(bad)[0])
                raise AssertionError(f"{w.name}/{w.layout} {key} seq {s} at {idx}: gpu {g[idx]!r} "
                                     f"ref {r[idx]!r}")
        pad_ml = gpu["max_logits"][s, :, P:]
        pad_es = gpu["exp_sums"][s, :, P:]
        assert np.all(np.isneginf(pad_ml)), f"{w.name} seq {s}: max_logits padding not -inf"
        assert np.all(pad_es == 0.0), f"{w.name} seq {s}: exp_sums padding not 0"
        g = gpu["tmp_out"][s, :, :P]
        r = ref["tmp_out"][s, :, :P]
        bad = _violations(g, r, atol, rtol) & ~unused[:, :, None]
        if bad.any():
            idx = tuple(np.argwhere(bad)[0])
            raise AssertionError(f"{w.name}/{w.layout} tmp_out seq {s} at {idx}: gpu {g[idx]!r} "
                                 f"ref {r[idx]!r}")

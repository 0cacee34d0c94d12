"""Pure-Python fp64 brute force for tiny inputs -- TEST INFRASTRUCTURE ONLY.

A second, independent statement of the computation, written in the order of
"paged_attention_v2_pytorch.py -- BI-V100 PagedAttention V2 implementation":
per sequence, gather the keys and values block by block through the block table
(key blocks [kv_heads, d/x, block, x] permuted to [block, kv_heads, d], value
blocks [kv_heads, d, block] permuted to [block, kv_heads, d]), expand the kv
heads to query heads (repeat_interleave), then for each 512-token partition form
the scores, the partition max, the exponential sum and the weighted value sum,
and finally merge the partitions with the log-sum-exp reduce of Phase 2.
Plain Python loops over Python floats; numpy only decodes storage types.
"""
from __future__ import annotations

import copy
import math

import numpy as np


def _decode(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype in ("e4m3", "e5m2"):  # fp8 caches: torch's own conversion
        import torch
        tdt = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
        return torch.from_numpy(np.ascontiguousarray(a)).view(tdt).double().numpy()
    return a.astype(np.float64)


def _gather(w, s):
    """keys[t][kvh][d], values[t][kvh][d] for sequence s (Python lists)."""
    cdt = getattr(w, "kv_dtype", None) or w.dtype
    kc = _decode(w.key_cache, cdt)
    vc = _decode(w.value_cache, cdt)
    bs, d, hkv = w.block_size, w.head_size, w.num_kv_heads
    L = int(w.seq_lens[s])
    nblk = (L + bs - 1) // bs
    keys, values = [], []
    for b in range(nblk):
        phys = int(w.block_tables[s][b])
        n_tok = min(bs, L - b * bs)
        for o in range(n_tok):
            krow, vrow = [], []
            for h in range(hkv):
                if w.layout == "split":
                    x = kc.shape[-1]
                    krow.append([float(kc[phys, h, dd // x, o, dd % x]) for dd in range(d)])
                    vrow.append([float(vc[phys, h, dd, o]) for dd in range(d)])
                else:
                    krow.append([float(kc[phys, h, o, dd]) for dd in range(d)])
                    vrow.append([float(vc[phys, h, o, dd]) for dd in range(d)])
            keys.append(krow)
            values.append(vrow)
    return keys, values


def brute_decode(w, partition_size: int = 512):
    """Several query tokens per sequence (w.query_start): query token i of a
    sequence with q_len tokens sees the keys up to position seq_len - q_len + i."""
    qs = getattr(w, "query_start", None)
    if qs is None:
        return _brute_single(w, partition_size)
    rows = int(qs[-1])
    res = None
    for s in range(w.num_seqs):
        qn = int(qs[s + 1] - qs[s])
        for qi in range(qn):
            one = copy.copy(w)
            one.num_seqs = 1
            one.query_start = None
            one.seq_lens = np.array([int(w.seq_lens[s]) - qn + 1 + qi], dtype=np.int32)
            one.block_tables = w.block_tables[s:s + 1]
            one.query = w.query[int(qs[s]) + qi:int(qs[s]) + qi + 1]
            r = _brute_single(one, partition_size)
            if res is None:
                res = {k: [None] * rows for k in r}
            for k in r:
                res[k][int(qs[s]) + qi] = r[k][0]
    return res


def _brute_single(w, partition_size: int = 512):
    """Returns dict(out, max_logits, exp_sums, tmp_out) as nested Python lists.

    out[s][h][d] is the Phase 2 reduce of the partitions; max_logits/exp_sums
    are [s][h][p] for the sequence's own partitions (unused ones are -inf / 0),
    tmp_out[s][h][p][d] the normalised partition outputs.
    """
    S, H, d = w.num_seqs, w.num_heads, w.head_size
    group = H // w.num_kv_heads
    q_all = _decode(w.query, w.dtype)
    P_max = max(1, -(-int(w.max_seq_len) // partition_size))
    out = [[[0.0] * d for _ in range(H)] for _ in range(S)]
    ml = [[[-math.inf] * P_max for _ in range(H)] for _ in range(S)]
    es = [[[0.0] * P_max for _ in range(H)] for _ in range(S)]
    tmp = [[[[0.0] * d for _ in range(P_max)] for _ in range(H)] for _ in range(S)]
    for s in range(S):
        L = int(w.seq_lens[s])
        if L == 0:
            continue
        keys, values = _gather(w, s)
        # "Apply k_scale if needed": dequantisation scales of the gathered keys / values
        ks, vs = getattr(w, "k_scale", 1.0), getattr(w, "v_scale", 1.0)
        if ks != 1.0:
            keys = [[[x * ks for x in row] for row in tok] for tok in keys]
        if vs != 1.0:
            values = [[[x * vs for x in row] for row in tok] for tok in values]
        n_parts = (L + partition_size - 1) // partition_size
        # sliding window: the query (position L-1) sees keys t >= L-1-window_left
        wl = getattr(w, "window_left", -1)
        lo = max(0, L - 1 - wl) if wl >= 0 else 0
        for h in range(H):
            kvh = h // group            # repeat_interleave of kv heads
            q = [float(v) for v in q_all[s, h]]
            slope = None if w.alibi_slopes is None else float(w.alibi_slopes[h])
            part_max, part_sum, part_out = [], [], []
            for p in range(n_parts):
                start, end = max(p * partition_size, lo), min((p + 1) * partition_size, L)
                if start >= end:
                    continue  # partition wholly before the window: unused
                scores = []
                for t in range(start, end):
                    z = w.scale * sum(q[i] * keys[t][kvh][i] for i in range(d))
                    if w.softcap > 0:
                        z = w.softcap * math.tanh(z / w.softcap)
                    if slope is not None:
                        z += slope * t
                    scores.append(z)
                m = max(scores)
                ex = [math.exp(z - m) for z in scores]
                ssum = sum(ex)
                acc = [0.0] * d
                for j, t in enumerate(range(start, end)):
                    for i in range(d):
                        acc[i] += ex[j] * values[t][kvh][i]
                acc = [a / ssum for a in acc]
                part_max.append(m)
                part_sum.append(ssum)
                part_out.append(acc)
                ml[s][h][p] = m
                es[s][h][p] = ssum
                tmp[s][h][p] = acc
            gmax = max(part_max)
            resc = [math.exp(m - gmax) * e for m, e in zip(part_max, part_sum)]
            total = sum(resc)
            out[s][h] = [sum(resc[j] * part_out[j][i] for j in range(len(part_out))) / total
                         for i in range(d)]
    return {"out": out, "max_logits": ml, "exp_sums": es, "tmp_out": tmp}

"""fp64 CPU oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports it, and this package never imports the product.

`oracle_decode` runs the plain C implementation in pa_oracle.c (dense softmax
attention gathered through the block table, plus the per-partition statistics
and their log-sum-exp reduce of Phase 1 / Phase 2 of
"paged_attention_v2_pytorch.py -- BI-V100 PagedAttention V2 implementation").
`brute` holds a second, pure-Python statement for tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "libpa_oracle.so"
_lock = threading.Lock()
_libs = {}

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3, "e5m2": 4}
LAYOUT_CODE = {"split": 0, "nhd": 1}
PARTITION_SIZE = 512


class OracleArgs(ctypes.Structure):
    _fields_ = [
        ("query", ctypes.c_void_p),
        ("key_cache", ctypes.c_void_p),
        ("value_cache", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p),
        ("alibi_slopes", ctypes.c_void_p),
        ("num_seqs", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_size", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("partition_size", ctypes.c_int32),
        ("max_num_partitions", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("softcap", ctypes.c_double),
        ("window_left", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("query_start", ctypes.c_void_p),
        ("num_query_tokens", ctypes.c_int32),
        ("k_scale", ctypes.c_double),
        ("v_scale", ctypes.c_double),
        ("seq_subset", ctypes.c_void_p),
        ("n_subset", ctypes.c_int32),
        ("num_threads", ctypes.c_int32),
        ("out", ctypes.c_void_p),
        ("out_v2", ctypes.c_void_p),
        ("max_logits", ctypes.c_void_p),
        ("exp_sums", ctypes.c_void_p),
        ("tmp_out", ctypes.c_void_p),
    ]


def compile_source(src: Path, out: Path) -> Path:
    """gcc a pa_oracle.c (this one or a copy) into a shared library."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", "-I", str(_HERE),
           "-o", str(out), str(src), "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> Path:
    """Compile pa_oracle.c with gcc into oracle/_build/libpa_oracle.so."""
    src = _HERE / "pa_oracle.c"
    hdr = _HERE / "pa_oracle.h"
    with _lock:
        if (not force and _LIB_PATH.exists()
                and _LIB_PATH.stat().st_mtime >= max(src.stat().st_mtime, hdr.stat().st_mtime)):
            return _LIB_PATH
        _BUILD.mkdir(exist_ok=True)
        tmp = _BUILD / f"libpa_oracle.{os.getpid()}.so"
        compile_source(src, tmp)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load(lib_path=None):
    """Load the oracle library (built on first use), or another build of
    pa_oracle.c given by path (the mutation tests use this)."""
    key = str(lib_path) if lib_path else None
    if key not in _libs:
        path = lib_path or build()
        lib = ctypes.CDLL(str(path))
        lib.oracle_decode.argtypes = [ctypes.POINTER(OracleArgs)]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_abi_version.restype = ctypes.c_int
        _libs[key] = lib
    return _libs[key]


def _ptr(a):
    return None if a is None else a.ctypes.data


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_decode(w, seq_subset=None, partials: bool = True, threads: int | None = None,
                  partition_size: int = PARTITION_SIZE, max_num_partitions: int | None = None,
                  lib_path=None):
    """Evaluate the oracle on a workloads.Workload (or any object with the same fields).

    Returns a dict of float64 arrays indexed by absolute query row (= sequence
    number with one query token per sequence; with w.query_start, rows
    query_start[s] .. query_start[s+1]-1 belong to sequence s):
      out        [rows, num_heads, head_size]   dense softmax attention
      out_v2     same, log-sum-exp reduce of the partitions (if partials)
      max_logits [num_seqs, num_heads, P_max]        (if partials)
      exp_sums   [num_seqs, num_heads, P_max]        (if partials)
      tmp_out    [num_seqs, num_heads, P_max, d]     (if partials)
    Rows of sequences outside `seq_subset` are left as NaN.
    """
    lib = _load(lib_path)
    S, H, d = w.num_seqs, w.num_heads, w.head_size
    qs = getattr(w, "query_start", None)
    qs = None if qs is None else np.ascontiguousarray(qs, dtype=np.int32)
    R = S if qs is None else int(qs[-1])  # rows: query tokens
    if max_num_partitions is None:
        max_num_partitions = max(1, -(-int(w.max_seq_len) // partition_size))
    P = max_num_partitions
    q = np.ascontiguousarray(w.query)
    k = np.ascontiguousarray(w.key_cache)
    v = np.ascontiguousarray(w.value_cache)
    bt = np.ascontiguousarray(w.block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(w.seq_lens, dtype=np.int32)
    al = None if w.alibi_slopes is None else np.ascontiguousarray(w.alibi_slopes, dtype=np.float32)
    sub = None if seq_subset is None else np.ascontiguousarray(seq_subset, dtype=np.int32)
    res = {"out": np.full((R, H, d), np.nan)}
    if partials:
        res["out_v2"] = np.full((R, H, d), np.nan)
        res["max_logits"] = np.full((R, H, P), np.nan)
        res["exp_sums"] = np.full((R, H, P), np.nan)
        res["tmp_out"] = np.full((R, H, P, d), np.nan)
    a = OracleArgs(
        query=_ptr(q), key_cache=_ptr(k), value_cache=_ptr(v), block_tables=_ptr(bt),
        seq_lens=_ptr(sl), alibi_slopes=_ptr(al),
        num_seqs=S, num_heads=H, num_kv_heads=w.num_kv_heads, head_size=d,
        block_size=w.block_size, num_blocks=w.num_blocks,
        max_blocks_per_seq=bt.shape[1], partition_size=partition_size,
        max_num_partitions=P, dtype=DTYPE_CODE[w.dtype], layout=LAYOUT_CODE[w.layout],
        scale=float(w.scale), softcap=float(w.softcap),
        window_left=int(getattr(w, "window_left", -1)),
        kv_dtype=DTYPE_CODE[w.kv_dtype] if getattr(w, "kv_dtype", None) else -1,
        query_start=_ptr(qs), num_query_tokens=R,
        k_scale=float(getattr(w, "k_scale", 1.0)), v_scale=float(getattr(w, "v_scale", 1.0)),
        seq_subset=_ptr(sub), n_subset=0 if sub is None else len(sub),
        num_threads=threads or default_threads(),
        out=_ptr(res["out"]),
        out_v2=_ptr(res.get("out_v2")), max_logits=_ptr(res.get("max_logits")),
        exp_sums=_ptr(res.get("exp_sums")), tmp_out=_ptr(res.get("tmp_out")),
    )
    rc = lib.oracle_decode(ctypes.byref(a))
    if rc != 0:
        raise ValueError(f"oracle_decode rejected its arguments (code {rc})")
    return res

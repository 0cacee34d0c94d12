"""Paged-KV decode attention for GB300 (sm_103a): Python binding of libpa_decode.so.

This module only marshals torch tensors (device memory and the current CUDA
stream) into the C ABI of include/pa_decode.h; every step of the computation
runs in the library's CUDA kernels.  It raises if the library is missing.

    out = torch.empty_like(query)
    ws = alloc_workspace(num_seqs, num_heads, head_size, max_seq_len, query.device)
    pa_decode(out, query, key_cache, value_cache, block_tables, seq_lens,
              num_kv_heads=..., scale=..., max_seq_len=..., layout="split", **ws)
"""
from __future__ import annotations

import ctypes

from . import _abi
from ._abi import (PA_BLOCK_SIZE, PA_DEVERR_BLOCK_ID, PA_DEVERR_SEQ_LEN, PA_DEVERR_TIMEOUT,
                   PA_PARTITION_SIZE, LibraryMissing)

__all__ = ["pa_decode", "pa_decode_static_workspace", "alloc_workspace", "max_num_partitions", "choose_mode",
           "plan", "plan_for", "status_str",
           "PaDecodeError", "PA_PARTITION_SIZE", "PA_BLOCK_SIZE", "PA_DEVERR_BLOCK_ID",
           "PA_DEVERR_SEQ_LEN", "PA_DEVERR_TIMEOUT", "LibraryMissing", "library"]

_LAYOUTS = {"split": _abi.PA_LAYOUT_SPLIT, "nhd": _abi.PA_LAYOUT_NHD}
_MODES = {"auto": _abi.PA_MODE_AUTO, "v1": _abi.PA_MODE_V1, "v2": _abi.PA_MODE_V2}
_KV = {None: _abi.PA_KV_SAME, "e4m3": _abi.PA_KV_FP8_E4M3, "e5m2": _abi.PA_KV_FP8_E5M2}


class PaDecodeError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"pa_decode failed: {status_str(status)} (status {status})")
        self.status = status


def library():
    return _abi.load()


def status_str(status: int) -> str:
    return library().pa_status_str(int(status)).decode()


def max_num_partitions(max_seq_len: int) -> int:
    return int(library().pa_max_num_partitions(int(max_seq_len)))


def choose_mode(num_seqs: int, num_kv_heads: int, max_seq_len: int, sm_count: int,
                seq_lens_host=None, ctas_per_sm: int = 2) -> str:
    """The library's AUTO rule as a pure host function (pa_choose_mode, or
    pa_choose_mode_for_lengths with seq_lens_host, host int32 lengths);
    ctas_per_sm is the partition kernel's resident CTAs per SM (plan())."""
    if seq_lens_host is None:
        m = library().pa_choose_mode(num_seqs, num_kv_heads, max_seq_len, sm_count, ctas_per_sm)
    else:
        import numpy as np
        lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
        if lens.shape != (num_seqs,):
            raise ValueError("seq_lens_host must hold num_seqs lengths")
        m = library().pa_choose_mode_for_lengths(num_seqs, num_kv_heads, max_seq_len, sm_count,
                                                 ctas_per_sm, lens.ctypes.data)
    return "v1" if m == _abi.PA_MODE_V1 else "v2"


def plan(args: _abi.PaDecodeArgs) -> dict:
    """What pa_decode would launch for a prepared argument struct on the current
    device (pa_plan): mode, in-kernel merge, kernels per call, the partition
    kernel's CTAs per SM, grid and tile count."""
    pl = _abi.PaLaunchPlan()
    st = library().pa_plan(ctypes.byref(args), ctypes.byref(pl))
    if st != _abi.PA_OK:
        raise PaDecodeError(st)
    return {"mode": "v1" if pl.mode == _abi.PA_MODE_V1 else "v2",
            "merge_in_kernel": bool(pl.merge_in_kernel), "kernels": int(pl.kernels),
            "ctas_per_sm": int(pl.ctas_per_sm), "grid": int(pl.grid),
            "dynamic_schedule": bool(pl.dynamic_schedule), "tiles": int(pl.tiles)}


def plan_for(out, query, key_cache, value_cache, block_tables, seq_lens, **kw) -> dict:
    """plan() for the tensors and keywords pa_decode takes."""
    import torch
    args = make_args(out, query, key_cache, value_cache, block_tables, seq_lens, **kw)
    with torch.cuda.device(query.device):
        return plan(args)


def _dtype_code(t):
    import torch
    return {torch.float32: _abi.PA_DTYPE_F32, torch.float16: _abi.PA_DTYPE_F16,
            torch.bfloat16: _abi.PA_DTYPE_BF16}[t.dtype]


def alloc_workspace(num_seqs: int, num_heads: int, head_size: int, max_seq_len: int, device,
                    num_kv_heads: int | None = None, num_query_tokens: int | None = None,
                    tile_counters: bool = False):
    """torch-allocated v2 workspace: dict(exp_sums, max_logits, tmp_out), plus
    zeroed partition_counters when num_kv_heads is given (fused merge) and
    zeroed tile_counters when asked for (dynamic tile schedule).  With
    several query tokens per sequence the statistics have one row per query
    token (num_query_tokens rows)."""
    import torch
    P = max_num_partitions(max_seq_len)
    rows = num_seqs if num_query_tokens is None else num_query_tokens
    extra = {}
    if num_kv_heads is not None:
        extra["partition_counters"] = torch.zeros((num_seqs, num_kv_heads), dtype=torch.int32,
                                                  device=device)
    if tile_counters:
        extra["tile_counters"] = torch.zeros(2, dtype=torch.int32, device=device)
    return {**extra,
        "exp_sums": torch.empty((rows, num_heads, P), dtype=torch.float32, device=device),
        "max_logits": torch.empty((rows, num_heads, P), dtype=torch.float32, device=device),
        "tmp_out": torch.empty((rows, num_heads, P, head_size), dtype=torch.float32,
                               device=device),
    }


def _ptr(t):
    return None if t is None else t.data_ptr()


def make_args(out, query, key_cache, value_cache, block_tables, seq_lens, *, num_kv_heads: int,
              scale: float, max_seq_len: int, block_size: int = PA_BLOCK_SIZE,
              alibi_slopes=None, softcap: float = 0.0, layout: str = "split", mode: str = "auto",
              exp_sums=None, max_logits=None, tmp_out=None, dev_error=None,
              event_begin=None, event_end=None, partition_counters=None,
              window_left: int = -1, kv_dtype: str | None = None, k_scale: float = 1.0,
              v_scale: float = 1.0, query_start=None,
              max_query_len: int | None = None, seq_lens_host=None,
              tile_counters=None, metadata_ready: bool = False) -> _abi.PaDecodeArgs:
    """Build the C argument struct.  The library validates sizes and types it can
    see; this also checks what only the tensors know: the caches' element size
    and element count against kv_dtype, head_size and num_kv_heads.

    window_left follows AttnDispatchConfig (-1 = no window; the query sees the
    keys t >= seq_len - 1 - window_left) and becomes sliding_window = window_left + 1.
    kv_dtype "e4m3" / "e5m2" marks fp8 caches (raw uint8 tensors) holding K / k_scale
    and V / v_scale; the query dtype sets the compute and output type.
    query_start ([num_seqs + 1] int32 offsets) gives several query tokens per
    sequence: query / out rows are query tokens, and max_query_len (>= every
    sequence's token count) is required with it.  seq_lens_host (a host copy of
    seq_lens: numpy array or CPU tensor) lets mode "auto" choose by the actual
    lengths; the struct keeps a reference to it.  tile_counters (int32 [2],
    zeroed once, e.g. from alloc_workspace(..., tile_counters=True)) turns on
    the dynamic tile schedule.  metadata_ready promises that no earlier kernel
    in the stream writes block_tables, seq_lens or query_start (the kernel may
    read them before it waits for that kernel)."""
    num_rows, num_heads, head_size = query.shape
    num_seqs = seq_lens.shape[0]
    if tuple(out.shape) != tuple(query.shape):
        raise ValueError(f"out shape {tuple(out.shape)} != query shape {tuple(query.shape)}")
    if query_start is None:
        if num_rows != num_seqs:
            raise ValueError(f"query has {num_rows} rows for {num_seqs} sequences")
    else:
        if max_query_len is None:
            raise ValueError("max_query_len is required with query_start")
        if query_start.dtype.itemsize != 4 or query_start.numel() != num_seqs + 1:
            raise ValueError("query_start must be int32 [num_seqs + 1]")
    num_blocks = key_cache.shape[0]
    kv_bytes = 1 if kv_dtype in ("e4m3", "e5m2") else query.element_size()
    page = num_kv_heads * block_size * head_size  # elements of one block of one cache
    for name, c in (("key_cache", key_cache), ("value_cache", value_cache)):
        if c.element_size() != kv_bytes:
            raise ValueError(f"{name} has {c.element_size()}-byte elements, kv_dtype "
                             f"{kv_dtype or 'same as query'} needs {kv_bytes}")
        if c.numel() != num_blocks * page:
            raise ValueError(f"{name} holds {c.numel()} elements, expected "
                             f"num_blocks {num_blocks} x {page}")
    host_lens = None
    if seq_lens_host is not None:
        import numpy as np
        src = seq_lens_host.numpy() if hasattr(seq_lens_host, "numpy") else seq_lens_host
        host_lens = np.ascontiguousarray(np.asarray(src, dtype=np.int32))
        if host_lens.shape != (num_seqs,):
            raise ValueError("seq_lens_host must hold num_seqs lengths")
    a = _abi.PaDecodeArgs(
        out=_ptr(out), query=_ptr(query), key_cache=_ptr(key_cache),
        value_cache=_ptr(value_cache), block_tables=_ptr(block_tables), seq_lens=_ptr(seq_lens),
        num_seqs=num_seqs, num_heads=num_heads, num_kv_heads=num_kv_heads, head_size=head_size,
        num_blocks=num_blocks, block_size=block_size, max_seq_len=max_seq_len,
        max_blocks_per_seq=block_tables.shape[1] if block_tables.dim() == 2 else 0,
        scale=scale, softcap=softcap, alibi_slopes=_ptr(alibi_slopes), dtype=_dtype_code(query),
        layout=_LAYOUTS[layout], mode=_MODES[mode], exp_sums=_ptr(exp_sums),
        max_logits=_ptr(max_logits), tmp_out=_ptr(tmp_out), dev_error=_ptr(dev_error),
        event_main_begin=None if event_begin is None else event_begin.cuda_event,
        event_main_end=None if event_end is None else event_end.cuda_event,
        partition_counters=_ptr(partition_counters),
        sliding_window=int(window_left) + 1 if window_left >= 0 else 0,
        kv_dtype=_KV[kv_dtype], k_scale=float(k_scale), v_scale=float(v_scale),
        query_start=_ptr(query_start), num_query_tokens=num_rows if query_start is not None else 0,
        max_query_len=int(max_query_len) if query_start is not None else 0,
        seq_lens_host=None if host_lens is None else host_lens.ctypes.data,
        tile_counters=_ptr(tile_counters), metadata_ready=1 if metadata_ready else 0,
    )
    a._keep_host_lens = host_lens  # the pointer above stays valid as long as the struct lives
    return a


def pa_decode(out, query, key_cache, value_cache, block_tables, seq_lens, *, stream=None,
              **kw) -> None:
    """Enqueue paged decode attention on `stream` (default: torch's current stream).

    Tensors must be contiguous CUDA tensors: query/out [num_seqs, num_heads,
    head_size] (fp32, fp16 or bf16; [num_query_tokens, ...] with query_start),
    key_cache/value_cache in the split or NHD layout, block_tables [num_seqs,
    max_blocks_per_seq] int32, seq_lens [num_seqs] int32, optional alibi_slopes
    [num_heads] fp32, v2 workspace from alloc_workspace().  Raises PaDecodeError
    with the library's status on failure.
    """
    import torch
    for t in (out, query, key_cache, value_cache, block_tables, seq_lens):
        if not t.is_contiguous():
            raise ValueError("pa_decode needs contiguous tensors")
    args = make_args(out, query, key_cache, value_cache, block_tables, seq_lens, **kw)
    if stream is None:
        stream = torch.cuda.current_stream(query.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    # the library sizes its grid for (and caches attributes of) the current device
    with torch.cuda.device(query.device):
        st = library().pa_decode(ctypes.byref(args), ctypes.c_void_p(handle))
    if st != _abi.PA_OK:
        raise PaDecodeError(st)


def decode_args_call(args: _abi.PaDecodeArgs, stream_handle: int) -> int:
    """Call pa_decode with a prepared argument struct (for tight timing loops)."""
    return library().pa_decode(ctypes.byref(args), ctypes.c_void_p(stream_handle))


def pa_decode_static_workspace(out, query, key_cache, value_cache, block_tables, seq_lens, *,
                               stream=None, **kw) -> None:
    """pa_decode (v2) with the partition workspace in the library's own device
    array, for callers that cannot allocate device memory (see the C header).
    Workspace arguments and `mode` are ignored.  Raises PaDecodeError, e.g.
    PA_ERR_WORKSPACE when the batch needs more than PA_STATIC_WORKSPACE_FLOATS."""
    import torch
    for t in (out, query, key_cache, value_cache, block_tables, seq_lens):
        if not t.is_contiguous():
            raise ValueError("pa_decode_static_workspace needs contiguous tensors")
    args = make_args(out, query, key_cache, value_cache, block_tables, seq_lens, **kw)
    if stream is None:
        stream = torch.cuda.current_stream(query.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    # the array used is the current device's: make the tensors' device current
    with torch.cuda.device(query.device):
        st = library().pa_decode_static_workspace(ctypes.byref(args), ctypes.c_void_p(handle))
    if st != _abi.PA_OK:
        raise PaDecodeError(st)

"""ctypes view of include/pa_decode.h and loading of libpa_decode.so.

Loading fails loudly when the library has not been built: there is no other
implementation behind this package.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "_build" / "libpa_decode.so"

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE = 3
PA_ERR_LAUNCH = 4
PA_ERR_DEVICE_CHECK = 5
PA_ERR_DEVICE_TIMEOUT = 6

PA_DTYPE_F32, PA_DTYPE_F16, PA_DTYPE_BF16 = 0, 1, 2
PA_LAYOUT_SPLIT, PA_LAYOUT_NHD = 0, 1
PA_MODE_AUTO, PA_MODE_V1, PA_MODE_V2 = 0, 1, 2
PA_KV_SAME, PA_KV_FP8_E4M3, PA_KV_FP8_E5M2 = 0, 3, 4

PA_DEVERR_BLOCK_ID = 1
PA_DEVERR_SEQ_LEN = 2
PA_DEVERR_TIMEOUT = 4
PA_DEVERR_QUERY_RANGE = 8

PA_PARTITION_SIZE = 512
PA_BLOCK_SIZE = 16

# every function include/pa_decode.h declares
EXPORTED = ("pa_decode", "pa_max_num_partitions", "pa_workspace_elems", "pa_choose_mode",
            "pa_choose_mode_for_lengths", "pa_workspace_bytes", "pa_partition_size", "pa_plan",
            "pa_status_str", "pa_version", "pa_decode_static_workspace", "pa_debug_withhold_page")

PA_STATIC_WORKSPACE_FLOATS = 4 * 1024 * 1024
PA_FUSED_MAX_PARTITIONS = 8


class PaDecodeArgs(ctypes.Structure):
    _fields_ = [
        ("out", ctypes.c_void_p),
        ("query", ctypes.c_void_p),
        ("key_cache", ctypes.c_void_p),
        ("value_cache", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p),
        ("num_seqs", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("alibi_slopes", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("mode", ctypes.c_int32),
        ("exp_sums", ctypes.c_void_p),
        ("max_logits", ctypes.c_void_p),
        ("tmp_out", ctypes.c_void_p),
        ("dev_error", ctypes.c_void_p),
        ("event_main_begin", ctypes.c_void_p),
        ("event_main_end", ctypes.c_void_p),
        ("partition_counters", ctypes.c_void_p),
        ("sliding_window", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("query_start", ctypes.c_void_p),
        ("num_query_tokens", ctypes.c_int32),
        ("max_query_len", ctypes.c_int32),
        ("seq_lens_host", ctypes.c_void_p),
        ("tile_counters", ctypes.c_void_p),
        ("metadata_ready", ctypes.c_int32),
    ]


class PaLaunchPlan(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int32),
        ("merge_in_kernel", ctypes.c_int32),
        ("kernels", ctypes.c_int32),
        ("ctas_per_sm", ctypes.c_int32),
        ("grid", ctypes.c_int32),
        ("dynamic_schedule", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("tiles", ctypes.c_int64),
    ]


_lib = None


class LibraryMissing(RuntimeError):
    pass


def load(path: Path | None = None):
    """Load libpa_decode.so (built by paged_kv_attention_v2_gb300.build)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path else LIB_PATH
    if not p.exists():
        raise LibraryMissing(
            f"{p} is missing: build it with `python -m paged_kv_attention_v2_gb300.build` "
            "(or __graft_entry__.build()); there is no fallback implementation")
    lib = ctypes.CDLL(str(p))
    lib.pa_decode.argtypes = [ctypes.POINTER(PaDecodeArgs), ctypes.c_void_p]
    lib.pa_decode.restype = ctypes.c_int
    lib.pa_max_num_partitions.argtypes = [ctypes.c_int32]
    lib.pa_max_num_partitions.restype = ctypes.c_int32
    lib.pa_workspace_elems.argtypes = [ctypes.c_int32] * 4 + [ctypes.POINTER(ctypes.c_int64)] * 2
    lib.pa_workspace_elems.restype = ctypes.c_int
    lib.pa_choose_mode.argtypes = [ctypes.c_int32] * 5
    lib.pa_choose_mode.restype = ctypes.c_int32
    lib.pa_workspace_bytes.argtypes = [ctypes.c_int32] * 4
    lib.pa_workspace_bytes.restype = ctypes.c_size_t
    lib.pa_partition_size.argtypes = []
    lib.pa_partition_size.restype = ctypes.c_int32
    lib.pa_choose_mode_for_lengths.argtypes = [ctypes.c_int32] * 5 + [ctypes.c_void_p]
    lib.pa_choose_mode_for_lengths.restype = ctypes.c_int32
    lib.pa_status_str.argtypes = [ctypes.c_int32]
    lib.pa_status_str.restype = ctypes.c_char_p
    lib.pa_version.restype = ctypes.c_int32
    lib.pa_decode_static_workspace.argtypes = [ctypes.POINTER(PaDecodeArgs), ctypes.c_void_p]
    lib.pa_decode_static_workspace.restype = ctypes.c_int
    lib.pa_plan.argtypes = [ctypes.POINTER(PaDecodeArgs), ctypes.POINTER(PaLaunchPlan)]
    lib.pa_plan.restype = ctypes.c_int
    lib.pa_debug_withhold_page.argtypes = [ctypes.c_int32, ctypes.c_int64]
    lib.pa_debug_withhold_page.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib

"""Host-side tests of the C ABI (no GPU needed): the library loads and exports
every function include/pa_decode.h declares, the size helpers, the v1/v2
choice, and the argument checks that return before anything is launched."""
import ctypes
import json
import math
import pathlib
import re

import pytest

import paged_kv_attention_v2_gb300 as pa
from paged_kv_attention_v2_gb300 import _abi

ROOT = pathlib.Path(__file__).resolve().parents[1]
GOLDEN = json.loads((ROOT / "tests" / "golden" / "pages_facts.json").read_text())


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_v2_gb300 import build
    build.build()
    return _abi.load()


def _declared_functions():
    names = set()
    for h in (ROOT / "include").glob("*.h"):
        text = h.read_text()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_function(lib):
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert declared == set(_abi.EXPORTED), declared ^ set(_abi.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_version(lib):
    assert lib.pa_version() >> 16 == 1


def test_partition_counts(lib):
    assert lib.pa_max_num_partitions(0) == 1
    assert lib.pa_max_num_partitions(1) == 1
    assert lib.pa_max_num_partitions(512) == 1
    assert lib.pa_max_num_partitions(513) == 2
    g = GOLDEN["partitions_at_100k"]
    assert lib.pa_max_num_partitions(g["seq_len"]) == g["num_partitions"]
    assert g["full_partitions"] * 512 + g["last_partition_tokens"] == g["seq_len"]


def test_workspace_elems(lib):
    s, t = ctypes.c_int64(), ctypes.c_int64()
    assert lib.pa_workspace_elems(4, 28, 128, 100000, ctypes.byref(s), ctypes.byref(t)) == 0
    assert s.value == 4 * 28 * 196 and t.value == 4 * 28 * 196 * 128
    assert lib.pa_workspace_elems(-1, 28, 128, 10, ctypes.byref(s), ctypes.byref(t)) == 1


def test_choose_mode(lib):
    """Without host lengths every sequence counts as max_seq_len long: v1 once
    the (sequence, kv head) tiles are at least one per SM."""
    assert pa.choose_mode(32, 4, 512, 152) == "v1"       # one partition
    assert pa.choose_mode(32, 4, 4096, 152) == "v2"      # 128 tiles < 152 SMs
    assert pa.choose_mode(4, 4, 100000, 152) == "v2"     # 16 tiles
    assert pa.choose_mode(38, 4, 4096, 152) == "v1"      # 152 tiles
    assert pa.choose_mode(128, 8, 16384, 152) == "v1"    # 1024 tiles, 4 equal rounds
    for c in (1, 2, 3, 0):
        assert pa.choose_mode(128, 8, 16384, 152, ctas_per_sm=c) == "v1"
    assert lib.pa_choose_mode(0, 8, 16384, 152, 2) == _abi.PA_MODE_V2
    assert lib.pa_choose_mode(8, 8, 16384, 0, 2) == _abi.PA_MODE_V2


def test_choose_mode_models_the_resident_ctas_of_the_path():
    """The balance test runs on the grid of the kernel that is launched: the
    same lengths can be even on one grid and uneven on another.  76 sequences
    x 4 kv heads = 304 tiles, the first 38 sequences twice as long: one CTA per
    SM (fp32 with two n-tiles) gives 152 CTAs that each take one long and one
    short tile; two or three per SM (16-bit, fp8 split) give one tile per CTA,
    so the long tiles set the time."""
    import numpy as np
    lens = np.array([8192] * 38 + [4096] * 38, dtype=np.int32)
    assert pa.choose_mode(76, 4, 8192, 152, lens, ctas_per_sm=1) == "v1"
    assert pa.choose_mode(76, 4, 8192, 152, lens, ctas_per_sm=2) == "v2"
    assert pa.choose_mode(76, 4, 8192, 152, lens, ctas_per_sm=3) == "v2"
    # interleaved long / short: every CTA of the 152-CTA grid gets two of a kind
    inter = np.array([8192, 4096] * 38, dtype=np.int32)
    assert pa.choose_mode(76, 4, 8192, 152, inter, ctas_per_sm=1) == "v2"


def test_pages_dispatch_rule_worked_example():
    """The page's own rule and worked example (16-SM part, 4 kv heads): v2 iff
    num_kv_heads * ceil(seq_len / 512) > 2 * 16, i.e. seq_len > 4096."""
    g = GOLDEN["dispatch_rule_bi_v100"]

    def pages_rule(seq_len):
        return g["num_kv_heads"] * math.ceil(seq_len / 512) > g["threshold_factor"] * g["sm_count"]

    for seq_len, expect in g["cases"]:
        assert pages_rule(seq_len) == expect
    assert not pages_rule(g["page_threshold_seq_len"]) and pages_rule(g["page_threshold_seq_len"] + 1)


def test_status_strings(lib):
    for code in range(7):
        assert lib.pa_status_str(code)
    assert pa.status_str(0) == "ok"


def _args(**over):
    a = _abi.PaDecodeArgs(
        out=16, query=16, key_cache=16, value_cache=16, block_tables=16, seq_lens=16,
        num_seqs=2, num_heads=8, num_kv_heads=2, head_size=128, num_blocks=10, block_size=16,
        max_seq_len=100, max_blocks_per_seq=7, scale=0.1, softcap=0.0, alibi_slopes=None,
        dtype=_abi.PA_DTYPE_F16, layout=_abi.PA_LAYOUT_SPLIT, mode=_abi.PA_MODE_V2,
        exp_sums=16, max_logits=16, tmp_out=16)
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,expect", [
    ({"num_heads": 7}, _abi.PA_ERR_INVALID_ARG),           # not a multiple of kv heads
    ({"num_kv_heads": 0}, _abi.PA_ERR_INVALID_ARG),
    ({"num_seqs": -1}, _abi.PA_ERR_INVALID_ARG),
    ({"head_size": 96}, _abi.PA_ERR_UNSUPPORTED),
    ({"block_size": 32}, _abi.PA_ERR_UNSUPPORTED),
    ({"num_heads": 34, "num_kv_heads": 2}, _abi.PA_ERR_UNSUPPORTED),   # group 17
    ({"dtype": 7}, _abi.PA_ERR_INVALID_ARG),
    ({"layout": 5}, _abi.PA_ERR_INVALID_ARG),
    ({"mode": 9}, _abi.PA_ERR_INVALID_ARG),
    ({"scale": float("nan")}, _abi.PA_ERR_INVALID_ARG),
    ({"query": None}, _abi.PA_ERR_INVALID_ARG),
    ({"block_tables": None}, _abi.PA_ERR_INVALID_ARG),
    ({"out": 8}, _abi.PA_ERR_INVALID_ARG),                 # misaligned
    ({"max_blocks_per_seq": 6}, _abi.PA_ERR_INVALID_ARG),  # 6 * 16 < 100
    ({"num_blocks": 0}, _abi.PA_ERR_INVALID_ARG),
    ({"tmp_out": None}, _abi.PA_ERR_WORKSPACE),
    ({"exp_sums": None}, _abi.PA_ERR_WORKSPACE),
    ({"tmp_out": 24}, _abi.PA_ERR_WORKSPACE),              # misaligned workspace
    ({"kv_dtype": _abi.PA_KV_FP8_E5M2, "dtype": _abi.PA_DTYPE_F32}, _abi.PA_ERR_UNSUPPORTED),
    ({"kv_dtype": 9}, _abi.PA_ERR_INVALID_ARG),
    ({"k_scale": float("inf")}, _abi.PA_ERR_INVALID_ARG),
    ({"query_start": 16, "num_query_tokens": 4, "max_query_len": 0}, _abi.PA_ERR_INVALID_ARG),
    ({"query_start": 18, "num_query_tokens": 4, "max_query_len": 2}, _abi.PA_ERR_INVALID_ARG),
    ({"query_start": 16, "num_query_tokens": -1, "max_query_len": 2}, _abi.PA_ERR_INVALID_ARG),
    # 3 query tokens x group 4 > 16 rows of one tile (group 8 x 2 = 16 fits)
    ({"query_start": 16, "num_query_tokens": 6, "max_query_len": 5}, _abi.PA_ERR_UNSUPPORTED),
    ({"query_start": 16, "num_query_tokens": 6, "max_query_len": 3, "num_heads": 16},
     _abi.PA_ERR_UNSUPPORTED),
    ({"num_seqs": 0}, _abi.PA_OK),                         # empty batch: no-op
])
def test_host_argument_checks(lib, over, expect):
    a = _args(**over)
    assert lib.pa_decode(ctypes.byref(a), None) == expect


def test_null_args(lib):
    assert lib.pa_decode(None, None) == _abi.PA_ERR_INVALID_ARG


def test_binding_struct_layouts_match_the_header(tmp_path):
    """The ctypes structs mirror include/pa_decode.h field by field: size and
    every field offset, as a C compiler lays them out (no GPU)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc = pathlib.Path(__file__).resolve().parents[1] / "include"
    lines = ['#include <stdio.h>', '#include "pa_decode.h"', "int main(void) {"]
    for cname, cls in (("pa_decode_args", _abi.PaDecodeArgs), ("pa_launch_plan", _abi.PaLaunchPlan)):
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", str(inc), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        name, field, val = line.split()
        got[(name, field)] = int(val)
    for cname, cls in (("pa_decode_args", _abi.PaDecodeArgs), ("pa_launch_plan", _abi.PaLaunchPlan)):
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert got[(cname, f)] == getattr(cls, f).offset, (cname, f)


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(_abi.LibraryMissing):
        _abi.load(tmp_path / "missing.so")


def test_binding_rejects_cache_tensors_that_do_not_match_the_declared_type():
    """fp8 caches passed without kv_dtype (or the reverse) would make the kernels
    read past the buffers: the binding refuses them before any call."""
    import torch
    q = torch.zeros((2, 8, 128), dtype=torch.float16)
    k8 = torch.zeros((10, 2, 8, 16, 16), dtype=torch.uint8)      # fp8 split key cache
    k16 = torch.zeros((10, 2, 16, 16, 8), dtype=torch.float16)   # fp16 split key cache
    bt = torch.zeros((2, 4), dtype=torch.int32)
    sl = torch.zeros(2, dtype=torch.int32)
    kw = dict(num_kv_heads=2, scale=0.1, max_seq_len=64)
    with pytest.raises(ValueError):
        pa.make_args(q, q, k8, k8, bt, sl, **kw)
    with pytest.raises(ValueError):
        pa.make_args(q, q, k16, k16, bt, sl, kv_dtype="e4m3", **kw)
    with pytest.raises(ValueError):
        pa.make_args(q, q, k16[:5].clone(), k16, bt, sl, **kw)
    pa.make_args(q, q, k8, k8, bt, sl, kv_dtype="e4m3", **kw)
    pa.make_args(q, q, k16, k16, bt, sl, **kw)


def test_binding_multi_token_rows():
    """With query_start the query / out rows are query tokens (any count), the
    sequence count comes from seq_lens, and max_query_len is required."""
    import torch
    k16 = torch.zeros((10, 2, 16, 16, 8), dtype=torch.float16)
    bt = torch.zeros((2, 4), dtype=torch.int32)
    sl = torch.zeros(2, dtype=torch.int32)
    q5 = torch.zeros((5, 8, 128), dtype=torch.float16)
    qs = torch.tensor([0, 2, 5], dtype=torch.int32)
    kw = dict(num_kv_heads=2, scale=0.1, max_seq_len=64)
    with pytest.raises(ValueError):
        pa.make_args(q5, q5, k16, k16, bt, sl, **kw)                 # 5 rows, 2 sequences
    with pytest.raises(ValueError):
        pa.make_args(q5, q5, k16, k16, bt, sl, query_start=qs, **kw)  # no max_query_len
    with pytest.raises(ValueError):
        pa.make_args(q5, q5, k16, k16, bt, sl, query_start=qs[:2], max_query_len=3, **kw)
    a = pa.make_args(q5, q5, k16, k16, bt, sl, query_start=qs, max_query_len=3, **kw)
    assert (a.num_seqs, a.num_query_tokens, a.max_query_len) == (2, 5, 3)
    b = pa.make_args(q5[:2], q5[:2], k16, k16, bt, sl, **kw)
    assert (b.num_seqs, b.query_start, b.num_query_tokens) == (2, None, 0)


def test_withhold_page_hook_arguments(lib):
    assert lib.pa_debug_withhold_page(0, -1) == _abi.PA_ERR_INVALID_ARG
    assert lib.pa_debug_withhold_page(0, 0) == _abi.PA_OK


def test_length_aware_dispatch():
    """v1 for batches whose (sequence, kv head) tiles fill the GPU evenly; v2 for
    few tiles or a ragged mix; max_seq_len <= 512 is always v1."""
    import numpy as np
    sm = 152
    assert pa.choose_mode(128, 8, 16384, sm, np.full(128, 16384)) == "v1"      # 1024 equal tiles
    assert pa.choose_mode(64, 4, 4096, sm, np.full(64, 4096)) == "v1"         # 256 equal tiles
    assert pa.choose_mode(32, 4, 4096, sm, np.full(32, 4096)) == "v2"         # 128 tiles < SMs
    assert pa.choose_mode(4, 4, 100000, sm, np.full(4, 100000)) == "v2"       # 16 tiles
    rng = np.random.default_rng(0)
    ragged = np.clip(np.round(2.0 ** (15 * rng.random(256))), 1, 32768).astype(np.int32)
    assert pa.choose_mode(256, 8, 32768, sm, ragged) == "v2"                  # imbalanced
    lens = np.full(128, 16384)
    lens[7] = 100                                                            # one short sequence
    assert pa.choose_mode(128, 8, 16384, sm, lens) == "v1"
    assert pa.choose_mode(8, 2, 512, sm, np.full(8, 512)) == "v1"
    assert pa.choose_mode(128, 8, 16384, sm) == "v1"                          # no host lengths: even
    with pytest.raises(ValueError):
        pa.choose_mode(4, 2, 4096, sm, np.full(3, 4096))


def test_length_aware_dispatch_edges(lib):
    """Degenerate inputs of the host rule: no usable lengths or SM count fall
    back to v2; lengths outside [0, max_seq_len] are clamped before the load
    balance is judged (an all-empty batch is trivially even)."""
    import numpy as np
    sm = 152
    lens = np.full(128, 16384, dtype=np.int32)
    ptr = lens.ctypes.data
    assert lib.pa_choose_mode_for_lengths(128, 8, 16384, 0, 2, ptr) == _abi.PA_MODE_V2
    assert lib.pa_choose_mode_for_lengths(0, 8, 16384, sm, 2, ptr) == _abi.PA_MODE_V2
    # no lengths: every sequence max_seq_len long, an even batch
    assert lib.pa_choose_mode_for_lengths(128, 8, 16384, sm, 2, None) == _abi.PA_MODE_V1
    assert lib.pa_choose_mode_for_lengths(128, 8, 300, sm, 2, None) == _abi.PA_MODE_V1
    zeros = np.zeros(128, dtype=np.int32)
    assert lib.pa_choose_mode_for_lengths(128, 8, 16384, sm, 2, zeros.ctypes.data) == _abi.PA_MODE_V1
    # lengths beyond max_seq_len count as max_seq_len, negative ones as 0
    over = np.full(128, 1 << 30, dtype=np.int32)
    assert lib.pa_choose_mode_for_lengths(128, 8, 16384, sm, 2, over.ctypes.data) == _abi.PA_MODE_V1
    mixed = lens.copy()
    mixed[::2] = -5  # every other sequence empty: the round-robin load is uneven
    assert lib.pa_choose_mode_for_lengths(128, 8, 16384, sm, 2, mixed.ctypes.data) == _abi.PA_MODE_V2


def test_workspace_bytes_and_partition_size(lib):
    assert lib.pa_partition_size() == 512
    # 4 x 100000 tokens, 28 heads, d 128: 196 partitions per row
    assert lib.pa_workspace_bytes(4, 28, 128, 100000) == 4 * 28 * 196 * (128 + 2) * 4
    assert lib.pa_workspace_bytes(-1, 28, 128, 100000) == 0

"""pa_decode_static_workspace: the decode entry point that allocates nothing.

Callers such as a memory pool or allocator that must not re-enter cudaMalloc,
or a plug-in whose host application owns every device allocation, cannot hand
the library a freshly allocated workspace.  This entry point keeps the
partition workspace in a fixed device array inside the library instead.  The
GPU test calls it through the C ABI twice in a row and checks each result
against the regular pa_decode entry point, within the tolerance the parity tests
use, after a call that leaves NaN in the part of the array the checked calls
use (contents left by an earlier call must not matter).  (This file is named
so that pytest collects it last.)
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from paged_kv_attention_v2_gb300 import _abi


def _args(**over):
    a = _abi.PaDecodeArgs(
        out=256, query=256, key_cache=256, value_cache=256, block_tables=256, seq_lens=256,
        num_seqs=256, num_heads=32, num_kv_heads=8, head_size=128, num_blocks=60000,
        block_size=16, max_seq_len=32768, max_blocks_per_seq=2048, scale=0.08, softcap=0.0,
        dtype=_abi.PA_DTYPE_F16, layout=_abi.PA_LAYOUT_SPLIT, mode=_abi.PA_MODE_AUTO)
    for k, v in over.items():
        setattr(a, k, v)
    return a


def test_batch_beyond_static_capacity_is_rejected():
    from paged_kv_attention_v2_gb300 import build
    build.build()
    lib = _abi.load()
    # 256 * 32 * 64 partitions * (128 + 2) floats > PA_STATIC_WORKSPACE_FLOATS: refused, no launch
    assert lib.pa_decode_static_workspace(ctypes.byref(_args()), None) == _abi.PA_ERR_WORKSPACE
    assert lib.pa_decode_static_workspace(None, None) == _abi.PA_ERR_INVALID_ARG
    # with several query tokens per sequence the workspace has one row per token:
    # 8 sequences fit, 8 sequences of 64 tokens do not
    small = dict(num_seqs=8, max_seq_len=4096, max_blocks_per_seq=256)
    assert lib.pa_decode_static_workspace(
        ctypes.byref(_args(**small, query_start=256, num_query_tokens=512, max_query_len=64)),
        None) == _abi.PA_ERR_WORKSPACE
    # sizes whose product would wrap a 64-bit integer are refused, not wrapped
    # into a small footprint (rows ~2^31, 2^24 heads, 1024 partitions)
    huge = dict(num_seqs=8, num_heads=1 << 24, num_kv_heads=1 << 20, max_seq_len=1 << 19,
                max_blocks_per_seq=1 << 15, query_start=256, num_query_tokens=(1 << 31) - 1,
                max_query_len=1)
    assert lib.pa_decode_static_workspace(ctypes.byref(_args(**huge)), None) == _abi.PA_ERR_WORKSPACE
    for rows, heads, msl in ((1 << 30, 1 << 20, 1 << 30), (1, 1, (1 << 31) - 1), (1 << 20, 8, 1 << 20)):
        a = _args(num_seqs=8, num_heads=heads, num_kv_heads=1, max_seq_len=msl,
                  max_blocks_per_seq=(msl + 15) // 16, query_start=256, num_query_tokens=rows,
                  max_query_len=1)
        assert lib.pa_decode_static_workspace(ctypes.byref(a), None) == _abi.PA_ERR_WORKSPACE


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["gqa4k-split", "alibi-bf16-nhd", "multi-token-f16"])
def test_static_workspace_matches_pa_decode_on_two_calls(case):
    import torch

    from parity_util import OUT_TOL, run_gpu, to_device, torch_dtype

    if case == "gqa4k-split":
        w = W.make_workload("gqa4k", "split")
    elif case == "alibi-bf16-nhd":
        w = W.make_workload(W.small_spec(name="static_ws", num_seqs=5, num_heads=16,
                                         num_kv_heads=4, head_size=128, dtype="bf16",
                                         seq_lens=(1, 511, 513, 3000, 1800), alibi=True,
                                         softcap=30.0, value_mult=2.0), "nhd")
    else:
        w = W.make_workload(W.small_spec(name="static_ws_mt", num_seqs=4, num_heads=8,
                                         num_kv_heads=2, head_size=128, dtype="f16",
                                         seq_lens=(3, 513, 1030, 2600), q_len=[1, 4, 2, 3]),
                            "split")
    dev = to_device(w)
    ref = run_gpu(w, mode="v2", dev=dev)
    assert ref["dev_error"] == 0

    lib = _abi.load()
    multi = dev["query_start"] is not None
    out = torch.empty((w.num_query_tokens, w.num_heads, w.head_size), dtype=torch_dtype(w.dtype),
                      device="cuda:0")
    err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    args = _abi.PaDecodeArgs(
        out=out.data_ptr(), query=dev["query"].data_ptr(), key_cache=dev["key_cache"].data_ptr(),
        value_cache=dev["value_cache"].data_ptr(), block_tables=dev["block_tables"].data_ptr(),
        seq_lens=dev["seq_lens"].data_ptr(), num_seqs=w.num_seqs, num_heads=w.num_heads,
        num_kv_heads=w.num_kv_heads, head_size=w.head_size, num_blocks=w.num_blocks,
        block_size=w.block_size, max_seq_len=w.max_seq_len,
        max_blocks_per_seq=w.block_tables.shape[1], scale=w.scale, softcap=w.softcap,
        alibi_slopes=None if dev["alibi_slopes"] is None else dev["alibi_slopes"].data_ptr(),
        dtype={"f32": 0, "f16": 1, "bf16": 2}[w.dtype],
        layout={"split": 0, "nhd": 1}[w.layout], mode=_abi.PA_MODE_AUTO, dev_error=err.data_ptr(),
        query_start=dev["query_start"].data_ptr() if multi else None,
        num_query_tokens=w.num_query_tokens if multi else 0,
        max_query_len=w.max_query_len if multi else 0,
        # the multi-token case also reads its metadata before the grid wait
        metadata_ready=1 if multi else 0)
    stream = torch.cuda.current_stream().cuda_stream

    # Leave NaN in every entry of the array the checked calls can touch: a call
    # of the same rows and heads with twice the partitions, all of them used,
    # and a NaN value cache writes NaN partition outputs over more than the
    # whole footprint of the checked calls.  A checked call that read an entry
    # it did not write itself would then return NaN.
    R = w.num_query_tokens
    P2 = 2 * max(1, -(-w.max_seq_len // 512))
    lens2 = torch.full((R,), P2 * 512, dtype=torch.int32, device="cuda:0")
    bt2 = torch.zeros((R, P2 * 32), dtype=torch.int32, device="cuda:0")
    v_nan = torch.full_like(dev["value_cache"], float("nan"))
    out2 = torch.zeros_like(out)
    poison = _abi.PaDecodeArgs(
        out=out2.data_ptr(), query=dev["query"].data_ptr(), key_cache=dev["key_cache"].data_ptr(),
        value_cache=v_nan.data_ptr(), block_tables=bt2.data_ptr(), seq_lens=lens2.data_ptr(),
        num_seqs=R, num_heads=w.num_heads, num_kv_heads=w.num_kv_heads, head_size=w.head_size,
        num_blocks=w.num_blocks, block_size=w.block_size, max_seq_len=P2 * 512,
        max_blocks_per_seq=P2 * 32, scale=w.scale, softcap=0.0,
        dtype={"f32": 0, "f16": 1, "bf16": 2}[w.dtype], layout={"split": 0, "nhd": 1}[w.layout],
        mode=_abi.PA_MODE_AUTO, dev_error=err.data_ptr())
    assert lib.pa_decode_static_workspace(ctypes.byref(poison), ctypes.c_void_p(stream)) == _abi.PA_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isnan(out2.float()).all(), "the poisoning call did not leave NaN behind"

    atol, rtol = OUT_TOL[w.dtype]
    for call in range(2):
        out.fill_(float("nan"))
        st = lib.pa_decode_static_workspace(ctypes.byref(args), ctypes.c_void_p(stream))
        assert st == _abi.PA_OK, (call, st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = out.double().cpu().numpy()
        bad = ~(np.abs(got - ref["out"]) <= atol + rtol * np.abs(ref["out"]))
        assert not bad.any(), (call, int(bad.sum()))

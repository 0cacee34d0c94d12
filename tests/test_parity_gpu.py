"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle,
element by element on the same seeded inputs.

Covers every workload (tiny, gqa4k, long100k, ragged at full size; large_batch
at full size on sampled sequences the oracle computes one by one), both cache
layouts, v1 / v2 / auto, and the edge cases: empty and one-token sequences,
page and partition boundaries, GQA groups from 1 to 16 (two n-tiles),
head size 64, fp32 / fp16 / bf16, ALiBi, softcap, out-of-range block ids and
sequence lengths (device error bits, no fault), NaN in unused cache slots;
sliding windows, fp8 (E4M3 / E5M2) caches with scales, and several query
tokens per sequence (1 to 16 tokens, ragged counts, bad offsets flagged).
"""
from __future__ import annotations

import functools

import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from parity_util import check_out, check_stats, run_gpu, to_device  # noqa: E402


@functools.lru_cache(maxsize=2)
def _workload(name, layout):
    return W.make_workload(name, layout)


FULL = [("tiny", "split"), ("tiny", "nhd"), ("gqa4k", "split"), ("gqa4k", "nhd"),
        ("long100k", "split"), ("long100k", "nhd"), ("ragged", "split"), ("ragged", "nhd"),
        ("gqa4k_fp8", "split"), ("gqa4k_fp8", "nhd"), ("long100k_fp8", "split"),
        ("long100k_fp8", "nhd"), ("spec4k", "split"), ("spec4k", "nhd"), ("spec4k_fp8", "split"),
        ("spec4k_fp8", "nhd")]


@pytest.mark.parametrize("name,layout", FULL, ids=[f"{n}-{l}" for n, l in FULL])
def test_workload_parity(name, layout):
    """Full-size workload, every output and partition statistic, v1 / v2 / auto."""
    w = _workload(name, layout)
    ref = oracle.oracle_decode(w)
    dev = to_device(w)
    for mode in ("auto", "v1", "v2", "v2f"):
        g = run_gpu(w, mode=mode, dev=dev, calls=2 if mode == "v2f" else 1)
        assert g["dev_error"] == 0, (mode, g["dev_error"])
        check_out(w, g["out"], ref["out"], what=f"out[{mode}]")
        if g["plan"]["mode"] == "v2":
            check_stats(w, g, ref)
    del dev
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["gqa4k_f32", "long100k_f32"])
def test_f32_full_size(name):
    """The 4K and 100K workloads with fp32 query and cache (the tf32 tensor-core
    consumer), both layouts, every output and partition statistic within the
    1e-5 tolerance.  Prints the share of the tolerance the worst element uses."""
    for layout in ("split", "nhd"):
        w = _workload(name, layout)
        ref = oracle.oracle_decode(w)
        for mode in ("v1", "v2", "v2f"):
            g = run_gpu(w, mode=mode)
            assert g["dev_error"] == 0
            used = check_out(w, g["out"], ref["out"], what=f"out[{mode}]")
            print(f"fp32 tolerance used: {name}/{layout}/{mode}: {used:.3f} of (1e-5 + 1e-5 |ref|)")
            if g["plan"]["mode"] == "v2":
                check_stats(w, g, ref)
        torch.cuda.empty_cache()


def test_large_batch_sampled():
    """128 x 16384 bf16 with softcap 30 at full size; the oracle checks sampled
    sequences, every output row is checked for finiteness and boundedness."""
    for layout in ("split", "nhd"):
        w = W.make_workload("large_batch", layout)
        sample = [0, 41, 86, 127]
        ref = oracle.oracle_decode(w, seq_subset=sample)
        g = run_gpu(w, mode="v2f")
        assert g["dev_error"] == 0
        check_out(w, g["out"], ref["out"], seqs=sample)
        check_stats(w, g, ref, seqs=sample)
        vmax = float(np.abs(W.storage_to_f64(w.value_cache[:1024], w.dtype)).max())
        assert np.all(np.isfinite(g["out"]))
        ml = g["max_logits"]
        assert np.nanmax(ml) <= 30.0 + 1e-3  # softcap bounds every logit
        assert np.abs(g["out"]).max() <= 4 * vmax
        # v1, which the length-aware dispatch picks for this even batch
        g1 = run_gpu(w, mode="v1")
        assert g1["dev_error"] == 0
        check_out(w, g1["out"], ref["out"], seqs=sample)
        assert np.all(np.isfinite(g1["out"]))
        del w


def test_v1_equals_v2():
    """The page's correctness claim: the partitioned result equals the single pass."""
    for name in ("gqa4k", "ragged"):
        w = _workload(name, "split")
        a = run_gpu(w, mode="v1")["out"]
        b = run_gpu(w, mode="v2")["out"]
        atol = 2e-3
        assert np.all(np.abs(a - b) <= atol + 1e-2 * np.abs(b))


EDGE = [
    # name, dtype, layout, H, Hkv, d, lens, alibi, softcap, mult
    ("lens_boundaries", "f16", "split", 8, 2, 128, (1, 15, 16, 17, 511, 512, 513, 1024, 1025), False, 0.0, 1.0),
    ("with_empty", "f16", "nhd", 4, 2, 128, (0, 37, 0, 600), False, 0.0, 1.0),
    ("group1", "bf16", "split", 4, 4, 128, (100, 700), False, 0.0, 1.0),
    ("group8", "f16", "nhd", 16, 2, 128, (300, 1500), True, 0.0, 1.0),
    ("group9_two_ntiles", "f16", "split", 18, 2, 128, (33, 900), False, 0.0, 1.0),
    ("group16", "bf16", "nhd", 32, 2, 128, (1, 2000), False, 20.0, 2.0),
    ("group12_split_alibi_softcap", "f16", "split", 24, 2, 128, (15, 513, 1700), True, 30.0, 2.0),
    ("group16_head64_split", "bf16", "split", 32, 2, 64, (16, 1030), False, 0.0, 1.0),
    ("head64_f16", "f16", "split", 8, 4, 64, (17, 530, 1200), True, 0.0, 1.0),
    ("head64_bf16_nhd", "bf16", "nhd", 6, 3, 64, (5, 1030), False, 10.0, 3.0),
    ("f32_head128", "f32", "split", 6, 2, 128, (40, 555), True, 0.0, 1.0),
    ("f32_nhd_g16", "f32", "nhd", 16, 1, 64, (3, 1100), False, 5.0, 2.0),
    ("f32_split_g8_softcap", "f32", "split", 16, 2, 128, (1, 16, 513, 1025), False, 30.0, 4.0),
    ("f32_split_g1_alibi", "f32", "split", 4, 4, 64, (17, 2100), True, 0.0, 1.0),
    ("f32_nhd_head64", "f32", "nhd", 8, 2, 64, (5, 515, 1300), True, 20.0, 1.0),
    ("f32_group16_split", "f32", "split", 32, 2, 128, (1, 700, 2100), True, 10.0, 1.0),
    ("f32_group12_nhd_head64", "f32", "nhd", 24, 2, 64, (17, 1500), False, 0.0, 3.0),
    ("alibi_softcap", "bf16", "split", 8, 2, 128, (511, 2049), True, 30.0, 2.0),
]


@pytest.mark.parametrize("case", EDGE, ids=[c[0] for c in EDGE])
@pytest.mark.parametrize("mode", ["v1", "v2", "v2f"])
def test_edge_cases(case, mode):
    name, dtype, layout, H, Hkv, d, lens, alibi, cap, mult = case
    spec = W.small_spec(name=name, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv,
                        head_size=d, dtype=dtype, seq_lens=lens, alibi=alibi, softcap=cap,
                        value_mult=mult)
    w = W.make_workload(spec, layout)
    ref = oracle.oracle_decode(w)
    g = run_gpu(w, mode=mode, calls=2)
    assert g["dev_error"] == 0
    used = check_out(w, g["out"], ref["out"])
    if dtype == "f32":
        print(f"fp32 tolerance used: {name}/{layout}/{mode}: {used:.3f} of (1e-5 + 1e-5 |ref|)")
    if mode in ("v2", "v2f"):
        check_stats(w, g, ref)


def test_bad_block_id_is_flagged_not_faulted():
    spec = W.small_spec(name="badblk", num_seqs=2, num_heads=4, num_kv_heads=2, head_size=128,
                        dtype="f16", seq_lens=(40, 600))
    w = W.make_workload(spec, "split")
    dev = to_device(w)
    bt = dev["block_tables"].clone()
    bt[1, 3] = w.num_blocks + 7
    bt[0, 0] = -5
    for mode in ("v1", "v2"):
        g = run_gpu(w, mode=mode, dev=dev, block_tables=bt)
        assert g["dev_error"] & 1, g["dev_error"]
    # the rest of the batch is still computed: a clean run afterwards matches
    g = run_gpu(w, mode="v2", dev=dev)
    assert g["dev_error"] == 0
    check_out(w, g["out"], oracle.oracle_decode(w)["out"])


def test_seq_len_beyond_max_is_clamped_and_flagged():
    spec = W.small_spec(name="badlen", num_seqs=2, num_heads=4, num_kv_heads=2, head_size=128,
                        dtype="bf16", seq_lens=(700, 1200))
    w = W.make_workload(spec, "nhd")
    dev = to_device(w)
    # max_seq_len 1024 < 1200: sequence 1 is clamped to 1024 tokens
    for mode in ("v1", "v2"):
        g = run_gpu(w, mode=mode, dev=dev, max_seq_len=1024)
        assert g["dev_error"] & 2
        w2 = W.make_workload(spec, "nhd")
        w2.seq_lens = np.array([700, 1024], dtype=np.int32)
        w2.max_seq_len = 1024
        ref = oracle.oracle_decode(w2)
        check_out(w2, g["out"], ref["out"])


@pytest.mark.parametrize("lens", [(4096, 0, 1, 3000, 0, 513), (32768, 0, 1, 20000, 0, 513)],
                         ids=["merge-in-kernel", "beyond-fused-limit"])
def test_partition_counters_with_empty_sequences(lens):
    """Counters given: the first batch (at most 8 partitions per sequence, one
    round of tiles) merges inside the partition kernel, the second exceeds the
    limit and uses the reduce kernel.  Empty sequences in the batch, counters
    reused over several calls and back at zero after each."""
    spec = W.small_spec(name="counters", num_seqs=6, num_heads=8, num_kv_heads=2, head_size=128,
                        dtype="bf16", seq_lens=lens, alibi=True)
    w = W.make_workload(spec, "split")
    ref = oracle.oracle_decode(w)
    counters = torch.zeros((w.num_seqs, w.num_kv_heads), dtype=torch.int32, device="cuda:0")
    for _ in range(2):
        g = run_gpu(w, mode="v2f", counters=counters, calls=3)
        assert g["dev_error"] == 0
        check_out(w, g["out"], ref["out"])
        check_stats(w, g, ref)


WINDOWS = [
    # name, dtype, layout, H, Hkv, d, lens, alibi, softcap, window_left
    ("w0", "f16", "split", 8, 2, 128, (1, 17, 700), False, 0.0, 0),
    ("w15_page_edge", "bf16", "nhd", 8, 2, 128, (16, 33, 1025), True, 0.0, 15),
    ("w100", "f16", "nhd", 14, 2, 128, (99, 101, 2000), False, 0.0, 100),
    ("w511_partition_edge", "bf16", "split", 8, 1, 128, (512, 1024, 1537), False, 30.0, 511),
    ("w600_alibi", "f16", "split", 32, 8, 128, (1, 600, 601, 5000), True, 0.0, 600),
    ("w_beyond_len", "f16", "split", 4, 2, 64, (40, 900), False, 0.0, 5000),
    ("w_f32", "f32", "nhd", 6, 2, 128, (300, 1100), True, 0.0, 333),
    ("w_f32_split", "f32", "split", 8, 2, 64, (15, 512, 1300), True, 0.0, 100),
]


@pytest.mark.parametrize("case", WINDOWS, ids=[c[0] for c in WINDOWS])
@pytest.mark.parametrize("mode", ["v1", "v2", "v2f"])
def test_sliding_window(case, mode):
    name, dtype, layout, H, Hkv, d, lens, alibi, cap, wl = case
    spec = W.small_spec(name=name, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv,
                        head_size=d, dtype=dtype, seq_lens=lens, alibi=alibi, softcap=cap)
    w = W.make_workload(spec, layout)
    w.window_left = wl
    ref = oracle.oracle_decode(w)
    g = run_gpu(w, mode=mode, calls=2)
    assert g["dev_error"] == 0
    check_out(w, g["out"], ref["out"])
    if mode in ("v2", "v2f"):
        check_stats(w, g, ref)


def test_sliding_window_ragged_full_size():
    """The ragged workload (256 sequences up to 32768 tokens, ALiBi) with a
    4096-key window: partitions wholly before the window are skipped."""
    w = _workload("ragged", "split")
    w.window_left = 4095
    try:
        ref = oracle.oracle_decode(w)
        for mode in ("v1", "v2"):
            g = run_gpu(w, mode=mode)
            assert g["dev_error"] == 0
            check_out(w, g["out"], ref["out"])
            if mode == "v2":
                check_stats(w, g, ref)
    finally:
        w.window_left = -1


FP8 = [
    # name, query dtype, kv dtype, H, Hkv, d, lens, alibi, softcap, window_left, k_scale, v_scale
    ("e4m3_f16", "f16", "e4m3", 8, 2, 128, (1, 15, 17, 513, 1100), False, 0.0, -1, 2 ** -6, 2 ** -6),
    ("e4m3_bf16_alibi", "bf16", "e4m3", 16, 2, 128, (600, 2049), True, 0.0, -1, 0.05, 0.02),
    ("e5m2_f16_softcap", "f16", "e5m2", 7, 1, 128, (33, 1500), False, 30.0, -1, 0.5, 0.25),
    ("e5m2_bf16_head64", "bf16", "e5m2", 6, 3, 64, (5, 1030), False, 0.0, -1, 1.0, 1.0),
    ("e4m3_group16_window", "bf16", "e4m3", 32, 2, 128, (1, 3000), True, 0.0, 700, 2 ** -5, 2 ** -4),
    ("e4m3_group9", "f16", "e4m3", 18, 2, 64, (100, 513), False, 0.0, -1, 0.01, 0.03),
    ("e4m3_window_head64_g3", "f16", "e4m3", 12, 4, 64, (1, 700, 3000), True, 20.0, 600, 2 ** -5, 2 ** -4),
    ("e5m2_bf16_group7", "bf16", "e5m2", 14, 2, 128, (16, 511, 513, 2100), False, 0.0, -1, 0.5, 0.25),
    ("e4m3_group1_six_kv", "f16", "e4m3", 6, 6, 128, (40, 1030), True, 0.0, -1, 0.1, 0.1),
]


@pytest.mark.parametrize("case", FP8, ids=[c[0] for c in FP8])
@pytest.mark.parametrize("mode", ["v1", "v2", "v2f"])
@pytest.mark.parametrize("layout", ["split", "nhd"])
def test_fp8_cache(case, mode, layout):
    name, dtype, kv, H, Hkv, d, lens, alibi, cap, wl, ks, vs = case
    spec = W.small_spec(name=name, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv,
                        head_size=d, dtype=dtype, seq_lens=lens, alibi=alibi, softcap=cap,
                        kv_dtype=kv, k_scale=ks, v_scale=vs)
    w = W.make_workload(spec, layout)
    w.window_left = wl
    ref = oracle.oracle_decode(w)
    g = run_gpu(w, mode=mode, calls=2)
    assert g["dev_error"] == 0
    check_out(w, g["out"], ref["out"])
    if mode in ("v2", "v2f"):
        check_stats(w, g, ref)


MULTI = [
    # name, query dtype, kv dtype, layout, H, Hkv, d, lens, q_len, alibi, softcap, window_left
    ("q2_f16_short", "f16", None, "split", 8, 2, 128, (1, 2, 16, 513, 514, 1100), 2,
     False, 0.0, -1),
    ("q4_bf16_nhd_alibi", "bf16", None, "nhd", 8, 2, 128, (3, 17, 512, 513, 3000), 4,
     True, 0.0, -1),
    ("q_mixed_window", "f16", None, "split", 12, 3, 128, (5, 600, 1025, 2000), [1, 3, 0, 4],
     False, 0.0, 511),
    ("q8_group2_head64", "f16", None, "nhd", 4, 2, 64, (9, 1030, 520), 8, False, 30.0, 100),
    ("q16_mha", "bf16", None, "split", 3, 3, 128, (20, 531), 16, True, 0.0, -1),
    ("q3_f32_alibi_window", "f32", None, "nhd", 8, 2, 128, (100, 700), 3, True, 0.0, 200),
    ("q5_f32_head64", "f32", None, "split", 6, 2, 64, (4, 515), 5, False, 0.0, -1),
    ("q2_f32_split_group4", "f32", None, "split", 8, 2, 128, (1, 16, 600, 1030), 2,
     True, 20.0, 300),
    ("q2_f32_nhd_group4_head64", "f32", None, "nhd", 8, 2, 64, (3, 600, 1030), 2,
     False, 10.0, 200),
    ("q2_e4m3_group8", "bf16", "e4m3", "split", 16, 2, 128, (600, 2049), 2, True, 0.0, -1),
    ("q3_e5m2_window", "f16", "e5m2", "split", 6, 2, 64, (33, 1500), 3, False, 30.0, 100),
    ("q2_e4m3_nhd_group8", "bf16", "e4m3", "nhd", 16, 2, 128, (600, 2049), 2, True, 0.0, -1),
    ("q3_e5m2_nhd_head64", "f16", "e5m2", "nhd", 6, 2, 64, (33, 1500), 3, False, 30.0, 100),
]


@pytest.mark.parametrize("case", MULTI, ids=[c[0] for c in MULTI])
@pytest.mark.parametrize("mode", ["auto", "v1", "v2", "v2f"])
def test_multi_token(case, mode):
    """Several query tokens per sequence (each the single-token decode of the
    sequence cut after its position): outputs and every row's statistics."""
    name, dtype, kv, layout, H, Hkv, d, lens, ql, alibi, cap, wl = case
    spec = W.small_spec(name=name, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv,
                        head_size=d, dtype=dtype, seq_lens=lens, alibi=alibi, softcap=cap,
                        kv_dtype=kv, k_scale=2 ** -5 if kv else 1.0,
                        v_scale=2 ** -4 if kv else 1.0, q_len=ql)
    w = W.make_workload(spec, layout)
    w.window_left = wl
    ref = oracle.oracle_decode(w)
    g = run_gpu(w, mode=mode, calls=2)
    assert g["dev_error"] == 0
    check_out(w, g["out"], ref["out"])
    if g["plan"]["mode"] == "v2":
        check_stats(w, g, ref)


def test_multi_token_full_size():
    """The 32 x 4096 GQA workload (28 heads over 4 kv heads) with two query
    tokens per sequence, both cache layouts."""
    import dataclasses
    spec = dataclasses.replace(W.SPECS["gqa4k"], name="gqa4k_q2", q_len=2)
    for layout in ("split", "nhd"):
        w = W.make_workload(spec, layout)
        ref = oracle.oracle_decode(w)
        for mode in ("v1", "v2", "v2f"):
            g = run_gpu(w, mode=mode)
            assert g["dev_error"] == 0
            check_out(w, g["out"], ref["out"], what=f"out[{mode}]")
            if mode != "v1":
                check_stats(w, g, ref)


def test_multi_token_bad_query_start_is_flagged_not_faulted():
    """Offsets beyond the query rows or a count above max_query_len: the kernels
    clamp them to existing rows, set PA_DEVERR_SEQ_LEN and never fault."""
    spec = W.small_spec(name="badqs", num_seqs=3, num_heads=8, num_kv_heads=2, head_size=128,
                        dtype="f16", seq_lens=(40, 600, 1200), q_len=2)
    w = W.make_workload(spec, "split")
    dev = to_device(w)
    # sequence 1 claims rows [2, 9): more than max_query_len (2) and past the 6 rows
    dev["query_start"] = torch.tensor([0, 2, 9, 6], dtype=torch.int32, device="cuda:0")
    for mode in ("v1", "v2", "v2f"):
        g = run_gpu(w, mode=mode, dev=dev)
        assert g["dev_error"] & 2, mode  # PA_DEVERR_SEQ_LEN
    ref = oracle.oracle_decode(w)
    check_out(w, g["out"][:2], ref["out"][:2])  # sequence 0 is untouched


EARLY = [
    # name, dtype, kv, layout, H, Hkv, lens, q_len, window_left, mode
    ("early_uniform_v2", "f16", None, "split", 28, 4, (2048,) * 40, None, -1, "v2"),
    ("early_ragged_dynamic", "bf16", None, "nhd", 16, 4, tuple(17 + 331 * i for i in range(48)), None, -1,
     "auto"),
    ("early_fused_one_round", "f16", None, "split", 8, 2, (1025, 3000, 77, 0), None, -1, "v2f"),
    ("early_v1_window", "bf16", None, "split", 8, 2, (300, 1500, 2600), None, 700, "v1"),
    ("early_tokens_fp8", "f16", "e4m3", "split", 8, 2, (600, 1300, 2049), [2, 1, 3], -1, "v2"),
]


@pytest.mark.parametrize("case", EARLY, ids=[c[0] for c in EARLY])
def test_metadata_ready_reads_before_the_grid_wait(case):
    """metadata_ready: the partition kernel reads block tables and lengths
    (and walks to its first tile) before it waits for the previous kernel in
    the stream.  Three calls back to back, so each starts while the previous
    call's kernels run: outputs and statistics against the oracle, the
    counters back at zero (static, dynamic and in-kernel-merge paths, v1)."""
    name, dtype, kv, layout, H, Hkv, lens, ql, wl, mode = case
    spec = W.small_spec(name=name, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv, head_size=128,
                        dtype=dtype, seq_lens=lens, q_len=ql, kv_dtype=kv)
    w = W.make_workload(spec, layout)
    w.window_left = wl
    ref = oracle.oracle_decode(w)
    g = run_gpu(w, mode=mode, calls=3, metadata_ready=True)
    assert g["dev_error"] == 0
    check_out(w, g["out"], ref["out"])
    if g["plan"]["mode"] == "v2":
        check_stats(w, g, ref)


@pytest.mark.parametrize("mode", ["v1", "v2"])
def test_cuda_graph_capture_replays_the_same_result(mode):
    """pa_decode allocates nothing and never synchronises, so a CUDA graph can
    capture it (both kernels of v2, with their programmatic dependency) and
    replay it with the same result as an eager call."""
    import paged_kv_attention_v2_gb300 as pa
    from parity_util import torch_dtype
    spec = W.small_spec(name="graph", num_seqs=5, num_heads=16, num_kv_heads=4, head_size=128,
                        dtype="bf16", seq_lens=(1, 511, 513, 3000, 1800), alibi=True)
    w = W.make_workload(spec, "split")
    dev = to_device(w)
    H, d = w.num_heads, w.head_size
    out = torch.empty((w.num_seqs, H, d), dtype=torch_dtype(w.dtype), device="cuda:0")
    ws = pa.alloc_workspace(w.num_seqs, H, d, w.max_seq_len, "cuda:0")
    kw = dict(num_kv_heads=w.num_kv_heads, scale=w.scale, max_seq_len=w.max_seq_len,
              alibi_slopes=dev["alibi_slopes"], mode=mode, **ws)
    pa.pa_decode(out, dev["query"], dev["key_cache"], dev["value_cache"], dev["block_tables"],
                 dev["seq_lens"], **kw)
    torch.cuda.synchronize()
    eager = out.clone()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.capture_begin()
        pa.pa_decode(out, dev["query"], dev["key_cache"], dev["value_cache"], dev["block_tables"],
                     dev["seq_lens"], stream=s, **kw)
        g.capture_end()
    torch.cuda.synchronize()
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    check_out(w, out.double().cpu().numpy(), oracle.oracle_decode(w)["out"])


def _plan(name, H, Hkv, d, dtype, lens, layout="split", kv=None, mode="auto", counters=True,
          q_len=None, dynamic=False):
    """pa_plan for a batch shape; the tensors only carry shapes (plan reads no memory)."""
    S, L = len(lens), int(max(lens))
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    rows = S if q_len is None else S * q_len
    q = torch.zeros((rows, H, d), dtype=tdt, device="cuda:0")
    cdt = torch.uint8 if kv else tdt
    nb = 4
    k = torch.zeros((nb, Hkv, 16, d), dtype=cdt, device="cuda:0")
    bt = torch.zeros((S, -(-L // 16)), dtype=torch.int32, device="cuda:0")
    sl = torch.zeros(S, dtype=torch.int32, device="cuda:0")
    import paged_kv_attention_v2_gb300 as pa
    ws = pa.alloc_workspace(S, H, d, L, "cuda:0", num_kv_heads=Hkv if counters else None,
                            num_query_tokens=None if q_len is None else rows, tile_counters=dynamic)
    extra = {}
    if q_len is not None:
        extra = dict(query_start=torch.arange(0, rows + 1, q_len, dtype=torch.int32, device="cuda:0"),
                     max_query_len=q_len)
    return pa.plan_for(q, q, k, k, bt, sl, num_kv_heads=Hkv, scale=0.1, max_seq_len=L, layout=layout,
                       mode=mode, kv_dtype=kv, seq_lens_host=np.asarray(lens, dtype=np.int32), **extra,
                       **ws)


def test_plan_reports_each_path():
    """pa_plan: what pa_decode launches per path -- mode, merge, kernels per call,
    resident CTAs per SM of the partition kernel and its equal-round grid."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    g = _plan("gqa4k", 28, 4, 128, "f16", [4096] * 32)
    assert (g["mode"], g["merge_in_kernel"], g["kernels"]) == ("v2", False, 2)   # several rounds
    assert g["ctas_per_sm"] == 2 and g["tiles"] == 1024
    rounds = -(-1024 // (sm * 2))
    assert g["grid"] == -(-1024 // rounds)
    g = _plan("gqa4k", 28, 4, 128, "f16", [4096] * 32, dynamic=True)   # equal tiles: static
    assert (g["dynamic_schedule"], g["grid"]) == (False, 256 if sm == 152 else g["grid"])
    g = _plan("mixed", 28, 4, 128, "f16", [4096, 2000] * 16, dynamic=True)  # every resident CTA
    assert (g["dynamic_schedule"], g["grid"]) == (True, min(g["tiles"], sm * 2))
    g = _plan("one_round", 28, 4, 128, "f16", [4096] * 4)           # 128 tiles: one round
    assert (g["mode"], g["merge_in_kernel"], g["kernels"], g["grid"]) == ("v2", True, 1, 128)
    g = _plan("one_round", 28, 4, 128, "f16", [4096] * 4, counters=False)
    assert (g["merge_in_kernel"], g["kernels"]) == (False, 2)
    g = _plan("long100k", 28, 4, 128, "bf16", [100000] * 4)
    assert (g["mode"], g["merge_in_kernel"], g["kernels"], g["tiles"]) == ("v2", False, 2, 3136)
    assert g["grid"] == -(-3136 // -(-3136 // (sm * 2)))
    assert _plan("fp8", 28, 4, 128, "f16", [4096] * 32, kv="e4m3")["ctas_per_sm"] == 3
    assert _plan("fp8", 28, 4, 128, "f16", [4096] * 32, kv="e4m3", layout="nhd")["ctas_per_sm"] == 3
    assert _plan("f32", 28, 4, 128, "f32", [4096] * 32)["ctas_per_sm"] == 2
    assert _plan("f32", 64, 4, 128, "f32", [4096] * 32)["ctas_per_sm"] == 1   # group 16: two n-tiles
    g = _plan("large", 64, 8, 128, "bf16", [16384] * 128)
    assert (g["mode"], g["kernels"], g["tiles"]) == ("v1", 1, 1024)
    g = _plan("ragged", 32, 8, 128, "f16", [20000, 30, 5000, 12] * 64)
    assert (g["mode"], g["merge_in_kernel"]) == ("v2", False)
    g = _plan("tokens", 8, 2, 128, "f16", [1030, 1500, 1200, 1536], q_len=2)   # several tokens
    assert (g["mode"], g["merge_in_kernel"], g["kernels"]) == ("v2", True, 1)
    assert _plan("short", 8, 2, 128, "f16", [300, 400])["mode"] == "v1"



MERGE = [
    # name, dtype, layout, H, Hkv, lens, alibi, softcap, q_len, merged in the kernel
    ("mk_f16_split", "f16", "split", 28, 4, (3073, 3200, 3584, 3333, 3500), False, 0.0, None, True),
    ("mk_bf16_nhd_alibi_cap", "bf16", "nhd", 16, 4, (1025, 1536, 100), True, 20.0, None, True),
    ("mk_tokens", "f16", "split", 8, 2, (1030, 1500, 1200, 1536), False, 0.0, [1, 4, 2, 3], True),
    ("mk_several_rounds", "f16", "split", 28, 4, tuple(3585 + 13 * i for i in range(40)), False, 0.0, None,
     False),
]


@pytest.mark.parametrize("case", MERGE, ids=[c[0] for c in MERGE])
def test_merge_in_kernel_plan_and_parity(case):
    """With partition counters, batches that fit in one round of the persistent
    grid (and at most PA_FUSED_MAX_PARTITIONS partitions) merge in the partition
    kernel (one launch); a batch of several rounds launches the reduce kernel.
    Both agree with the oracle on two calls in a row (the counters return to
    zero)."""
    name, dtype, layout, H, Hkv, lens, alibi, cap, ql, merged = case
    spec = W.small_spec(name=name, num_seqs=len(lens), num_heads=H, num_kv_heads=Hkv, head_size=128,
                        dtype=dtype, seq_lens=lens, alibi=alibi, softcap=cap, q_len=ql)
    w = W.make_workload(spec, layout)
    ref = oracle.oracle_decode(w)
    g = run_gpu(w, mode="v2f", calls=2)
    assert g["plan"]["merge_in_kernel"] == merged and g["plan"]["kernels"] == (1 if merged else 2)
    assert g["dev_error"] == 0
    check_out(w, g["out"], ref["out"])
    check_stats(w, g, ref)

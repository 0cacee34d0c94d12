"""Failure detection without a GPU fault: the kernels' barrier waits are
bounded.  A test hook of the library withholds one page copy, so the consumer
warp waiting for it gives up after a short limit; the call must report
PA_DEVERR_TIMEOUT through the device error word, end, and leave the context
usable for the next (correct) call.
"""
from __future__ import annotations

import time

import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from parity_util import check_out, run_gpu, to_device  # noqa: E402

PA_DEVERR_TIMEOUT = 4


@pytest.mark.parametrize("dtype,kv,mode", [("f16", None, "v2"), ("bf16", "e4m3", "v1"),
                                           ("f32", None, "v2")])
def test_withheld_page_times_out_and_context_survives(dtype, kv, mode):
    from paged_kv_attention_v2_gb300 import _abi
    lib = _abi.load()
    spec = W.small_spec(name="stall", num_seqs=3, num_heads=8, num_kv_heads=2, head_size=128,
                        dtype=dtype, seq_lens=(700, 1300, 90), kv_dtype=kv,
                        k_scale=0.05 if kv else 1.0, v_scale=0.05 if kv else 1.0)
    w = W.make_workload(spec, "split")
    dev = to_device(w)
    assert lib.pa_debug_withhold_page(1, 50_000_000) == 0  # 50 ms per wait
    try:
        t0 = time.perf_counter()
        g = run_gpu(w, mode=mode, dev=dev)
        dt = time.perf_counter() - t0
    finally:
        assert lib.pa_debug_withhold_page(0, 0) == 0
    assert g["dev_error"] & PA_DEVERR_TIMEOUT, g["dev_error"]
    assert dt < 30.0
    g2 = run_gpu(w, mode=mode, dev=dev)
    assert g2["dev_error"] == 0
    check_out(w, g2["out"], oracle.oracle_decode(w)["out"])

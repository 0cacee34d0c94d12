"""Pins of the fp64 oracle to things other than itself.

Each pin_* function takes `run(workload, **kw) -> dict` (the oracle, or a build
of it with a planted mistake) and raises AssertionError when the oracle
disagrees with what the pages or the mathematics fix:

  brute force     a pure-Python statement in the order of
                  "paged_attention_v2_pytorch.py -- BI-V100 PagedAttention V2
                  implementation" (oracle/brute.py), on tiny inputs
  library         torch scaled_dot_product_attention in fp64 (identity block
                  table; GQA by repeat_interleave as in the page's "GQA
                  expansion" step)
  closed forms    two-token softmax and softcap, ALiBi geometric weights
  invariants      partitioned == dense (the page's claim that the log-sum-exp
                  reduce equals a full softmax), seq_len 1, identical V rows,
                  pool permutation, split == NHD, zero query, bounds on exp_sums
  pages' numbers  tests/golden/pages_facts.json (partition count at 100K tokens)

`run_all` runs every pin and reports which ones failed; the mutation test uses
it against oracle builds with planted mistakes.
"""
from __future__ import annotations

import copy
import json
import math
import pathlib
import sys

import numpy as np

ROOT = pathlib.Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import workloads as W  # noqa: E402

GOLDEN = json.loads((ROOT / "tests" / "golden" / "pages_facts.json").read_text())


def _close(a, b, rtol=1e-11, atol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    ok = both_inf | np.isclose(a, b, rtol=rtol, atol=atol)
    if not ok.all():
        idx = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: mismatch at {tuple(idx)}: {a[tuple(idx)]} vs {b[tuple(idx)]}")


def _clone(w, **changes):
    w2 = copy.copy(w)
    for k, v in changes.items():
        setattr(w2, k, v)
    return w2


def _logical_kv(w):
    """Logical [blocks, kv_heads, block_size, d] float64 views of the caches."""
    k = W.storage_to_f64(w.key_cache, w.dtype)
    v = W.storage_to_f64(w.value_cache, w.dtype)
    nb, hkv, bs, d = w.num_blocks, w.num_kv_heads, w.block_size, w.head_size
    if w.layout == "split":
        k = k.transpose(0, 1, 3, 2, 4).reshape(nb, hkv, bs, d)
        v = v.transpose(0, 1, 3, 2)
    return k, v


def _from_logical(w, k_log, v_log):
    """Replace the caches of w by logical fp values (rounded to w.dtype)."""
    k = W.round_to_storage(np.asarray(k_log, dtype=np.float32), w.dtype)
    v = W.round_to_storage(np.asarray(v_log, dtype=np.float32), w.dtype)
    return _clone(w, key_cache=W.logical_to_layout(k, "k", w.layout, w.dtype),
                  value_cache=W.logical_to_layout(v, "v", w.layout, w.dtype))


def _identity_tables(w):
    bs = w.block_size
    t = np.zeros_like(w.block_tables)
    off = 0
    for s in range(w.num_seqs):
        nb = -(-int(w.seq_lens[s]) // bs)
        t[s, :nb] = np.arange(off, off + nb)
        off += nb
    return t


def _spec(**kw):
    kw.setdefault("pool_extra", 3)
    return W.small_spec(**kw)


# ------------------------------------------------------------------ pins

def pin_brute(run):
    """C oracle == pure-Python brute force (tiny workload and small random shapes)."""
    from oracle.brute import brute_decode
    cases = [W.make_workload("tiny", "split"), W.make_workload("tiny", "nhd")]
    cases.append(W.make_workload(_spec(name="b1", num_seqs=3, num_heads=4, num_kv_heads=2,
                                       head_size=4, dtype="f32",
                                       seq_lens=(1, 15, 17), block_size=2), "nhd"))
    cases.append(W.make_workload(_spec(name="b2", num_seqs=4, num_heads=6, num_kv_heads=3,
                                       head_size=8, dtype="f16",
                                       seq_lens=(16, 511, 513, 1025), alibi=True), "split"))
    cases.append(W.make_workload(_spec(name="b3", num_seqs=3, num_heads=2, num_kv_heads=1,
                                       head_size=8, dtype="bf16", seq_lens=(512, 4, 600),
                                       softcap=3.0, value_mult=3.0, block_size=4), "split"))
    cases.append(W.make_workload(_spec(name="b4", num_seqs=2, num_heads=4, num_kv_heads=4,
                                       head_size=4, dtype="f32", seq_lens=(5, 1030),
                                       block_size=1, alibi=True, softcap=5.0), "split"))
    for w in cases:
        r = run(w)
        b = brute_decode(w)
        what = f"{w.name}/{w.layout}"
        _close(r["out"], b["out"], what=what + " out")
        _close(r["out_v2"], b["out"], what=what + " out_v2")
        _close(r["max_logits"], b["max_logits"], what=what + " max_logits")
        _close(r["exp_sums"], b["exp_sums"], what=what + " exp_sums")
        _close(r["tmp_out"], b["tmp_out"], what=what + " tmp_out")


def pin_sdpa(run):
    """Identity block table, no ALiBi / softcap: equals torch SDPA in fp64 with
    the kv heads repeat-interleaved to the query heads."""
    import torch
    for dtype, layout, H, Hkv, d in (("f32", "split", 4, 2, 8), ("f16", "nhd", 6, 2, 16),
                                     ("bf16", "split", 8, 8, 16), ("f16", "split", 4, 1, 8)):
        spec = _spec(name="sdpa", num_seqs=3, num_heads=H, num_kv_heads=Hkv, head_size=d,
                     dtype=dtype, seq_lens=(1, 300, 777))
        spec.poison = False
        w = W.make_workload(spec, layout)
        w = _clone(w, block_tables=_identity_tables(w))
        r = run(w)
        k_log, v_log = _logical_kv(w)
        q = W.storage_to_f64(w.query, w.dtype)
        off = 0
        for s in range(w.num_seqs):
            L = int(w.seq_lens[s])
            nb = -(-L // w.block_size)
            ks = k_log[off:off + nb].transpose(0, 2, 1, 3).reshape(nb * w.block_size, Hkv, d)[:L]
            vs = v_log[off:off + nb].transpose(0, 2, 1, 3).reshape(nb * w.block_size, Hkv, d)[:L]
            off += nb
            kt = torch.from_numpy(np.ascontiguousarray(ks.transpose(1, 0, 2)))
            vt = torch.from_numpy(np.ascontiguousarray(vs.transpose(1, 0, 2)))
            kt = kt.repeat_interleave(H // Hkv, dim=0)
            vt = vt.repeat_interleave(H // Hkv, dim=0)
            qt = torch.from_numpy(np.ascontiguousarray(q[s]))[:, None, :]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, kt, vt, scale=w.scale)[:, 0, :].numpy()
            _close(r["out"][s], ref, rtol=1e-9, atol=1e-12, what=f"sdpa {dtype}/{layout} seq {s}")


def pin_partitioned_equals_dense(run):
    """The Phase 2 reduce of the partition statistics equals the dense softmax."""
    for alibi, cap, mult in ((False, 0.0, 1.0), (True, 0.0, 1.0), (False, 4.0, 3.0)):
        w = W.make_workload(_spec(name="pd", num_seqs=4, num_heads=4, num_kv_heads=2,
                                  head_size=16, dtype="f16", seq_lens=(512, 513, 1600, 2049),
                                  alibi=alibi, softcap=cap, value_mult=mult), "split")
        r = run(w)
        _close(r["out_v2"], r["out"], rtol=1e-10, atol=1e-13, what="partitioned vs dense")
        # the partition statistics, recombined, give the dense normaliser
        for s in range(w.num_seqs):
            P = -(-int(w.seq_lens[s]) // 512)
            assert np.all(np.isfinite(r["max_logits"][s, :, :P]))


def pin_seq_len_one(run):
    """seq_len 1: output is that token's V row, exp_sum 1, max_logit its logit."""
    w = W.make_workload(_spec(name="one", num_seqs=3, num_heads=4, num_kv_heads=2,
                              head_size=16, dtype="f16", seq_lens=(1, 1, 1), alibi=True),
                        "split")
    r = run(w)
    k_log, v_log = _logical_kv(w)
    q = W.storage_to_f64(w.query, w.dtype)
    group = w.num_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        blk = int(w.block_tables[s, 0])
        for h in range(w.num_heads):
            kvh = h // group
            _close(r["out"][s, h], v_log[blk, kvh, 0], what="seq_len 1 out")
            logit = w.scale * float(np.dot(q[s, h], k_log[blk, kvh, 0]))  # ALiBi at t=0 adds 0
            _close(r["max_logits"][s, h, 0], logit, what="seq_len 1 max_logit")
            _close(r["exp_sums"][s, h, 0], 1.0, what="seq_len 1 exp_sum")


def pin_identical_v_rows(run):
    """All V rows of a kv head equal to one row r: the output is r."""
    w = W.make_workload(_spec(name="iv", num_seqs=2, num_heads=4, num_kv_heads=2,
                              head_size=8, dtype="f32", seq_lens=(700, 33), alibi=True),
                        "split")
    k_log, v_log = _logical_kv(w)
    rows = np.array([[0.5, -1.25, 2.0, 0.0, 3.5, -0.75, 1.0, 0.125],
                     [-2.0, 0.25, 0.0, 1.5, -3.0, 0.5, 4.0, -1.0]])
    v_new = np.empty_like(v_log)
    v_new[:] = rows[None, :, None, :]
    w = _from_logical(w, np.nan_to_num(k_log), v_new)
    r = run(w)
    for h in range(w.num_heads):
        _close(r["out"][:, h], np.broadcast_to(rows[h // 2], (2, 8)), rtol=1e-13,
               what="identical V rows")


def pin_pool_permutation(run):
    """Moving the physical blocks and rewriting the table leaves the result bit-identical."""
    w = W.make_workload(_spec(name="perm", num_seqs=3, num_heads=4, num_kv_heads=2,
                              head_size=8, dtype="bf16", seq_lens=(40, 513, 1000)), "split")
    r1 = run(w)
    rng = np.random.default_rng(5)
    pi = rng.permutation(w.num_blocks)
    kc = np.empty_like(w.key_cache)
    vc = np.empty_like(w.value_cache)
    kc[pi] = w.key_cache
    vc[pi] = w.value_cache
    w2 = _clone(w, key_cache=kc, value_cache=vc, block_tables=pi[w.block_tables].astype(np.int32))
    r2 = run(w2)
    for key in ("out", "max_logits", "exp_sums"):
        assert np.array_equal(r1[key], r2[key], equal_nan=True), key


def pin_split_equals_nhd(run):
    """The split layout and the NHD layout of the same logical cache give the same result."""
    for dtype in ("f32", "f16"):
        spec = _spec(name="lay", num_seqs=2, num_heads=4, num_kv_heads=2, head_size=16,
                     dtype=dtype, seq_lens=(100, 530))
        a = run(W.make_workload(spec, "split"))
        b = run(W.make_workload(spec, "nhd"))
        for key in ("out", "max_logits", "exp_sums"):
            assert np.array_equal(a[key], b[key], equal_nan=True), (dtype, key)


def pin_zero_query(run):
    """q = 0: uniform weights, so out = mean of V, max_logit 0, exp_sum = partition length."""
    w = W.make_workload(_spec(name="zq", num_seqs=2, num_heads=2, num_kv_heads=1,
                              head_size=8, dtype="f16", seq_lens=(515, 1024)), "nhd")
    w = _clone(w, query=np.zeros_like(w.query))
    r = run(w)
    _, v_log = _logical_kv(w)
    for s in range(w.num_seqs):
        L = int(w.seq_lens[s])
        nb = -(-L // w.block_size)
        vs = v_log[w.block_tables[s, :nb], 0].reshape(nb * w.block_size, -1)[:L]
        for h in range(w.num_heads):
            _close(r["out"][s, h], vs.mean(axis=0), rtol=1e-12, atol=1e-14, what="q=0 mean")
            P = -(-L // 512)
            lens = [min(512, L - 512 * p) for p in range(P)]
            _close(r["exp_sums"][s, h, :P], lens, what="q=0 exp_sums")
            _close(r["max_logits"][s, h, :P], np.zeros(P), what="q=0 max_logits")


def pin_exp_sum_bounds(run):
    """1 <= exp_sum_p <= tokens in partition p; unused partitions are -inf / 0."""
    w = W.make_workload(_spec(name="eb", num_seqs=3, num_heads=4, num_kv_heads=2,
                              head_size=16, dtype="f16", seq_lens=(3, 600, 1500),
                              value_mult=2.0), "split")
    r = run(w)
    for s in range(w.num_seqs):
        L = int(w.seq_lens[s])
        P = -(-L // 512)
        for p in range(r["exp_sums"].shape[2]):
            e = r["exp_sums"][s, :, p]
            if p < P:
                n = min(512, L - 512 * p)
                assert np.all(e >= 1.0 - 1e-12) and np.all(e <= n + 1e-9), (s, p, e)
            else:
                assert np.all(e == 0.0) and np.all(np.isneginf(r["max_logits"][s, :, p]))


def pin_softcap(run):
    """Two tokens with logits a and 0: weights sigmoid(c), 1 - sigmoid(c) with
    c = cap * tanh(a / cap); every max_logit stays below cap."""
    spec = _spec(name="cap", num_seqs=1, num_heads=1, num_kv_heads=1, head_size=4,
                 dtype="f32", seq_lens=(2,), softcap=2.0)
    spec.poison = False
    w = W.make_workload(spec, "nhd")
    w = _clone(w, block_tables=_identity_tables(w), scale=1.0)
    k = np.zeros((w.num_blocks, 1, w.block_size, 4))
    v = np.zeros_like(k)
    k[0, 0, 0, 0] = 3.0
    v[0, 0, 0, 0] = 1.0
    v[0, 0, 1, 1] = 1.0
    w = _from_logical(w, k, v)
    w = _clone(w, query=np.array([[[1.0, 0, 0, 0]]], dtype=np.float32))
    r = run(w)
    c = 2.0 * math.tanh(3.0 / 2.0)
    sig = 1.0 / (1.0 + math.exp(-c))
    _close(r["out"][0, 0, :2], [sig, 1.0 - sig], rtol=1e-13, what="softcap two-token")
    _close(r["max_logits"][0, 0, 0], c, what="softcap max_logit")
    _close(r["exp_sums"][0, 0, 0], 1.0 + math.exp(-c), what="softcap exp_sum")
    # large logits stay below the cap
    w2 = W.make_workload(_spec(name="cap2", num_seqs=2, num_heads=4, num_kv_heads=2,
                               head_size=16, dtype="bf16", seq_lens=(300, 900),
                               softcap=5.0, value_mult=4.0), "split")
    r2 = run(w2)
    ml = r2["max_logits"][np.isfinite(r2["max_logits"])]
    assert ml.max() <= 5.0 and ml.max() > 4.0


def pin_two_token_softmax(run):
    """Logits 1 and 0, V rows e0 and e1: out = (sigmoid(1), 1 - sigmoid(1))."""
    spec = _spec(name="two", num_seqs=1, num_heads=1, num_kv_heads=1, head_size=4,
                 dtype="f32", seq_lens=(2,))
    spec.poison = False
    w = W.make_workload(spec, "split")
    w = _clone(w, block_tables=_identity_tables(w), scale=0.5)
    k = np.zeros((w.num_blocks, 1, w.block_size, 4))
    v = np.zeros_like(k)
    k[0, 0, 0, 2] = 1.0
    v[0, 0, 0, 0] = 1.0
    v[0, 0, 1, 1] = 1.0
    w = _from_logical(w, k, v)
    w = _clone(w, query=np.array([[[0, 0, 2.0, 0]]], dtype=np.float32))
    r = run(w)
    sig = 1.0 / (1.0 + math.exp(-1.0))
    _close(r["out"][0, 0], [sig, 1.0 - sig, 0.0, 0.0], rtol=1e-14, atol=1e-15, what="two-token")
    _close(r["max_logits"][0, 0, 0], 1.0, what="two-token max_logit")
    _close(r["exp_sums"][0, 0, 0], 1.0 + math.exp(-1.0), what="two-token exp_sum")


def pin_alibi_closed_form(run):
    """q = 0 with ALiBi: logit of token t is slope * t (absolute position), so the
    weights are geometric, r^t with r = e^slope; with V_t = (1, t, 0, 0):
    out = (1, sum t r^t / sum r^t, 0, 0); per partition max_logit = slope*(last
    token) and exp_sum = (1 - e^{-slope n}) / (1 - e^{-slope})."""
    spec = _spec(name="alibi", num_seqs=1, num_heads=2, num_kv_heads=1, head_size=4,
                 dtype="f32", seq_lens=(1100,), alibi=True)
    spec.poison = False
    w = W.make_workload(spec, "nhd")
    w = _clone(w, block_tables=_identity_tables(w), query=np.zeros_like(w.query))
    L = 1100
    nb = -(-L // w.block_size)
    k = np.zeros((w.num_blocks, 1, w.block_size, 4))
    v = np.zeros_like(k)
    t = np.arange(nb * w.block_size)
    v[:nb, 0, :, 0] = 1.0
    v[:nb, 0, :, 1] = t.reshape(nb, w.block_size)
    w = _from_logical(w, k, v)
    r = run(w)
    for h in range(2):
        sl = float(w.alibi_slopes[h])
        rr = math.exp(sl)
        denom = (rr ** L - 1.0) / (rr - 1.0)
        num = rr * (1.0 - L * rr ** (L - 1) + (L - 1) * rr ** L) / (1.0 - rr) ** 2
        _close(r["out"][0, h], [1.0, num / denom, 0.0, 0.0], rtol=1e-9, atol=1e-12,
               what="alibi closed form")
        for p in range(3):
            n = min(512, L - 512 * p)
            _close(r["max_logits"][0, h, p], sl * (512 * p + n - 1), what="alibi max_logit")
            _close(r["exp_sums"][0, h, p], (1 - math.exp(-sl * n)) / (1 - math.exp(-sl)),
                   rtol=1e-10, what="alibi exp_sum")


def pin_gqa_mapping(run):
    """Query head h reads kv head h // (num_heads / num_kv_heads): give each kv head
    a constant V row equal to its index; out[h] = h // group."""
    w = W.make_workload(_spec(name="gqa", num_seqs=1, num_heads=6, num_kv_heads=3,
                              head_size=4, dtype="f32", seq_lens=(40,)), "split")
    k_log, v_log = _logical_kv(w)
    v_new = np.zeros_like(v_log)
    for kvh in range(3):
        v_new[:, kvh] = kvh
    w = _from_logical(w, np.nan_to_num(k_log), v_new)
    r = run(w)
    for h in range(6):
        _close(r["out"][0, h], np.full(4, h // 2), what="gqa mapping")


def pin_poison_never_read(run):
    """Spare pool blocks, unused table entries and tail slots hold NaN; the
    result is finite."""
    for layout in ("split", "nhd"):
        r = run(W.make_workload("tiny", layout))
        for key in ("out", "exp_sums", "tmp_out"):
            assert np.all(np.isfinite(r[key])), key


def pin_partitions_at_100k(run):
    """The pages' partition count at 100K tokens: 195 full 512-token partitions
    plus one of 160 tokens (q = 0 makes exp_sum the partition length)."""
    g = GOLDEN["partitions_at_100k"]
    spec = _spec(name="p100k", num_seqs=1, num_heads=1, num_kv_heads=1, head_size=4,
                 dtype="f32", seq_lens=(g["seq_len"],))
    w = W.make_workload(spec, "nhd")
    w = _clone(w, query=np.zeros_like(w.query))
    r = run(w, max_num_partitions=g["num_partitions"] + 1)
    es = r["exp_sums"][0, 0]
    assert int(np.sum(es == GOLDEN["partition_size"]["value"])) == g["full_partitions"]
    assert es[g["num_partitions"] - 1] == g["last_partition_tokens"]
    assert es[g["num_partitions"]] == 0.0
    assert int(np.sum(np.isfinite(r["max_logits"][0, 0]))) == g["num_partitions"]


def pin_sliding_window(run):
    """Sliding window (query at position L-1 sees keys t >= L-1-W): matches the
    brute force; W >= L-1 is bit-identical to no window; W = 0 returns the last
    V row with exp_sum 1 in the last partition and every other partition unused;
    q = 0 gives the mean of V over the window and exp_sum = in-window tokens."""
    from oracle.brute import brute_decode
    spec = _spec(name="win", num_seqs=3, num_heads=4, num_kv_heads=2, head_size=8,
                 dtype="f16", seq_lens=(1, 513, 1100), alibi=True)
    base = W.make_workload(spec, "split")
    for wl in (0, 5, 511, 600, 2000):
        w = _clone(base, window_left=wl)
        r = run(w)
        b = brute_decode(w)
        _close(r["out"], b["out"], what=f"window {wl} out")
        _close(r["max_logits"], b["max_logits"], what=f"window {wl} max_logits")
        _close(r["exp_sums"], b["exp_sums"], what=f"window {wl} exp_sums")
    r_none = run(base)
    r_big = run(_clone(base, window_left=1099))
    for key in ("out", "max_logits", "exp_sums"):
        assert np.array_equal(r_none[key], r_big[key], equal_nan=True), key
    r0 = run(_clone(base, window_left=0))
    _, v_log = _logical_kv(base)
    group = base.num_heads // base.num_kv_heads
    for s in range(base.num_seqs):
        L = int(base.seq_lens[s])
        blk = int(base.block_tables[s, (L - 1) // base.block_size])
        P = -(-L // 512)
        for h in range(base.num_heads):
            _close(r0["out"][s, h], v_log[blk, h // group, (L - 1) % base.block_size],
                   what="window 0 out")
            _close(r0["exp_sums"][s, h, P - 1], 1.0, what="window 0 exp_sum")
            assert np.all(r0["exp_sums"][s, h, :P - 1] == 0.0)
            assert np.all(np.isneginf(r0["max_logits"][s, h, :P - 1]))
    wq = _clone(base, query=np.zeros_like(base.query), alibi_slopes=None, window_left=600)
    rq = run(wq)
    for s in range(base.num_seqs):
        L = int(base.seq_lens[s])
        lo = max(0, L - 1 - 600)
        nb = -(-L // base.block_size)
        vs = v_log[base.block_tables[s, :nb], 0].reshape(nb * base.block_size, -1)[lo:L]
        _close(rq["out"][s, 0], vs.mean(axis=0), rtol=1e-12, atol=1e-14, what="window q=0 mean")
        for p in range(-(-L // 512)):
            n = max(0, min(512 * p + 512, L) - max(512 * p, lo))
            _close(rq["exp_sums"][s, 0, p], float(n), what="window q=0 exp_sum")


def pin_fp8_cache(run):
    """fp8 caches: every bit pattern decodes as torch's fp8 conversion does
    (seq_len 1, q = 0: the output is v_scale * the V row); k_scale scales the
    logits and v_scale the output linearly; an fp8 cache gives the result of an
    fp32 cache holding its decoded, scaled values; the brute force agrees."""
    import torch
    from oracle.brute import brute_decode
    for kind, tdt in (("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)):
        spec = _spec(name="fp8bits", num_seqs=16, num_heads=1, num_kv_heads=1, head_size=16,
                     dtype="f16", seq_lens=(1,) * 16, kv_dtype=kind)
        spec.poison = False
        w = W.make_workload(spec, "nhd")
        bits = np.arange(256, dtype=np.uint8).reshape(16, 16)
        vc = np.zeros_like(w.value_cache)
        for s in range(16):
            vc[w.block_tables[s, 0], 0, 0, :] = bits[s]
        w = _clone(w, value_cache=vc, query=np.zeros_like(w.query), v_scale=1.0)
        r = run(w)
        expect = torch.from_numpy(bits.copy()).view(tdt).double().numpy()
        got = r["out"][:, 0, :]
        assert np.array_equal(np.isnan(got), np.isnan(expect)), kind
        fin = ~np.isnan(expect)
        assert np.array_equal(got[fin], expect[fin]), kind
    spec = _spec(name="fp8", num_seqs=3, num_heads=4, num_kv_heads=2, head_size=16, dtype="bf16",
                 seq_lens=(1, 300, 700), kv_dtype="e4m3", k_scale=2.0 ** -5, v_scale=2.0 ** -4)
    w = W.make_workload(spec, "split")
    r = run(w)
    b = brute_decode(w)
    _close(r["out"], b["out"], what="fp8 brute out")
    _close(r["max_logits"], b["max_logits"], what="fp8 brute max_logits")
    # linearity in the scales: seq_len 1 logit ~ k_scale, output ~ v_scale
    r2 = run(_clone(w, k_scale=2 * w.k_scale, v_scale=3 * w.v_scale))
    _close(r2["max_logits"][0], 2 * r["max_logits"][0], rtol=1e-14, what="k_scale linear")
    _close(r2["out"][0], 3 * r["out"][0], rtol=1e-14, what="v_scale linear")
    # same logical values in an fp32 cache (split layout with x = 4)
    k8 = W.storage_to_f64(w.key_cache, "e4m3").transpose(0, 1, 3, 2, 4).reshape(
        w.num_blocks, 2, w.block_size, 16) * w.k_scale
    v8 = W.storage_to_f64(w.value_cache, "e4m3").transpose(0, 1, 3, 2) * w.v_scale
    q32 = W.storage_to_f64(w.query, "bf16").astype(np.float32)
    w32 = _clone(w, dtype="f32", kv_dtype=None, k_scale=1.0, v_scale=1.0, query=q32)
    w32 = _from_logical(w32, k8, v8)
    r32 = run(w32)
    _close(r["out"], r32["out"], rtol=1e-12, what="fp8 vs decoded fp32 cache")
    _close(r["exp_sums"], r32["exp_sums"], rtol=1e-12, what="fp8 vs decoded fp32 exp_sums")


def pin_multi_token(run):
    """Several query tokens per sequence: matches the brute force; query token i
    equals the single-token decode of the sequence cut after its position (bit
    for bit); one token per sequence through query_start equals the default."""
    from oracle.brute import brute_decode
    spec = _spec(name="mq", num_seqs=4, num_heads=4, num_kv_heads=2, head_size=8, dtype="f16",
                 seq_lens=(3, 514, 1024, 1100), alibi=True, q_len=3)
    w = W.make_workload(spec, "split")
    for wl in (-1, 600):
        ww = _clone(w, window_left=wl)
        r = run(ww)
        b = brute_decode(ww)
        _close(r["out"], b["out"], what=f"multi-token brute (window {wl})")
        _close(r["max_logits"], b["max_logits"], what="multi-token max_logits")
        _close(r["exp_sums"], b["exp_sums"], what="multi-token exp_sums")
        qs = ww.query_start
        for s in range(ww.num_seqs):
            qn = int(qs[s + 1] - qs[s])
            for qi in range(qn):
                row = int(qs[s]) + qi
                one = _clone(ww, num_seqs=1, query_start=None, block_tables=ww.block_tables[s:s + 1],
                             seq_lens=np.array([int(ww.seq_lens[s]) - qn + 1 + qi], dtype=np.int32),
                             query=ww.query[row:row + 1])
                r1 = run(one, max_num_partitions=r["max_logits"].shape[2])
                for key in ("out", "max_logits", "exp_sums"):
                    assert np.array_equal(r[key][row], r1[key][0], equal_nan=True), (s, qi, key)
    w1 = W.make_workload(_spec(name="mq1", num_seqs=3, num_heads=4, num_kv_heads=2, head_size=8,
                               dtype="bf16", seq_lens=(5, 600, 1030), q_len=1), "nhd")
    a = run(w1)
    b = run(_clone(w1, query_start=None))
    for key in ("out", "max_logits", "exp_sums"):
        assert np.array_equal(a[key], b[key], equal_nan=True), key


ALL_PINS = [
    pin_brute, pin_sdpa, pin_partitioned_equals_dense, pin_seq_len_one,
    pin_identical_v_rows, pin_pool_permutation, pin_split_equals_nhd, pin_zero_query,
    pin_exp_sum_bounds, pin_softcap, pin_two_token_softmax, pin_alibi_closed_form,
    pin_gqa_mapping, pin_poison_never_read, pin_partitions_at_100k, pin_sliding_window,
    pin_fp8_cache, pin_multi_token,
]


def run_all(lib_path=None):
    """Run every pin against an oracle build; returns {pin name: error or None}."""
    import oracle

    def run(w, **kw):
        return oracle.oracle_decode(w, lib_path=lib_path, **kw)

    res = {}
    for pin in ALL_PINS:
        try:
            with np.errstate(invalid="ignore"):
                pin(run)
            res[pin.__name__] = None
        except Exception as e:  # noqa: BLE001 -- a planted mistake may raise anything
            res[pin.__name__] = f"{type(e).__name__}: {e}"
    return res


if __name__ == "__main__":
    out = run_all(sys.argv[1] if len(sys.argv) > 1 else None)
    failed = [k for k, v in out.items() if v]
    print(json.dumps(out))
    sys.exit(1 if failed else 0)

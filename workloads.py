"""Seeded synthetic inputs for paged-KV decode attention.

This module is the one piece shared by the CUDA path's tests/bench and by the
fp64 oracle: it draws the query, the paged K/V pool, the block tables and the
sequence lengths, rounds them to the storage dtype and lays them out.  It holds
none of the attention arithmetic.

Workloads (sizes from the paged_attention_v2 problem statement of
"paged_attention_v2_pytorch.py -- BI-V100 PagedAttention V2 implementation"
and the AttnDispatchConfig defaults of "ex_engine/factors/attn_dispatch.py"):

  tiny         2 seqs, lens {37, 600}, 4 heads / 2 kv heads, d=64, fp32
  gqa4k        32 x 4096, 28 / 4 heads, d=128, fp16
  long100k     4 x 100000 (196 partitions of 512), 28 / 4 heads, d=128, bf16
  ragged       256 seqs, lens log-uniform in [1, 32768], 32 / 8 heads, d=128,
               fp16, ALiBi slopes 2^(-8(i+1)/32)
  large_batch  128 x 16384, 64 / 8 heads, d=128, bf16 with Q/K/V scaled x2,
               logit softcap 30

Recipe: numpy PCG64 streams keyed by (seed, stream name, chunk); values are
N(0,1) fp32 draws (times the workload's multiplier), rounded to the storage
dtype with round-to-nearest-even.  Physical blocks are assigned to sequences
through a seeded permutation of the pool.  Pool blocks that no sequence uses
and the unused slots of each sequence's last block are filled with NaN, and
unused block-table entries point at a NaN block, so that any read past the
valid tokens shows up in the output.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BLOCK_SIZE = 16
PARTITION_SIZE = 512

DTYPES = ("f32", "f16", "bf16")
LAYOUTS = ("split", "nhd")

# storage numpy dtype per dtype name (bf16 is carried as raw uint16 bits)
_STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "e4m3": np.uint8,
            "e5m2": np.uint8}
_ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1, "e5m2": 1}
_NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "e4m3": 0x7F, "e5m2": 0x7E}
KV_FP8 = ("e4m3", "e5m2")

# blocks generated per RNG chunk; fixed so values do not depend on memory limits
_CHUNK_BLOCKS = 512


@dataclass
class Spec:
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    dtype: str
    seq_lens: Optional[list] = None       # explicit lengths
    seq_len: Optional[int] = None         # uniform length
    log_uniform_max: Optional[int] = None # lens = clamp(round(2^(log2(max) u)), 1, max)
    block_size: int = BLOCK_SIZE
    pool_blocks: Optional[int] = None     # None: exactly the blocks in use (+1 NaN block if needed)
    value_mult: float = 1.0
    alibi: bool = False
    softcap: float = 0.0
    seed_index: int = 0
    poison: bool = True
    kv_dtype: Optional[str] = None        # "e4m3" / "e5m2": fp8 cache holding K / k_scale, V / v_scale
    k_scale: float = 1.0
    v_scale: float = 1.0
    q_len: object = None                  # query tokens per sequence (int or list); None = 1


SPECS = {
    "tiny": Spec("tiny", 2, 4, 2, 64, "f32", seq_lens=[37, 600], pool_blocks=64, seed_index=0),
    "gqa4k": Spec("gqa4k", 32, 28, 4, 128, "f16", seq_len=4096, seed_index=1),
    "long100k": Spec("long100k", 4, 28, 4, 128, "bf16", seq_len=100000, seed_index=2),
    "ragged": Spec("ragged", 256, 32, 8, 128, "f16", log_uniform_max=32768, alibi=True,
                   seed_index=3),
    "large_batch": Spec("large_batch", 128, 64, 8, 128, "bf16", seq_len=16384, value_mult=2.0,
                        softcap=30.0, seed_index=4),
    # fp8 KV caches (kv_cache_dtype / k_scale / v_scale): the 4K and 100K workloads
    "gqa4k_fp8": Spec("gqa4k_fp8", 32, 28, 4, 128, "f16", seq_len=4096, seed_index=5,
                      kv_dtype="e4m3", k_scale=2.0 ** -6, v_scale=2.0 ** -6),
    "long100k_fp8": Spec("long100k_fp8", 4, 28, 4, 128, "bf16", seq_len=100000, seed_index=6,
                         kv_dtype="e4m3", k_scale=2.0 ** -6, v_scale=2.0 ** -6),
    # several query tokens per sequence (speculative decoding: 4 drafted tokens
    # verified at once): 32 x 4096, 32/8 heads (group 4, 16 rows per tile)
    "spec4k": Spec("spec4k", 32, 32, 8, 128, "bf16", seq_len=4096, seed_index=7, q_len=4),
    # the same with an fp8 e4m3 KV cache
    "spec4k_fp8": Spec("spec4k_fp8", 32, 32, 8, 128, "bf16", seq_len=4096, seed_index=10, q_len=4,
                       kv_dtype="e4m3", k_scale=2.0 ** -6, v_scale=2.0 ** -6),
    # fp32 query and cache: the 4K and 100K shapes (tf32 tensor-core path, 1e-5 tolerance)
    "gqa4k_f32": Spec("gqa4k_f32", 32, 28, 4, 128, "f32", seq_len=4096, seed_index=8),
    "long100k_f32": Spec("long100k_f32", 4, 28, 4, 128, "f32", seq_len=100000, seed_index=9),
}

DESCRIPTIONS = {
    "tiny": "2 seqs, lens {37,600}, 4/2 heads, d=64, fp32, pool 64 blocks (NaN-poisoned spares)",
    "gqa4k": "GQA decode: 32 seqs x 4096, 28/4 heads, d=128, block 16, fp16",
    "long100k": "long context: 4 seqs x 100000 (196 partitions), 28/4 heads, d=128, block 16, bf16",
    "ragged": "ragged batch: 256 seqs, lens log-uniform [1,32768], 32/8 heads, d=128, fp16, ALiBi",
    "large_batch": "large batch: 128 seqs x 16384, 64/8 heads, d=128, bf16 (x2), softcap 30",
    "gqa4k_fp8": "GQA decode, fp8 e4m3 KV cache (scales 2^-6): 32 seqs x 4096, 28/4 heads, d=128, fp16 query",
    "long100k_fp8": "long context, fp8 e4m3 KV cache (scales 2^-6): 4 seqs x 100000, 28/4 heads, d=128, bf16 query",
    "spec4k": "speculative decode: 32 seqs x 4096 with 4 query tokens each (causal), 32/8 heads, d=128, bf16",
    "spec4k_fp8": "speculative decode, fp8 e4m3 KV cache (scales 2^-6): 32 seqs x 4096 with 4 query tokens each, 32/8 heads, d=128, bf16 query",
    "gqa4k_f32": "GQA decode, fp32 query and KV: 32 seqs x 4096, 28/4 heads, d=128",
    "long100k_f32": "long context, fp32 query and KV: 4 seqs x 100000, 28/4 heads, d=128",
}


@dataclass
class Workload:
    name: str
    dtype: str
    layout: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    max_seq_len: int
    scale: float
    softcap: float
    query: np.ndarray
    key_cache: np.ndarray
    value_cache: np.ndarray
    block_tables: np.ndarray
    seq_lens: np.ndarray
    alibi_slopes: Optional[np.ndarray]
    meta: dict = field(default_factory=dict)
    window_left: int = -1  # sliding window: keys t >= seq_len - 1 - window_left (-1 = none)
    kv_dtype: Optional[str] = None  # fp8 cache type, None = same as dtype
    k_scale: float = 1.0
    v_scale: float = 1.0
    # several query tokens per sequence: query rows of sequence s are
    # query_start[s] .. query_start[s+1]-1; None = one row per sequence
    query_start: Optional[np.ndarray] = None

    @property
    def num_query_tokens(self) -> int:
        return self.num_seqs if self.query_start is None else int(self.query_start[-1])

    @property
    def max_query_len(self) -> int:
        return 1 if self.query_start is None else int(np.diff(self.query_start).max(initial=0))

    @property
    def cache_dtype(self) -> str:
        return self.kv_dtype or self.dtype

    @property
    def elem_bytes(self) -> int:
        """Bytes per element of the K / V caches."""
        return _ELEM_BYTES[self.cache_dtype]

    @property
    def max_num_partitions(self) -> int:
        return max(1, -(-self.max_seq_len // PARTITION_SIZE))

    @property
    def kv_bytes(self) -> int:
        """Bytes of K and V the method must read: sum_s len_s * kv_heads * d * 2 * elem."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * \
            self.head_size * 2 * self.elem_bytes


# ---------------------------------------------------------------- rounding

def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 values to the storage dtype (round-to-nearest-even)."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f32":
        return x.copy()
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        u = x.view(np.uint32)  # finite inputs: the rounding add cannot overflow 32 bits
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        return r.astype(np.uint16)
    raise ValueError(dtype)


def quantize_fp8(x: np.ndarray, kind: str) -> np.ndarray:
    """fp32 values -> fp8 bits (uint8) with torch's casts (saturated to the finite range)."""
    import torch
    lim = 448.0 if kind == "e4m3" else 57344.0
    t = torch.from_numpy(np.clip(np.asarray(x, dtype=np.float32), -lim, lim))
    tdt = torch.float8_e4m3fn if kind == "e4m3" else torch.float8_e5m2
    return t.to(tdt).view(torch.uint8).numpy()


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of storage values to float64 (for tests)."""
    if dtype in ("f32", "f16"):
        return a.astype(np.float64)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype in KV_FP8:
        import torch
        tdt = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
        return torch.from_numpy(np.ascontiguousarray(a)).view(tdt).double().numpy()
    raise ValueError(dtype)


def _nan_value(dtype: str):
    if dtype == "f32":
        return np.float32(np.nan)
    if dtype == "f16":
        return np.uint16(_NAN_BITS["f16"]).view(np.float16)
    if dtype in KV_FP8:
        return np.uint8(_NAN_BITS[dtype])
    return np.uint16(_NAN_BITS["bf16"])


def _gen_threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(32, n))


def _rng(seed: int, stream: str, chunk: int = 0) -> np.random.Generator:
    key = [seed, sum(ord(c) * 131 ** i for i, c in enumerate(stream)) % (2 ** 31), chunk]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


# ---------------------------------------------------------------- layouts

def logical_to_layout(kv: np.ndarray, which: str, layout: str, dtype: str) -> np.ndarray:
    """kv: logical [blocks, kv_heads, block_size, d] -> storage layout.

    split key   : [blocks, kv_heads, d/x, block_size, x], x = 16 / elem_bytes
    split value : [blocks, kv_heads, d, block_size]
    nhd         : [blocks, kv_heads, block_size, d]
    """
    nb, hkv, bs, d = kv.shape
    if layout == "nhd":
        return np.ascontiguousarray(kv)
    if which == "k":
        x = 16 // _ELEM_BYTES[dtype]
        return np.ascontiguousarray(kv.reshape(nb, hkv, bs, d // x, x).transpose(0, 1, 3, 2, 4))
    return np.ascontiguousarray(kv.transpose(0, 1, 3, 2))


def layout_shape(which: str, layout: str, dtype: str, nb: int, hkv: int, bs: int, d: int):
    if layout == "nhd":
        return (nb, hkv, bs, d)
    if which == "k":
        x = 16 // _ELEM_BYTES[dtype]
        return (nb, hkv, d // x, bs, x)
    return (nb, hkv, d, bs)


# ---------------------------------------------------------------- generation

def _seq_lens(spec: Spec, seed: int) -> np.ndarray:
    if spec.seq_lens is not None:
        return np.asarray(spec.seq_lens, dtype=np.int32)
    if spec.seq_len is not None:
        return np.full(spec.num_seqs, spec.seq_len, dtype=np.int32)
    u = _rng(seed, "lens").random(spec.num_seqs)
    top = math.log2(spec.log_uniform_max)
    lens = np.clip(np.rint(np.exp2(top * u)), 1, spec.log_uniform_max)
    return lens.astype(np.int32)


def alibi_slopes(num_heads: int) -> np.ndarray:
    """ALiBi slopes 2^(-8(i+1)/num_heads), fp32."""
    i = np.arange(num_heads, dtype=np.float64)
    return np.exp2(-8.0 * (i + 1) / num_heads).astype(np.float32)


def make_workload(spec, layout: str = "split", seed: Optional[int] = None,
                  shuffle_seed: Optional[int] = None) -> Workload:
    """Build a workload from a Spec or the name of one in SPECS."""
    if isinstance(spec, str):
        spec = SPECS[spec]
    assert layout in LAYOUTS and spec.dtype in DTYPES
    seed = 1234 + spec.seed_index if seed is None else seed
    shuffle_seed = 99 + spec.seed_index if shuffle_seed is None else shuffle_seed
    bs, d, hkv = spec.block_size, spec.head_size, spec.num_kv_heads
    lens = _seq_lens(spec, seed)
    max_seq_len = int(lens.max()) if len(lens) else 0
    max_blocks = max(1, -(-max_seq_len // bs))
    blocks_per_seq = (lens.astype(np.int64) + bs - 1) // bs
    used = int(blocks_per_seq.sum())
    need_spare = spec.poison and bool((blocks_per_seq < max_blocks).any())
    if spec.pool_blocks is not None:
        pool = spec.pool_blocks
        assert pool >= used + (1 if need_spare else 0), "pool too small"
    else:
        pool = used + (1 if need_spare else 0)
    perm = _rng(shuffle_seed, "perm").permutation(pool).astype(np.int32)
    assigned, spares = perm[:used], perm[used:]
    tables = np.empty((spec.num_seqs, max_blocks), dtype=np.int32)
    fill = int(spares[0]) if len(spares) else 0
    tables[:] = fill
    # valid slots per physical block (0 = block no sequence uses)
    valid_slots = np.zeros(pool, dtype=np.int32)
    off = 0
    for s in range(spec.num_seqs):
        nb = int(blocks_per_seq[s])
        tables[s, :nb] = assigned[off:off + nb]
        if nb:
            valid_slots[assigned[off:off + nb]] = bs
            tail = int(lens[s]) - (nb - 1) * bs
            valid_slots[assigned[off + nb - 1]] = tail
        off += nb

    cdt = spec.kv_dtype or spec.dtype  # storage type of the caches
    sdt = _STORAGE[cdt]
    kshape = layout_shape("k", layout, cdt, pool, hkv, bs, d)
    vshape = layout_shape("v", layout, cdt, pool, hkv, bs, d)
    key_cache = np.empty(kshape, dtype=sdt)
    value_cache = np.empty(vshape, dtype=sdt)
    nan = _nan_value(cdt)

    def fill(job):
        c0, which = job
        dst = key_cache if which == "k" else value_cache
        c1 = min(pool, c0 + _CHUNK_BLOCKS)
        n = c1 - c0
        g = _rng(seed, "kv_" + which, c0 // _CHUNK_BLOCKS)
        x = g.standard_normal((n, hkv, bs, d), dtype=np.float32)
        if spec.value_mult != 1.0:
            x *= np.float32(spec.value_mult)
        if spec.kv_dtype:
            sc = spec.k_scale if which == "k" else spec.v_scale
            st = quantize_fp8(x / np.float32(sc), spec.kv_dtype)
        else:
            st = round_to_storage(x, spec.dtype)
        if spec.poison:
            for i in np.nonzero(valid_slots[c0:c1] < bs)[0]:
                st[i, :, valid_slots[c0 + i]:, :] = nan
        dst[c0:c1] = logical_to_layout(st, which, layout, cdt)

    jobs = [(c0, which) for c0 in range(0, pool, _CHUNK_BLOCKS) for which in ("k", "v")]
    with ThreadPoolExecutor(max_workers=_gen_threads()) as ex:
        list(ex.map(fill, jobs))
    query_start = None
    rows = spec.num_seqs
    if spec.q_len is not None:
        ql = np.broadcast_to(np.asarray(spec.q_len, dtype=np.int64), (spec.num_seqs,))
        ql = np.minimum(ql, lens.astype(np.int64))  # a sequence cannot have more queries than keys
        query_start = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
        rows = int(query_start[-1])
    q = _rng(seed, "query").standard_normal((rows, spec.num_heads, d), dtype=np.float32)
    if spec.value_mult != 1.0:
        q *= np.float32(spec.value_mult)
    query = round_to_storage(q, spec.dtype)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    return Workload(
        name=spec.name, dtype=spec.dtype, layout=layout, num_seqs=spec.num_seqs,
        num_heads=spec.num_heads, num_kv_heads=hkv, head_size=d, block_size=bs,
        num_blocks=pool, max_blocks_per_seq=max_blocks, max_seq_len=max_seq_len,
        scale=scale, softcap=float(spec.softcap), query=query, key_cache=key_cache,
        value_cache=value_cache, block_tables=tables, seq_lens=lens,
        alibi_slopes=alibi_slopes(spec.num_heads) if spec.alibi else None,
        meta={"seed": seed, "shuffle_seed": shuffle_seed, "spec": spec},
        kv_dtype=spec.kv_dtype, k_scale=float(np.float32(spec.k_scale)),
        v_scale=float(np.float32(spec.v_scale)), query_start=query_start,
    )


def small_spec(name="small", num_seqs=3, num_heads=4, num_kv_heads=2, head_size=64,
               dtype="f16", seq_lens=(1, 513, 1100), alibi=False, softcap=0.0,
               value_mult=1.0, pool_extra=5, seed_index=7, block_size=BLOCK_SIZE,
               kv_dtype=None, k_scale=1.0, v_scale=1.0, q_len=None) -> Spec:
    """A Spec for tests: explicit lengths, a pool with NaN-poisoned spare blocks."""
    lens = list(seq_lens)
    used = sum(-(-l // block_size) for l in lens)
    return Spec(name, num_seqs, num_heads, num_kv_heads, head_size, dtype,
                seq_lens=lens, pool_blocks=used + pool_extra, alibi=alibi, softcap=softcap,
                value_mult=value_mult, seed_index=seed_index, block_size=block_size,
                kv_dtype=kv_dtype, k_scale=k_scale, v_scale=v_scale, q_len=q_len)

// pa_kernels.cuh -- device code of the paged decode attention path (sm_103a).
//
// Partition kernel (Phase 1 of "paged_attention_v2_pytorch.py -- BI-V100
// PagedAttention V2 implementation", and the whole v1 pass):
//   persistent CTAs walk (sequence, kv head, 512-token partition) tiles; in v1
//   mode a tile is a whole (sequence, kv head).  Warp NC is the producer: it
//   walks seq_lens with a warp scan to find its tiles, reads each tile's block
//   table slice with one coalesced warp load, and streams every K/V page of
//   the tile into a STAGES-deep shared-memory ring with bulk (TMA) copies,
//   one mbarrier per stage.  Warps 0..NC-1 consume pages round-robin: the
//   whole GQA query group of the kv head is packed into the N dimension of
//   m16n8k16 tensor-core MMAs (tokens on M for Q.K^T, head dims on M for P.V),
//   so each page is read from HBM once for all heads of the group; the softmax
//   state stays online in registers.  At the end of a tile the consumer warps
//   merge their partial (max, sum, acc) through shared memory and write the
//   partition statistics (v2) or the output row (v1).
// Reduce kernel (Phase 2): per (sequence, head), M = max_p m_p,
//   w_p = exp(m_p - M) * e_p, out = sum_p w_p tmp_p / sum_p w_p.
#pragma once

#include <stdint.h>

#include <type_traits>

#include "pa_decode.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kPart = PA_PARTITION_SIZE;  // tokens per partition
constexpr int kBS = PA_BLOCK_SIZE;        // tokens per page
constexpr int kSplit = PA_LAYOUT_SPLIT;
constexpr int kNHD = PA_LAYOUT_NHD;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legal wait (default)
constexpr float kLog2e = 1.4426950408889634f;

// Cache element kinds (template parameter KV of the partition kernel).
constexpr int kKvSame = 0;      // same 16-bit / 32-bit type as the query
constexpr int kKvE4M3 = 1;      // fp8 E4M3
constexpr int kKvE5M2 = 2;      // fp8 E5M2

// Shape of the partition kernel.  Ring stages per cache type, one 16-token
// page of K and V each.  One n-tile of 16-bit or fp32 pages: five consumer
// warps, with 10 stages (16-bit) or 5 stages of 16 KB (fp32), two CTAs of
// ~110 KB per SM; two n-tiles: four warps, 10 stages for 16-bit pages (two
// page streams of two warps, one n-tile each) or 8 stages of 16 KB for fp32
// (one CTA per SM); fp8 pages: four warps and 12 stages, so that three CTAs
// share an SM.  The stages are a multiple of the page streams.
constexpr int kStages16 = 10;      // 16-bit caches, one n-tile
constexpr int kStages16x2 = 10;    // 16-bit caches, two n-tiles (paired page streams)
constexpr int kStagesFp8 = 12;     // fp8 caches (three CTAs per SM fit)
constexpr int kStagesF32 = 5;      // fp32 caches, one n-tile (two CTAs per SM)
constexpr int kStagesF32x2 = 8;    // fp32 caches, two n-tiles (one CTA per SM)
constexpr int kConsumerWarps = 4;  // consumer warps per CTA
constexpr int kConsumerWarps5 = 5; // consumer warps per CTA, 16-bit or fp32 caches with one n-tile
constexpr int kPrefetchPages = 16; // pages of the first tile prefetched into L2 before the grid wait
constexpr int kReduceWarpMaxParts = 64;  // warp-per-row reduce up to this many partitions per row

constexpr int kReduceWarpsPerCta = 8;  // warp-per-row reduce: rows per CTA

struct Params {
    const void* query;
    const void* key_cache;
    const void* value_cache;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const float* alibi;
    void* out;
    float* exp_sums;
    float* max_logits;
    float* tmp_out;
    int32_t* dev_error;
    int num_seqs, num_heads, num_kv_heads, group;
    int num_blocks, max_blocks_per_seq, max_seq_len, max_parts;
    float scale, softcap, inv_softcap;  // scale includes k_scale for fp8 caches
    float v_scale;                       // fp8 caches: applied to the partition outputs
    int v1;
    int32_t* counters;  // [num_seqs][num_kv_heads] finished partitions (fused v2 only)
    int window_left;    // < 0: no window; else keys t >= pos - window_left (pos: the query's position)
    const int32_t* query_start;  // [num_seqs + 1] query rows per sequence, or NULL (one row each)
    int max_q_len;               // upper bound of query tokens per sequence (1 without query_start)
    int num_q_rows;              // rows of query / out / workspace
    int fused;          // v2 with the log-sum-exp merge done by the last CTA of each (seq, kv head)
    uint64_t wait_limit_ns;  // limit of every barrier wait (0: kWaitLimitNs)
    int withhold_page;       // test hook: CTA 0 withholds its first page copy (a wait runs out)
    int kv_evict_first;      // KV page copies marked evict_first (partition outputs small against L2)
    int32_t* tile_ctr;       // [2] dynamic schedule: tiles claimed, CTAs done (NULL: static schedule)
    int metadata_ready;      // block tables / lengths / query_start final: read before the grid wait
};

struct TileDesc {
    int seq, kvh, part, tok_begin, tok_end, len, flags, q0, qn, pad[3];
};
constexpr int kTileStop = 1;

__device__ __forceinline__ void report(const Params& p, int bits) {
    if (p.dev_error) atomicOr(p.dev_error, bits);
}

__device__ __forceinline__ int clamp_len(const Params& p, int raw) {
    return raw < 0 ? 0 : (raw > p.max_seq_len ? p.max_seq_len : raw);
}

// First key inside the sliding window of a query at position pos (0 without one).
__device__ __forceinline__ int window_lo_at(const Params& p, int pos) {
    if (p.window_left < 0) return 0;
    const int lo = pos - p.window_left;
    return lo > 0 ? lo : 0;
}

// First key any query token of a sequence sees: the window of its first query
// token, at position len - qn.
__device__ __forceinline__ int window_lo(const Params& p, int len, int qn = 1) {
    return window_lo_at(p, len - qn);
}

// Query rows of sequence s: first row and count, clamped to max_q_len tokens
// and to the rows that exist.
__device__ __forceinline__ void query_rows(const Params& p, int s, int& q0, int& qn) {
    if (!p.query_start) {
        q0 = s;
        qn = 1;
        return;
    }
    q0 = __ldg(p.query_start + s);
    qn = __ldg(p.query_start + s + 1) - q0;
    if (qn < 0 || qn > p.max_q_len || q0 < 0 || q0 > p.num_q_rows - min(max(qn, 0), p.max_q_len)) {
        report(p, PA_DEVERR_SEQ_LEN);
        qn = qn < 0 ? 0 : min(qn, p.max_q_len);
        if (q0 < 0 || q0 > p.num_q_rows) {
            q0 = 0;
            qn = 0;
        } else if (q0 + qn > p.num_q_rows) {
            qn = p.num_q_rows - q0;
        }
    }
}

// Pages covering tokens [tb, te): from page tb/16 to page ceil(te/16) - 1.
__device__ __forceinline__ int tile_pages(int tb, int te) {
    return te > tb ? (te + kBS - 1) / kBS - tb / kBS : 0;
}

// ------------------------------------------------------------------ config

template <typename T, int HEAD, int NT, int LAYOUT, int STAGES, int NC, int KV = kKvSame,
          bool MQ = false>
struct Cfg {
    static constexpr bool kMQ = MQ;  // several query tokens per sequence (query_start given)
    static constexpr bool kF32 = std::is_same<T, float>::value;
    static constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    static constexpr int kElem = sizeof(T);                // query / output element
    static constexpr int kKvElem = KV == kKvSame ? (int)sizeof(T) : 1;
    static constexpr int kPageBytes = kBS * HEAD * kKvElem;  // one page of K (or of V)
    // One page of K and one of V per ring stage.  (Two pages per fp8 NHD stage
    // halve its barrier rounds, max reductions and rescales, but their 8 KB
    // stages leave room for two CTAs per SM, against three with one-page
    // stages: measured, long100k_fp8 NHD 83.1 -> 75.9 µs and gqa4k_fp8 NHD
    // 34.2 -> 32.7 µs for the one-page stages.)
    static constexpr int kStageBytes = 2 * kPageBytes;  // K page, then V page
    static constexpr int kMaxG = NT * 8;                   // rows (heads x query tokens) handled
    // 16-bit caches with two n-tiles: warps in pairs of page streams, one
    // n-tile each (consumer_mma); every page is consumed by two warps.
    static constexpr bool kPairs = NT == 2 && KV == kKvSame && !kF32;
    static constexpr int kMergeRows = kPairs ? 8 : kMaxG;  // merge-buffer rows per warp
    static constexpr int kPageWarps = kPairs ? 2 : 1;      // warps that release each page
    static constexpr int kQBytes = kMaxG * HEAD * kElem;
    static constexpr int kTD = 2;                          // tile descriptor ring depth
    static constexpr int kMergeStride = HEAD + 4;          // floats; +4 breaks bank conflicts
    static constexpr int kThreads = (NC + 1) * 32;
    // NHD pages arrive through tensor maps with the 128-byte swizzle (3-D for
    // 16-bit and fp32, 2-D for fp8)
    static constexpr bool kTensorMap = LAYOUT == kNHD;
    static_assert(KV == kKvSame || !kF32, "fp8 caches: 16-bit query");

    static constexpr int oRing = 0;
    static constexpr int oQ = oRing + STAGES * kStageBytes;
    static constexpr int oMerge = oQ + kTD * kQBytes;
    static constexpr int oML = oMerge + NC * kMergeRows * kMergeStride * 4;
    static constexpr int oDesc = oML + NC * kMergeRows * 8;
    static constexpr int oBar = (oDesc + kTD * (int)sizeof(TileDesc) + 7) & ~7;
    static constexpr int oAbort = oBar + (2 * STAGES + 2 * kTD + 1) * 8;
    static constexpr int kSmemBytes = oAbort + 16 + 1024;  // + slack for 1024-B alignment

    static_assert(kPageBytes % 1024 == 0 || !kTensorMap, "swizzled pages need 1024-B alignment");
    // Within a tile, page j goes to page stream j % (NC / kPageWarps) (one
    // warp, or two with paired streams, each releasing it) and to ring stage
    // (base + j) % STAGES.  With STAGES a multiple of the streams every page of
    // a stage inside one tile belongs to the same stream, so no warp ever waits
    // on a stage's full barrier more than one phase ahead (a parity wait
    // cannot tell phase n from phase n + 2): the stage is refilled only once
    // both warps of a pair released it.  Across tiles the tile-end barrier of
    // the consumer warps gives the same guarantee.
    static_assert(STAGES % (NC / kPageWarps) == 0, "ring stages must be a multiple of the page streams");
    static_assert(STAGES <= 32, "one producer lane per stage");
    static_assert(kQBytes % 16 == 0, "bulk copy size");
};

struct Smem {
    uint32_t ring;       // shared address of stage 0
    uint32_t q;          // shared address of Q slot 0
    float* merge;
    float2* ml;
    TileDesc* desc;
    uint32_t full, empty, td_full, td_empty;  // shared addresses of barrier arrays
    uint32_t merge_bar;  // consumer warps: partial states written / epilogue reads done
    volatile int* abort;     // [0] give-up flag, [1] never set (drain waits), [2] last-arriver flag
    uint64_t wait_ns;        // limit of every barrier wait
};

// Ring stage and phase parity of the page NC pages further on (a consumer
// warp's next page of the tile): no division per page.
template <int STAGES, int NC>
__device__ __forceinline__ void advance_stage(uint32_t& st, uint32_t& ph) {
    static_assert(NC <= STAGES, "a warp's next page is at most one lap ahead");
    st += NC;
    if (st >= STAGES) {
        st -= STAGES;
        ph ^= 1u;
    }
}

// Bounded wait by every lane of a warp; the result is the same in all lanes.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
    const bool ok = mbar_wait(bar, parity, abort, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Barrier among the NC consumer warps on an mbarrier of count NC (bounded,
// unlike bar.sync, so a warp that gave up cannot strand the others).
__device__ __forceinline__ bool consumer_sync(const Smem& sm, uint32_t& phase, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.merge_bar);
    const bool ok = warp_wait(sm.merge_bar, phase & 1, sm.abort, sm.wait_ns);
    ++phase;
    return ok;
}

// ------------------------------------------------------------------ producer

// The (sequence, partition) of tile unit u when every sequence of the batch
// has max_parts partitions and there is no window (v1: one unit per
// sequence).  The producer's walk of seq_lens finds the real one; this guess
// lets the first tile's loads start before that walk.
__device__ __forceinline__ void guess_unit(const Params& p, int u, int& seq, int& part) {
    if (p.v1) {
        seq = u;
        part = 0;
    } else {
        seq = u / p.max_parts;
        part = u - seq * p.max_parts;
    }
}

// Run before the wait for the previous grid in the stream (programmatic
// dependent launch), while that grid finishes: prefetch into L2 the first
// pages of K and V of this CTA's first tile (guessed as above) and its query
// rows.  The inputs may still be written by the previous grid, so everything
// read here only steers the prefetch: lengths and block ids are read through
// L2 only (no L1 line is left behind for the reads after the wait), lengths
// are clamped and block ids outside the pool are skipped.
template <class C, int HEAD>
__device__ void prefetch_first_tile(const Params& p, int lane) {
    if (p.window_left >= 0 || p.withhold_page) return;
    const int Hkv = p.num_kv_heads;
    const int u = (int)blockIdx.x / Hkv, kvh = (int)blockIdx.x - u * Hkv;
    int seq, part;
    guess_unit(p, u, seq, part);
    if (seq >= p.num_seqs) return;
    const int len = clamp_len(p, __ldcg(p.seq_lens + seq));
    const int tb = part * kPart;
    const int te = p.v1 ? len : min(len, tb + kPart);
    const int npg = min(kPrefetchPages, tile_pages(tb, te));
    if (lane < npg) {
        const int blk = __ldcg(p.block_tables + (int64_t)seq * p.max_blocks_per_seq + tb / kBS + lane);
        if ((unsigned)blk < (unsigned)p.num_blocks) {
            const int64_t off = ((int64_t)blk * Hkv + kvh) * C::kPageBytes;
            bulk_prefetch_l2(static_cast<const char*>(p.key_cache) + off, C::kPageBytes);
            bulk_prefetch_l2(static_cast<const char*>(p.value_cache) + off, C::kPageBytes);
        }
    }
    if (!C::kMQ && lane == 31)
        bulk_prefetch_l2(static_cast<const char*>(p.query) +
                             ((int64_t)seq * p.num_heads + (int64_t)kvh * p.group) * HEAD * C::kElem,
                         (uint32_t)(p.group * HEAD * C::kElem));
}

struct ProducerTile {
    int seq, kvh, part, tb, te, len, npages, q0, qn;
    bool valid;
};

template <class C, int HEAD, int STAGES>
__device__ void producer(const Params& p, const Smem& sm, const CUtensorMap* tmk,
                         const CUtensorMap* tmv, int lane) {
    const int S = p.num_seqs, Hkv = p.num_kv_heads;
    const char* kbase = static_cast<const char*>(p.key_cache);
    const char* vbase = static_cast<const char*>(p.value_cache);
    const char* qbase = static_cast<const char*>(p.query);
    const uint32_t qbytes = (uint32_t)(p.group * HEAD * C::kElem);
    // KV pages are read once: first to leave L2, ahead of the partition outputs
    // (measured: a gain while those fit in L2, a loss once they overflow it)
    const uint64_t kvpol = p.kv_evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();

    // Walk of seq_lens in chunks of 32 sequences: lane i holds sequence cb+i.
    int cb = 0, cu = 0;  // first sequence of the chunk, tile units before the chunk
    int c_len = 0, c_units = 0, c_p0 = 0, c_q0 = 0, c_qn = 0, c_incl = 0, c_total = 0;
    auto load_chunk = [&](int base) {
        const int s = base + lane;
        c_len = 0;
        c_units = 0;
        c_p0 = 0;
        c_q0 = 0;
        c_qn = 0;
        if (s < S) {
            const int raw = __ldg(p.seq_lens + s);
            c_len = clamp_len(p, raw);
            if (c_len != raw) report(p, PA_DEVERR_SEQ_LEN);
            query_rows(p, s, c_q0, c_qn);  // a token at a negative position sees no key
            // v1: one tile per sequence; v2: one per partition that has keys in
            // the window (fused v2 keeps one empty tile for an empty sequence so
            // that its output row is written)
            c_p0 = window_lo(p, c_len, c_qn) / kPart;
            c_units = p.v1 ? 1 : (c_len + kPart - 1) / kPart - c_p0;
            if (p.fused && c_units == 0) c_units = 1;
        }
        c_incl = c_units;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, c_incl, o);
            if (lane >= o) c_incl += v;
        }
        c_total = __shfl_sync(0xffffffffu, c_incl, 31);
    };
    // Ramp: in a batch whose sequences all have max_parts partitions the first
    // tile of this CTA is known before seq_lens is read; load its block ids now,
    // in parallel with the walk, and keep them only if the walk confirms the tile.
    int spec_seq = -1, spec_tb = 0, spec_ids = 0;
    if (!p.v1 && p.window_left < 0) {
        int spec_part;
        guess_unit(p, (int)blockIdx.x / Hkv, spec_seq, spec_part);
        spec_tb = spec_part * kPart;
        const int idx = spec_tb / kBS + lane;
        if (spec_seq < S && idx < p.max_blocks_per_seq)
            spec_ids = __ldg(p.block_tables + (int64_t)spec_seq * p.max_blocks_per_seq + idx);
    }
    load_chunk(0);
    // Final metadata: lengths and block ids are read before the wait for the
    // previous grid, which must be done before the grid-wide tile counter
    // (dynamic schedule: here), the copies and the workspace are touched.
    if (p.metadata_ready && p.tile_ctr) pdl_wait_primary();

    // Tiles of this CTA (kv head fastest): blockIdx.x, then blockIdx.x +
    // gridDim.x, ... (static schedule) or, with tile counters, whatever tile
    // index the grid-wide counter hands out next (dynamic schedule: a CTA
    // that streams faster takes more tiles).  A claim is made one tile ahead
    // by lane 0, so its round trip overlaps a whole tile; the claimed indices
    // of a CTA increase, as the walk of seq_lens below needs.
    int tile = blockIdx.x;
    const bool dyn = p.tile_ctr != nullptr;
    int claimed = 0;  // lane 0: the tile after `tile` (dynamic schedule)
    auto claim = [&]() {
        if (lane == 0) claimed = (int)gridDim.x + atomicAdd(p.tile_ctr, 1);
    };
    if (dyn) claim();
    auto next_tile = [&]() {
        ProducerTile t;
        t.valid = false;
        t.seq = t.part = t.tb = t.te = t.len = t.npages = t.q0 = t.qn = 0;
        const int u = tile / Hkv;
        t.kvh = tile - u * Hkv;
        if (dyn) {
            tile = __shfl_sync(0xffffffffu, claimed, 0);
            claim();
        } else {
            tile += gridDim.x;
        }
        while (cb < S && u >= cu + c_total) {
            cu += c_total;
            cb += 32;
            load_chunk(cb);
        }
        if (cb >= S) return t;
        const int rel = u - cu;
        const unsigned hit = __ballot_sync(0xffffffffu, c_incl > rel);
        const int j = __ffs(hit) - 1;
        t.seq = cb + j;
        const int excl = __shfl_sync(0xffffffffu, c_incl - c_units, j);
        t.len = __shfl_sync(0xffffffffu, c_len, j);
        t.q0 = __shfl_sync(0xffffffffu, c_q0, j);
        t.qn = __shfl_sync(0xffffffffu, c_qn, j);
        const int lo = window_lo(p, t.len, t.qn);
        t.part = __shfl_sync(0xffffffffu, c_p0, j) + rel - excl;
        t.tb = p.v1 ? lo : max(t.part * kPart, lo);
        t.te = p.v1 ? t.len : min(t.len, t.part * kPart + kPart);
        t.npages = tile_pages(t.tb, t.te);
        t.valid = true;
        return t;
    };
    // Block ids of pages [pc, pc + 32) of tile t, one per lane.  The load is
    // only issued here; its range check (check_ids) comes where the ids are
    // used, so that no copy waits on the load.
    auto load_ids = [&](const ProducerTile& t, int pc) {
        return (t.valid && pc + lane < t.npages)
                   ? __ldg(p.block_tables + (int64_t)t.seq * p.max_blocks_per_seq + t.tb / kBS + pc + lane)
                   : 0;
    };
    auto check_ids = [&](int blk) {
        if ((unsigned)blk >= (unsigned)p.num_blocks) {
            report(p, PA_DEVERR_BLOCK_ID);
            blk = 0;
        }
        return blk;
    };

    uint32_t g = 0;  // pages issued by this CTA
    int k = 0;       // tiles issued by this CTA
    bool ok = true;
    ProducerTile cur = next_tile();
    int ids = check_ids((cur.valid && cur.seq == spec_seq && cur.tb == spec_tb) ? (lane < cur.npages ? spec_ids : 0)
                                                                                  : load_ids(cur, 0));
    if (p.metadata_ready && !p.tile_ctr) pdl_wait_primary();  // static schedule: first tile found
    while (ok && cur.valid) {
        // The next tile is walked to, and its first block ids loaded, only once
        // the first batch of this tile's copies is out (the walk may load
        // lengths): nothing delays the first copies of a tile.
        ProducerTile nxt;
        nxt.valid = false;
        bool have_nxt = false;

        const int slot = k % C::kTD;
        if (lane == 0) {
            ok = mbar_wait(sm.td_empty + slot * 8, ((k / C::kTD) & 1) ^ 1, sm.abort, sm.wait_ns);
            if (ok) {
                TileDesc& d = sm.desc[slot];
                d.seq = cur.seq;
                d.kvh = cur.kvh;
                d.part = cur.part;
                d.tok_begin = cur.tb;
                d.tok_end = cur.te;
                d.len = cur.len;
                d.q0 = cur.q0;
                d.qn = cur.qn;
                d.flags = 0;
                // the group's rows of every query token of the sequence: slot row
                // i * group + g holds query token i, head kvh * group + g
                mbar_arrive_expect_tx(sm.td_full + slot * 8, qbytes * (uint32_t)cur.qn);
                for (int qi = 0; qi < cur.qn; ++qi)
                    bulk_g2s(sm.q + slot * C::kQBytes + (uint32_t)qi * qbytes,
                             qbase + ((int64_t)(cur.q0 + qi) * p.num_heads + (int64_t)cur.kvh * p.group) *
                                         HEAD * C::kElem,
                             qbytes, sm.td_full + slot * 8);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);

        for (int pc = 0; pc < cur.npages && ok; pc += 32) {
            const int n = min(32, cur.npages - pc);
            int ids_next = 0;  // block ids of the next 32 pages (this tile or the next one)
            // Issue in batches of up to STAGES pages, one stage per lane: the
            // stages of a batch are distinct, so each lane waits for exactly the
            // previous use of its own stage.
            for (int b0 = 0; b0 < n && ok; b0 += STAGES) {
                const int nb = min(STAGES, n - b0);
                const int blk = __shfl_sync(0xffffffffu, ids, (b0 + lane) & 31);
                bool lok = true;
                if (lane < nb) {
                    const uint32_t gg = g + (uint32_t)lane;
                    const uint32_t st = gg % STAGES, ph = (gg / STAGES) & 1;
                    lok = mbar_wait(sm.empty + st * 8, ph ^ 1, sm.abort, sm.wait_ns);
                    // test hook: CTA 0 never issues its first stage, so the consumer
                    // waiting for it runs out of time (bounded, no fault)
                    const bool withhold = p.withhold_page && blockIdx.x == 0 && gg == 0;
                    if (lok && !withhold) {
                        const uint32_t fb = sm.full + st * 8;
                        const uint32_t dk = sm.ring + st * C::kStageBytes, dv = dk + C::kPageBytes;
                        mbar_arrive_expect_tx(fb, 2 * C::kPageBytes);
                        const int64_t page = (int64_t)blk * Hkv + cur.kvh;
                        if constexpr (C::kTensorMap && C::kKvElem == 1) {
                            // fp8 NHD: one box of 16 token rows x HEAD bytes per page
                            const int y = (int)(page * kBS);
                            tensor2d_g2s_hint(dk, tmk, 0, y, fb, kvpol);
                            tensor2d_g2s_hint(dv, tmv, 0, y, fb, kvpol);
                        } else if constexpr (C::kTensorMap) {
                            // 16-bit / fp32 NHD: the whole page in one box of the
                            // 3-D view (128-byte chunk of a row, row, chunk index),
                            // staged as HEAD * elem / 128 blocks of 16 rows x 128 bytes
                            const int y = (int)(page * kBS);
                            tensor3d_g2s_hint(dk, tmk, 0, y, 0, fb, kvpol);
                            tensor3d_g2s_hint(dv, tmv, 0, y, 0, fb, kvpol);
                        } else {
                            bulk_g2s_hint(dk, kbase + page * C::kPageBytes, C::kPageBytes, fb, kvpol);
                            bulk_g2s_hint(dv, vbase + page * C::kPageBytes, C::kPageBytes, fb, kvpol);
                        }
                    }
                }
                ok = __all_sync(0xffffffffu, lok);
                g += (uint32_t)nb;
                if (b0 == 0) {  // first batch out: load the next ids while the rest streams
                    if (pc + 32 < cur.npages) {
                        ids_next = load_ids(cur, pc + 32);
                    } else {
                        if (!have_nxt) {
                            nxt = next_tile();
                            have_nxt = true;
                        }
                        ids_next = load_ids(nxt, 0);
                    }
                }
            }
            ids = check_ids(ids_next);
        }
        if (!have_nxt) {
            nxt = next_tile();
            if (cur.npages == 0) ids = check_ids(load_ids(nxt, 0));
        }
        ++k;
        cur = nxt;
    }

    if (lane == 0) {
        if (ok) {
            const int slot = k % C::kTD;
            ok = mbar_wait(sm.td_empty + slot * 8, ((k / C::kTD) & 1) ^ 1, sm.abort, sm.wait_ns);
            if (ok) {
                sm.desc[slot].flags = kTileStop;
                mbar_arrive(sm.td_full + slot * 8);
            }
        }
        if (!ok) {
            report(p, PA_DEVERR_TIMEOUT);
            *sm.abort = 1;
        }
        // No bulk copy may still be writing shared memory when the CTA exits:
        // wait (bounded) for the last phase issued on every stage.
        for (uint32_t st = 0; st < STAGES && st < g; ++st) {
            const uint32_t last = g - 1 - ((g - 1 - st) % STAGES);
            mbar_wait(sm.full + st * 8, (last / STAGES) & 1, sm.abort + 1, sm.wait_ns);
        }
        // Dynamic schedule: the last CTA to be done with claiming (its arrival
        // releases its claims) sets both counters back to zero for the next call.
        if (dyn && atom_add_acq_rel_gpu(p.tile_ctr + 1, 1) == (int)gridDim.x - 1) {
            p.tile_ctr[0] = 0;
            p.tile_ctr[1] = 0;
        }
    }
}

// ------------------------------------------------------------------ epilogue

// Merge the NC consumer warps' partial states of one tile and write either the
// partition statistics (v2) or the final output row (v1).  Each thread owns up
// to ITEMS (row, 4-column) items; all their shared-memory loads are issued
// before any arithmetic, so the merge costs one dependency chain, not ITEMS.
template <class C, typename T, int HEAD, int NC>
__device__ void tile_epilogue(const Params& p, const TileDesc& d, const Smem& sm, int tid) {
    constexpr int D4 = HEAD / 4;
    constexpr int ITEMS = (C::kMaxG * D4 + NC * 32 - 1) / (NC * 32);
    const int G = p.group;
    // row v of the merge buffers: query token v / G, head kvh * G + v % G
    const int qn = C::kMQ ? d.qn : 1;
    const int n = qn * G * D4;
    // warps holding a partial state of row h: all of them, or with paired page
    // streams the WR warps of the row's n-tile (its rows at h % 8 of their buffers)
    constexpr int WR = NC / C::kPageWarps;
    float2 e[ITEMS][WR];
    float4 a[ITEMS][WR];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int idx = tid + it * NC * 32;
        const int h = idx / D4, d4 = idx - h * D4;
        const int w0 = C::kPairs ? (h >> 3) * WR : 0, hl = C::kPairs ? (h & 7) : h;
#pragma unroll
        for (int w = 0; w < WR; ++w) {
            if (idx < n) {
                e[it][w] = sm.ml[(w0 + w) * C::kMergeRows + hl];
                a[it][w] = *reinterpret_cast<const float4*>(
                    sm.merge + ((w0 + w) * C::kMergeRows + hl) * C::kMergeStride + 4 * d4);
            } else {
                e[it][w] = make_float2(-INFINITY, 0.f);
                a[it][w] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int idx = tid + it * NC * 32;
        if (idx >= n) break;
        const int h = idx / D4, d4 = idx - h * D4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < WR; ++w) M = fmaxf(M, e[it][w].x);
        float L = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < WR; ++w) {
            const float c = (e[it][w].x == -INFINITY) ? 0.f : exp2f((e[it][w].x - M) * kLog2e);
            L += c * e[it][w].y;
            o.x += c * a[it][w].x;
            o.y += c * a[it][w].y;
            o.z += c * a[it][w].z;
            o.w += c * a[it][w].w;
        }
        const float inv = L > 0.f ? p.v_scale / L : 0.f;
        o.x *= inv;
        o.y *= inv;
        o.z *= inv;
        o.w *= inv;
        const int qi = C::kMQ ? h / G : 0;
        const int head = d.kvh * G + (h - qi * G);
        const int64_t sh = (int64_t)(d.q0 + qi) * p.num_heads + head;
        if (p.v1) {
            T* dst = static_cast<T*>(p.out) + sh * HEAD + 4 * d4;
            if constexpr (C::kF32) {
                *reinterpret_cast<float4*>(dst) = o;
            } else {
                uint2 v;
                v.x = pack2<C::kBF16>(o.x, o.y);
                v.y = pack2<C::kBF16>(o.z, o.w);
                *reinterpret_cast<uint2*>(dst) = v;
            }
        } else {
            const int64_t ps = sh * p.max_parts + d.part;
            // kept in L2 for the reduce that follows (the read demotes it)
            st_global_v4_hint(p.tmp_out + ps * HEAD + 4 * d4, o, l2_policy_evict_last());
            if (d4 == 0) {
                float m = M;
                // logits are kept relative to the tile's last token; move the
                // partition max into the sequence frame (last token of the
                // sequence) -- the reduce kernel finishes the shift to absolute
                // positions after merging.
                if (p.alibi) m += __ldg(p.alibi + head) * (float)(d.tok_end - d.len);
                p.max_logits[ps] = m;
                p.exp_sums[ps] = L;
            }
        }
    }
}

template <typename T, int HEAD, bool L2ONLY>
__device__ __forceinline__ void merge_row_warp(const Params& p, int64_t row, int h, int len, int qn, int qi,
                                               int lane);

// The rows of one (sequence, kv head), one per consumer warp at a time.  Not
// inlined: its loads then never share a register allocation with the page
// loop (three fp8 CTAs per SM need the kernel within 128 registers).
template <typename T, int HEAD, int NC, bool MQ>
__device__ __noinline__ void merge_group(const Params& p, int seq_kvh_base, int q0, int qn, int len, int warp,
                                         int lane) {
    const int G = p.group;
    for (int r = warp; r < qn * G; r += NC) {
        const int qi = MQ ? r / G : 0;
        merge_row_warp<T, HEAD, true>(p, (int64_t)q0 + qi, seq_kvh_base + (r - qi * G), len, qn, qi, lane);
    }
}

// End of a tile for the consumer warps: epilogue (merge of the warps' partial
// states, partition statistics or output row), then in fused v2 mode the
// arrival count of the (sequence, kv head) and, for its last partition, the
// Phase 2 merge: one (query row, head) per consumer warp at a time, the same
// row merge as the reduce kernel, with L2-only loads.  Returns false if a
// bounded wait gave up.
template <class C, typename T, int HEAD, int NC>
__device__ bool tile_finish(const Params& p, const TileDesc& d, const Smem& sm, int warp, int lane,
                            uint32_t& mphase) {
    const int tid = warp * 32 + lane;
    tile_epilogue<C, T, HEAD, NC>(p, d, sm, tid);
    if (!consumer_sync(sm, mphase, lane)) return false;  // epilogue done, merge buffers free
    if (!p.fused || p.v1) return true;
    if (tid == 0) {
        const int P = (d.len + kPart - 1) / kPart - window_lo(p, d.len, d.qn) / kPart;
        int* counter = p.counters + (int64_t)d.seq * p.num_kv_heads + d.kvh;
        // releases this CTA's partition results (every warp's, seen through the
        // barrier above) before the count; acquires the others' with it
        const int last = atom_add_acq_rel_gpu(counter, 1) == (P > 0 ? P : 1) - 1;
        if (last) *counter = 0;  // every tile has arrived: zero again for the next call
        sm.abort[2] = last ? 1 : 0;
    }
    if (!consumer_sync(sm, mphase, lane)) return false;
    if (sm.abort[2])
        merge_group<T, HEAD, NC, C::kMQ>(p, d.kvh * p.group, d.q0, C::kMQ ? d.qn : 1, d.len, warp, lane);
    return true;
}

// ------------------------------------------------------------ online softmax

// Logits may exceed the running reference max by this much (natural-log units,
// 8 ln 2) before the reference moves: p = exp(z - m) then stays below 2^8,
// well inside the range of the fp16 / bf16 P operand.
constexpr float kLazyMax = 5.545177444479562f;

// One page of the online softmax (running max and sum, rescaled as new
// logits arrive) with which a tile streams one partition of Phase 1
// ("paged_attention_v2_pytorch.py -- BI-V100 PagedAttention V2", per-partition
// attention): rows are the page's tokens, columns this lane's heads.  z holds
// the logits (-inf where masked) and becomes p = exp(z - m).  The reference m
// of each head is the same in every lane of the warp; it moves only when some
// logit exceeds it by more than kLazyMax, and then to the running max of the
// whole warp (three shuffle rounds), with l and acc rescaled.  Otherwise a
// page costs no shuffle and no rescale.  mx keeps this lane's running max, for
// the exact statistics at the end of the tile (settle_max).
template <int NT, int KT, bool MQ>
__device__ __forceinline__ void softmax_page(float (&z)[NT][4], float (&m)[NT][2], float (&mx)[NT][2],
                                             float (&l)[NT][2], float (&acc)[KT][NT][4], bool edge) {
    bool need = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float a = fmaxf(z[nt][0], z[nt][2]), b = fmaxf(z[nt][1], z[nt][3]);
        mx[nt][0] = fmaxf(mx[nt][0], a);
        mx[nt][1] = fmaxf(mx[nt][1], b);
        need |= (a - m[nt][0] > kLazyMax) || (b - m[nt][1] > kLazyMax);  // -inf - -inf: false
    }
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float mn0 = mx[nt][0], mn1 = mx[nt][1];
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mn0 = fmaxf(mn0, __shfl_xor_sync(0xffffffffu, mn0, o));
                mn1 = fmaxf(mn1, __shfl_xor_sync(0xffffffffu, mn1, o));
            }
            // several query tokens: a row with no key in its range so far keeps
            // max -inf (masked pages only); take 0 as reference so no -inf - -inf
            // appears.  One token: every page holds a key of every row.
            const float mr0 = (MQ && mn0 == -INFINITY) ? 0.f : mn0;
            const float mr1 = (MQ && mn1 == -INFINITY) ? 0.f : mn1;
            const float al0 = exp2f((m[nt][0] - mr0) * kLog2e);
            const float al1 = exp2f((m[nt][1] - mr1) * kLog2e);
            m[nt][0] = mn0;
            m[nt][1] = mn1;
            l[nt][0] *= al0;
            l[nt][1] *= al1;
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
                acc[mt][nt][0] *= al0;
                acc[mt][nt][1] *= al1;
                acc[mt][nt][2] *= al0;
                acc[mt][nt][3] *= al1;
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float mr0 = (MQ && edge && m[nt][0] == -INFINITY) ? 0.f : m[nt][0];
        const float mr1 = (MQ && edge && m[nt][1] == -INFINITY) ? 0.f : m[nt][1];
        z[nt][0] = exp2f((z[nt][0] - mr0) * kLog2e);
        z[nt][1] = exp2f((z[nt][1] - mr1) * kLog2e);
        z[nt][2] = exp2f((z[nt][2] - mr0) * kLog2e);
        z[nt][3] = exp2f((z[nt][3] - mr1) * kLog2e);
        l[nt][0] += z[nt][0] + z[nt][2];
        l[nt][1] += z[nt][1] + z[nt][3];
    }
}

// End of a warp's pages of a tile: move the reference of each head to the
// warp's exact running max (what the partition statistics hold), rescaling l
// and acc once.
template <int NT, int KT>
__device__ __forceinline__ void settle_max(float (&m)[NT][2], float (&mx)[NT][2], float (&l)[NT][2],
                                           float (&acc)[KT][NT][4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float mn0 = mx[nt][0], mn1 = mx[nt][1];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mn0 = fmaxf(mn0, __shfl_xor_sync(0xffffffffu, mn0, o));
            mn1 = fmaxf(mn1, __shfl_xor_sync(0xffffffffu, mn1, o));
        }
        // equal (also both -inf: no key seen): nothing to move
        const float al0 = mn0 == m[nt][0] ? 1.f : exp2f((m[nt][0] - mn0) * kLog2e);
        const float al1 = mn1 == m[nt][1] ? 1.f : exp2f((m[nt][1] - mn1) * kLog2e);
        m[nt][0] = mn0;
        m[nt][1] = mn1;
        l[nt][0] *= al0;
        l[nt][1] *= al1;
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
            acc[mt][nt][0] *= al0;
            acc[mt][nt][1] *= al1;
            acc[mt][nt][2] *= al0;
            acc[mt][nt][3] *= al1;
        }
    }
}

// ------------------------------------------------------------------ consumers

// Byte offset of this lane's ldmatrix row address inside a K page for k-step kk
// (A operand of Q.K^T: rows = 16 tokens, columns = head dims 16kk..16kk+15).
template <int LAYOUT>
__device__ __forceinline__ uint32_t k_frag_off(int lane, int kk) {
    const int j = lane >> 3, r = lane & 7;
    const int tok = r + ((j & 1) << 3);
    const int c = 2 * kk + (j >> 1);  // 8-element chunk of the head dim
    if constexpr (LAYOUT == kSplit) {
        return (uint32_t)((c * kBS + tok) * 16);  // [d/8][token][8]
    } else {
        // NHD page staged as [d/64][token][64] with the 128-byte swizzle
        return (uint32_t)((c >> 3) * 2048 + tok * 128 + (((c & 7) ^ (tok & 7)) << 4));
    }
}

// Byte offset of this lane's ldmatrix row address inside a V page for m-tile mt
// (A operand of P.V: rows = head dims 16mt..16mt+15, columns = 16 tokens).
template <int LAYOUT>
__device__ __forceinline__ uint32_t v_frag_off(int lane, int mt) {
    const int j = lane >> 3, r = lane & 7;
    if constexpr (LAYOUT == kSplit) {
        const int d = mt * 16 + r + ((j & 1) << 3);  // [d][token]: row d holds 16 tokens
        return (uint32_t)(d * 32 + (j >> 1) * 16);
    } else {
        const int tok = r + ((j >> 1) << 3);  // stored as token rows: loaded transposed
        const int c = 2 * mt + (j & 1);
        return (uint32_t)((c >> 3) * 2048 + tok * 128 + (((c & 7) ^ (tok & 7)) << 4));
    }
}

// Zero the V entries of tokens >= valid in a staged 16-bit page so that the
// P.V product never sees unused slots (which may hold anything, even NaN).
template <int LAYOUT, int HEAD>
__device__ __forceinline__ void zero_v_tail16(uint32_t vpage, int valid, int lane) {
    if constexpr (LAYOUT == kSplit) {
        for (int d = lane; d < HEAD; d += 32)
            for (int t = valid; t < kBS; ++t)
                asm volatile("st.shared.u16 [%0], %1;" ::"r"(vpage + (uint32_t)(d * kBS + t) * 2),
                             "h"((unsigned short)0)
                             : "memory");
    } else {
        const int rows = (kBS - valid) * (HEAD / 64);
        for (int i = lane; i < rows * 8; i += 32) {
            const int rowi = i >> 3, chunk = i & 7;
            const int tok = valid + rowi / (HEAD / 64), half = rowi % (HEAD / 64);
            const uint32_t a = vpage + (uint32_t)(half * 2048 + tok * 128 + chunk * 16);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
        }
    }
}

// Zero the fp32 V entries of tokens >= valid in a staged page: split [d][16
// tokens], or NHD as HEAD / 32 swizzled blocks of 16 token rows x 128 bytes
// (the swizzle permutes 16-byte chunks within a row, so a row stays one token's).
template <int LAYOUT, int HEAD>
__device__ __forceinline__ void zero_v_tail32(uint32_t vpage, int valid, int lane) {
    if constexpr (LAYOUT == kSplit) {
        for (int d = lane; d < HEAD; d += 32)
            for (int t = valid; t < kBS; ++t)
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(vpage + (uint32_t)(d * kBS + t) * 4), "r"(0u)
                             : "memory");
    } else {
        const int rows = (kBS - valid) * (HEAD / 32);
        for (int i = lane; i < rows * 8; i += 32) {
            const int rowi = i >> 3, chunk = i & 7;
            const int tok = valid + rowi / (HEAD / 32), bx = rowi % (HEAD / 32);
            const uint32_t a = vpage + (uint32_t)(bx * 2048 + tok * 128 + chunk * 16);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
        }
    }
}

// Zero the fp8 V entries of tokens >= valid in a staged split page [d][16 tokens].
template <int HEAD>
__device__ __forceinline__ void zero_v_tail8(uint32_t vpage, int valid, int lane) {
    for (int d = lane; d < HEAD; d += 32)
        for (int t = valid; t < kBS; ++t)
            asm volatile("st.shared.u8 [%0], %1;" ::"r"(vpage + (uint32_t)(d * kBS + t)),
                         "h"((unsigned short)0)
                         : "memory");
}

template <class C, typename T, int HEAD, int NT, int LAYOUT, int STAGES, int NC>
__device__ void consumer_mma(const Params& p, const Smem& sm, int warp, int lane) {
    constexpr bool BF = C::kBF16;
    constexpr int KT = HEAD / 16;  // k-steps of Q.K^T, m-tiles of P.V
    // Two n-tiles: the warps work in pairs of page streams, one n-tile each
    // (rows nt0 * 8 .. nt0 * 8 + 7) on the pages j = pfirst (mod PSTRIDE), so
    // every page is read by two warps, each with one n-tile's registers.
    constexpr bool kPairs = C::kPairs;
    constexpr int NTW = kPairs ? 1 : NT;          // n-tiles per warp
    constexpr int PSTRIDE = kPairs ? NC / 2 : NC; // warps per page stream
    const int nt0 = kPairs ? warp / PSTRIDE : 0;
    const int pfirst = kPairs ? warp % PSTRIDE : warp;
    const int G = p.group;
    const int r = lane >> 2, cq = lane & 3;
    const bool has_alibi = p.alibi != nullptr;
    const bool has_cap = p.softcap > 0.f;
    uint32_t gbase = 0;
    uint32_t mphase = 0;
    for (int k = 0;; ++k) {
        const int slot = k % C::kTD;
        if (!warp_wait(sm.td_full + slot * 8, (k / C::kTD) & 1, sm.abort, sm.wait_ns)) {
            report(p, PA_DEVERR_TIMEOUT);
            *sm.abort = 1;
            return;
        }
        const TileDesc d = sm.desc[slot];
        if (d.flags & kTileStop) return;
        const int qn = C::kMQ ? d.qn : 1;
        const int GE = qn * G;  // rows of N: query token v / G, head kvh * G + v % G

        // Q as B fragments: B[k = head dim][n = row], rows >= GE are zero.
        uint32_t qb[NTW][KT][2];
        const uint32_t qs = sm.q + slot * C::kQBytes;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            const int h = (nt0 + nt) * 8 + r;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                uint32_t b0 = 0, b1 = 0;
                if (h < GE) {
                    const uint32_t a = qs + (uint32_t)((h * HEAD + kk * 16 + 2 * cq) * 2);
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(b0) : "r"(a));
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(b1) : "r"(a + 16));
                }
                qb[nt][kk][0] = b0;
                qb[nt][kk][1] = b1;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.td_empty + slot * 8);  // Q and descriptor are in registers

        float sl[NTW][2];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = (nt0 + nt) * 8 + 2 * cq + e;
                sl[nt][e] = (has_alibi && h < GE) ? __ldg(p.alibi + d.kvh * G + h % G) : 0.f;
            }
        // key range of each of this lane's rows: its query token's position and
        // window, within the tile (padded rows get the tile's range)
        int klo[NTW][2], khi[NTW][2];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int v = (nt0 + nt) * 8 + 2 * cq + e;
                int lo = d.tok_begin, hi = d.tok_end - 1;
                if (C::kMQ && v < GE) {
                    const int pos = d.len - qn + v / G;
                    hi = min(hi, pos);
                    lo = max(lo, window_lo_at(p, pos));
                }
                klo[nt][e] = lo;
                khi[nt][e] = hi;
            }
        // keys inside every row's range: a page within [lo_all, hi_all] needs no mask
        // (one query token: the tile's own range)
        const int hi_all = C::kMQ ? min(d.tok_end - 1, d.len - qn) : d.tok_end - 1;
        const int lo_all = C::kMQ ? max(d.tok_begin, window_lo_at(p, d.len - 1)) : d.tok_begin;
        const int origin = d.tok_end - 1;  // ALiBi positions are taken relative to this token

        float m[NTW][2], l[NTW][2], mx[NTW][2];  // reference max, sum, this lane's running max
        float acc[KT][NTW][4];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            m[nt][0] = m[nt][1] = mx[nt][0] = mx[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < KT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
        }

        const int npages = tile_pages(d.tok_begin, d.tok_end);
        const int page0 = d.tok_begin / kBS * kBS;  // first token of the tile's first page
        // stage and phase of page j: advanced per page with one n-tile per warp,
        // computed per page with two (whose registers are all taken)
        uint32_t st = (gbase + (uint32_t)pfirst) % STAGES, ph = ((gbase + (uint32_t)pfirst) / STAGES) & 1;
        for (int j = pfirst; j < npages; j += PSTRIDE, advance_stage<STAGES, PSTRIDE>(st, ph)) {
            if constexpr (NTW > 1) {
                st = (gbase + (uint32_t)j) % STAGES;
                ph = ((gbase + (uint32_t)j) / STAGES) & 1;
            }
            if (!warp_wait(sm.full + st * 8, ph, sm.abort, sm.wait_ns)) {
                report(p, PA_DEVERR_TIMEOUT);
                *sm.abort = 1;
                return;
            }
            const uint32_t kp = sm.ring + st * C::kStageBytes;
            const uint32_t vp = kp + C::kPageBytes;
            const int tok0 = page0 + j * kBS;
            const int valid = min(kBS, d.tok_end - tok0);  // slots >= valid: past the sequence
            const bool edge = tok0 < lo_all || tok0 + kBS - 1 > hi_all;  // some key masked
            if (valid < kBS) {
                zero_v_tail16<LAYOUT, HEAD>(vp, valid, lane);
                fence_proxy_async_smem();
                __syncwarp();
            }

            // S^T[token][head] = K . Q^T
            // two accumulator chains (even / odd k-steps) for MMA latency hiding
            float s[NTW][4], s2[NTW][4];
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] = s2[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kp + k_frag_off<LAYOUT>(lane, kk), a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt) {
                    if (kk & 1)
                        mma_16816<BF>(s2[nt], a0, a1, a2, a3, qb[nt][kk][0], qb[nt][kk][1]);
                    else
                        mma_16816<BF>(s[nt], a0, a1, a2, a3, qb[nt][kk][0], qb[nt][kk][1]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];

            // One n-tile: the page's V fragments go to registers here and the
            // stage back to the producer, before the softmax and P.V, so the
            // stage is refilled while they run (two n-tiles have no registers
            // to spare and load V in the P.V loop).
            constexpr bool kEarlyV = NTW == 1;
            uint32_t vf[kEarlyV ? KT : 1][4];
            if constexpr (kEarlyV) {
#pragma unroll
                for (int mt = 0; mt < KT; ++mt) {
                    if constexpr (LAYOUT == kSplit)
                        ldsm_x4(vp + v_frag_off<LAYOUT>(lane, mt), vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3]);
                    else
                        ldsm_x4_trans(vp + v_frag_off<LAYOUT>(lane, mt), vf[mt][0], vf[mt][1], vf[mt][2],
                                      vf[mt][3]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.empty + st * 8);
            }

            // logits, online softmax, P as B fragments of P.V
            const int tlo = tok0 + r;  // this thread's tokens: tlo (e=0,1), tlo+8 (e=2,3)
            uint32_t pb[NTW][2], pbl[NTW][2];
            float z[NTW][4];
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = s[nt][e] * p.scale;
                    if (has_cap) v = p.softcap * tanhf(v * p.inv_softcap);
                    if (has_alibi) v += sl[nt][e & 1] * (float)(tlo + ((e >> 1) << 3) - origin);
                    z[nt][e] = v;
                }
                if (edge) {
                    const int t0 = tok0 + r, t1 = t0 + 8;
                    if (t0 < klo[nt][0] || t0 > khi[nt][0]) z[nt][0] = -INFINITY;
                    if (t0 < klo[nt][1] || t0 > khi[nt][1]) z[nt][1] = -INFINITY;
                    if (t1 < klo[nt][0] || t1 > khi[nt][0]) z[nt][2] = -INFINITY;
                    if (t1 < klo[nt][1] || t1 > khi[nt][1]) z[nt][3] = -INFINITY;
                }
            }
            softmax_page<NTW, KT, C::kMQ>(z, m, mx, l, acc, edge);
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
                const float p0 = z[nt][0], p1 = z[nt][1], p2 = z[nt][2], p3 = z[nt][3];
                const uint32_t x0 = pack2<BF>(p0, p1);  // token r,   heads 2cq, 2cq+1
                const uint32_t x1 = pack2<BF>(p2, p3);  // token r+8
                pb[nt][0] = movmatrix_trans(x0);         // -> B[k = token 2cq..][n = head r]
                pb[nt][1] = movmatrix_trans(x1);
                if constexpr (BF) {
                    // bf16 keeps 8 significant bits; carry the rounding residue
                    // of P in a second bf16 term so P.V keeps ~16 bits.
                    const float2 h0 = unpack2<BF>(x0), h1 = unpack2<BF>(x1);
                    pbl[nt][0] = movmatrix_trans(pack2<BF>(p0 - h0.x, p1 - h0.y));
                    pbl[nt][1] = movmatrix_trans(pack2<BF>(p2 - h1.x, p3 - h1.y));
                }
            }

            // acc^T[head dim][head] += V^T . P^T
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
                uint32_t a0, a1, a2, a3;
                if constexpr (kEarlyV) {
                    a0 = vf[mt][0];
                    a1 = vf[mt][1];
                    a2 = vf[mt][2];
                    a3 = vf[mt][3];
                } else if constexpr (LAYOUT == kSplit) {
                    ldsm_x4(vp + v_frag_off<LAYOUT>(lane, mt), a0, a1, a2, a3);
                } else {
                    ldsm_x4_trans(vp + v_frag_off<LAYOUT>(lane, mt), a0, a1, a2, a3);
                }
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt) {
                    mma_16816<BF>(acc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                    if constexpr (BF) mma_16816<BF>(acc[mt][nt], a0, a1, a2, a3, pbl[nt][0], pbl[nt][1]);
                }
            }
            if constexpr (!kEarlyV) {
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.empty + st * 8);
            }
        }

        // this warp's partial state -> shared memory
        settle_max<NTW, KT>(m, mx, l, acc);
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], o);
                l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], o);
            }
        }
        float* mw = sm.merge + warp * C::kMergeRows * C::kMergeStride;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
            const int h0 = nt * 8 + 2 * cq;
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
                const int d0 = mt * 16 + r;
                mw[h0 * C::kMergeStride + d0] = acc[mt][nt][0];
                mw[(h0 + 1) * C::kMergeStride + d0] = acc[mt][nt][1];
                mw[h0 * C::kMergeStride + d0 + 8] = acc[mt][nt][2];
                mw[(h0 + 1) * C::kMergeStride + d0 + 8] = acc[mt][nt][3];
            }
            if (r == 0) {
                sm.ml[warp * C::kMergeRows + h0] = make_float2(m[nt][0], l[nt][0]);
                sm.ml[warp * C::kMergeRows + h0 + 1] = make_float2(m[nt][1], l[nt][1]);
            }
        }
        if (!consumer_sync(sm, mphase, lane)) {  // all partial states written
            report(p, PA_DEVERR_TIMEOUT);
            *sm.abort = 1;
            return;
        }
        if (!tile_finish<C, T, HEAD, NC>(p, d, sm, warp, lane, mphase)) {  // merge buffers free again
            report(p, PA_DEVERR_TIMEOUT);
            *sm.abort = 1;
            return;
        }
        gbase += (uint32_t)npages;
    }
}

// Four fp8 cache elements (one 32-bit word, lowest address in the low byte) as
// two f16x2 pairs: lo = elements 0, 1 and hi = elements 2, 3 (exact).
template <int KV>
__device__ __forceinline__ void fp8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    if constexpr (KV == kKvE4M3)
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
    else
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "cvt.rn.f16x2.e5m2x2 %0, l;\n\tcvt.rn.f16x2.e5m2x2 %1, h;\n\t}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
}

// Byte offset of 16-byte chunk c of token row t in an fp8 NHD page as the
// tensor copy leaves it: rows of HEAD bytes, chunks swizzled (128-byte swizzle:
// chunk ^ (t mod 8); 64-byte swizzle: chunk ^ ((t / 2) mod 4)), so the eight
// rows a warp reads at once fall in distinct banks.
template <int HEAD>
__device__ __forceinline__ uint32_t nhd8_off(int t, int c) {
    const int sw = HEAD == 128 ? (t & 7) : ((t >> 1) & 3);
    return (uint32_t)(t * HEAD + ((c ^ sw) << 4));
}

// ldmatrix.x4 row address of this lane in an fp8 key page for k-steps kk and
// kk + 1.  Matrix j = lane / 8 holds the 16-byte rows of the eight tokens of
// S^T rows 0-7 (j even) or 8-15 (j odd) in k-step kk + j / 2, so register j of
// lane (r, cq) is the word (token of row r or r + 8, head dims 16k + 4cq..+3).
template <int LAYOUT, int HEAD>
__device__ __forceinline__ uint32_t k8_frag_off(int lane, int kk) {
    const int j = lane >> 3, i = lane & 7;
    const int c = kk + (j >> 1);
    if constexpr (LAYOUT == kNHD) {
        return nhd8_off<HEAD>(i + ((j & 1) << 3), c);  // natural token order
    } else {
        const int tok = ((i >> 1) << 2) + (i & 1) + ((j & 1) << 1);  // tau(i), tau(i) + 2
        return (uint32_t)((c * kBS + tok) * 16);
    }
}

// ldmatrix.x4 row address of this lane in an fp8 value page for m-tiles mt and
// mt + 1: split [d][16 tokens] rows are head dims 16(mt + j/2) + i (+ 8 for odd
// j); NHD rows are tokens i (+ 8 for odd j), chunk mt + j/2.
template <int LAYOUT, int HEAD>
__device__ __forceinline__ uint32_t v8_frag_off(int lane, int mt) {
    const int j = lane >> 3, i = lane & 7;
    const int m = mt + (j >> 1);
    if constexpr (LAYOUT == kNHD) {
        return nhd8_off<HEAD>(i + ((j & 1) << 3), m);
    } else {
        return (uint32_t)((m * 16 + i + ((j & 1) << 3)) * kBS);
    }
}

// fp8 NHD value page: zero the rows of tokens >= valid (whole rows: the
// swizzle only permutes chunks inside a row).
template <int HEAD>
__device__ __forceinline__ void zero_v_tail8_nhd(uint32_t vpage, int valid, int lane) {
    for (int i = lane; i < (kBS - valid) * HEAD / 4; i += 32)
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(vpage + (uint32_t)(valid * HEAD + 4 * i)), "r"(0u)
                     : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// Consumer for fp8 caches (split layout).  The tensor-core inputs are fp16 for
// both query types: fp8 -> fp16 is exact; a bf16 query is converted once per
// tile (values beyond the fp16 range are clamped and PA_DEVERR_QUERY_RANGE is
// set); P is packed to fp16 (11 significant bits, no second term needed).
// Every lane fetches four fp8 values with one 32-bit shared load.  For that
// the reduction index of each MMA is permuted identically on both operands:
//   Q.K^T  k-index 2cq+j <-> head dim 4cq+j, 2cq+8+j <-> 4cq+2+j  (per 16-dim step)
//   P.V    k-index 2cq+j <-> token    4cq+j, 2cq+8+j <-> 4cq+2+j  (per page)
// so row rr of S^T (the M index of Q.K^T) holds token tau(rr) of the page:
//   tau(r) = 4*(r/2) + (r&1) and tau(r+8) = tau(r) + 2 for r < 8.
template <class C, typename T, int HEAD, int NT, int LAYOUT, int STAGES, int NC, int KV>
__device__ void consumer_mma_fp8(const Params& p, const Smem& sm, int warp, int lane) {
    constexpr bool QBF = C::kBF16;
    constexpr int KT = HEAD / 16;
    const int G = p.group;
    const int r = lane >> 2, cq = lane & 3;
    // page token of S^T rows r and r + 8: permuted for the split layout (see
    // above), natural for NHD, where the transposition of V is done by movmatrix
    const int tau = ((r >> 1) << 2) + (r & 1);
    const int tlo = LAYOUT == kNHD ? r : tau;
    const int thi = LAYOUT == kNHD ? r + 8 : tau + 2;
    const bool has_alibi = p.alibi != nullptr;
    const bool has_cap = p.softcap > 0.f;
    uint32_t gbase = 0;
    uint32_t mphase = 0;
    for (int k = 0;; ++k) {
        const int slot = k % C::kTD;
        if (!warp_wait(sm.td_full + slot * 8, (k / C::kTD) & 1, sm.abort, sm.wait_ns)) {
            report(p, PA_DEVERR_TIMEOUT);
            *sm.abort = 1;
            return;
        }
        const TileDesc d = sm.desc[slot];
        if (d.flags & kTileStop) return;
        const int qn = C::kMQ ? d.qn : 1;
        const int GE = qn * G;  // rows of N: query token v / G, head kvh * G + v % G

        // Q as fp16 B fragments in the permuted head-dim order.
        uint32_t qb[NT][KT][2];
        bool q_clamped = false;
        const uint32_t qs = sm.q + slot * C::kQBytes;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int h = nt * 8 + r;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                uint32_t w0 = 0, w1 = 0;
                if (h < GE) {
                    const uint32_t a = qs + (uint32_t)((h * HEAD + kk * 16 + 4 * cq) * 2);
                    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(a));
                    if constexpr (QBF) {
                        float2 f0 = unpack2<true>(w0), f1 = unpack2<true>(w1);
                        const float lim = 65504.f;
                        q_clamped |= fabsf(f0.x) > lim || fabsf(f0.y) > lim || fabsf(f1.x) > lim ||
                                     fabsf(f1.y) > lim;
                        w0 = pack2<false>(fminf(fmaxf(f0.x, -lim), lim), fminf(fmaxf(f0.y, -lim), lim));
                        w1 = pack2<false>(fminf(fmaxf(f1.x, -lim), lim), fminf(fmaxf(f1.y, -lim), lim));
                    }
                }
                qb[nt][kk][0] = w0;  // head dims 16kk + 4cq, +1  (k-index 2cq, 2cq+1)
                qb[nt][kk][1] = w1;  // head dims 16kk + 4cq+2, +3 (k-index 2cq+8, 2cq+9)
            }
        }
        if (q_clamped) report(p, PA_DEVERR_QUERY_RANGE);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.td_empty + slot * 8);

        float sl[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = nt * 8 + 2 * cq + e;
                sl[nt][e] = (has_alibi && h < GE) ? __ldg(p.alibi + d.kvh * G + h % G) : 0.f;
            }
        // key range of each of this lane's rows: its query token's position and
        // window, within the tile (padded rows get the tile's range)
        int klo[NT][2], khi[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int v = nt * 8 + 2 * cq + e;
                int lo = d.tok_begin, hi = d.tok_end - 1;
                if (C::kMQ && v < GE) {
                    const int pos = d.len - qn + v / G;
                    hi = min(hi, pos);
                    lo = max(lo, window_lo_at(p, pos));
                }
                klo[nt][e] = lo;
                khi[nt][e] = hi;
            }
        // keys inside every row's range: a page within [lo_all, hi_all] needs no mask
        // (one query token: the tile's own range)
        const int hi_all = C::kMQ ? min(d.tok_end - 1, d.len - qn) : d.tok_end - 1;
        const int lo_all = C::kMQ ? max(d.tok_begin, window_lo_at(p, d.len - 1)) : d.tok_begin;
        const int origin = d.tok_end - 1;

        float m[NT][2], l[NT][2], mx[NT][2];  // reference max, sum, this lane's running max
        float acc[KT][NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m[nt][0] = m[nt][1] = mx[nt][0] = mx[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < KT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
        }

        const int npages = tile_pages(d.tok_begin, d.tok_end);
        const int page0 = d.tok_begin / kBS * kBS;
        // stage and phase of page j: advanced per page with one n-tile, computed
        // per page with two (whose registers are all taken)
        uint32_t st = (gbase + (uint32_t)warp) % STAGES, ph = ((gbase + (uint32_t)warp) / STAGES) & 1;
        for (int j = warp; j < npages; j += NC, advance_stage<STAGES, NC>(st, ph)) {
            if constexpr (NT > 1) {
                st = (gbase + (uint32_t)j) % STAGES;
                ph = ((gbase + (uint32_t)j) / STAGES) & 1;
            }
            if (!warp_wait(sm.full + st * 8, ph, sm.abort, sm.wait_ns)) {
                report(p, PA_DEVERR_TIMEOUT);
                *sm.abort = 1;
                return;
            }
            const uint32_t kp = sm.ring + st * C::kStageBytes;
            const uint32_t vp = kp + C::kPageBytes;
            const int tok0 = page0 + j * kBS;
            const int valid = min(kBS, d.tok_end - tok0);  // slots >= valid: past the sequence
            const bool edge = tok0 < lo_all || tok0 + kBS - 1 > hi_all;  // some key masked
            if (valid < kBS) {
                if constexpr (LAYOUT == kNHD)
                    zero_v_tail8_nhd<HEAD>(vp, valid, lane);
                else
                    zero_v_tail8<HEAD>(vp, valid, lane);
                fence_proxy_async_smem();
                __syncwarp();
            }

            // S^T[row][head]: key page [d/16][token][16 bytes] (split) or [token][d]
            // with swizzled 16-byte chunks (NHD)
            float s[NT][4], s2[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] = s2[nt][e] = 0.f;
            // one ldmatrix.x4 fetches the four 32-bit words (tokens tlo / thi,
            // k-steps kk / kk + 1) that four separate loads would
#pragma unroll
            for (int kk = 0; kk < KT; kk += 2) {
                uint32_t w[4];
                ldsm_x4(kp + k8_frag_off<LAYOUT, HEAD>(lane, kk), w[0], w[1], w[2], w[3]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    uint32_t a0, a1, a2, a3;
                    fp8x4_to_f16<KV>(w[2 * u], a0, a2);
                    fp8x4_to_f16<KV>(w[2 * u + 1], a1, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (u)
                            mma_16816<false>(s2[nt], a0, a1, a2, a3, qb[nt][kk + u][0], qb[nt][kk + u][1]);
                        else
                            mma_16816<false>(s[nt], a0, a1, a2, a3, qb[nt][kk + u][0], qb[nt][kk + u][1]);
                    }
                }
            }

            // One n-tile: the page's V words go to registers here and the stage
            // back to the producer, before the softmax, the conversion and P.V.
            constexpr bool kEarlyV = NT == 1;
            uint32_t vw[kEarlyV ? KT / 2 : 1][4];
            if constexpr (kEarlyV) {
#pragma unroll
                for (int mt = 0; mt < KT; mt += 2)
                    ldsm_x4(vp + v8_frag_off<LAYOUT, HEAD>(lane, mt), vw[mt / 2][0], vw[mt / 2][1],
                            vw[mt / 2][2], vw[mt / 2][3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.empty + st * 8);
            }

            uint32_t pb[NT][2];
            float z[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = (s[nt][e] + s2[nt][e]) * p.scale;
                    if (has_cap) v = p.softcap * tanhf(v * p.inv_softcap);
                    if (has_alibi) v += sl[nt][e & 1] * (float)(tok0 + ((e >> 1) ? thi : tlo) - origin);
                    z[nt][e] = v;
                }
                if (edge) {
                    const int t0 = tok0 + tlo, t1 = tok0 + thi;
                    if (t0 < klo[nt][0] || t0 > khi[nt][0]) z[nt][0] = -INFINITY;
                    if (t0 < klo[nt][1] || t0 > khi[nt][1]) z[nt][1] = -INFINITY;
                    if (t1 < klo[nt][0] || t1 > khi[nt][0]) z[nt][2] = -INFINITY;
                    if (t1 < klo[nt][1] || t1 > khi[nt][1]) z[nt][3] = -INFINITY;
                }
            }
            softmax_page<NT, KT, C::kMQ>(z, m, mx, l, acc, edge);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                pb[nt][0] = movmatrix_trans(pack2<false>(z[nt][0], z[nt][1]));  // k-index 2cq.. = tokens tlo
                pb[nt][1] = movmatrix_trans(pack2<false>(z[nt][2], z[nt][3]));
            }

            // acc^T[head dim][head] += V^T . P^T.  Split value page [d][16
            // tokens]: one 32-bit load is four permuted tokens of a head dim.  NHD
            // page [token][d]: one load is four head dims of a token; movmatrix
            // turns each 8 x 8 block (tokens x head dims 16mt + 4cq + {0,1} or
            // {2,3}) into the A fragment, whose rows are then head dims 16mt +
            // tau(r) (rows r) and 16mt + tau(r) + 2 (rows r + 8).
#pragma unroll
            for (int mt = 0; mt < KT; mt += 2) {
                // words of rows r and r + 8 (head dims, or tokens for NHD) of
                // m-tiles mt and mt + 1 in one ldmatrix.x4
                uint32_t w[4];
                if constexpr (kEarlyV) {
                    w[0] = vw[mt / 2][0];
                    w[1] = vw[mt / 2][1];
                    w[2] = vw[mt / 2][2];
                    w[3] = vw[mt / 2][3];
                } else {
                    ldsm_x4(vp + v8_frag_off<LAYOUT, HEAD>(lane, mt), w[0], w[1], w[2], w[3]);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    uint32_t a0, a1, a2, a3;
                    if constexpr (LAYOUT == kNHD) {
                        uint32_t lo0, hi0, lo1, hi1;
                        fp8x4_to_f16<KV>(w[2 * u], lo0, hi0);
                        fp8x4_to_f16<KV>(w[2 * u + 1], lo1, hi1);
                        a0 = movmatrix_trans(lo0);
                        a1 = movmatrix_trans(hi0);
                        a2 = movmatrix_trans(lo1);
                        a3 = movmatrix_trans(hi1);
                    } else {
                        fp8x4_to_f16<KV>(w[2 * u], a0, a2);
                        fp8x4_to_f16<KV>(w[2 * u + 1], a1, a3);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_16816<false>(acc[mt + u][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
            }
            if constexpr (!kEarlyV) {
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.empty + st * 8);
            }
        }

        settle_max<NT, KT>(m, mx, l, acc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], o);
                l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], o);
            }
        }
        float* mw = sm.merge + warp * C::kMergeRows * C::kMergeStride;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int h0 = nt * 8 + 2 * cq;
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
                // head dims of accumulator rows r and r + 8 (see the P.V step)
                const int d0 = mt * 16 + (LAYOUT == kNHD ? tau : r);
                const int d1 = d0 + (LAYOUT == kNHD ? 2 : 8);
                mw[h0 * C::kMergeStride + d0] = acc[mt][nt][0];
                mw[(h0 + 1) * C::kMergeStride + d0] = acc[mt][nt][1];
                mw[h0 * C::kMergeStride + d1] = acc[mt][nt][2];
                mw[(h0 + 1) * C::kMergeStride + d1] = acc[mt][nt][3];
            }
            if (r == 0) {
                sm.ml[warp * C::kMergeRows + h0] = make_float2(m[nt][0], l[nt][0]);
                sm.ml[warp * C::kMergeRows + h0 + 1] = make_float2(m[nt][1], l[nt][1]);
            }
        }
        if (!consumer_sync(sm, mphase, lane)) {
            report(p, PA_DEVERR_TIMEOUT);
            *sm.abort = 1;
            return;
        }
        if (!tile_finish<C, T, HEAD, NC>(p, d, sm, warp, lane, mphase)) {
            report(p, PA_DEVERR_TIMEOUT);
            *sm.abort = 1;
            return;
        }
        gbase += (uint32_t)npages;
    }
}

// fp32 inputs: tensor cores with each fp32 operand carried as two tf32 terms
// (hi + lo) and three MMAs per product (hi.hi + hi.lo + lo.hi), which keeps
// each product to ~2^-20 relative, well inside the fp32 result's error budget.
// Tokens on M, query rows on N for Q.K^T (NT n-tiles of 8 rows); head dims on
// M, rows on N for P.V, as in the 16-bit consumer.  P moves from the S^T
// fragment to the B fragment with shuffles (there is no 32-bit movmatrix).
// One n-tile keeps Q split in registers for the whole tile; two keep the raw
// fp32 words (64 registers at head size 128 instead of 128) and split them at
// each use.
//
// Shared-memory reads.  Split pages: K [d/4][16 tokens][4] gives each k-step's
// A fragment as one ldmatrix.x4; V [d][16 tokens] likewise (its 64-byte rows
// cost 4-way bank conflicts whatever the order).  NHD pages (HEAD / 32 blocks
// of 16 token rows x 128 bytes, 16-byte chunks swizzled by token % 8): K by
// ldmatrix.x4 as well; V^T needs a transpose that ldmatrix does not do for
// 32-bit elements, so its fragments are single-word loads, with the k-step's
// tokens taken in the order 0, 2, 4, 6 | 1, 3, 5, 7 (k-index t -> token 2t, t + 4
// -> 2t + 1), which puts the 32 words of each load in 32 distinct banks; the
// P^T fragment follows the same order.
template <class C, int HEAD, int NT, int LAYOUT, int STAGES, int NC>
__device__ void consumer_tf32(const Params& p, const Smem& sm, int warp, int lane) {
    constexpr int KT = HEAD / 8;   // k-steps of Q.K^T (8 head dims each)
    constexpr int MT = HEAD / 16;  // m-tiles of P.V (16 head dims each)
    constexpr bool QSPLIT = NT == 1;  // Q held split for the whole tile
    const int G = p.group;
    const int r = lane >> 2, cq = lane & 3;
    const bool has_alibi = p.alibi != nullptr;
    const bool has_cap = p.softcap > 0.f;
    uint32_t gbase = 0;
    uint32_t mphase = 0;
    for (int k = 0;; ++k) {
        const int slot = k % C::kTD;
        if (!warp_wait(sm.td_full + slot * 8, (k / C::kTD) & 1, sm.abort, sm.wait_ns)) {
            report(p, PA_DEVERR_TIMEOUT);
            *sm.abort = 1;
            return;
        }
        const TileDesc d = sm.desc[slot];
        if (d.flags & kTileStop) return;
        const int qn = C::kMQ ? d.qn : 1;
        const int GE = qn * G;  // rows of N: query token v / G, head kvh * G + v % G

        // Q as B fragments (k = head dim 8kk + cq / + 4, n = row nt * 8 + r):
        // hi and lo terms (one n-tile) or the raw words (two)
        uint32_t qa[NT][KT][2];
        uint32_t qlo[QSPLIT ? KT : 1][2];
        {
            const float* q = reinterpret_cast<const float*>(
                __cvta_shared_to_generic(sm.q + slot * C::kQBytes));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int kk = 0; kk < KT; ++kk)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int row = nt * 8 + r;
                        const uint32_t x =
                            row < GE ? __float_as_uint(q[row * HEAD + kk * 8 + cq + 4 * e]) : 0u;
                        if constexpr (QSPLIT)
                            split_tf32(x, qa[nt][kk][e], qlo[kk][e]);
                        else
                            qa[nt][kk][e] = x;
                    }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.td_empty + slot * 8);  // Q and descriptor are in registers

        float sl[NT][2];
        int klo[NT][2], khi[NT][2];  // key range of this lane's rows within the tile
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int v = nt * 8 + 2 * cq + e;
                sl[nt][e] = (has_alibi && v < GE) ? __ldg(p.alibi + d.kvh * G + v % G) : 0.f;
                int lo = d.tok_begin, hi = d.tok_end - 1;
                if (C::kMQ && v < GE) {
                    const int pos = d.len - qn + v / G;
                    hi = min(hi, pos);
                    lo = max(lo, window_lo_at(p, pos));
                }
                klo[nt][e] = lo;
                khi[nt][e] = hi;
            }
        const int hi_all = C::kMQ ? min(d.tok_end - 1, d.len - qn) : d.tok_end - 1;
        const int lo_all = C::kMQ ? max(d.tok_begin, window_lo_at(p, d.len - 1)) : d.tok_begin;
        const int origin = d.tok_end - 1;

        float m[NT][2], l[NT][2], mx[NT][2];  // reference max, sum, this lane's running max
        float acc[MT][NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m[nt][0] = m[nt][1] = mx[nt][0] = mx[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
        }

        const int npages = tile_pages(d.tok_begin, d.tok_end);
        const int page0 = d.tok_begin / kBS * kBS;
        // ldmatrix row of this lane: matrix j = lane / 8, row i = lane % 8
        const int lj = lane >> 3, li = lane & 7;
        // P^T k-index cq holds token cq (split) or 2cq (NHD), cq + 4 token cq + 4 or 2cq + 1
        const int tk0 = LAYOUT == kSplit ? cq : 2 * cq, tk1 = LAYOUT == kSplit ? cq + 4 : 2 * cq + 1;
        const int src0 = 4 * tk0 + (r >> 1), src1 = 4 * tk1 + (r >> 1);
        // stage and phase of page j: advanced per page with one n-tile, computed
        // per page with two (whose registers are all taken)
        uint32_t st = (gbase + (uint32_t)warp) % STAGES, ph = ((gbase + (uint32_t)warp) / STAGES) & 1;
        for (int j = warp; j < npages; j += NC, advance_stage<STAGES, NC>(st, ph)) {
            if constexpr (NT > 1) {
                st = (gbase + (uint32_t)j) % STAGES;
                ph = ((gbase + (uint32_t)j) / STAGES) & 1;
            }
            if (!warp_wait(sm.full + st * 8, ph, sm.abort, sm.wait_ns)) {
                report(p, PA_DEVERR_TIMEOUT);
                *sm.abort = 1;
                return;
            }
            const uint32_t kp = sm.ring + st * C::kStageBytes;
            const uint32_t vp = kp + C::kPageBytes;
            const int tok0 = page0 + j * kBS;
            const int valid = min(kBS, d.tok_end - tok0);
            const bool edge = tok0 < lo_all || tok0 + kBS - 1 > hi_all;
            if (valid < kBS) {
                zero_v_tail32<LAYOUT, HEAD>(vp, valid, lane);
                fence_proxy_async_smem();
                __syncwarp();
            }

            // S^T[token][row] = K . Q^T; the four 8 x 4 blocks (tokens 0-7 /
            // 8-15, head dims 8kk..+3 / +4..+7) of a k-step are its A fragment,
            // one ldmatrix.x4 (this lane's row: block lj, row li).  Each
            // k-step's three products go to a fresh accumulator that is then
            // added with a rounded fp32 add, so that the tensor core's own
            // accumulation (which need not round to nearest) never carries a
            // sum across the k-steps of a page or, for P.V below, the pages of
            // a tile: without it a 24-head, group-12 fp32 case missed the 1e-5
            // tolerance even with the rounded split.
            float s[NT][4], s2[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] = s2[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                uint32_t a[4], ah[4], al[4];
                const int cg = 2 * kk + (lj >> 1);  // 16-byte chunk of the head dims
                const uint32_t ka =
                    LAYOUT == kSplit
                        ? kp + (uint32_t)((cg * kBS + li + ((lj & 1) << 3)) * 16)
                        : kp + (uint32_t)((cg >> 3) * 2048 + (li + ((lj & 1) << 3)) * 128 +
                                          (((cg & 7) ^ li) << 4));
                ldsm_x4(ka, a[0], a[1], a[2], a[3]);
#pragma unroll
                for (int e = 0; e < 4; ++e) split_tf32(a[e], ah[e], al[e]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    uint32_t bh[2], bl[2];
                    if constexpr (QSPLIT) {
                        bh[0] = qa[nt][kk][0];
                        bh[1] = qa[nt][kk][1];
                        bl[0] = qlo[kk][0];
                        bl[1] = qlo[kk][1];
                    } else {
                        split_tf32(qa[nt][kk][0], bh[0], bl[0]);
                        split_tf32(qa[nt][kk][1], bh[1], bl[1]);
                    }
                    float t[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_1688_tf32(t, al[0], al[1], al[2], al[3], bh[0], bh[1]);
                    mma_1688_tf32(t, ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
                    mma_1688_tf32(t, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
                    float (&sa)[4] = (kk & 1) ? s2[nt] : s[nt];
#pragma unroll
                    for (int e = 0; e < 4; ++e) sa[e] = __fadd_rn(sa[e], t[e]);
                }
            }

            // logits, online softmax, P^T as B fragments (hi and lo) per n-tile
            uint32_t pbh[NT][2][2], pbl[NT][2][2];
            float z[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = (s[nt][e] + s2[nt][e]) * p.scale;
                    if (has_cap) v = p.softcap * tanhf(v * p.inv_softcap);
                    if (has_alibi) v += sl[nt][e & 1] * (float)(tok0 + r + ((e >> 1) << 3) - origin);
                    z[nt][e] = v;
                }
                if (edge) {
                    const int t0 = tok0 + r, t1 = t0 + 8;
                    if (t0 < klo[nt][0] || t0 > khi[nt][0]) z[nt][0] = -INFINITY;
                    if (t0 < klo[nt][1] || t0 > khi[nt][1]) z[nt][1] = -INFINITY;
                    if (t1 < klo[nt][0] || t1 > khi[nt][0]) z[nt][2] = -INFINITY;
                    if (t1 < klo[nt][1] || t1 > khi[nt][1]) z[nt][3] = -INFINITY;
                }
            }
            softmax_page<NT, MT, C::kMQ>(z, m, mx, l, acc, edge);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // z[nt]: p of (token r, row 2cq), (token r, row 2cq + 1),
                // (token r + 8, row 2cq), (token r + 8, row 2cq + 1)
                const float* pv = z[nt];
                // B fragments of P^T for k-steps ks = 0, 1 (tokens 8ks..8ks+7):
                // b0 = P[row r][token 8ks + tk0], b1 = P[row r][token 8ks + tk1],
                // held by lanes (token % 8, row / 2), element by row parity and ks
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const float e0 = __shfl_sync(0xffffffffu, pv[2 * ks], src0);
                    const float o0 = __shfl_sync(0xffffffffu, pv[2 * ks + 1], src0);
                    const float e1 = __shfl_sync(0xffffffffu, pv[2 * ks], src1);
                    const float o1 = __shfl_sync(0xffffffffu, pv[2 * ks + 1], src1);
                    split_tf32(__float_as_uint((r & 1) ? o0 : e0), pbh[nt][ks][0], pbl[nt][ks][0]);
                    split_tf32(__float_as_uint((r & 1) ? o1 : e1), pbh[nt][ks][1], pbl[nt][ks][1]);
                }
            }

            // acc^T[head dim][row] += V^T . P^T; A fragment of (m-tile mt,
            // k-step ks): head dims 16mt + r / + 8 by k-indices cq / cq + 4
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    uint32_t a[4], ah[4], al[4];
                    if constexpr (LAYOUT == kSplit) {
                        // [d][16 tokens]: the four 8 x 4 blocks (head dims
                        // 16mt..+7 / +8..+15, tokens 8ks..+3 / +4..+7), one ldmatrix.x4
                        ldsm_x4(vp + (uint32_t)(((mt * 16 + li + ((lj & 1) << 3)) * kBS + 8 * ks +
                                                 4 * (lj >> 1)) * 4),
                                a[0], a[1], a[2], a[3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int dim = mt * 16 + r + ((e & 1) << 3);
                            const int tok = 8 * ks + ((e >> 1) ? tk1 : tk0);
                            const uint32_t va = vp + (uint32_t)((dim >> 5) * 2048 + tok * 128 +
                                                                ((((dim >> 2) & 7) ^ (tok & 7)) << 4) +
                                                                (dim & 3) * 4);
                            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a[e]) : "r"(va));
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) split_tf32(a[e], ah[e], al[e]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        float t[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_1688_tf32(t, al[0], al[1], al[2], al[3], pbh[nt][ks][0], pbh[nt][ks][1]);
                        mma_1688_tf32(t, ah[0], ah[1], ah[2], ah[3], pbl[nt][ks][0], pbl[nt][ks][1]);
                        mma_1688_tf32(t, ah[0], ah[1], ah[2], ah[3], pbh[nt][ks][0], pbh[nt][ks][1]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[mt][nt][e] = __fadd_rn(acc[mt][nt][e], t[e]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.empty + st * 8);
        }

        float* mw = sm.merge + warp * C::kMergeRows * C::kMergeStride;
        settle_max<NT, MT>(m, mx, l, acc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], o);
                l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], o);
            }
            const int h0 = nt * 8 + 2 * cq;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int d0 = mt * 16 + r;
                mw[h0 * C::kMergeStride + d0] = acc[mt][nt][0];
                mw[(h0 + 1) * C::kMergeStride + d0] = acc[mt][nt][1];
                mw[h0 * C::kMergeStride + d0 + 8] = acc[mt][nt][2];
                mw[(h0 + 1) * C::kMergeStride + d0 + 8] = acc[mt][nt][3];
            }
            if (r == 0) {
                sm.ml[warp * C::kMergeRows + h0] = make_float2(m[nt][0], l[nt][0]);
                sm.ml[warp * C::kMergeRows + h0 + 1] = make_float2(m[nt][1], l[nt][1]);
            }
        }
        if (!consumer_sync(sm, mphase, lane)) {
            report(p, PA_DEVERR_TIMEOUT);
            *sm.abort = 1;
            return;
        }
        if (!tile_finish<C, float, HEAD, NC>(p, d, sm, warp, lane, mphase)) {
            report(p, PA_DEVERR_TIMEOUT);
            *sm.abort = 1;
            return;
        }
        gbase += (uint32_t)npages;
    }
}

// ------------------------------------------------------------------ kernels

// Two n-tiles hold 16 rows of accumulators (~200 registers uncapped), and the
// fp32 tensor-core consumer holds Q as two tf32 terms (~213): cap them so that
// two CTAs share an SM, as they do for one n-tile of 16-bit inputs.  fp32 with
// two n-tiles fills an SM's shared memory with one CTA (16 KB stages): no cap.
// fp8 with one n-tile: capped for three CTAs per SM (128 registers: fifteen
// warps put four on some SM sub-partition, whose register file is 16 K).
template <typename T, int HEAD, int NT, int LAYOUT, int STAGES, int NC, int KV, bool MQ>
__global__ void __launch_bounds__((NC + 1) * 32,
                                  (std::is_same<T, float>::value && NT > 1)
                                      ? 1
                                      : ((NT > 1 || std::is_same<T, float>::value) ? 2 : (KV != kKvSame ? 3 : 1)))
    pa_partition_kernel(const Params p, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv) {
    using C = Cfg<T, HEAD, NT, LAYOUT, STAGES, NC, KV, MQ>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gen = smem_raw + (base - raw);

    Smem sm;
    sm.ring = base + C::oRing;
    sm.q = base + C::oQ;
    sm.merge = reinterpret_cast<float*>(gen + C::oMerge);
    sm.ml = reinterpret_cast<float2*>(gen + C::oML);
    sm.desc = reinterpret_cast<TileDesc*>(gen + C::oDesc);
    sm.full = base + C::oBar;
    sm.empty = sm.full + STAGES * 8;
    sm.td_full = sm.empty + STAGES * 8;
    sm.td_empty = sm.td_full + C::kTD * 8;
    sm.merge_bar = sm.td_empty + C::kTD * 8;
    sm.abort = reinterpret_cast<volatile int*>(gen + C::oAbort);
    sm.wait_ns = p.wait_limit_ns ? p.wait_limit_ns : kWaitLimitNs;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == NC) prefetch_first_tile<C, HEAD>(p, lane);
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(sm.full + s * 8, 1);
            mbar_init(sm.empty + s * 8, C::kPageWarps);
        }
        for (int s = 0; s < C::kTD; ++s) {
            mbar_init(sm.td_full + s * 8, 1);
            mbar_init(sm.td_empty + s * 8, NC);
        }
        mbar_init(sm.merge_bar, NC);
        sm.abort[0] = 0;
        sm.abort[1] = 0;
        sm.abort[2] = 0;
        fence_mbar_init();
    }
    if constexpr (C::kTensorMap) {
        if (threadIdx.x == NC * 32) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
    }
    __syncthreads();
    pdl_launch_dependents();  // the reduce kernel may be scheduled; it waits for our completion
    // Earlier work in the stream (inputs, workspace readers) must be done.
    // With final metadata only the producer waits, once it has its first tile
    // (producer); every other warp reaches global memory only after that
    // through the producer's barriers.
    if (!p.metadata_ready) pdl_wait_primary();

    if (warp == NC) {
        producer<C, HEAD, STAGES>(p, sm, &tmk, &tmv, lane);
    } else if constexpr (C::kF32) {
        consumer_tf32<C, HEAD, NT, LAYOUT, STAGES, NC>(p, sm, warp, lane);
    } else {
        if constexpr (KV == kKvSame)
            consumer_mma<C, T, HEAD, NT, LAYOUT, STAGES, NC>(p, sm, warp, lane);
        else
            consumer_mma_fp8<C, T, HEAD, NT, LAYOUT, STAGES, NC, KV>(p, sm, warp, lane);
    }
}

// Phase 2: one CTA of 32*WARPS threads per (sequence, head), one pass.  Each
// lane owns four head dims (a float4 column) of one partition row and keeps U
// partition rows in flight; it carries its own running max, so no separate
// pass over max_logits is needed.  The rows are then combined with the usual
// max rescale in shared memory.
template <typename T, int HEAD, int WARPS, int U, bool MQ>
__global__ void __launch_bounds__(WARPS * 32) pa_reduce_kernel(const Params p) {
    constexpr int D4 = HEAD / 4;          // float4 columns of a partition row
    constexpr int RPW = 32 / D4;          // partition rows per warp (1 or 2)
    constexpr int RSTEP = WARPS * RPW;    // partition rows per CTA round (U rounds in flight)
    constexpr int NT = WARPS * 32;
    __shared__ float4 part[RSTEP][D4];
    __shared__ float rowm[RSTEP], roww[RSTEP];

    // one CTA per (sequence, query token, head); query tokens beyond the
    // sequence's count return at once
    const int bid = blockIdx.x;
    const int sq = bid / p.num_heads, h = bid - sq * p.num_heads;
    const int s = MQ ? sq / p.max_q_len : sq, qi = MQ ? sq - s * p.max_q_len : 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();  // the next launch may start its prologue; it waits for us
    pdl_wait_primary();

    int q0 = s, qn = 1;
    if constexpr (MQ) {
        query_rows(p, s, q0, qn);
        if (qi >= qn) return;
    }
    const int len = clamp_len(p, p.seq_lens[s]);
    const int hi = len - qn + qi;                      // the query token's position
    const int P = hi >= 0 ? (hi + kPart) / kPart : 0;  // partitions holding its keys
    const int p0 = window_lo_at(p, hi) / kPart;        // partitions before p0: outside the window
    const int64_t row = (int64_t)q0 + qi;
    const int64_t sb = (row * p.num_heads + h) * p.max_parts;
    float* ml = p.max_logits + sb;
    float* es = p.exp_sums + sb;
    const float* tmp = p.tmp_out + sb * HEAD;
    const uint64_t pol = l2_policy_evict_first();  // partition outputs: last use
    T* o = static_cast<T*>(p.out) + (row * p.num_heads + h) * HEAD;

    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (P > 0) {
        const int prow = warp * RPW + lane / D4, d4 = lane % D4;
        float M = -INFINITY, W = 0.f;
        for (int qb = p0 + prow; qb < P; qb += RSTEP * U) {
            float mq[U], eq[U];
            float4 t[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = qb + u * RSTEP;
                if (q < P) {
                    mq[u] = ml[q];
                    eq[u] = es[q];
                    t[u] = ld_global_v4_hint(tmp + (int64_t)q * HEAD + 4 * d4, pol);
                } else {
                    mq[u] = -INFINITY;
                    eq[u] = 0.f;
                    t[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (mq[u] == -INFINITY) continue;
                if (mq[u] > M) {
                    const float sc = (M == -INFINITY) ? 0.f : expf(M - mq[u]);
                    a.x *= sc;
                    a.y *= sc;
                    a.z *= sc;
                    a.w *= sc;
                    W *= sc;
                    M = mq[u];
                }
                const float c = expf(mq[u] - M) * eq[u];
                a.x += c * t[u].x;
                a.y += c * t[u].y;
                a.z += c * t[u].z;
                a.w += c * t[u].w;
                W += c;
            }
        }
        part[prow][d4] = a;
        if (d4 == 0) {
            rowm[prow] = M;
            roww[prow] = W;
        }
        __syncthreads();
        if (tid < D4) {
            float Mg = -INFINITY;
#pragma unroll
            for (int i = 0; i < RSTEP; ++i) Mg = fmaxf(Mg, rowm[i]);
            float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
            float Wg = 0.f;
#pragma unroll
            for (int i = 0; i < RSTEP; ++i) {
                if (rowm[i] == -INFINITY) continue;
                const float c = expf(rowm[i] - Mg);
                const float4 v = part[i][tid];
                sum.x += c * v.x;
                sum.y += c * v.y;
                sum.z += c * v.z;
                sum.w += c * v.w;
                Wg += c * roww[i];
            }
            const float inv = 1.f / Wg;
            a = make_float4(sum.x * inv, sum.y * inv, sum.z * inv, sum.w * inv);
        }
        // statistics: sequence frame -> absolute ALiBi positions (every read of
        // max_logits above happened before the barrier)
        if (p.alibi) {
            const float shift = __ldg(p.alibi + h) * (float)(len - 1);
            for (int q = p0 + tid; q < P; q += NT) ml[q] += shift;
        }
    }
    if (tid < D4) {
        T* dst = o + 4 * tid;
        if constexpr (std::is_same<T, float>::value) {
            *reinterpret_cast<float4*>(dst) = a;
        } else {
            constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
            uint2 v;
            v.x = pack2<BF>(a.x, a.y);
            v.y = pack2<BF>(a.z, a.w);
            *reinterpret_cast<uint2*>(dst) = v;
        }
    }
    for (int q = P + tid; q < p.max_parts; q += NT) {
        ml[q] = -INFINITY;
        es[q] = 0.f;
    }
    for (int q = tid; q < p0 && q < P; q += NT) {
        ml[q] = -INFINITY;
        es[q] = 0.f;
    }
}

// Phase 2 of one (query row, head) by one warp: M = max_p m_p, w_p = exp(m_p
// - M) e_p / sum, out = sum_p w_p tmp_p.  Lane i holds the statistics of
// partitions p0 + i, p0 + i + 32, ... and HEAD/32 columns of every partition
// output; the first eight partition outputs are loaded together with the
// statistics, so a row of up to eight partitions costs one round trip.  Then
// the row's statistics move to absolute ALiBi positions and its unused
// partitions are padded (every read of them is above, in this warp).
// L2ONLY: every load through L2 only (the merge inside the partition kernel
// reads what other CTAs of the same grid wrote); otherwise the partition
// outputs are read with an evict_first hint (their last use).
template <typename T, int HEAD, bool L2ONLY>
__device__ __forceinline__ void merge_row_warp(const Params& p, int64_t row, int h, int len, int qn, int qi,
                                               int lane) {
    constexpr int VEC = HEAD / 32;  // columns per lane: 4 (HEAD 128) or 2 (HEAD 64)
    constexpr int PRE = 8;          // partition outputs loaded before the weights are known
    const int hi = len - qn + qi;                      // the query token's position
    const int P = hi >= 0 ? (hi + kPart) / kPart : 0;  // partitions holding its keys
    const int p0 = window_lo_at(p, hi) / kPart;        // partitions before p0: outside the window
    const int64_t sb = (row * p.num_heads + h) * p.max_parts;
    float* ml = p.max_logits + sb;
    float* es = p.exp_sums + sb;
    const float* tmp = p.tmp_out + sb * HEAD + lane * VEC;

    // partition outputs p0 .. p0 + 7 and this lane's first statistics, all in flight
    const uint64_t pol = l2_policy_evict_first();  // partition outputs: last use
    auto load_out = [&](int q, float (&t)[VEC]) {
        if constexpr (VEC == 4) {
            const float4 v = L2ONLY ? __ldcg(reinterpret_cast<const float4*>(tmp + (int64_t)q * HEAD))
                                    : ld_global_v4_hint(tmp + (int64_t)q * HEAD, pol);
            t[0] = v.x; t[1] = v.y; t[2] = v.z; t[3] = v.w;
        } else {
            const float2 v = L2ONLY ? __ldcg(reinterpret_cast<const float2*>(tmp + (int64_t)q * HEAD))
                                    : ld_global_v2_hint(tmp + (int64_t)q * HEAD, pol);
            t[0] = v.x; t[1] = v.y;
        }
    };
    auto ld_stat = [&](const float* a) { return L2ONLY ? __ldcg(a) : *a; };
    float pre[PRE][VEC];
#pragma unroll
    for (int k = 0; k < PRE; ++k) {
        if (p0 + k < P) {
            load_out(p0 + k, pre[k]);
        } else {
#pragma unroll
            for (int v = 0; v < VEC; ++v) pre[k][v] = 0.f;
        }
    }
    const int q1 = p0 + lane;
    const float m1 = q1 < P ? ld_stat(ml + q1) : -INFINITY;
    const float e1 = q1 < P ? ld_stat(es + q1) : 0.f;

    // global max and weight sum over the row's partitions (lanes, then the warp)
    float M = m1, W = m1 == -INFINITY ? 0.f : e1;
    for (int q = q1 + 32; q < P; q += 32) {
        const float m = ld_stat(ml + q), e = ld_stat(es + q);
        if (m == -INFINITY) continue;
        if (m > M) {
            W = (M == -INFINITY) ? 0.f : W * expf(M - m);
            M = m;
        }
        W += expf(m - M) * e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float Mo = __shfl_xor_sync(0xffffffffu, M, o), Wo = __shfl_xor_sync(0xffffffffu, W, o);
        const float Mn = fmaxf(M, Mo);
        W = (M == -INFINITY ? 0.f : W * expf(M - Mn)) + (Mo == -INFINITY ? 0.f : Wo * expf(Mo - Mn));
        M = Mn;
    }
    const float invW = W > 0.f ? 1.f / W : 0.f;

    // weighted sum of the partition outputs; lane i holds the weight of
    // partition p0 + 32j + i for the current group j of 32
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
    float c = m1 == -INFINITY ? 0.f : expf(m1 - M) * e1 * invW;
#pragma unroll
    for (int k = 0; k < PRE; ++k) {
        const float ck = __shfl_sync(0xffffffffu, c, k);
#pragma unroll
        for (int v = 0; v < VEC; ++v) acc[v] = fmaf(ck, pre[k][v], acc[v]);
    }
    for (int qb = p0 + PRE; qb < P; qb += PRE) {
        if (((qb - p0) & 31) == 0) {  // next group of 32 partitions
            const int q = qb + lane;
            c = 0.f;
            if (q < P) {
                const float m = ld_stat(ml + q);
                c = m == -INFINITY ? 0.f : expf(m - M) * ld_stat(es + q) * invW;
            }
        }
        float t[PRE][VEC];
#pragma unroll
        for (int k = 0; k < PRE; ++k) {
            if (qb + k < P) {
                load_out(qb + k, t[k]);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v) t[k][v] = 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < PRE; ++k) {
            const float ck = __shfl_sync(0xffffffffu, c, (qb - p0 + k) & 31);
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc[v] = fmaf(ck, t[k][v], acc[v]);
        }
    }

    T* dst = static_cast<T*>(p.out) + (row * p.num_heads + h) * HEAD + lane * VEC;
    if constexpr (std::is_same<T, float>::value) {
        if constexpr (VEC == 4)
            *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        else
            *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
    } else {
        constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
        if constexpr (VEC == 4) {
            uint2 v;
            v.x = pack2<BF>(acc[0], acc[1]);
            v.y = pack2<BF>(acc[2], acc[3]);
            *reinterpret_cast<uint2*>(dst) = v;
        } else {
            *reinterpret_cast<uint32_t*>(dst) = pack2<BF>(acc[0], acc[1]);
        }
    }
    // statistics: sequence frame -> absolute ALiBi positions; unused partitions
    // padded (every read of this row's statistics is above, in this warp)
    __syncwarp();
    const float shift = p.alibi ? __ldg(p.alibi + h) * (float)(len - 1) : 0.f;
    for (int q = lane; q < p.max_parts; q += 32) {
        if (q >= p0 && q < P) {
            if (p.alibi) ml[q] += shift;
        } else {
            ml[q] = -INFINITY;
            es[q] = 0.f;
        }
    }
}

// Phase 2 with one warp per (sequence, query token, head) row, for batches of
// many rows with few partitions each (a CTA per row would need several waves
// of mostly idle CTAs).  No shared memory, no block barrier.
template <typename T, int HEAD, bool MQ>
__global__ void __launch_bounds__(kReduceWarpsPerCta * 32) pa_reduce_warp_kernel(const Params p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait_primary();

    const int64_t rid = (int64_t)blockIdx.x * kReduceWarpsPerCta + warp;
    const int64_t nrows = (int64_t)p.num_seqs * (MQ ? p.max_q_len : 1) * p.num_heads;
    if (rid >= nrows) return;
    const int sq = (int)(rid / p.num_heads), h = (int)(rid - (int64_t)sq * p.num_heads);
    const int s = MQ ? sq / p.max_q_len : sq, qi = MQ ? sq - s * p.max_q_len : 0;
    int q0 = s, qn = 1;
    if constexpr (MQ) {
        query_rows(p, s, q0, qn);
        if (qi >= qn) return;
    }
    const int len = clamp_len(p, p.seq_lens[s]);
    merge_row_warp<T, HEAD, false>(p, (int64_t)q0 + qi, h, len, qn, qi, lane);
}

}  // namespace pa

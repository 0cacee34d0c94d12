// pa_launch.cuh -- host-side launch of the partition (or v1) kernel and of the
// reduce kernel for one (dtype, head size) family.  Included by the
// per-dtype translation units so they compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "pa_kernels.cuh"

namespace pa {

// What a launch would do, reported instead of launching (see LaunchArgs::query).
struct LaunchOut {
    int occ = 0;        // resident CTAs per SM of the partition kernel
    int64_t grid = 0;   // CTAs of its persistent grid
    bool fused = false; // Phase 2 merge inside the partition kernel (no reduce launch)
};

struct LaunchArgs {
    cudaStream_t stream;
    LaunchOut* query;        // non-null: fill it and launch nothing
    const CUtensorMap* tmk;  // NHD 16-bit only (otherwise unused placeholders)
    const CUtensorMap* tmv;
    int sm_count;
    int64_t tiles_upper;     // upper bound on tiles (persistent grid never exceeds it)
    int group_tiles;         // 1 or 2: n-tiles of 8 query heads
    int layout;
    int head_size;
    int dtype;               // pa_dtype of the query
    void* ev_begin;
    void* ev_end;
};

constexpr int kMaxDevices = 64;

// Launch the partition (or v1) kernel.  *fused reports whether the Phase 2
// merge runs inside it: only with partition counters, a v2 batch that fits in
// one round of the persistent grid (each CTA finishes at most one tile, so at
// most one merge) and at most PA_FUSED_MAX_PARTITIONS partitions per sequence
// (a short merge).  With several rounds the CTA that merges falls behind and
// becomes the last arriver of the next group too, so merges pile up on a few
// CTAs; the separate reduce kernel spreads them over the whole GPU instead.
template <typename T, int HEAD, int NT, int LAYOUT, int KV, bool MQ>
cudaError_t launch_main(const Params& p_in, const LaunchArgs& la, bool* fused) {
    constexpr int STAGES = std::is_same<T, float>::value ? (NT == 1 ? kStagesF32 : kStagesF32x2)
                           : (KV == kKvSame ? (NT == 1 ? kStages16 : kStages16x2) : kStagesFp8);
    constexpr int NC = (KV == kKvSame && NT == 1) ? kConsumerWarps5 : kConsumerWarps;
    using C = Cfg<T, HEAD, NT, LAYOUT, STAGES, NC, KV, MQ>;
    auto kern = pa_partition_kernel<T, HEAD, NT, LAYOUT, STAGES, NC, KV, MQ>;

    static std::atomic<int> occ_cache[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int occ = (dev >= 0 && dev < kMaxDevices) ? occ_cache[dev].load() : 0;
    if (occ <= 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::kThreads, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        if (dev >= 0 && dev < kMaxDevices) occ_cache[dev].store(occ);
    }
    int64_t grid = (int64_t)la.sm_count * occ;
    if (grid > la.tiles_upper) grid = la.tiles_upper;
    if (grid < 1) grid = 1;
    // Equal rounds: the fewest CTAs that keep the number of rounds of the
    // static tile schedule, so that in a uniform batch every CTA gets the same
    // number of tiles instead of a last round that leaves most CTAs idle
    // (1024 tiles: 256 CTAs x 4 instead of 304 CTAs with 112 doing a 4th).
    // tiles_upper is exact for equal lengths and only an upper bound otherwise.
    // The dynamic schedule keeps every resident CTA: its tiles go to whichever
    // CTA is free, so no CTA waits on a fixed share.
    if (!p_in.tile_ctr) {
        const int64_t rounds = (la.tiles_upper + grid - 1) / grid;
        grid = (la.tiles_upper + rounds - 1) / rounds;
    }
    Params p = p_in;
    p.fused = (!p.v1 && p.counters && p.max_parts <= PA_FUSED_MAX_PARTITIONS &&
               la.tiles_upper <= grid) ? 1 : 0;
    *fused = p.fused != 0;
    if (la.query) {
        la.query->occ = occ;
        la.query->grid = grid;
        la.query->fused = *fused;
        return cudaSuccess;
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = la.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (la.ev_begin) {
        e = cudaEventRecord(static_cast<cudaEvent_t>(la.ev_begin), la.stream);
        if (e != cudaSuccess) return e;
    }
    e = cudaLaunchKernelEx(&cfg, kern, p, *la.tmk, *la.tmv);
    if (e != cudaSuccess) return e;
    if (la.ev_end) e = cudaEventRecord(static_cast<cudaEvent_t>(la.ev_end), la.stream);
    return e;
}

// Reduce shape by partition count: few partitions need one round of rows,
// long sequences (hundreds of partitions, few (sequence, head) CTAs) want as
// many independent row loads in flight per CTA as possible.
template <typename T, int HEAD, int WARPS, int U, bool MQ>
cudaError_t launch_reduce_shape(const Params& p, const LaunchArgs& la) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)p.num_seqs * p.max_q_len * p.num_heads));
    cfg.blockDim = dim3(WARPS * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = la.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pa_reduce_kernel<T, HEAD, WARPS, U, MQ>, p);
}

template <typename T, int HEAD, bool MQ>
cudaError_t launch_reduce_warp(const Params& p, const LaunchArgs& la, int64_t rows) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + kReduceWarpsPerCta - 1) / kReduceWarpsPerCta));
    cfg.blockDim = dim3(kReduceWarpsPerCta * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = la.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pa_reduce_warp_kernel<T, HEAD, MQ>, p);
}

template <typename T, int HEAD, bool MQ>
cudaError_t launch_reduce(const Params& p, const LaunchArgs& la) {
    // Few (sequence, head) rows of many partitions (4 x 28 rows of 196): a
    // wide CTA per row; otherwise one warp per row, so that a batch of
    // thousands of short rows runs in one wave instead of several waves of
    // CTAs that each wait on one round trip.
    const int64_t rows = (int64_t)p.num_seqs * p.max_q_len * p.num_heads;
    if (p.max_parts > 32 && rows <= 2 * (int64_t)la.sm_count)
        return launch_reduce_shape<T, HEAD, 16, 8, MQ>(p, la);
    if (p.max_parts <= kReduceWarpMaxParts) return launch_reduce_warp<T, HEAD, MQ>(p, la, rows);
    return launch_reduce_shape<T, HEAD, 8, 4, MQ>(p, la);
}

template <typename T, int HEAD, int NT, int KV, bool MQ>
cudaError_t launch_layout_mq(const Params& p, const LaunchArgs& la, bool* fused) {
    return la.layout == kNHD ? launch_main<T, HEAD, NT, kNHD, KV, MQ>(p, la, fused)
                             : launch_main<T, HEAD, NT, kSplit, KV, MQ>(p, la, fused);
}

// Single-token decode and several query tokens per sequence are separate
// instantiations, so the common single-token path carries no per-row ranges.
template <typename T, int HEAD, int NT, int KV>
cudaError_t launch_layout(const Params& p, const LaunchArgs& la, bool* fused) {
    return p.query_start ? launch_layout_mq<T, HEAD, NT, KV, true>(p, la, fused)
                         : launch_layout_mq<T, HEAD, NT, KV, false>(p, la, fused);
}

// Whole operation for one (query type, cache type) pair.
template <typename T, int KV = kKvSame>
cudaError_t launch_family(const Params& p, const LaunchArgs& la) {
    cudaError_t e;
    bool fused = false;
    if (la.head_size == 128) {
        e = la.group_tiles == 2 ? launch_layout<T, 128, 2, KV>(p, la, &fused)
                                : launch_layout<T, 128, 1, KV>(p, la, &fused);
    } else {
        e = la.group_tiles == 2 ? launch_layout<T, 64, 2, KV>(p, la, &fused)
                                : launch_layout<T, 64, 1, KV>(p, la, &fused);
    }
    if (e != cudaSuccess || p.v1 || fused || la.query) return e;
    if (p.query_start)
        return la.head_size == 128 ? launch_reduce<T, 128, true>(p, la) : launch_reduce<T, 64, true>(p, la);
    return la.head_size == 128 ? launch_reduce<T, 128, false>(p, la) : launch_reduce<T, 64, false>(p, la);
}

cudaError_t launch_f32(const Params& p, const LaunchArgs& la);
cudaError_t launch_f16(const Params& p, const LaunchArgs& la);
cudaError_t launch_bf16(const Params& p, const LaunchArgs& la);
cudaError_t launch_f16_fp8(const Params& p, const LaunchArgs& la, int kv);   // kv: kKvE4M3 / kKvE5M2
cudaError_t launch_bf16_fp8(const Params& p, const LaunchArgs& la, int kv);

}  // namespace pa

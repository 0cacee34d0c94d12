// pa_decode.cu -- the C ABI of include/pa_decode.h: argument checks, v1/v2
// choice, grid sizing, tensor maps for the NHD layout, launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "pa_decode.h"
#include "pa_launch.cuh"

namespace {

using pa::Params;

constexpr int kMaxDevices = pa::kMaxDevices;

// ---------------------------------------------------------------- device info

int sm_count_for_current_device(int* out) {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    int v = (dev >= 0 && dev < kMaxDevices) ? cache[dev].load() : 0;
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        if (dev >= 0 && dev < kMaxDevices) cache[dev].store(v);
    }
    *out = v;
    return 0;
}

int l2_bytes_for_current_device(int* out) {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    int v = (dev >= 0 && dev < kMaxDevices) ? cache[dev].load() : 0;
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return -1;
        if (dev >= 0 && dev < kMaxDevices) cache[dev].store(v);
    }
    *out = v;
    return 0;
}

// ---------------------------------------------------------------- tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// NHD page of one kv head = 16 rows of head_size elements.  The map views a
// cache as 3-D: (E = 128 / elem elements of a row: one 128-byte chunk, the
// rows [num_blocks * num_kv_heads * 16], the head_size / E chunks of a row),
// strides (row: head_size * elem bytes, chunk: 128 bytes), and moves a whole
// page as one box (E, 16, head_size / E): in shared memory the page lands as
// head_size / E blocks of 16 rows x 128 bytes, each with the 128-byte swizzle,
// so that the kernel's shared-memory reads are free of bank conflicts -- the
// layout of one 2-D box per chunk, with one copy instead of two (16-bit) or
// four (fp32).
bool make_nhd_map(CUtensorMap* map, const void* base, int64_t rows, int head_size, pa_dtype dt) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int elem = dt == PA_DTYPE_F32 ? 4 : 2;
    const int e = 128 / elem;  // elements of a 128-byte chunk
    cuuint64_t dims[3] = {(cuuint64_t)e, (cuuint64_t)rows, (cuuint64_t)(head_size / e)};
    cuuint64_t strides[2] = {(cuuint64_t)head_size * elem, 128};
    cuuint32_t box[3] = {(cuuint32_t)e, 16, (cuuint32_t)(head_size / e)};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType t = dt == PA_DTYPE_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : dt == PA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(map, t, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// fp8 NHD page of one kv head = 16 rows of head_size bytes: one box of the
// whole page, swizzled by 128 bytes (head_size 128) or 64 bytes (64) so the
// kernel's four-byte reads of eight token rows fall in distinct banks.
bool make_nhd_map_fp8(CUtensorMap* map, const void* base, int64_t rows, int head_size) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)head_size, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_size};
    cuuint32_t box[2] = {(cuuint32_t)head_size, 16};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    head_size == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Test hook of pa_debug_withhold_page (process-wide).
std::atomic<int> g_withhold_page{0};
std::atomic<int64_t> g_wait_limit_ns{0};

/*
 * v1 / v2 choice.  The pages pick v2 when the v2 tiles of one sequence (kv
 * heads x partitions) exceed twice the SM count of their 16-SM part
 * (should_use_paged_v2 in "ex_engine/factors/attn_dispatch.py").  Here both
 * modes run the same persistent kernel, so the choice compares its two grids:
 * v1 makes one tile per (sequence, kv head) over the whole sequence and writes
 * the output directly; v2 makes one tile per 512-token partition and adds the
 * partition statistics round trip, an epilogue per partition and the reduce.
 * v1 measured 2-4 % faster than v2 when its tiles fill the GPU evenly (128 x
 * 16384 on GB300: 1232 against 1288 us; 64 x 4096: 82.4 against 85.1 us) and
 * far slower when one long sequence holds a CTA while the others idle.  So:
 *  - one partition per sequence (max_seq_len <= 512): v1 (v2 would only add
 *    the round trip);
 *  - v1 tiles (num_seqs x num_kv_heads) fewer than the SMs: v2;
 *  - otherwise v1 if the persistent grid's static round-robin of the v1 tiles
 *    (sm_count x ctas_per_sm resident CTAs, cut to equal rounds, as the launch
 *    does) loads its busiest CTA with at most 10 % more pages than the mean,
 *    else v2.
 * `len(i)` is the length of sequence i, clamped into [0, max_seq_len].
 */
template <class Len>
int32_t choose_by_balance(int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len, int32_t sm_count,
                          int32_t ctas_per_sm, Len len) {
    if (max_seq_len <= PA_PARTITION_SIZE) return PA_MODE_V1;
    if (num_seqs <= 0 || num_kv_heads <= 0 || sm_count <= 0) return PA_MODE_V2;
    const int64_t tiles = (int64_t)num_seqs * num_kv_heads;
    if (tiles < sm_count) return PA_MODE_V2;
    const int64_t resident = (int64_t)sm_count * (ctas_per_sm > 0 ? ctas_per_sm : 2);
    const int64_t rounds = (tiles + resident - 1) / resident;
    const int64_t grid = (tiles + rounds - 1) / rounds;
    std::vector<int64_t> load((size_t)grid, 0);
    int64_t total = 0;
    for (int32_t sq = 0; sq < num_seqs; ++sq) {
        int64_t l = len(sq);
        l = l < 0 ? 0 : (l > max_seq_len ? max_seq_len : l);
        const int64_t pages = (l + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
        for (int32_t h = 0; h < num_kv_heads; ++h) load[(size_t)(((int64_t)sq * num_kv_heads + h) % grid)] += pages;
        total += pages * num_kv_heads;
    }
    int64_t mx = 0;
    for (int64_t v : load) mx = v > mx ? v : mx;
    return (double)mx * grid <= 1.1 * (double)total ? PA_MODE_V1 : PA_MODE_V2;
}


// Arguments of one call, checked and turned into kernel parameters.
struct Prepared {
    Params p;
    pa::LaunchArgs la;
    alignas(64) CUtensorMap tmk;
    alignas(64) CUtensorMap tmv;
    int kv = PA_KV_SAME;
    int ctas_per_sm = 0;
    bool empty = false;  // num_seqs == 0: nothing to launch
};

// The kernels of the (query type, cache type) pair: launch them, or with
// `out` only report the partition kernel's occupancy, grid and merge choice.
pa_status dispatch(Prepared& pr, pa::LaunchOut* out) {
    pr.la.query = out;
    const int kvk = pr.kv == PA_KV_FP8_E4M3 ? pa::kKvE4M3 : pa::kKvE5M2;
    cudaError_t e;
    switch (pr.la.dtype) {
    case PA_DTYPE_F32: e = pa::launch_f32(pr.p, pr.la); break;
    case PA_DTYPE_F16: e = pr.kv == PA_KV_SAME ? pa::launch_f16(pr.p, pr.la) : pa::launch_f16_fp8(pr.p, pr.la, kvk); break;
    default: e = pr.kv == PA_KV_SAME ? pa::launch_bf16(pr.p, pr.la) : pa::launch_bf16_fp8(pr.p, pr.la, kvk); break;
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}

// Host-visible checks of pa_decode (every error returned before any launch),
// then the kernel parameters, the v1 / v2 choice and the tile order.
pa_status prepare(const pa_decode_args* a, void* stream, Prepared& pr) {
    if (!a) return PA_ERR_INVALID_ARG;
    if (a->num_seqs < 0 || a->num_heads <= 0 || a->num_kv_heads <= 0 || a->max_seq_len < 0 ||
        a->num_blocks < 0 || a->max_blocks_per_seq < 0)
        return PA_ERR_INVALID_ARG;
    if (a->num_heads % a->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (a->dtype != PA_DTYPE_F32 && a->dtype != PA_DTYPE_F16 && a->dtype != PA_DTYPE_BF16)
        return PA_ERR_INVALID_ARG;
    if (a->layout != PA_LAYOUT_SPLIT && a->layout != PA_LAYOUT_NHD) return PA_ERR_INVALID_ARG;
    if (a->mode != PA_MODE_AUTO && a->mode != PA_MODE_V1 && a->mode != PA_MODE_V2)
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(a->scale) || !std::isfinite(a->softcap) || !std::isfinite(a->k_scale) ||
        !std::isfinite(a->v_scale))
        return PA_ERR_INVALID_ARG;
    const int kv = a->kv_dtype;
    if (kv != PA_KV_SAME && kv != PA_KV_FP8_E4M3 && kv != PA_KV_FP8_E5M2) return PA_ERR_INVALID_ARG;
    if (kv != PA_KV_SAME && a->dtype == PA_DTYPE_F32) return PA_ERR_UNSUPPORTED;
    if (a->block_size != PA_BLOCK_SIZE) return PA_ERR_UNSUPPORTED;
    if (a->head_size != 64 && a->head_size != 128) return PA_ERR_UNSUPPORTED;
    const int group = a->num_heads / a->num_kv_heads;
    if (group > 16) return PA_ERR_UNSUPPORTED;
    // several query tokens per sequence: all tokens of a (sequence, kv head)
    // share one tile, their group rows side by side (at most 16)
    const bool multi = a->query_start != nullptr;
    const int max_q = multi ? a->max_query_len : 1;
    if (multi && (a->max_query_len < 1 || a->num_query_tokens < 0 || !aligned(a->query_start, 4)))
        return PA_ERR_INVALID_ARG;
    if ((int64_t)max_q * group > 16) return PA_ERR_UNSUPPORTED;
    if (a->num_seqs == 0) {
        pr.empty = true;
        return PA_OK;
    }
    if (!a->out || !a->query || !a->key_cache || !a->value_cache || !a->block_tables || !a->seq_lens)
        return PA_ERR_INVALID_ARG;
    if (a->num_blocks == 0) return PA_ERR_INVALID_ARG;
    if ((int64_t)a->max_blocks_per_seq * PA_BLOCK_SIZE < (int64_t)a->max_seq_len)
        return PA_ERR_INVALID_ARG;
    if (!aligned(a->out, 16) || !aligned(a->query, 16) || !aligned(a->key_cache, 16) ||
        !aligned(a->value_cache, 16) || !aligned(a->block_tables, 4) || !aligned(a->seq_lens, 4) ||
        !aligned(a->alibi_slopes, 4) || !aligned(a->partition_counters, 4) || !aligned(a->tile_counters, 4))
        return PA_ERR_INVALID_ARG;
    const int max_parts = pa_max_num_partitions(a->max_seq_len);
    auto workspace_ok = [a] {
        return a->exp_sums && a->max_logits && a->tmp_out && aligned(a->tmp_out, 16) &&
               aligned(a->exp_sums, 4) && aligned(a->max_logits, 4);
    };
    // v2 asked for: the workspace is checked before anything touches the device
    // (AUTO checks it once the mode is chosen)
    if (a->mode == PA_MODE_V2 && !workspace_ok()) return PA_ERR_WORKSPACE;
    if ((int64_t)a->num_seqs * max_q * a->num_heads >= (int64_t)1 << 31) return PA_ERR_UNSUPPORTED;
    if ((int64_t)a->num_seqs * max_parts * a->num_kv_heads >= (int64_t)1 << 31) return PA_ERR_UNSUPPORTED;

    int sm = 0;
    if (sm_count_for_current_device(&sm) != 0) return PA_ERR_LAUNCH;

    Params& p = pr.p;
    std::memset(&p, 0, sizeof p);
    p.query = a->query;
    p.key_cache = a->key_cache;
    p.value_cache = a->value_cache;
    p.block_tables = a->block_tables;
    p.seq_lens = a->seq_lens;
    p.alibi = a->alibi_slopes;
    p.out = a->out;
    p.exp_sums = a->exp_sums;
    p.max_logits = a->max_logits;
    p.tmp_out = a->tmp_out;
    p.dev_error = a->dev_error;
    p.num_seqs = a->num_seqs;
    p.num_heads = a->num_heads;
    p.num_kv_heads = a->num_kv_heads;
    p.group = group;
    p.num_blocks = a->num_blocks;
    p.max_blocks_per_seq = a->max_blocks_per_seq;
    p.max_seq_len = a->max_seq_len;
    p.max_parts = max_parts;
    const float k_scale = (kv != PA_KV_SAME && a->k_scale > 0.f) ? a->k_scale : 1.f;
    p.scale = a->scale * k_scale;  // q.(k_scale k8) = k_scale (q.k8): folded into the logit scale
    p.v_scale = (kv != PA_KV_SAME && a->v_scale > 0.f) ? a->v_scale : 1.f;
    p.softcap = a->softcap > 0.f ? a->softcap : 0.f;
    p.inv_softcap = a->softcap > 0.f ? 1.f / a->softcap : 0.f;
    p.counters = a->partition_counters;
    p.window_left = a->sliding_window > 0 ? a->sliding_window - 1 : -1;
    p.query_start = a->query_start;
    p.max_q_len = max_q;
    p.num_q_rows = multi ? a->num_query_tokens : a->num_seqs;
    p.fused = 0;  // decided at launch, once the persistent grid size is known
    p.wait_limit_ns = (uint64_t)g_wait_limit_ns.load();
    p.withhold_page = g_withhold_page.load();
    p.tile_ctr = nullptr;  // set below once the mode is known
    p.metadata_ready = a->metadata_ready ? 1 : 0;

    pa::LaunchArgs& la = pr.la;
    std::memset(&la, 0, sizeof la);
    la.stream = static_cast<cudaStream_t>(stream);
    la.tmk = &pr.tmk;
    la.tmv = &pr.tmv;
    std::memset(&pr.tmk, 0, sizeof pr.tmk);
    std::memset(&pr.tmv, 0, sizeof pr.tmv);
    la.sm_count = sm;
    la.group_tiles = max_q * group > 8 ? 2 : 1;
    la.layout = a->layout;
    la.head_size = a->head_size;
    la.dtype = a->dtype;
    la.ev_begin = a->event_main_begin;
    la.ev_end = a->event_main_end;
    pr.kv = kv;

    // resident CTAs per SM of the partition kernel of this call (the same
    // kernel runs v1 and v2): the persistent grid and the v1 / v2 choice use it
    {
        pa::LaunchOut lo;
        la.tiles_upper = 1;
        if (dispatch(pr, &lo) != PA_OK) return PA_ERR_LAUNCH;
        pr.ctas_per_sm = lo.occ;
    }
    int mode = a->mode;
    if (mode == PA_MODE_AUTO)
        mode = pa_choose_mode_for_lengths(a->num_seqs, a->num_kv_heads, a->max_seq_len, sm, pr.ctas_per_sm,
                                          a->seq_lens_host);
    const bool v1 = mode == PA_MODE_V1;
    if (!v1 && !workspace_ok()) return PA_ERR_WORKSPACE;
    p.v1 = v1 ? 1 : 0;
    la.tiles_upper = (int64_t)a->num_seqs * (v1 ? 1 : max_parts) * a->num_kv_heads;
    // Dynamic tile schedule: only for batches whose tiles differ in size (the
    // host lengths hold sequences of different page counts in v1, partition
    // counts in v2), where it balanced the ragged workload (551 -> 536 us);
    // for equal tiles the static equal-round grid measured faster (gqa4k 47.1
    // against 49.6 us; large_batch v1 1224 against 1300 us).
    if (a->tile_counters && a->seq_lens_host) {
        auto units_of = [&](int32_t i) {
            int64_t l = a->seq_lens_host[i];
            l = l < 0 ? 0 : (l > a->max_seq_len ? a->max_seq_len : l);
            return v1 ? (l + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE : (l + PA_PARTITION_SIZE - 1) / PA_PARTITION_SIZE;
        };
        bool varied = false;
        const int64_t u0 = units_of(0);
        for (int32_t i = 1; i < a->num_seqs && !varied; ++i) varied = units_of(i) != u0;
        if (varied) p.tile_ctr = a->tile_counters;
    }
    // KV copies marked evict_first while the partition outputs (at most the
    // workspace) take no more than half of L2; with larger workspaces it was
    // measured to slow the partition kernel (128 x 16384: +1.6 %)
    {
        int l2 = 0;
        if (l2_bytes_for_current_device(&l2) != 0) return PA_ERR_LAUNCH;
        const int64_t rows = multi ? a->num_query_tokens : a->num_seqs;
        const int64_t tmp_bytes = v1 ? 0 : rows * a->num_heads * (int64_t)max_parts * a->head_size * 4;
        p.kv_evict_first = tmp_bytes <= (int64_t)l2 / 2 ? 1 : 0;
    }
    return PA_OK;
}

}  // namespace

extern "C" {

int32_t pa_version(void) { return (1 << 16) | 0; }

int32_t pa_max_num_partitions(int32_t max_seq_len) {
    if (max_seq_len <= 0) return 1;
    return (int32_t)(((int64_t)max_seq_len + PA_PARTITION_SIZE - 1) / PA_PARTITION_SIZE);
}

pa_status pa_workspace_elems(int32_t num_seqs, int32_t num_heads, int32_t head_size,
                             int32_t max_seq_len, int64_t* stats_elems, int64_t* tmp_elems) {
    if (num_seqs < 0 || num_heads <= 0 || head_size <= 0 || max_seq_len < 0) return PA_ERR_INVALID_ARG;
    const int64_t s = (int64_t)num_seqs * num_heads * pa_max_num_partitions(max_seq_len);
    if (stats_elems) *stats_elems = s;
    if (tmp_elems) *tmp_elems = s * head_size;
    return PA_OK;
}

size_t pa_workspace_bytes(int32_t rows, int32_t num_heads, int32_t head_size, int32_t max_seq_len) {
    int64_t stats = 0, tmp = 0;
    if (pa_workspace_elems(rows, num_heads, head_size, max_seq_len, &stats, &tmp) != PA_OK) return 0;
    return (size_t)(2 * stats + tmp) * sizeof(float);
}

int32_t pa_partition_size(void) { return PA_PARTITION_SIZE; }

/* Without host lengths every sequence is taken to be max_seq_len long (the
 * pages' rule decides from one length too). */
int32_t pa_choose_mode(int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len, int32_t sm_count,
                       int32_t ctas_per_sm) {
    return choose_by_balance(num_seqs, num_kv_heads, max_seq_len, sm_count, ctas_per_sm,
                             [max_seq_len](int32_t) { return (int64_t)max_seq_len; });
}

int32_t pa_choose_mode_for_lengths(int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len,
                                   int32_t sm_count, int32_t ctas_per_sm, const int32_t* seq_lens_host) {
    if (!seq_lens_host) return pa_choose_mode(num_seqs, num_kv_heads, max_seq_len, sm_count, ctas_per_sm);
    return choose_by_balance(num_seqs, num_kv_heads, max_seq_len, sm_count, ctas_per_sm,
                             [seq_lens_host](int32_t i) { return (int64_t)seq_lens_host[i]; });
}


const char* pa_status_str(int32_t status) {
    switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_WORKSPACE: return "v2 workspace (exp_sums / max_logits / tmp_out) missing or misaligned";
    case PA_ERR_LAUNCH: return "CUDA launch failed";
    case PA_ERR_DEVICE_CHECK: return "device-side argument check failed";
    case PA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
    }
}

pa_status pa_debug_withhold_page(int32_t enable, int64_t wait_limit_ns) {
    if (wait_limit_ns < 0) return PA_ERR_INVALID_ARG;
    g_wait_limit_ns.store(wait_limit_ns);
    g_withhold_page.store(enable ? 1 : 0);
    return PA_OK;
}

pa_status pa_plan(const pa_decode_args* a, pa_launch_plan* plan) {
    if (!plan) return PA_ERR_INVALID_ARG;
    std::memset(plan, 0, sizeof *plan);
    Prepared pr;
    const pa_status st = prepare(a, nullptr, pr);
    if (st != PA_OK || pr.empty) return st;
    pa::LaunchOut lo;
    const pa_status q = dispatch(pr, &lo);
    if (q != PA_OK) return q;
    plan->mode = pr.p.v1 ? PA_MODE_V1 : PA_MODE_V2;
    plan->merge_in_kernel = lo.fused ? 1 : 0;
    plan->kernels = (pr.p.v1 || lo.fused) ? 1 : 2;
    plan->ctas_per_sm = pr.ctas_per_sm;
    plan->grid = (int32_t)lo.grid;
    plan->dynamic_schedule = pr.p.tile_ctr ? 1 : 0;
    plan->tiles = pr.la.tiles_upper;
    return PA_OK;
}

pa_status pa_decode(const pa_decode_args* a, void* stream) {
    Prepared pr;
    const pa_status st = prepare(a, stream, pr);
    if (st != PA_OK || pr.empty) return st;
    // NHD pages come through tensor maps
    if (a->layout == PA_LAYOUT_NHD) {
        const int64_t rows = (int64_t)a->num_blocks * a->num_kv_heads * PA_BLOCK_SIZE;
        if (rows > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;  // tensor-map row coordinate is int32
        const bool ok = pr.kv != PA_KV_SAME
                            ? make_nhd_map_fp8(&pr.tmk, a->key_cache, rows, a->head_size) &&
                                  make_nhd_map_fp8(&pr.tmv, a->value_cache, rows, a->head_size)
                            : make_nhd_map(&pr.tmk, a->key_cache, rows, a->head_size, (pa_dtype)a->dtype) &&
                                  make_nhd_map(&pr.tmv, a->value_cache, rows, a->head_size, (pa_dtype)a->dtype);
        if (!ok) return PA_ERR_LAUNCH;
    }
    return dispatch(pr, nullptr);
}

}  // extern "C"

/*
 * pa_decode.h -- C ABI of the GB300 (sm_103a) paged-KV decode attention library.
 *
 * One query token per sequence (or several, see query_start) attends over
 * that sequence's keys and values, which live in fixed-size pages ("blocks")
 * of a shared cache and are found through a per-sequence block table.  The operation is the one of
 * "paged_attention_v2_pytorch.py -- BI-V100 PagedAttention V2 implementation"
 * (function paged_attention_v2_pytorch, Phase 1 per-partition attention and
 * Phase 2 log-sum-exp reduce), with the NHD cache layout and the `softcap`
 * field of "ex_engine/factors/attn_dispatch.py" (AttnDispatchConfig,
 * dispatch_decode).
 *
 * For sequence s, query head h (kv head g = h / (num_heads / num_kv_heads))
 * and token t < seq_lens[s]:
 *     z_t = scale * <query[s][h], K_g(t)>
 *     z_t = softcap * tanh(z_t / softcap)          if softcap > 0
 *     z_t = z_t + alibi_slopes[h] * t              if alibi_slopes != NULL
 *     out[s][h] = sum_t exp(z_t - max z) V_g(t) / sum_t exp(z_t - max z)
 * (t restricted to the last sliding_window keys when sliding_window > 0).
 * K_g(t) is read from physical block block_tables[s][t / block_size] at slot
 * t % block_size.  Sequences are cut into partitions of PA_PARTITION_SIZE
 * tokens; for partition p (tokens [512p, min(512p+512, seq_len))):
 *     max_logits[s][h][p] = max z_t
 *     exp_sums[s][h][p]   = sum exp(z_t - max_logits[s][h][p])
 *     tmp_out[s][h][p][:] = sum exp(z_t - max_logits) V(t) / exp_sums[s][h][p]
 * and the output is their log-sum-exp merge (equal to the dense softmax).
 *
 * Conventions for every entry point below:
 *  - All tensor pointers are DEVICE pointers (global memory of the current
 *    device), caller-owned and caller-allocated, except seq_lens_host (host
 *    memory, read during the call); the library allocates no device memory
 *    and keeps no state except per-device cached attributes (and the array of
 *    pa_decode_static_workspace).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous on that stream and never synchronise the host.
 *  - Errors the host can see are returned before anything is launched.
 *    Data-dependent errors are reported through the optional device word
 *    `dev_error` (bit flags PA_DEVERR_*), set with atomicOr; the kernels
 *    clamp the offending value and continue, they never trap.
 */
#ifndef PA_DECODE_H
#define PA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Tokens per partition (module constant _PARTITION_SIZE of
 * paged_attention_v2_pytorch.py). */
#define PA_PARTITION_SIZE 512

/* Tokens per cache page supported by this library. */
#define PA_BLOCK_SIZE 16

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer     */
    PA_ERR_UNSUPPORTED = 2,   /* valid but not built: head_size, block_size ... */
    PA_ERR_WORKSPACE = 3,     /* v2 selected but exp_sums/max_logits/tmp_out NULL */
    PA_ERR_LAUNCH = 4,        /* CUDA reported an error while launching         */
    PA_ERR_DEVICE_CHECK = 5,  /* reserved for callers mapping dev_error bits    */
    PA_ERR_DEVICE_TIMEOUT = 6 /* reserved for callers mapping dev_error bits    */
} pa_status;

/* Storage type of query and out (and of the caches unless kv_dtype says otherwise). */
typedef enum pa_dtype { PA_DTYPE_F32 = 0, PA_DTYPE_F16 = 1, PA_DTYPE_BF16 = 2 } pa_dtype;

/* Storage type of key_cache / value_cache (kv_cache_dtype / k_scale / v_scale of
 * paged_attention_v2_pytorch.py): the caches hold K / k_scale and V / v_scale. */
typedef enum pa_kv_dtype {
    PA_KV_SAME = 0,      /* same as dtype */
    PA_KV_FP8_E4M3 = 3,  /* OCP fp8 E4M3 (bias 7, no infinities); f16/bf16 query */
    PA_KV_FP8_E5M2 = 4   /* OCP fp8 E5M2 (bias 15); f16/bf16 query */
} pa_kv_dtype;

/*
 * Cache layouts.
 *  PA_LAYOUT_SPLIT: key_cache   [num_blocks][num_kv_heads][head_size/x][block_size][x],
 *                   x = 16 / sizeof(element) (16 for fp8, 8 for f16/bf16, 4 for f32);
 *                   value_cache [num_blocks][num_kv_heads][head_size][block_size]
 *                   (key_cache / value_cache shape comments of
 *                   paged_attention_v2_pytorch.py).
 *  PA_LAYOUT_NHD:   key_cache and value_cache [num_blocks][num_kv_heads][block_size][head_size]
 *                   (dispatch_decode argument comments of attn_dispatch.py).
 * All arrays are dense, row-major, without padding.
 */
typedef enum pa_layout { PA_LAYOUT_SPLIT = 0, PA_LAYOUT_NHD = 1 } pa_layout;

/*
 * PA_MODE_V2: partition kernel over (sequence, kv head, 512-token partition)
 *             tiles, then the log-sum-exp reduce (needs the workspace).
 * PA_MODE_V1: one pass per (sequence, kv head) over the whole sequence that
 *             writes `out` directly (no workspace, no statistics).
 * PA_MODE_AUTO: the library picks (pa_choose_mode).
 */
typedef enum pa_mode { PA_MODE_AUTO = 0, PA_MODE_V1 = 1, PA_MODE_V2 = 2 } pa_mode;

/* dev_error bits */
#define PA_DEVERR_BLOCK_ID   1  /* a block table entry outside [0, num_blocks); page 0 read instead */
#define PA_DEVERR_SEQ_LEN    2  /* seq_lens[s] < 0 or > max_seq_len; clamped into [0, max_seq_len] */
#define PA_DEVERR_TIMEOUT    4  /* an internal pipeline wait exceeded its limit; results invalid   */
#define PA_DEVERR_QUERY_RANGE 8 /* fp8 caches with a bf16 query: |q| > 65504 clamped (fp16 MMAs)  */

typedef struct pa_decode_args {
    /* [rows][num_heads][head_size], dtype; written.  16-byte aligned.
     * rows = num_seqs, or num_query_tokens with query_start (below). */
    void* out;
    /* [rows][num_heads][head_size], dtype.  16-byte aligned. */
    const void* query;
    /* layout-dependent, see pa_layout; 16-byte aligned. */
    const void* key_cache;
    const void* value_cache;
    /* [num_seqs][max_blocks_per_seq] int32 physical block ids; only the first
     * ceil(seq_lens[s] / block_size) entries of row s are read. */
    const int32_t* block_tables;
    /* [num_seqs] int32 tokens per sequence, each in [0, max_seq_len]. */
    const int32_t* seq_lens;
    int32_t num_seqs;
    int32_t num_heads;
    int32_t num_kv_heads;        /* num_heads % num_kv_heads == 0, group <= 16 */
    int32_t head_size;           /* 64 or 128 */
    int32_t num_blocks;          /* pages in each cache */
    int32_t block_size;          /* must be PA_BLOCK_SIZE */
    int32_t max_seq_len;         /* upper bound of seq_lens; sets max_num_partitions */
    int32_t max_blocks_per_seq;  /* row stride of block_tables, >= ceil(max_seq_len/block_size) */
    float scale;                 /* logit scale, e.g. 1/sqrt(head_size) */
    float softcap;               /* > 0: z = softcap * tanh(z / softcap); <= 0: off */
    /* [num_heads] fp32 ALiBi slopes, or NULL. */
    const float* alibi_slopes;
    int32_t dtype;               /* pa_dtype */
    int32_t layout;              /* pa_layout */
    int32_t mode;                /* pa_mode */
    /* Workspace (required for v2, ignored by v1); P = pa_max_num_partitions(max_seq_len):
     *   exp_sums, max_logits [rows][num_heads][P] fp32,
     *   tmp_out [rows][num_heads][P][head_size] fp32 (16-byte aligned).
     * After a v2 call they hold the Phase 1 statistics of every partition
     * p < ceil(seq_lens[s]/512); for p beyond that max_logits = -inf and
     * exp_sums = 0, tmp_out is left unspecified. */
    float* exp_sums;
    float* max_logits;
    float* tmp_out;
    /* Optional device int32 receiving PA_DEVERR_* bits (never cleared by the library). */
    int32_t* dev_error;
    /* Optional cudaEvent_t (as void*) recorded on `stream` immediately before and
     * after the main (partition or v1) kernel, for timing; NULL = none. */
    void* event_main_begin;
    void* event_main_end;
    /* Optional [num_seqs][num_kv_heads] int32 partition counters, all zero
     * before the first call.  When given, the v2 path has at most
     * PA_FUSED_MAX_PARTITIONS partitions per sequence and the whole batch fits
     * in one round of the persistent grid (num_seqs * num_kv_heads * P no more
     * than the resident CTAs), the Phase 2 merge of a (sequence, kv head) is
     * done inside the partition kernel by the CTA that finishes its last
     * partition, and no second kernel is launched (pa_plan tells); otherwise
     * the counters are not touched.  Each completed call leaves every counter at zero again;
     * after a PA_DEVERR_TIMEOUT the caller must zero them.  Calls that share
     * counters must not overlap on the GPU.  NULL = separate reduce kernel. */
    int32_t* partition_counters;
    /* Sliding window, in keys visible to the query including its own token:
     * 0 (or < 0) = off, so a zero-initialised struct has no window; otherwise
     * the query, at position seq_lens[s] - 1, attends the keys
     * t >= seq_lens[s] - sliding_window.  This is window_left + 1 for the
     * window_left of AttnDispatchConfig in attn_dispatch.py (-1 there = off).
     * Partitions with no key in the window are skipped (unused: max_logits
     * -inf, exp_sums 0). */
    int32_t sliding_window;
    /* pa_kv_dtype of the caches (0 = same as dtype).  For fp8 caches the split
     * key layout packs x = 16 elements per 16 bytes. */
    int32_t kv_dtype;
    /* Dequantisation scales of fp8 caches: K = k_scale * fp8(K), V = v_scale *
     * fp8(V); values <= 0 mean 1.0 (so a zero-initialised struct has none). */
    float k_scale;
    float v_scale;
    /* Several query tokens per sequence (speculative / multi-token decode, the
     * qo_len of "[Refactor] Uniform PoDAttention API with Horizontal Fusion SMs
     * Schedule #967").  NULL = one query token per sequence, rows of query /
     * out / workspace indexed by sequence (the fields below are ignored).
     * Otherwise [num_seqs + 1] int32 offsets, query_start[0] = 0,
     * nondecreasing, query_start[num_seqs] = num_query_tokens: sequence s owns
     * the rows [query_start[s], query_start[s+1]) of query and out (and of the
     * workspace's first dimension).  Its qn = query_start[s+1] - query_start[s]
     * tokens are the last qn cache entries: token i sits at position
     * seq_lens[s] - qn + i and attends the keys t <= that position (causal),
     * within its own sliding window, so its result is the single-token decode
     * of the sequence cut after that position; a token at a negative position
     * sees no key and gets a zero row.  qn > max_query_len is reported as
     * PA_DEVERR_SEQ_LEN and clamped. */
    const int32_t* query_start;
    int32_t num_query_tokens;  /* rows of query / out / workspace */
    int32_t max_query_len;     /* >= every qn, >= 1; max_query_len * group <= 16 */
    /* Optional HOST copy of seq_lens ([num_seqs] int32, read during the call,
     * never by the device).  PA_MODE_AUTO picks v1 or v2 with
     * pa_choose_mode_for_lengths on it (NULL: every sequence taken as
     * max_seq_len long). */
    const int32_t* seq_lens_host;
    /* Optional [2] int32 device counters, both zero before the first call.
     * Given, and seq_lens_host shows sequences of different partition counts
     * (v2) or page counts (v1), the persistent partition kernel hands out its
     * tiles dynamically: each CTA starts on its own first tile and claims
     * every later one from a grid-wide counter, so CTAs whose tiles are
     * shorter take more of them and the CTAs finish closer together
     * (pa_plan tells); otherwise the counters are not touched and the tiles
     * go round-robin over a grid cut to equal rounds.  Each completed call
     * leaves both at zero; after a PA_DEVERR_TIMEOUT the caller must zero
     * them.  Calls that share them must not overlap on the GPU. */
    int32_t* tile_counters;
    /* 1: block_tables, seq_lens and query_start are final when pa_decode is
     * enqueued -- no kernel earlier in the stream writes them (a host copy
     * before the call is fine).  The partition kernel then reads them, and
     * walks to its first tile, before it waits for the previous kernel in the
     * stream (programmatic dependent launch), so that wait no longer covers a
     * round trip to memory.  The query, the caches and the workspace are still
     * touched only after that wait.  0 (a zero-initialised struct): every
     * input is read after the wait. */
    int32_t metadata_ready;
} pa_decode_args;

/* Largest partition count per sequence for which the merge runs inside the
 * partition kernel (longer sequences use the separate reduce kernel, whose
 * many CTAs read the partitions of one sequence in parallel). */
#define PA_FUSED_MAX_PARTITIONS 8

/*
 * Paged decode attention (the whole operation: partition kernel + reduce for
 * v2, or the single v1 pass).  Returns PA_OK once the work is enqueued.
 * num_seqs == 0 is a no-op.
 */
pa_status pa_decode(const pa_decode_args* args, void* stream);

/* Capacity, in floats, of the device array used by pa_decode_static_workspace
 * (4 Mi floats = 16 MiB). */
#define PA_STATIC_WORKSPACE_FLOATS (4 * 1024 * 1024)

/*
 * The same decode as pa_decode in v2 mode, for callers that cannot allocate
 * device memory -- code running inside a memory pool or allocator that must not
 * re-enter cudaMalloc, plug-ins whose host application owns all device
 * allocations, or code that must not allocate after set-up.  (The pages have no
 * counterpart of this entry point.)
 *
 * The caller passes inputs and `out` as for pa_decode; args->mode,
 * exp_sums, max_logits and tmp_out are ignored.  The partition statistics and
 * partial outputs live in one library-owned __device__ array of
 * PA_STATIC_WORKSPACE_FLOATS floats instead, which every GPU that loads the
 * library keeps until the process exits.  Allocates nothing.
 *  - Returns PA_ERR_WORKSPACE, before launching anything, when
 *    rows * num_heads * P * (head_size + 2) > PA_STATIC_WORKSPACE_FLOATS
 *    (rows = num_seqs, or num_query_tokens with query_start),
 *    P = pa_max_num_partitions(max_seq_len); other errors as pa_decode.
 *  - The array used is the one of the CURRENT device (cudaGetDevice): make
 *    the device of `stream` and of the tensors current before the call.  The
 *    first call on a device looks up the array's address on that device; make
 *    that first call before any stream capture.  The address is cached for the
 *    life of the process: after a cudaDeviceReset of that device it is no
 *    longer valid, so do not call this entry point again on it.
 *  - All calls on a device share the array, which keeps the last call's
 *    contents; nothing in it needs to start at zero.  Calls whose kernels
 *    overlap on the GPU (unordered streams) race on it: order them.
 */
pa_status pa_decode_static_workspace(const pa_decode_args* args, void* stream);

/* ceil(max_seq_len / PA_PARTITION_SIZE), at least 1: the max_num_partitions
 * of "paged_attention_v2_pytorch.py -- BI-V100 PagedAttention V2
 * implementation" (the third dimension of exp_sums / max_logits / tmp_output
 * in the signature of paged_attention_v2_pytorch; a sequence of seq_len
 * tokens uses the first ceil(seq_len / 512) of them).  It is the partition
 * stride of the workspace rows.  Pure host function; no error case
 * (max_seq_len <= 0 gives 1). */
int32_t pa_max_num_partitions(int32_t max_seq_len);

/* Element counts of the v2 workspace, from the shapes in the signature of
 * paged_attention_v2_pytorch ("paged_attention_v2_pytorch.py -- BI-V100
 * PagedAttention V2 implementation"): exp_sums and max_logits
 * [num_seqs][num_heads][max_num_partitions], tmp_output
 * [num_seqs][num_heads][max_num_partitions][head_size].  *stats_elems gets
 * the count of each of exp_sums and max_logits, *tmp_elems that of tmp_out
 * (either pointer may be NULL).  num_seqs is the row count: pass
 * num_query_tokens when query_start gives several tokens per sequence.
 * Pure host function.  Returns PA_ERR_INVALID_ARG on negative sizes or a
 * non-positive num_heads / head_size, writing nothing. */
pa_status pa_workspace_elems(int32_t num_seqs, int32_t num_heads, int32_t head_size,
                             int32_t max_seq_len, int64_t* stats_elems, int64_t* tmp_elems);

/* Bytes of the whole fp32 v2 workspace (the same shapes: exp_sums +
 * max_logits + tmp_out, as in pa_workspace_elems) for `rows` query rows.
 * Pure host function; returns 0 on the sizes pa_workspace_elems rejects. */
size_t pa_workspace_bytes(int32_t rows, int32_t num_heads, int32_t head_size, int32_t max_seq_len);

/* Tokens per partition of the v2 workspace (PA_PARTITION_SIZE). */
int32_t pa_partition_size(void);

/*
 * v1 / v2 choice used by PA_MODE_AUTO, as a pure host function.  The pages
 * decide by tiles against SMs (should_use_paged_v2 in
 * "ex_engine/factors/attn_dispatch.py": v2 when num_kv_heads *
 * ceil(seq_len/512) > 2 * SM_COUNT on a 16-SM part, with the one seq_len of
 * the batch); this library retunes that rule for its persistent kernel, which
 * runs both modes: v1 (one tile per (sequence, kv head), no partition
 * statistics, no reduce launch) when max_seq_len <= PA_PARTITION_SIZE, or
 * when the v1 tiles (num_seqs * num_kv_heads) are at least sm_count and the
 * persistent grid's static assignment of them (sm_count * ctas_per_sm
 * resident CTAs cut to equal rounds, as the launch does) gives its busiest
 * CTA at most 10 % more pages than the mean; otherwise v2.
 * pa_choose_mode takes every sequence to be max_seq_len long (callers with
 * unequal lengths should pass them: pa_choose_mode_for_lengths, or
 * seq_lens_host in the arguments).  sm_count is the device's multiprocessor
 * count, ctas_per_sm the resident CTAs per SM of the partition kernel that
 * the call runs (pa_plan reports it; <= 0 means 2, the figure of 16-bit
 * caches).  Returns PA_MODE_V1 or PA_MODE_V2; sizes <= 0 give PA_MODE_V2
 * (PA_MODE_V1 when max_seq_len <= PA_PARTITION_SIZE).
 */
int32_t pa_choose_mode(int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len, int32_t sm_count,
                       int32_t ctas_per_sm);

/* The same choice with the lengths known on the host (seq_lens_host,
 * [num_seqs] int32, each clamped into [0, max_seq_len]; NULL behaves as
 * pa_choose_mode). */
int32_t pa_choose_mode_for_lengths(int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len,
                                   int32_t sm_count, int32_t ctas_per_sm, const int32_t* seq_lens_host);

/* What pa_decode runs for a set of arguments (filled by pa_plan). */
typedef struct pa_launch_plan {
    int32_t mode;             /* PA_MODE_V1 or PA_MODE_V2 */
    int32_t merge_in_kernel;  /* 1: the v2 Phase 2 merge runs in the partition kernel */
    int32_t kernels;          /* kernels launched per call: 1 or 2 */
    int32_t ctas_per_sm;      /* resident CTAs per SM of the partition kernel */
    int32_t grid;             /* CTAs of the persistent partition-kernel grid */
    int32_t dynamic_schedule; /* 1: tiles claimed from tile_counters */
    int32_t reserved;
    int64_t tiles;            /* tiles of the partition kernel (an upper bound for unequal lengths) */
} pa_launch_plan;

/*
 * The launch pa_decode would make for `args` on the current device, without
 * launching anything: the mode (AUTO resolved as pa_decode resolves it),
 * whether the merge runs in the partition kernel, the kernels per call and
 * the partition kernel's grid.  Returns what pa_decode would return for the
 * host-visible checks (pointers are checked for presence and alignment only,
 * never read), PA_ERR_INVALID_ARG for a NULL plan, PA_ERR_LAUNCH when the
 * device cannot be queried; `*plan` is zeroed first and stays zero for an
 * empty batch.  (The pages have no counterpart.)
 */
pa_status pa_plan(const pa_decode_args* args, pa_launch_plan* plan);

/*
 * Test hook for the bounded waits of the kernels (failure detection without a
 * GPU fault).  While `enable` is non-zero, every later pa_decode call of this
 * process withholds the copy of the first page of one CTA, so the consumer
 * warp waiting for it gives up after `wait_limit_ns`; the kernels then set
 * PA_DEVERR_TIMEOUT in dev_error, stop, and return (results of that call are
 * invalid; the CUDA context stays usable).  `wait_limit_ns` (0 = 2 s, the
 * default) is the limit of every barrier wait of later calls, enabled or not.
 * pa_debug_withhold_page(0, 0) restores normal operation.  Not thread-safe
 * against concurrent pa_decode calls.  Returns PA_ERR_INVALID_ARG for a
 * negative limit.  (The pages have no counterpart.)
 */
pa_status pa_debug_withhold_page(int32_t enable, int64_t wait_limit_ns);

/* Static string for a pa_status value. */
const char* pa_status_str(int32_t status);

/* Library version, (major << 16) | minor. */
int32_t pa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PA_DECODE_H */

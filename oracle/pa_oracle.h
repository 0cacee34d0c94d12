/*
 * pa_oracle.h -- interface of the fp64 CPU oracle (test infrastructure only;
 * see pa_oracle.c).  Independent of include/pa_decode.h: nothing here is
 * shared with the CUDA library.
 */
#ifndef PA_ORACLE_H
#define PA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_ABI_VERSION 1

enum { ORACLE_OK = 0, ORACLE_ERR_ARG = 1, ORACLE_ERR_NOMEM = 2 };
enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2, ORACLE_FP8_E4M3 = 3, ORACLE_FP8_E5M2 = 4 };
enum { ORACLE_LAYOUT_SPLIT = 0, ORACLE_LAYOUT_NHD = 1 };

typedef struct oracle_args {
    /* inputs (host memory, raw storage bytes of `dtype`) */
    const void* query;            /* [num_query_tokens][num_heads][head_size] */
    const void* key_cache;        /* split or NHD, see pa_oracle.c */
    const void* value_cache;
    const int32_t* block_tables;  /* [num_seqs][max_blocks_per_seq] */
    const int32_t* seq_lens;      /* [num_seqs] */
    const float* alibi_slopes;    /* [num_heads] or NULL */
    int32_t num_seqs, num_heads, num_kv_heads, head_size, block_size;
    int32_t num_blocks, max_blocks_per_seq;
    int32_t partition_size, max_num_partitions;
    int32_t dtype, layout;
    double scale, softcap;
    int32_t window_left;          /* < 0: no window; else keys t >= seq_len - 1 - window_left */
    int32_t kv_dtype;             /* storage type of the caches; < 0: same as dtype */
    /* Several query tokens per sequence: query / out / statistics rows are
     * flattened over query tokens, sequence s owning rows
     * [query_start[s], query_start[s+1]); NULL = one token (row) per sequence. */
    const int32_t* query_start;   /* [num_seqs + 1] or NULL */
    int32_t num_query_tokens;     /* rows of query / out (num_seqs when query_start is NULL) */
    double k_scale, v_scale;      /* dequantisation scales of the caches (1.0 = none) */
    /* optional subset of sequences to evaluate (NULL = all) */
    const int32_t* seq_subset;
    int32_t n_subset;
    int32_t num_threads;
    /* outputs (fp64, indexed by absolute sequence number) */
    double* out;          /* [num_query_tokens][num_heads][head_size], dense softmax */
    double* out_v2;       /* same shape, reduce of the partitions; may be NULL */
    double* max_logits;   /* [num_query_tokens][num_heads][max_num_partitions]; may be NULL */
    double* exp_sums;     /* same shape; may be NULL */
    double* tmp_out;      /* [num_query_tokens][num_heads][max_num_partitions][head_size]; may be NULL */
} oracle_args;

int oracle_decode(const oracle_args* a);
int oracle_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif

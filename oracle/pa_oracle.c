/*
 * pa_oracle.c -- plain fp64 CPU oracle for single-token decode attention over a
 * paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may build, load or call this code.
 * It shares no code, header, table or helper with the CUDA library; the two
 * meet only through the seeded input generator, which holds no arithmetic of
 * the method.
 *
 * What it computes (sources are the page titles and sections they come from):
 *
 *  - "paged_attention_v2_pytorch.py -- BI-V100 PagedAttention V2
 *    implementation", block gather loop: logical token t of sequence s lives in
 *    physical block block_tables[s][t / block_size] at slot t % block_size;
 *    only ceil(seq_len / block_size) table entries are read.
 *  - same page, key/value cache shape comments: split key layout
 *    [num_blocks][num_kv_heads][head_size/x][block_size][x] with
 *    x = 16 / element_size, value layout [num_blocks][num_kv_heads][head_size]
 *    [block_size].
 *  - "ex_engine/factors/attn_dispatch.py", dispatch_decode signature: NHD
 *    layout [num_blocks][num_kv_heads][block_size][head_dim] for both caches.
 *  - GQA expansion (repeat_interleave): query head h reads kv head
 *    h / (num_heads / num_kv_heads).
 *  - Phase 1: logits z = scale * q.k (then softcap, then ALiBi
 *    slope[h] * absolute position), per 512-token partition: m_p = max z,
 *    e_p = sum exp(z - m_p), tmp_p = sum exp(z - m_p) v / e_p.
 *  - Phase 2 (log-sum-exp reduce): M = max m_p, r_p = exp(m_p - M) e_p,
 *    out = sum r_p tmp_p / sum r_p, stated on the page to equal the full
 *    softmax -- so the dense result out = sum exp(z - Z) v / sum exp(z - Z)
 *    is computed independently and both are returned.
 *  - Unused partitions (p >= ceil(seq_len/512)): m = -inf, e = 0, tmp = 0.
 *  - same page, arguments kv_cache_dtype / k_scale / v_scale: the gathered
 *    keys are multiplied by k_scale and the values by v_scale.  Reading: an
 *    fp8 cache ("fp8_e4m3" / "fp8_e5m2") holds the keys / values divided by
 *    their scale, so K = k_scale * decode(K8), V = v_scale * decode(V8); the
 *    query and the output keep the query's type.
 *  - Several query tokens per sequence (speculative / multi-token decode, the
 *    qo_len of "[Refactor] Uniform PoDAttention API with Horizontal Fusion SMs
 *    Schedule #967"): reading: a sequence with q_len query tokens holds their
 *    keys as its last q_len cache entries; query token i sits at position
 *    seq_len - q_len + i and attends the keys up to its own position (causal).
 *    Its result is the single-token decode of the sequence cut after that
 *    position.
 *  - "ex_engine/factors/attn_dispatch.py", AttnDispatchConfig window_left /
 *    window_right (-1 = no window), passed to the decode call: the single
 *    query token sits at position seq_len - 1 and attends the keys
 *    t >= seq_len - 1 - window_left (window_right cannot matter: no key lies
 *    after the query).  Partitions with no key inside the window are unused.
 *
 * Readings where the pages are silent or inconsistent:
 *  - tmp_p is stored normalised by e_p (the reduce on the page is only equal
 *    to a full softmax with that reading).
 *  - softcap (the `softcap` field of AttnDispatchConfig, formula not printed):
 *    z = cap * tanh(z / cap), applied to the scaled logit, before ALiBi;
 *    cap <= 0 means off.
 *  - seq_len == 0: output row is zero, all partitions unused.
 *
 * All arithmetic is in double; inputs are decoded exactly from their storage
 * type (fp32, IEEE binary16, bfloat16).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "pa_oracle.h"

/* ---- exact decoding of the storage types into double ------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);     /* (1.f) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 (the "FN" variant): 1 sign, 4 exponent bits (bias 7), 3
 * fraction bits, no infinities, S.1111.111 is NaN, largest finite 448. */
static double e4m3_bits_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int f = b & 0x7;
    double v;
    if (e == 15 && f == 7) return NAN;
    if (e == 0) v = ldexp((double)f, -9);             /* subnormal: f/8 * 2^-6 */
    else v = ldexp((double)(8 + f), e - 10);          /* (1.f) * 2^(e-7) */
    return sign ? -v : v;
}

/* OCP FP8 E5M2: 1 sign, 5 exponent bits (bias 15), 2 fraction bits, IEEE-style
 * infinities and NaNs. */
static double e5m2_bits_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 2) & 0x1f;
    int f = b & 0x3;
    double v;
    if (e == 31) v = f ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)f, -16);       /* subnormal: f/4 * 2^-14 */
    else v = ldexp((double)(4 + f), e - 17);          /* (1.f) * 2^(e-15) */
    return sign ? -v : v;
}

static double load_elem(const void* base, int64_t idx, int dtype) {
    switch (dtype) {
    case ORACLE_F32: return (double)((const float*)base)[idx];
    case ORACLE_F16: return half_bits_to_double(((const uint16_t*)base)[idx]);
    case ORACLE_BF16: return bf16_bits_to_double(((const uint16_t*)base)[idx]);
    case ORACLE_FP8_E4M3: return e4m3_bits_to_double(((const uint8_t*)base)[idx]);
    case ORACLE_FP8_E5M2: return e5m2_bits_to_double(((const uint8_t*)base)[idx]);
    default: return NAN;
    }
}

static int elem_bytes(int dtype) {
    return dtype == ORACLE_F32 ? 4 : (dtype == ORACLE_FP8_E4M3 || dtype == ORACLE_FP8_E5M2) ? 1 : 2;
}

static int cache_dtype(const oracle_args* a) { return a->kv_dtype < 0 ? a->dtype : a->kv_dtype; }

/* ---- page addressing ----------------------------------------------------- */

/* Element index of K[token slot o][dim d] inside physical block `blk`,
 * kv head `kvh`. */
static int64_t key_index(const oracle_args* a, int64_t blk, int kvh, int o, int d) {
    int64_t base = (blk * a->num_kv_heads + kvh) * (int64_t)a->head_size * a->block_size;
    if (a->layout == ORACLE_LAYOUT_SPLIT) {
        int x = 16 / elem_bytes(cache_dtype(a));
        /* [head_size/x][block_size][x] */
        return base + ((int64_t)(d / x) * a->block_size + o) * x + (d % x);
    }
    /* NHD: [block_size][head_size] */
    return base + (int64_t)o * a->head_size + d;
}

static int64_t value_index(const oracle_args* a, int64_t blk, int kvh, int o, int d) {
    int64_t base = (blk * a->num_kv_heads + kvh) * (int64_t)a->head_size * a->block_size;
    if (a->layout == ORACLE_LAYOUT_SPLIT) {
        /* [head_size][block_size] */
        return base + (int64_t)d * a->block_size + o;
    }
    return base + (int64_t)o * a->head_size + d;
}

/* ---- one (sequence, head) --------------------------------------------- */

typedef struct {
    double* z;       /* logits, length seq_len */
    double* vrow;    /* one value row, length head_size */
} scratch_t;

static int query_count(const oracle_args* a, int s) {
    return a->query_start ? a->query_start[s + 1] - a->query_start[s] : 1;
}

/* Query token qi of sequence s, head h. */
static void compute_head(const oracle_args* a, int s, int qi, int h, scratch_t* sc) {
    const int d_sz = a->head_size;
    const int group = a->num_heads / a->num_kv_heads;
    const int kvh = h / group;
    const int qn = query_count(a, s);
    /* keys visible to this query token: positions 0 .. seq_len - qn + qi */
    const int len = a->seq_lens[s] - qn + 1 + qi;
    const int64_t row = (a->query_start ? a->query_start[s] : s) + qi;
    const int P_max = a->max_num_partitions;
    const int PS = a->partition_size;
    const int32_t* table = a->block_tables + (int64_t)s * a->max_blocks_per_seq;
    const int64_t qoff = (row * a->num_heads + h) * d_sz;
    double* out = a->out + qoff;
    double* out_v2 = a->out_v2 ? a->out_v2 + qoff : NULL;
    const int64_t stat_off = (row * a->num_heads + h) * P_max;
    const int num_parts = (len + PS - 1) / PS;
    /* first key inside the sliding window (0 without a window) */
    int t_lo = 0;
    if (a->window_left >= 0 && len - 1 - a->window_left > 0) t_lo = len - 1 - a->window_left;

    /* unused partitions: beyond the sequence, or wholly before the window */
    for (int p = 0; p < P_max; ++p) {
        if (p < num_parts && (p + 1) * PS > t_lo) continue;
        if (a->max_logits) a->max_logits[stat_off + p] = -INFINITY;
        if (a->exp_sums) a->exp_sums[stat_off + p] = 0.0;
        if (a->tmp_out)
            for (int d = 0; d < d_sz; ++d) a->tmp_out[(stat_off + p) * d_sz + d] = 0.0;
    }
    if (len <= 0) {
        for (int d = 0; d < d_sz; ++d) out[d] = 0.0;
        if (out_v2) for (int d = 0; d < d_sz; ++d) out_v2[d] = 0.0;
        return;
    }

    /* logits */
    double Z = -INFINITY;
    for (int t = t_lo; t < len; ++t) {
        int64_t blk = table[t / a->block_size];
        int o = t % a->block_size;
        double dot = 0.0;
        for (int d = 0; d < d_sz; ++d)
            dot += load_elem(a->query, qoff + d, a->dtype) *
                   (a->k_scale * load_elem(a->key_cache, key_index(a, blk, kvh, o, d), cache_dtype(a)));
        double z = a->scale * dot;
        if (a->softcap > 0.0) z = a->softcap * tanh(z / a->softcap);
        if (a->alibi_slopes) z += (double)a->alibi_slopes[h] * (double)t;
        sc->z[t] = z;
        if (z > Z) Z = z;
    }

    /* dense softmax-weighted sum of V */
    double denom = 0.0;
    for (int d = 0; d < d_sz; ++d) out[d] = 0.0;
    for (int t = t_lo; t < len; ++t) {
        int64_t blk = table[t / a->block_size];
        int o = t % a->block_size;
        double w = exp(sc->z[t] - Z);
        denom += w;
        for (int d = 0; d < d_sz; ++d)
            out[d] += w * (a->v_scale * load_elem(a->value_cache, value_index(a, blk, kvh, o, d), cache_dtype(a)));
    }
    for (int d = 0; d < d_sz; ++d) out[d] /= denom;

    if (!(a->max_logits || a->exp_sums || a->tmp_out || out_v2)) return;

    /* per-partition statistics (Phase 1) and the oracle's own reduce (Phase 2) */
    double M = -INFINITY;
    for (int p = 0; p < num_parts; ++p) {
        int t0 = p * PS, t1 = t0 + PS < len ? t0 + PS : len;
        if (t0 < t_lo) t0 = t_lo;
        double m = -INFINITY;
        for (int t = t0; t < t1; ++t) if (sc->z[t] > m) m = sc->z[t];
        if (m > M) M = m;
    }
    double r_total = 0.0;
    if (out_v2) for (int d = 0; d < d_sz; ++d) out_v2[d] = 0.0;
    for (int p = 0; p < num_parts; ++p) {
        int t0 = p * PS, t1 = t0 + PS < len ? t0 + PS : len;
        if (t0 < t_lo) t0 = t_lo;
        if (t0 >= t1) continue;   /* wholly before the window: unused (written above) */
        double m = -INFINITY;
        for (int t = t0; t < t1; ++t) if (sc->z[t] > m) m = sc->z[t];
        double e = 0.0;
        for (int d = 0; d < d_sz; ++d) sc->vrow[d] = 0.0;
        for (int t = t0; t < t1; ++t) {
            int64_t blk = table[t / a->block_size];
            int o = t % a->block_size;
            double w = exp(sc->z[t] - m);
            e += w;
            for (int d = 0; d < d_sz; ++d)
                sc->vrow[d] += w * (a->v_scale * load_elem(a->value_cache, value_index(a, blk, kvh, o, d), cache_dtype(a)));
        }
        for (int d = 0; d < d_sz; ++d) sc->vrow[d] /= e;      /* tmp_p, normalised */
        if (a->max_logits) a->max_logits[stat_off + p] = m;
        if (a->exp_sums) a->exp_sums[stat_off + p] = e;
        if (a->tmp_out)
            for (int d = 0; d < d_sz; ++d) a->tmp_out[(stat_off + p) * d_sz + d] = sc->vrow[d];
        double r = exp(m - M) * e;
        r_total += r;
        if (out_v2) for (int d = 0; d < d_sz; ++d) out_v2[d] += r * sc->vrow[d];
    }
    if (out_v2) for (int d = 0; d < d_sz; ++d) out_v2[d] /= r_total;
}

/* ---- threading over the selected (sequence, head) pairs ----------------- */

typedef struct {
    const oracle_args* a;
    const int32_t* pair_seq;  /* per (sequence, query token) pair: sequence */
    const int32_t* pair_q;    /* ... and query token within the sequence */
    int64_t n_items;
    int64_t next;
    pthread_mutex_t lock;
    int max_len;
    int failed;
} pool_t;

static void* worker(void* arg) {
    pool_t* pool = (pool_t*)arg;
    const oracle_args* a = pool->a;
    scratch_t sc;
    sc.z = (double*)malloc(sizeof(double) * (size_t)(pool->max_len > 0 ? pool->max_len : 1));
    sc.vrow = (double*)malloc(sizeof(double) * (size_t)a->head_size);
    if (!sc.z || !sc.vrow) {
        pthread_mutex_lock(&pool->lock);
        pool->failed = 1;
        pthread_mutex_unlock(&pool->lock);
        free(sc.z); free(sc.vrow);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&pool->lock);
        int64_t i = pool->next++;
        pthread_mutex_unlock(&pool->lock);
        if (i >= pool->n_items) break;
        int64_t pi = i / a->num_heads;
        int h = (int)(i % a->num_heads);
        compute_head(a, pool->pair_seq[pi], pool->pair_q[pi], h, &sc);
    }
    free(sc.z);
    free(sc.vrow);
    return NULL;
}

int oracle_decode(const oracle_args* a) {
    if (!a || !a->query || !a->key_cache || !a->value_cache || !a->block_tables ||
        !a->seq_lens || !a->out)
        return ORACLE_ERR_ARG;
    if (a->num_heads <= 0 || a->num_kv_heads <= 0 || a->num_heads % a->num_kv_heads)
        return ORACLE_ERR_ARG;
    if (a->head_size <= 0 || a->block_size <= 0 || a->partition_size <= 0)
        return ORACLE_ERR_ARG;
    if (a->dtype != ORACLE_F32 && a->dtype != ORACLE_F16 && a->dtype != ORACLE_BF16)
        return ORACLE_ERR_ARG;
    if (a->kv_dtype >= 0 && a->kv_dtype != ORACLE_FP8_E4M3 && a->kv_dtype != ORACLE_FP8_E5M2 &&
        a->kv_dtype != a->dtype)
        return ORACLE_ERR_ARG;
    if (a->layout == ORACLE_LAYOUT_SPLIT && a->head_size % (16 / elem_bytes(cache_dtype(a))))
        return ORACLE_ERR_ARG;
    int n_seq = a->seq_subset ? a->n_subset : a->num_seqs;
    int max_len = 0;
    for (int i = 0; i < n_seq; ++i) {
        int s = a->seq_subset ? a->seq_subset[i] : i;
        if (s < 0 || s >= a->num_seqs) return ORACLE_ERR_ARG;
        int len = a->seq_lens[s];
        if (len < 0) return ORACLE_ERR_ARG;
        if (query_count(a, s) < 0 || (len > 0 && query_count(a, s) > len) ||
            (len == 0 && query_count(a, s) > 1))
            return ORACLE_ERR_ARG;
        if ((len + a->block_size - 1) / a->block_size > a->max_blocks_per_seq) return ORACLE_ERR_ARG;
        if ((len + a->partition_size - 1) / a->partition_size > a->max_num_partitions &&
            (a->max_logits || a->exp_sums || a->tmp_out))
            return ORACLE_ERR_ARG;
        int nb = (len + a->block_size - 1) / a->block_size;
        const int32_t* table = a->block_tables + (int64_t)s * a->max_blocks_per_seq;
        for (int b = 0; b < nb; ++b)
            if (table[b] < 0 || table[b] >= a->num_blocks) return ORACLE_ERR_ARG;
        if (len > max_len) max_len = len;
    }
    /* (sequence, query token) pairs of the selected sequences */
    int64_t n_pairs = 0;
    for (int i = 0; i < n_seq; ++i) n_pairs += query_count(a, a->seq_subset ? a->seq_subset[i] : i);
    int32_t* pair_seq = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_pairs > 0 ? n_pairs : 1));
    int32_t* pair_q = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_pairs > 0 ? n_pairs : 1));
    if (!pair_seq || !pair_q) {
        free(pair_seq);
        free(pair_q);
        return ORACLE_ERR_NOMEM;
    }
    n_pairs = 0;
    for (int i = 0; i < n_seq; ++i) {
        int s = a->seq_subset ? a->seq_subset[i] : i;
        for (int qi = 0; qi < query_count(a, s); ++qi) {
            pair_seq[n_pairs] = s;
            pair_q[n_pairs] = qi;
            ++n_pairs;
        }
    }
    pool_t pool;
    pool.a = a;
    pool.pair_seq = pair_seq;
    pool.pair_q = pair_q;
    pool.n_items = n_pairs * a->num_heads;
    pool.next = 0;
    pool.max_len = max_len;
    pool.failed = 0;
    pthread_mutex_init(&pool.lock, NULL);
    int nt = a->num_threads > 0 ? a->num_threads : 1;
    if (nt > 256) nt = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 0; i < nt; ++i) {
        if (pthread_create(&th[i], NULL, worker, &pool) != 0) break;
        ++started;
    }
    if (started == 0) worker(&pool);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&pool.lock);
    free(pair_seq);
    free(pair_q);
    return pool.failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

int oracle_abi_version(void) { return ORACLE_ABI_VERSION; }

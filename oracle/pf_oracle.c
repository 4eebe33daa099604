/*
 * CPU oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 restatement of what the hot path computes.  Only the test
 * suite, the smoke check and the bench's CPU-baseline leg may load it; the
 * product library never links, loads or calls it, and it shares no code,
 * header or table with the CUDA path.
 *
 * What it computes (no blocking, fusion or reordering beyond the definition):
 *
 *  - KV append: each new token i whose slot s = slot_mapping[i] is not -1 is
 *    copied, for every kv head h, into k_cache[s / bs][h][s % bs][:] (and the
 *    same for v).  This is the write side of "physical KV blocks with logical
 *    per-request block tables" (ForgeLLM README, feature list).
 *
 *  - Decode attention over the paged cache: for sequence i and query head h
 *    the kv head is kh = h / g (g = Hq / Hkv, grouped-query attention as in
 *    the ForgeLLM README's "Llama-family decoder" feature), token t < L_i is
 *    read from physical block block_tables[i][t / bs] at offset t % bs ("reads
 *    physical KV blocks directly", ForgeLLM README, "Decode-only block-table
 *    attention" feature), and
 *        s_t = scale * sum_c q[i][h][c] * K_t[c]
 *        w_t = exp(s_t - max_u s_u) / sum_u exp(s_u - max_u s_u)
 *        out[i][h][:] = sum_t w_t * V_t
 *    which is softmax(q K^T * scale) V.  L_i = 0 gives zeros.
 *
 *  - Split over context partitions (flash-decoding): the same sums restricted
 *    to tokens [k*P, (k+1)*P) intersected with [0, L_i) give, per partition,
 *        m_k = max s_t,  l_k = sum exp(s_t - m_k),
 *        o_k = sum exp(s_t - m_k) V_t / l_k,
 *    and the log-sum-exp merge over the non-empty partitions is
 *        M = max_k m_k,  w_k = l_k * exp(m_k - M),
 *        out = sum_k w_k o_k / sum_k w_k.
 *    Empty partitions are written as m = -inf, l = 0, o = 0.
 *
 *  - Several query tokens per sequence: the same attention for query row
 *    (i, j, h) over the tokens t <= L_i - q_len + j (see
 *    oracle_paged_attention_multi).  Block copy: whole physical blocks, bit
 *    for bit (oracle_copy_blocks).
 *
 * bf16 inputs are decoded here, independently of any CUDA header: a bf16 bit
 * pattern is the top half of an IEEE binary32, so widening is exact.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Address of element c of token `off` of kv head kh in physical block p. */
static size_t cache_index(int64_t p, int kh, int off, int c, int Hkv, int bs, int D) {
    return (((size_t)p * Hkv + kh) * bs + off) * D + c;
}

/* ----------------------------------------------------------------- append */

/* Returns the number of rows skipped because their slot is out of range
 * (anything negative other than -1, or >= num_blocks * block_size). */
int64_t oracle_reshape_and_cache(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                                 uint16_t* k_cache, uint16_t* v_cache, int64_t num_tokens,
                                 int num_kv_heads, int head_dim, int block_size, int64_t num_blocks) {
    int64_t bad = 0;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s == -1) continue;
        if (s < 0 || s >= num_blocks * block_size) { ++bad; continue; }
        int64_t p = s / block_size;
        int off = (int)(s % block_size);
        for (int h = 0; h < num_kv_heads; ++h)
            for (int c = 0; c < head_dim; ++c) {
                size_t src = ((size_t)i * num_kv_heads + h) * head_dim + c;
                size_t dst = cache_index(p, h, off, c, num_kv_heads, block_size, head_dim);
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
    }
    return bad;
}

/* ------------------------------------------------------------- block copy */

/* Copies whole physical blocks (every kv head, every offset) of both caches:
 * for pair j, block block_mapping[2j] -> block block_mapping[2j+1].  This is the
 * device side of giving a forked request its own copy of a shared block, on top
 * of "physical KV blocks with logical per-request block tables" (ForgeLLM README,
 * feature list).  Pairs with an id outside [0, num_blocks) are skipped and
 * counted (the return value). */
int64_t oracle_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, const int64_t* block_mapping,
                           int64_t num_pairs, int num_kv_heads, int head_dim, int block_size,
                           int64_t num_blocks) {
    int64_t bad = 0;
    const size_t per_block = (size_t)num_kv_heads * block_size * head_dim;
    for (int64_t j = 0; j < num_pairs; ++j) {
        int64_t src = block_mapping[2 * j], dst = block_mapping[2 * j + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { ++bad; continue; }
        for (size_t e = 0; e < per_block; ++e) {
            k_cache[(size_t)dst * per_block + e] = k_cache[(size_t)src * per_block + e];
            v_cache[(size_t)dst * per_block + e] = v_cache[(size_t)src * per_block + e];
        }
    }
    return bad;
}

/* ----------------------------------------------------- one (seq, head) pair */

typedef struct {
    const uint16_t* q;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int Hq, Hkv, D, bs, MB;
    double scale;
} problem_t;

/* Grouped-query map: query head h reads kv head h / g, g = Hq / Hkv. */
static int kv_head_of(const problem_t* P, int h) {
    int g = P->Hq / P->Hkv;
    return h / g;
}

/* The query vector of (sequence i, head h) in a [S][Hq][D] query. */
static const uint16_t* query_row(const problem_t* P, int i, int h) {
    return P->q + ((size_t)i * P->Hq + h) * P->D;
}

/* Scores s_t = scale * qv . K_t for tokens [t0, t1) of sequence i, kv head kh. */
static void scores(const problem_t* P, const uint16_t* qv, int i, int kh, int t0, int t1, double* s) {
    for (int t = t0; t < t1; ++t) {
        int64_t p = P->block_tables[(size_t)i * P->MB + t / P->bs];
        int off = t % P->bs;
        double dot = 0.0;
        for (int c = 0; c < P->D; ++c)
            dot += bf16_to_f64(qv[c]) * bf16_to_f64(P->k_cache[cache_index(p, kh, off, c, P->Hkv, P->bs, P->D)]);
        s[t - t0] = P->scale * dot;
    }
}

/* Softmax-weighted sum of V over tokens [t0, t1): o = sum_t e_t V_t / sum_t e_t with
 * e_t = exp(s_t - m), m = max s_t.  Also returns m and l = sum e_t. */
static void attend_range(const problem_t* P, const uint16_t* qv, int i, int kh, int t0, int t1, double* s,
                         double* o, double* m_out, double* l_out) {
    for (int c = 0; c < P->D; ++c) o[c] = 0.0;
    if (t1 <= t0) { *m_out = -INFINITY; *l_out = 0.0; return; }
    scores(P, qv, i, kh, t0, t1, s);
    double m = -INFINITY;
    for (int t = 0; t < t1 - t0; ++t) if (s[t] > m) m = s[t];
    double l = 0.0;
    for (int t = 0; t < t1 - t0; ++t) l += exp(s[t] - m);
    for (int t = t0; t < t1; ++t) {
        double w = exp(s[t - t0] - m) / l;
        int64_t p = P->block_tables[(size_t)i * P->MB + t / P->bs];
        int off = t % P->bs;
        for (int c = 0; c < P->D; ++c)
            o[c] += w * bf16_to_f64(P->v_cache[cache_index(p, kh, off, c, P->Hkv, P->bs, P->D)]);
    }
    *m_out = m;
    *l_out = l;
}

static void set_threads(int num_threads) {
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
}

/* ------------------------------------------------------- decode attention */

/* out: [S, Hq, D] fp64.  num_threads <= 0 uses the OpenMP default. */
void oracle_paged_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, double scale, double* out, int num_threads) {
    problem_t P = {q, k_cache, v_cache, block_tables, context_lens, num_q_heads, num_kv_heads,
                   head_dim, block_size, max_blocks_per_seq, scale};
    set_threads(num_threads);
    int64_t pairs = (int64_t)num_seqs * num_q_heads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t ph = 0; ph < pairs; ++ph) {
        int i = (int)(ph / num_q_heads), h = (int)(ph % num_q_heads);
        int L = context_lens[i];
        double* s = (double*)malloc(sizeof(double) * (L > 0 ? L : 1));
        double m, l;
        attend_range(&P, query_row(&P, i, h), i, kv_head_of(&P, h), 0, L, s, out + (size_t)ph * head_dim, &m, &l);
        free(s);
    }
}

/* ------------------------------------------------- multi-token query rows */

/* Several new tokens per sequence (a chunk of a long prompt interleaved with
 * decode -- "long prompts are split into bounded chunks and interleaved with
 * decode", ForgeLLM README -- or the draft tokens a speculative step verifies,
 * TokenForge post): sequence i has q_len new tokens at positions
 * L_i - q_len + j, j < q_len, already in the cache; query row (i, j, h) attends
 * to the tokens t <= L_i - q_len + j (causal among the new tokens).  A row whose
 * position is negative (L_i < q_len) is zero.
 * q, out: [S][q_len][Hq][D]. */
void oracle_paged_attention_multi(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                  const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                  int q_len, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, double scale, double* out, int num_threads) {
    problem_t P = {q, k_cache, v_cache, block_tables, context_lens, num_q_heads, num_kv_heads,
                   head_dim, block_size, max_blocks_per_seq, scale};
    set_threads(num_threads);
    int64_t rows = (int64_t)num_seqs * q_len * num_q_heads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        int i = (int)(r / ((int64_t)q_len * num_q_heads));
        int j = (int)((r / num_q_heads) % q_len);
        int h = (int)(r % num_q_heads);
        int pos = context_lens[i] - q_len + j;
        int t1 = pos + 1;
        const uint16_t* qv = q + (size_t)r * head_dim;
        double* s = (double*)malloc(sizeof(double) * (t1 > 0 ? t1 : 1));
        double m, l;
        attend_range(&P, qv, i, kv_head_of(&P, h), 0, t1 > 0 ? t1 : 0, s, out + (size_t)r * head_dim, &m, &l);
        free(s);
    }
}

/* --------------------------------------------------- split over partitions */

/* tmp_out: [S, Hq, NP, D], tmp_m / tmp_l: [S, Hq, NP], fp64; NP = max_partitions. */
void oracle_paged_attention_partition(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                      int block_size, int max_blocks_per_seq, double scale,
                                      int partition_size, int max_partitions, double* tmp_out,
                                      double* tmp_m, double* tmp_l, int num_threads) {
    problem_t P = {q, k_cache, v_cache, block_tables, context_lens, num_q_heads, num_kv_heads,
                   head_dim, block_size, max_blocks_per_seq, scale};
    set_threads(num_threads);
    int64_t pairs = (int64_t)num_seqs * num_q_heads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t ph = 0; ph < pairs; ++ph) {
        int i = (int)(ph / num_q_heads), h = (int)(ph % num_q_heads);
        int L = context_lens[i];
        double* s = (double*)malloc(sizeof(double) * (partition_size > 0 ? partition_size : 1));
        for (int k = 0; k < max_partitions; ++k) {
            int t0 = k * partition_size;
            int t1 = t0 + partition_size < L ? t0 + partition_size : L;
            size_t slot = (size_t)ph * max_partitions + k;
            attend_range(&P, query_row(&P, i, h), i, kv_head_of(&P, h), t0, t1, s, tmp_out + slot * head_dim,
                         &tmp_m[slot], &tmp_l[slot]);
        }
        free(s);
    }
}

/* Log-sum-exp merge of the non-empty partitions of each (seq, q head); out: [S, Hq, D] fp64. */
void oracle_merge(const double* tmp_out, const double* tmp_m, const double* tmp_l,
                  const int32_t* context_lens, int num_seqs, int num_q_heads, int head_dim,
                  int partition_size, int max_partitions, double* out) {
    for (int i = 0; i < num_seqs; ++i) {
        int L = context_lens[i];
        int np_i = L > 0 ? (L + partition_size - 1) / partition_size : 0;
        for (int h = 0; h < num_q_heads; ++h) {
            size_t base = ((size_t)i * num_q_heads + h) * max_partitions;
            double* o = out + ((size_t)i * num_q_heads + h) * head_dim;
            for (int c = 0; c < head_dim; ++c) o[c] = 0.0;
            if (np_i == 0) continue;
            double M = -INFINITY;
            for (int k = 0; k < np_i; ++k) if (tmp_m[base + k] > M) M = tmp_m[base + k];
            double W = 0.0;
            for (int k = 0; k < np_i; ++k) W += tmp_l[base + k] * exp(tmp_m[base + k] - M);
            for (int k = 0; k < np_i; ++k) {
                double w = tmp_l[base + k] * exp(tmp_m[base + k] - M) / W;
                for (int c = 0; c < head_dim; ++c) o[c] += w * tmp_out[(base + k) * head_dim + c];
            }
        }
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

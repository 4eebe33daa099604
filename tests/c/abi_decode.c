/*
 * A plain C caller of libpf.so: no Python, no torch.  It draws a small paged-KV
 * problem with the shared input generator, appends one new token per sequence
 * (one sequence appends nothing), runs the single-pass decode and the split
 * (partition + merge) through the C ABI with device memory it allocates itself,
 * and compares with the fp64 oracle: the caches bit for bit, the attention within
 * max |d| <= 2e-3.  Exit status 0 and "ok" on success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "pf.h"

/* the oracle (tests only) and the seeded generator */
int64_t oracle_reshape_and_cache(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                                 uint16_t* k_cache, uint16_t* v_cache, int64_t num_tokens, int num_kv_heads,
                                 int head_dim, int block_size, int64_t num_blocks);
void oracle_paged_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, double scale, double* out, int num_threads);
void wl_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t stream, int64_t offset, int num_threads);

#define S 3
#define HQ 8
#define HKV 2
#define D 128
#define BS 16
#define MB 8

static int fail(const char* what) {
    fprintf(stderr, "FAILED: %s\n", what);
    return 1;
}

#define CK(call)                                                        \
    do {                                                                \
        if ((call) != cudaSuccess) return fail(#call);                  \
    } while (0)
#define PF(call)                                                        \
    do {                                                                \
        pf_status st_ = (call);                                         \
        if (st_ != PF_OK) {                                             \
            fprintf(stderr, "%s: %s\n", #call, pf_status_string(st_));  \
            return 1;                                                   \
        }                                                               \
    } while (0)

int main(void) {
    const int32_t lens[S] = {1, 40, 100};
    int32_t tables[S * MB];
    int64_t nb = 0;
    for (int i = 0; i < S; ++i)
        for (int j = 0; j < MB; ++j) tables[i * MB + j] = j * BS < lens[i] ? (int32_t)nb++ : -1;
    /* reverse the pool so logical and physical order differ */
    for (int i = 0; i < S * MB; ++i)
        if (tables[i] >= 0) tables[i] = (int32_t)(nb - 1 - tables[i]);
    const size_t cache_n = (size_t)nb * HKV * BS * D, q_n = (size_t)S * HQ * D, new_n = (size_t)S * HKV * D;
    uint16_t *q = malloc(q_n * 2), *kc = malloc(cache_n * 2), *vc = malloc(cache_n * 2);
    uint16_t *nk = malloc(new_n * 2), *nv = malloc(new_n * 2);
    wl_normal_bf16(q, (int64_t)q_n, 7, 1, 0, 1);
    wl_normal_bf16(kc, (int64_t)cache_n, 7, 2, 0, 1);
    wl_normal_bf16(vc, (int64_t)cache_n, 7, 3, 0, 1);
    wl_normal_bf16(nk, (int64_t)new_n, 7, 4, 0, 1);
    wl_normal_bf16(nv, (int64_t)new_n, 7, 5, 0, 1);
    int64_t slots[S];
    for (int i = 0; i < S; ++i) {
        const int t = lens[i] - 1;
        slots[i] = i == 0 ? -1 : (int64_t)tables[i * MB + t / BS] * BS + t % BS;
    }
    const double scale = 1.0 / sqrt((double)D);

    /* device copies */
    void *dq, *dkc, *dvc, *dnk, *dnv, *dtab, *dlen, *dslot, *dout, *dsplit, *dws;
    CK(cudaMalloc(&dq, q_n * 2));
    CK(cudaMalloc(&dkc, cache_n * 2));
    CK(cudaMalloc(&dvc, cache_n * 2));
    CK(cudaMalloc(&dnk, new_n * 2));
    CK(cudaMalloc(&dnv, new_n * 2));
    CK(cudaMalloc(&dtab, sizeof tables));
    CK(cudaMalloc(&dlen, sizeof lens));
    CK(cudaMalloc(&dslot, sizeof slots));
    CK(cudaMalloc(&dout, q_n * 4));
    CK(cudaMalloc(&dsplit, q_n * 4));
    CK(cudaMemcpy(dq, q, q_n * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dkc, kc, cache_n * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dvc, vc, cache_n * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dnk, nk, new_n * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dnv, nv, new_n * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dtab, tables, sizeof tables, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dlen, lens, sizeof lens, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dslot, slots, sizeof slots, cudaMemcpyHostToDevice));

    /* the step through the C ABI, on the legacy default stream */
    PF(pf_reshape_and_cache(dnk, dnv, dslot, dkc, dvc, S, HKV, D, BS, nb, NULL));
    PF(pf_paged_attention_decode(dq, dkc, dvc, dtab, dlen, S, HQ, HKV, D, BS, MB, nb, (float)scale, dout, NULL));
    const int P = 32, max_len = MB * BS;
    const size_t ws_bytes = pf_paged_attention_partition_workspace_size(S, HQ, D, max_len, P);
    if (ws_bytes == 0) return fail("workspace size");
    CK(cudaMalloc(&dws, ws_bytes));
    PF(pf_paged_attention_decode_partition(dq, dkc, dvc, dtab, dlen, S, HQ, HKV, D, BS, MB, nb, (float)scale, P,
                                           max_len, dws, ws_bytes, NULL));
    PF(pf_paged_attention_merge(dws, dlen, S, HQ, D, P, max_len, dsplit, NULL));
    PF(pf_get_device_error(NULL));

    uint16_t *gk = malloc(cache_n * 2), *gv = malloc(cache_n * 2);
    float *out = malloc(q_n * 4), *split = malloc(q_n * 4);
    CK(cudaMemcpy(gk, dkc, cache_n * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gv, dvc, cache_n * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out, dout, q_n * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(split, dsplit, q_n * 4, cudaMemcpyDeviceToHost));

    /* the oracle */
    if (oracle_reshape_and_cache(nk, nv, slots, kc, vc, S, HKV, D, BS, nb) != 0) return fail("oracle slots");
    if (memcmp(gk, kc, cache_n * 2) != 0 || memcmp(gv, vc, cache_n * 2) != 0) return fail("append not bit-exact");
    double* ref = malloc(q_n * sizeof(double));
    oracle_paged_attention(q, kc, vc, tables, lens, S, HQ, HKV, D, BS, MB, scale, ref, 1);
    double worst = 0.0, worst_split = 0.0;
    for (size_t e = 0; e < q_n; ++e) {
        const double d1 = fabs((double)out[e] - ref[e]), d2 = fabs((double)split[e] - ref[e]);
        if (!(d1 <= worst)) worst = d1;         /* a NaN makes worst NaN */
        if (!(d2 <= worst_split)) worst_split = d2;
    }
    printf("max abs err: decode %.3e, split %.3e\n", worst, worst_split);
    if (!(worst <= 2e-3) || !(worst_split <= 2e-3)) return fail("attention beyond 2e-3");
    printf("ok\n");
    return 0;
}

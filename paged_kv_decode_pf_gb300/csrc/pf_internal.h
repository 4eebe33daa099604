// Host-side interfaces between the C ABI (pf_api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "pf.h"

namespace pf {

// Tokens per K/V tile that one bulk copy moves; block_size and the partition
// size must be multiples of it.
constexpr int kTileTokens = 16;

// Arguments of the decode / partition kernel; see pf.h for the meaning of each.
struct DecodeParams {
    const uint16_t* q;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* out;        // decode: out [S, Hq, D]; partition pass: tmp_out [S, Hq, NP, D]
    float* part_m;     // partition pass only: tmp_m [S, Hq, NP] (natural-log units)
    float* part_l;     // partition pass only: tmp_l [S, Hq, NP]
    uint16_t* out_bf16;  // single pass only: when set, out [S, Hq, D] in bf16 (each fp32 result rounded
                         // to nearest, ties to even) instead of `out`
    unsigned* err;     // device error word
    long long num_blocks;
    unsigned long long wait_limit_ns;
    float scale_log2;  // scale * log2(e): scores are kept in base-2 units
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int block_size;          // a multiple of 16
    int block_shift;         // log2(block_size) when it is a power of two, else -1
    int max_blocks_per_seq;
    int partition_size;      // partition pass: tokens per partition; cluster split: tokens per CTA
                             // (multiples of 16)
    int cluster_size;        // cluster split: CTAs per (sequence, kv head), 2, 4 or 8
    int num_partitions;      // partition pass: NP
    int max_context_len;     // partition pass: bound every context length must respect
    int order_mode;          // ORDER_NATURAL or ORDER_SORTED (see below)
    // decode with append only: the new token of sequence i, its slot, and writable caches
    const uint16_t* k_new;   // [S, Hkv, D]
    const uint16_t* v_new;
    const int64_t* slot_mapping;  // [S]
    uint16_t* k_cache_w;
    uint16_t* v_cache_w;
};

// What one launch of the decode kernel computes.
constexpr int MODE_DECODE = 0;          // single pass over each whole sequence
constexpr int MODE_PARTITION = 1;       // one context partition per CTA, partials to the workspace
constexpr int MODE_DECODE_APPEND = 2;   // single pass, after writing each sequence's new token
constexpr int MODE_CLUSTER = 3;         // a cluster of C CTAs per item, each one chunk of partition_size
                                        // tokens; the partials merge through distributed shared memory
constexpr int kClusterMaxSize = 8;      // CTAs per cluster at most (the portable cluster size)

// How CTAs map to work items.
//  ORDER_NATURAL: CTA b serves (sequence b / Hkv, kv head b % Hkv); partition pass:
//                 b -> (partition, kv head, sequence), empty partitions exit at once.
//  ORDER_SORTED:  decode: CTA b serves the sequence of rank b / Hkv when sequences
//                 are ordered longest first (ties by index), so that the hardware's
//                 in-order CTA dispatch approximates longest-processing-time-first
//                 scheduling; partition pass: CTA b serves the (b / Hkv)-th non-empty
//                 (sequence, partition) pair, so the empty ones form the grid's tail.
constexpr int ORDER_NATURAL = 0;
constexpr int ORDER_SORTED = 1;
constexpr int kMaxSortedSeqsDecode = 512;      // ranking costs O(S^2 / threads) per CTA
constexpr int kMaxSortedSeqsPartition = 1024;  // the prefix scan costs O(S / threads)

// Device address of the current device's error word (looked up once per device)
// and the current device's SM count; both defined in pf_api.cu.
cudaError_t error_word(unsigned** out);
cudaError_t sm_count(int* out);

// Host-side checks shared by the partition pass and the split that allocates
// nothing: the decode arguments (shapes, alignment, supported sizes) plus
// partition_size and max_context_len.  Returns PF_OK or the status the entry
// point reports; the workspace itself is not checked here.
pf_status check_split_arguments(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int max_blocks_per_seq, int64_t num_blocks, float scale, int partition_size,
                                int max_context_len);

// Launch the decode kernel in one of the MODE_* modes for one head_dim.
// Returns cudaSuccess or the launch error.
cudaError_t launch_decode_d64(const DecodeParams& p, int group, int mode, cudaStream_t stream);
cudaError_t launch_decode_d128(const DecodeParams& p, int group, int mode, cudaStream_t stream);

// Default bound of every device-side wait: long enough never to fire on a
// healthy GPU (a tile copy takes microseconds), short enough to end a broken call.
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;

}  // namespace pf

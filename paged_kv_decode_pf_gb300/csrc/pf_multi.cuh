// Shared by the multi-token query kernels (pf_multi.cu, pf_chunk.cu): their
// parameter block, the longest-first CTA order, and the launcher of the
// prompt-chunk kernel that the multi-query entry points dispatch to.
#pragma once

#include <cstdint>

#include <cuda.h>  // CUtensorMap
#include <cuda_runtime.h>

#include "pf_internal.h"

namespace pf {

struct MultiParams {
    const uint16_t* q;          // [S, q_len, Hq, D]
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* out;                 // [S, q_len, Hq, D]
    unsigned* err;
    long long num_blocks;
    unsigned long long wait_limit_ns;
    float scale_log2;
    int num_seqs, q_len, num_q_heads, num_kv_heads, group, rows;
    int block_size, block_shift, max_blocks_per_seq;
    int sorted;  // CTA b serves the sequence of rank b / Hkv, longest first (num_seqs <= kMultiSortMax)
};

constexpr int kMultiSortMax = 512;

// The sequence of rank r when the sequences are ordered longest first (ties by index):
// every CTA ranks the lengths in shared memory, so the hardware's in-order dispatch of
// the grid starts the longest items first and they do not form the launch's tail.
// keys: round_up(num_seqs, 4) ints of shared memory (16-byte aligned), s_seq one more.
template <int NT>
__device__ __forceinline__ int multi_sorted_seq_into(const MultiParams& p, int r, int* keys, int& s_seq) {
    const int S = p.num_seqs, Sp = (S + 3) & ~3;
    for (int i = threadIdx.x; i < Sp; i += NT) {
        int key = -1;
        if (i < S) {
            const int Li = min(max(__ldg(p.context_lens + i), 0), (1 << 20) - 1);
            key = (Li << 10) | (1023 - i);
        }
        keys[i] = key;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < S; i += NT) {
        const int ki = keys[i];
        int rank = 0;
        for (int j = 0; j < Sp; j += 4) {
            const int4 kj = *reinterpret_cast<const int4*>(keys + j);
            rank += int(kj.x > ki) + int(kj.y > ki) + int(kj.z > ki) + int(kj.w > ki);
        }
        if (rank == r) s_seq = i;
    }
    __syncthreads();
    return s_seq;
}

template <int NT>
__device__ __forceinline__ int multi_sorted_seq(const MultiParams& p, int r) {
    __shared__ __align__(16) int keys[kMultiSortMax];
    __shared__ int s_seq;
    return multi_sorted_seq_into<NT>(p, r, keys, s_seq);
}

// Query rows per kv head (g * q_len) above which the prompt-chunk kernel runs, and its
// upper limit.
constexpr int kChunkMinRows = 65;
constexpr int kChunkMaxRows = 1 << 16;

// At head_dim 128 the prompt-chunk kernel reads V in whole 16-token blocks: one 4 KiB TMA
// copy of a 3D view of the cache (64 elements, rows, the two dim halves 128 bytes apart),
// landing as [dim half][16 rows][128 bytes], instead of two 2 KiB copies (1-1.5 % faster
// there; the 33-64-row tcgen05 kernel, whose V copies go out from more lanes side by side,
// measured 1.6 % slower with it and keeps the 2 KiB boxes).  K stays in 16-row x 128-byte
// boxes: its MMA operand needs every dim half's rows at one stride across the tile.
#ifndef PF_V_BLOCK_COPIES
#define PF_V_BLOCK_COPIES 1
#endif
constexpr bool kVBlockCopies = PF_V_BLOCK_COPIES != 0;

// The cache as a 3D tensor {64 elements, rows = NB * Hkv * bs, 2 dim halves} (D = 128) read in
// boxes {64, 16, 2} with the 128-byte swizzle.
bool encode_cache_map_vblocks(CUtensorMap* map, const void* cache, long long rows);

// Launches the prompt-chunk kernel (pf_chunk.cu): one CTA per (sequence, kv head, 128-row
// tile), scores and P.V on tcgen05 with the query rows as the MMA's M side.
// head_dim 64 or 128; mk views the K cache as [NB * Hkv * bs, D] rows in boxes of 16 rows x
// 64 elements with the 128-byte swizzle; mv the V cache the same way, or at D = 128 with
// kVBlockCopies as encode_cache_map_vblocks does.
cudaError_t launch_chunk(const CUtensorMap& mk, const CUtensorMap& mv, const MultiParams& p, int head_dim,
                         cudaStream_t stream);

}  // namespace pf

// Block copy for the KV allocator: pf_copy_blocks.
//
// When a request forks (beam search, parallel sampling, a shared prompt whose
// last block is still being filled) the allocator gives the child its own copy
// of a shared physical block before either side appends to it -- the device
// half of "physical KV blocks with logical per-request block tables,
// worst-case admission reservation, reclamation" (ForgeLLM README, feature
// list).  The copy is a pure HBM stream: every CTA moves 16 KiB slices of one
// (pair, cache) block with 16-byte loads, four in flight per thread.
#include <cstdint>

#include "pf.h"
#include "pf_device.cuh"
#include "pf_internal.h"

namespace pf {

constexpr int kCopyThreads = 256;
constexpr int kCopyChunksPerGroup = 1024;  // 16 KiB of one block per CTA iteration

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(uint4* __restrict__ k_cache,
                                                                   uint4* __restrict__ v_cache,
                                                                   const int64_t* __restrict__ mapping,
                                                                   long long num_pairs, long long chunks_per_block,
                                                                   long long num_blocks, unsigned* err) {
    const long long groups = (chunks_per_block + kCopyChunksPerGroup - 1) / kCopyChunksPerGroup;
    const long long total = num_pairs * 2 * groups;
    for (long long g = blockIdx.x; g < total; g += gridDim.x) {
        const long long pair = g / (2 * groups);
        const long long rem = g - pair * 2 * groups;
        const int which = int(rem / groups);
        const long long grp = rem - which * groups;
        const long long src = __ldg(mapping + 2 * pair), dst = __ldg(mapping + 2 * pair + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (threadIdx.x == 0 && which == 0 && grp == 0) set_error(err, ERR_BOUNDS);
            continue;
        }
        uint4* cache = which ? v_cache : k_cache;
        const uint4* from = cache + src * chunks_per_block + grp * kCopyChunksPerGroup;
        uint4* to = cache + dst * chunks_per_block + grp * kCopyChunksPerGroup;
        const long long left = chunks_per_block - grp * kCopyChunksPerGroup;
        const int n = left < kCopyChunksPerGroup ? int(left) : kCopyChunksPerGroup;
        constexpr int U = kCopyChunksPerGroup / kCopyThreads;
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = threadIdx.x + u * kCopyThreads;
            if (c < n) x[u] = __ldcs(from + c);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = threadIdx.x + u * kCopyThreads;
            if (c < n) __stcs(to + c, x[u]);
        }
    }
}

}  // namespace pf

using namespace pf;

extern "C" pf_status pf_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping, int64_t num_pairs,
                                    int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                    pf_stream_t stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PF_ERR_INVALID_ARG;
    if (head_dim % 8 != 0) return PF_ERR_UNSUPPORTED;
    const long long chunks_per_block = (long long)num_kv_heads * block_size * (head_dim / 8);
    if (chunks_per_block <= 0 || chunks_per_block > (1ll << 40) / 16 || num_blocks > (1ll << 48) / chunks_per_block ||
        num_pairs > (1ll << 40))
        return PF_ERR_INVALID_ARG;
    if (num_pairs == 0) return PF_OK;
    if (k_cache == nullptr || v_cache == nullptr || block_mapping == nullptr ||
        reinterpret_cast<uintptr_t>(k_cache) % 16 || reinterpret_cast<uintptr_t>(v_cache) % 16 ||
        reinterpret_cast<uintptr_t>(block_mapping) % 8)
        return PF_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    int sms = 0;
    if (error_word(&err) != cudaSuccess || sm_count(&sms) != cudaSuccess) return PF_ERR_CUDA;
    const long long groups = (chunks_per_block + kCopyChunksPerGroup - 1) / kCopyChunksPerGroup;
    const long long total = num_pairs * 2 * groups;
    const long long cap = (long long)sms * 8;
    const unsigned blocks = unsigned(total < cap ? total : cap);
    copy_blocks_kernel<<<blocks, kCopyThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), block_mapping, num_pairs, chunks_per_block,
        num_blocks, err);
    return cudaGetLastError() == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

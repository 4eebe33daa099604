// Block copy for the KV allocator: pf_copy_blocks.
//
// When a request forks (beam search, parallel sampling, a shared prompt whose
// last block is still being filled) the allocator gives the child its own copy
// of a shared physical block before either side appends to it -- the device
// half of "physical KV blocks with logical per-request block tables,
// worst-case admission reservation, reclamation" (ForgeLLM README, feature
// list).  The copy is a pure HBM stream moved by the bulk-copy engine: 16 KiB
// chunks through shared memory, loads and stores both asynchronous.
#include <atomic>
#include <cstdint>

#include "pf.h"
#include "pf_device.cuh"
#include "pf_internal.h"

namespace pf {

// One warp per CTA; its lane 0 drives the copy engine: each (pair, cache, 16 KiB
// chunk) item is a bulk copy global -> shared (completing on the stage's
// mbarrier) and a bulk copy shared -> global (tracked by bulk async-groups).  A
// stage is refilled kCopyLag items after its store was issued, once the store has
// finished reading it, so about kCopyStages - kCopyLag loads and kCopyLag + 1
// stores are in flight per CTA.  The CTA takes pairs c, c + grid, ... and reads
// each pair's (src, dst) ids two pairs ahead of the copies.
#ifndef PF_COPY_CHUNK
#define PF_COPY_CHUNK 16384
#endif
#ifndef PF_COPY_STAGES
#define PF_COPY_STAGES 6
#endif
#ifndef PF_COPY_LAG
#define PF_COPY_LAG 2
#endif
#ifndef PF_COPY_CTAS_PER_SM
#define PF_COPY_CTAS_PER_SM 2
#endif
constexpr int kCopyChunk = PF_COPY_CHUNK;
constexpr int kCopyStages = PF_COPY_STAGES;
constexpr int kCopyLag = PF_COPY_LAG;
constexpr int kCopyCtasPerSm = PF_COPY_CTAS_PER_SM;

__device__ __forceinline__ void bulk_copy_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__global__ void __launch_bounds__(32) copy_blocks_kernel(unsigned char* k_cache, unsigned char* v_cache,
                                                         const int64_t* __restrict__ mapping, long long num_pairs,
                                                         long long block_bytes, long long num_blocks, unsigned* err,
                                                         unsigned long long wait_limit_ns) {
    extern __shared__ __align__(128) unsigned char smem[];  // kCopyStages x kCopyChunk
    __shared__ __align__(8) uint64_t bars[kCopyStages];
    __shared__ unsigned char* stage_dst[kCopyStages];
    __shared__ uint32_t stage_bytes[kCopyStages];
    if (threadIdx.x != 0) return;

    const long long groups = (block_bytes + kCopyChunk - 1) / kCopyChunk;
    const long long per_pair = 2 * groups;  // K and V chunks of one pair
    const long long my_pairs =
        num_pairs > (long long)blockIdx.x ? (num_pairs - 1 - (long long)blockIdx.x) / gridDim.x + 1 : 0;
    const long long n = my_pairs * per_pair;
    if (n == 0) return;
    const uint32_t bar0 = smem_u32(bars), buf0 = smem_u32(smem);
#pragma unroll
    for (int s = 0; s < kCopyStages; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_init_fence();
    const uint64_t policy = l2_policy_evict_first();

    long long ms[3], md[3];  // (src, dst) of CTA-local pairs q_load, q_load + 1, q_load + 2
    auto fetch = [&](long long q, long long& src, long long& dst) {
        if (q < my_pairs) {
            const long long gp = (long long)blockIdx.x + q * gridDim.x;
            src = __ldg(mapping + 2 * gp);
            dst = __ldg(mapping + 2 * gp + 1);
        } else {
            src = dst = -1;
        }
    };
#pragma unroll
    for (int i = 0; i < 3; ++i) fetch(i, ms[i], md[i]);
    long long q_load = 0, m = 0;  // pair of ms[0]; next item to load
    auto issue_load = [&]() {     // item m into stage m % kCopyStages
        const long long q = m / per_pair;
        if (q > q_load) {  // q grows by at most one per item
            ms[0] = ms[1]; md[0] = md[1];
            ms[1] = ms[2]; md[1] = md[2];
            fetch(q_load + 3, ms[2], md[2]);
            ++q_load;
        }
        const long long r = m - q * per_pair;
        const int which = int(r / groups);
        const long long off = (r - which * groups) * kCopyChunk;
        const uint32_t bytes = uint32_t(min(block_bytes - off, (long long)kCopyChunk));
        const int s = int(m % kCopyStages);
        const uint32_t bar = bar0 + 8 * s;
        unsigned char* cache = which ? v_cache : k_cache;
        if (ms[0] >= 0 && ms[0] < num_blocks && md[0] >= 0 && md[0] < num_blocks) {
            stage_dst[s] = cache + md[0] * block_bytes + off;
            stage_bytes[s] = bytes;
            mbar_arrive_expect_tx(bar, bytes);
            bulk_copy_g2s(buf0 + uint32_t(s) * kCopyChunk, cache + ms[0] * block_bytes + off, bytes, bar, policy);
        } else {
            if (r == 0) set_error(err, ERR_BOUNDS);  // the pair is skipped
            stage_bytes[s] = 0;
            mbar_arrive(bar);
        }
        ++m;
    };

    const long long prologue = n < kCopyStages ? n : kCopyStages;
    for (long long i = 0; i < prologue; ++i) issue_load();
    long long it = 0;
    for (; it < n; ++it) {
        const int s = int(it % kCopyStages);
        if (!mbar_wait_bounded(bar0 + 8 * s, uint32_t(it / kCopyStages) & 1u, wait_limit_ns)) {
            set_error(err, ERR_TIMEOUT);
            break;
        }
        if (stage_bytes[s]) bulk_copy_s2g(stage_dst[s], buf0 + uint32_t(s) * kCopyChunk, stage_bytes[s]);
        bulk_commit_group();  // one group per item (empty for a skipped pair)
        if (it >= kCopyLag && m < n) {
            bulk_wait_group_read<kCopyLag>();  // the store of item it - kCopyLag has read its stage
            issue_load();                      // item it - kCopyLag + kCopyStages into that stage
        }
    }
    // loads still in flight (only after a wait gave up), then every store to completion
    for (long long k = it; k < m; ++k)
        mbar_wait_bounded(bar0 + 8 * int(k % kCopyStages), uint32_t(k / kCopyStages) & 1u, wait_limit_ns);
    bulk_wait_group_all();
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
    static std::atomic<unsigned long long> configured{0};  // one bit per device ordinal
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PF_ERR_CUDA;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    constexpr int smem = kCopyStages * kCopyChunk;
    if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(copy_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return PF_ERR_CUDA;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const long long block_bytes = chunks_per_block * 16;
    const long long cap = (long long)sms * kCopyCtasPerSm;
    const unsigned blocks = unsigned(num_pairs < cap ? num_pairs : cap);
    copy_blocks_kernel<<<blocks, 32, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned char*>(k_cache), static_cast<unsigned char*>(v_cache), block_mapping, num_pairs,
        block_bytes, num_blocks, err, kDefaultWaitLimitNs);
    return cudaGetLastError() == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

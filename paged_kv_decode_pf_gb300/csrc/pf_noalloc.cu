// Split-K decode without allocation: pf_paged_attention_split_noalloc.
//
// Some callers cannot give the library a workspace -- a plugin inside a runtime
// that owns every byte of device memory, a decode loop that must never call
// cudaMalloc, a process whose memory another allocator has already reserved.
// For them the partials of the partition pass live in a fixed scratch array
// compiled into the library; the entry point runs the ordinary partition pass
// and log-sum-exp merge with that array as their workspace.
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "pf.h"
#include "pf_internal.h"

namespace {

// The scratch.  A device keeps it from its first use until the process exits.
static __device__ __align__(256) unsigned char g_split_scratch[PF_SPLIT_NOALLOC_SCRATCH_BYTES];

// Device address of g_split_scratch per device ordinal.  In host code the
// symbol is only a host-side stand-in, never a device address.
std::atomic<void*> g_scratch_address[64];

// Looks the address up once per device, with that device current.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    void* p = g_scratch_address[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        e = cudaGetSymbolAddress(&p, g_split_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_address[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" pf_status pf_paged_attention_split_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                      const int32_t* block_tables, const int32_t* context_lens,
                                                      int num_seqs, int num_q_heads, int num_kv_heads,
                                                      int head_dim, int block_size, int max_blocks_per_seq,
                                                      int64_t num_blocks, float scale, int partition_size,
                                                      int max_context_len, float* out, pf_stream_t stream) {
    // The same argument checks as the partition pass, so a bad argument is reported
    // as such whatever the size; only then the size of the partials against the scratch.
    pf_status st = pf::check_split_arguments(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                             num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                             num_blocks, scale, partition_size, max_context_len);
    if (st != PF_OK) return st;
    if (num_seqs == 0) return PF_OK;
    if (out == nullptr || reinterpret_cast<uintptr_t>(out) % 16 != 0) return PF_ERR_INVALID_ARG;
    const size_t need = pf_paged_attention_partition_workspace_size(num_seqs, num_q_heads, head_dim,
                                                                    max_context_len, partition_size);
    if (need == 0) return PF_ERR_INVALID_ARG;
    if (need > PF_SPLIT_NOALLOC_SCRATCH_BYTES) return PF_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return PF_ERR_CUDA;
    // Every partial the merge reads (partitions below ceil(L / P)) is written by the
    // partition pass of this same call, so the scratch needs no clearing.
    st = pf_paged_attention_decode_partition(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                                             num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                                             scale, partition_size, max_context_len, scratch,
                                             PF_SPLIT_NOALLOC_SCRATCH_BYTES, stream);
    if (st != PF_OK) return st;
    return pf_paged_attention_merge(scratch, context_lens, num_seqs, num_q_heads, head_dim, partition_size,
                                    max_context_len, out, stream);
}

/*
 * pf.h -- C ABI of libpf.so: paged-KV decode attention for NVIDIA GB300 (sm_103a).
 *
 * The operations follow the decode step of a paged KV cache:
 *   - "Physical KV blocks with logical per-request block tables" and
 *     "Decode-only block-table attention reads physical KV blocks directly; the
 *     Triton kernel uses online softmax without constructing padded batch-wide
 *     K/V" (ForgeLLM README, feature list), with "grouped-query attention"
 *     (same list, "Llama-family decoder");
 *   - "Paged KV cache allocates fixed-size blocks on demand" (LLM-Inference-Engine
 *     README, "Why paged KV cache?");
 *   - "Decode is memory-bound" (same README, "Why dynamic injection during
 *     decode?") -- every kernel here streams the cache once and is bounded by
 *     HBM bandwidth.
 *
 * Conventions shared by every call
 *   bf16       IEEE binary32 truncated to its upper 16 bits, stored as uint16.
 *   Layouts    (all row-major, contiguous, no padding)
 *              q             [num_seqs, num_q_heads, head_dim]          bf16
 *              k, v          [num_tokens, num_kv_heads, head_dim]       bf16
 *              k_cache,
 *              v_cache       [num_blocks, num_kv_heads, block_size, head_dim] bf16
 *              block_tables  [num_seqs, max_blocks_per_seq]             int32
 *              context_lens  [num_seqs]                                 int32
 *              out           [num_seqs, num_q_heads, head_dim]          fp32
 *   Paging     token t of sequence i is stored in physical block
 *              block_tables[i][t / block_size] at offset t % block_size.
 *              Table entries at or past ceil(context_lens[i] / block_size) are
 *              never read.
 *   GQA        query head h reads kv head h / (num_q_heads / num_kv_heads)
 *              (contiguous groups).
 *   Memory     every pointer is device memory owned by the caller; nothing is
 *              retained after a call returns.  q, k, v, the caches, out and the
 *              workspace must be 16-byte aligned (workspace: 256-byte),
 *              block_tables / context_lens 4-byte, slot_mapping 8-byte.
 *   Streams    every call is asynchronous and stream-ordered on `stream`
 *              (a cudaStream_t; NULL is the legacy default stream).  Calls are
 *              thread-safe.  The current CUDA device must own all pointers.
 *   Devices    the first call on a device looks up, with that device current,
 *              the device addresses of the library's per-device variables (the
 *              error word; the scratch of pf_paged_attention_split_noalloc) and
 *              keeps them for the life of the process.  cudaDeviceReset after a
 *              call of this library is therefore not supported: the module may
 *              be loaded again at another address.
 *   Errors     problems visible on the host (null or misaligned pointers,
 *              non-positive sizes, overflowing sizes) return PF_ERR_INVALID_ARG
 *              and shapes outside the compiled set return PF_ERR_UNSUPPORTED,
 *              both before anything is launched; a failed launch returns
 *              PF_ERR_CUDA.  Problems only the device can see -- a slot or a
 *              block id out of range, a context length the table or the
 *              partition grid cannot hold, a bounded wait that gave up -- never
 *              trap: the kernel skips the offending row (append) or writes NaN
 *              to the affected output rows (attention), sets a bit in a
 *              per-device error word, and pf_get_device_error() reports it.
 */
#ifndef PF_H
#define PF_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PF_API __attribute__((visibility("default")))
#else
#define PF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA header. */
typedef struct CUstream_st* pf_stream_t;

typedef enum pf_status {
    PF_OK = 0,
    PF_ERR_INVALID_ARG = 1,     /* host-visible argument error; nothing launched */
    PF_ERR_UNSUPPORTED = 2,     /* valid but not compiled: head_dim, block_size or group */
    PF_ERR_CUDA = 3,            /* a CUDA runtime call or launch failed */
    PF_ERR_DEVICE_BOUNDS = 4,   /* device saw a slot / block id / length out of range */
    PF_ERR_DEVICE_TIMEOUT = 5   /* a bounded device-side wait gave up */
} pf_status;

/*
 * KV append ("reshape_and_cache"): writes each new token's K and V into its
 * physical slot -- the write side of the ForgeLLM README's "Physical KV blocks
 * with logical per-request block tables".
 *
 *   for every token i < num_tokens with s = slot_mapping[i] != -1, every kv head h:
 *     k_cache[s / block_size][h][s % block_size][:] = k[i][h][:]
 *     v_cache[s / block_size][h][s % block_size][:] = v[i][h][:]
 *
 * Bit-exact copy.  Slots equal to -1 are padding and are skipped.  Any other
 * negative slot or a slot >= num_blocks * block_size is skipped and flags
 * PF_ERR_DEVICE_BOUNDS.  Valid slots must be distinct within one call (the
 * result is unspecified otherwise).  head_dim must be a multiple of 8;
 * any block_size >= 1.  num_tokens == 0 launches nothing.
 */
PF_API pf_status pf_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping,
                               void* k_cache, void* v_cache, int64_t num_tokens,
                               int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, pf_stream_t stream);

/*
 * Block copy for the allocator: when a request forks (beam search, parallel
 * sampling, a shared prompt whose last block is still being filled) it gets its
 * own copy of a shared physical block before either side appends to it -- the
 * device half of "physical KV blocks with logical per-request block tables ...
 * reclamation" (ForgeLLM README, feature list).
 *
 *   for every pair j < num_pairs, with (src, dst) = (block_mapping[2j], block_mapping[2j+1]):
 *     k_cache[dst][:][:][:] = k_cache[src][:][:][:];  v_cache likewise
 *
 * block_mapping is int64 [num_pairs][2] in device memory.  Bit-exact copy of
 * whole blocks (every kv head and offset).  Destinations must be distinct and
 * no destination may also be a source in the same call (the result is
 * unspecified otherwise); src == dst is a no-op.  A pair with an id outside
 * [0, num_blocks) is skipped and flags PF_ERR_DEVICE_BOUNDS.  head_dim must be
 * a multiple of 8.  num_pairs == 0 launches nothing.
 */
PF_API pf_status pf_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping, int64_t num_pairs,
                                int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                pf_stream_t stream);

/*
 * Decode attention over the paged cache, one query token per sequence, in a
 * single pass (ForgeLLM README, feature list: decode-only block-table attention
 * with online softmax, grouped-query heads):
 *
 *   out[i][h][:] = sum_t softmax_t(scale * q[i][h] . K_t) V_t,   t < context_lens[i],
 *   K_t, V_t = k_cache/v_cache[block_tables[i][t / bs]][h / g][t % bs][:]
 *
 * fp32 accumulation and an fp32 online softmax; out is fp32.
 * context_lens[i] == 0 gives a zero row.  Supported: head_dim in {64, 128},
 * block_size a multiple of 16 (the configurations use 16 and 32),
 * g = num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 * A context length above max_blocks_per_seq * block_size, or a table entry
 * outside [0, num_blocks), flags PF_ERR_DEVICE_BOUNDS and NaN-fills the rows
 * of that (sequence, kv head).
 */
PF_API pf_status pf_paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, const int32_t* context_lens,
                                    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                    float scale, float* out, pf_stream_t stream);

/*
 * The same single pass with a bf16 output: out is [num_seqs][num_q_heads][head_dim]
 * bf16 (16-byte aligned, device), each element the fp32 result of
 * pf_paged_attention_decode rounded once to bf16, to nearest with ties to even --
 * bit for bit that rounding of the fp32 call's output.  The source pages fix no
 * output precision (the fp32 entry above is the reading this library takes); this
 * variant is for callers that feed the attention output straight into a bf16
 * projection.  Its error against the exact result is the fp32 error plus one bf16
 * rounding (a relative 2^-9), so it meets |d| <= 2e-3 + 1e-2 |exact| but not the
 * fp32 entry's 2e-3 absolute bound on outputs of magnitude >= 0.5.  Arguments,
 * supported shapes and error behaviour are those of pf_paged_attention_decode.
 */
PF_API pf_status pf_paged_attention_decode_bf16(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                         int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                         float scale, void* out, pf_stream_t stream);

/*
 * One decode step in one launch: append each sequence's new token, then attend
 * over the cache that includes it (the write and the read sides of "physical KV
 * blocks with logical per-request block tables" and "decode-only block-table
 * attention", ForgeLLM README, feature list, fused).  The result -- the caches
 * after the call and out -- is that of
 *     pf_reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache, num_seqs, ...)
 *     pf_paged_attention_decode(q, k_cache, v_cache, ...)
 * for the decode case in which token i is the newest token of sequence i:
 * slot_mapping[i] is -1 (sequence i appends nothing; it attends over its
 * context_lens[i] cached tokens) or the slot of its position context_lens[i]-1,
 * block_tables[i][(L-1)/bs]*bs + (L-1)%bs.  Any other slot flags
 * PF_ERR_DEVICE_BOUNDS, writes nothing for that sequence and NaN-fills its rows.
 * The new token's K/V enter the attention from k_new / v_new directly, so the
 * slot's previous contents are never read.
 *
 *   k_new, v_new   [num_seqs, num_kv_heads, head_dim] bf16, 16-byte aligned
 *   slot_mapping   [num_seqs] int64, 8-byte aligned
 * Other arguments, shapes and errors as pf_paged_attention_decode.
 */
PF_API pf_status pf_paged_attention_decode_append(const void* q, const void* k_new, const void* v_new,
                                                  const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                                  const int32_t* block_tables, const int32_t* context_lens,
                                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                                  int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                                  float scale, float* out, pf_stream_t stream);

/*
 * Several new tokens per sequence at once: the draft tokens a speculative step
 * verifies ("paired the main model with a tiny draft model to guess tokens
 * ahead of time", TokenForge post) or a short prompt chunk interleaved with
 * decode ("long prompts are split into bounded chunks and interleaved with
 * decode", ForgeLLM README).  The q_len new tokens of sequence i are its last
 * positions L_i - q_len + j, already in the cache; query row (j, h) attends to
 * the tokens t <= L_i - q_len + j:
 *
 *   out[i][j][h][:] = sum_{t <= L_i - q_len + j} softmax_t(scale * q[i][j][h] . K_t) V_t
 *
 * A row whose position is negative (L_i < q_len) is zero.  A NaN or infinite
 * key at a position a row cannot see leaves that row alone (its score is
 * replaced); a NaN or infinite *value* there may make the row NaN, since the
 * tensor-core P.V product multiplies it by the row's zero probability.  Finite
 * caches are unaffected.  The scores and P.V
 * run on tensor cores (bf16 inputs, fp32 accumulation; the probabilities enter
 * P.V as a bf16 high part plus a bf16 remainder).  By rows per kv head
 * (g * q_len): up to 16, one CTA's four warps split the tokens (mma.sync); 17 to
 * 32, and 33 to 64 at head_dim 64, each 16-row tile has its own warp and one or
 * two producer warps stream K/V to all of them (mma.sync); 33 to 64 at head_dim
 * 128 run the kernel of pf_paged_attention_multi_query_tcgen05.  Past 64 rows --
 * a prompt chunk of tens to hundreds of tokens -- the prompt-chunk kernel runs:
 * one CTA per (sequence, kv head, tile of 128 rows), the rows as the M side of
 * tcgen05.mma, Q, S, P and O in tensor memory, K and V tiles by TMA.
 *
 *   q    [num_seqs, q_len, num_q_heads, head_dim] bf16, 16-byte aligned
 *   out  [num_seqs, q_len, num_q_heads, head_dim] fp32
 * Supported: head_dim in {64, 128}, block_size a multiple of 16,
 * (num_q_heads / num_kv_heads) * q_len <= 65536, num_blocks * num_kv_heads *
 * block_size < 2^31; other arguments and errors as pf_paged_attention_decode.
 */
PF_API pf_status pf_paged_attention_multi_query(const void* q, const void* k_cache, const void* v_cache,
                                                const int32_t* block_tables, const int32_t* context_lens,
                                                int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                                int head_dim, int block_size, int max_blocks_per_seq,
                                                int64_t num_blocks, float scale, float* out, pf_stream_t stream);

/*
 * The same operation as pf_paged_attention_multi_query, with both products on
 * the fifth-generation tensor cores (tcgen05.mma, accumulators in tensor
 * memory), computed transposed so that a tile's 128 tokens (and the 128 head
 * dimensions) fill the MMA's 128 lanes and the query rows are its N side:
 * S^T = K Q^T, then O^T += V^T P^T with P as bf16 high part plus remainder.
 * One CTA per (sequence, kv head) streams 128-token K and V tiles (TMA copies of
 * the cache blocks, three- and two-deep rings) straight into the swizzled
 * operand layout.  Results agree with the mma.sync kernels to fp32 rounding.
 * pf_paged_attention_multi_query runs it for 33-64 rows at head_dim 128, where
 * it is the faster one (Llama-3-8B-shaped batch: 886 and 905 us at 48 and 64
 * rows against 1,148 and 1,211 us); at 32 rows and below the mma.sync kernels
 * are faster (827 against 864 us at 32 rows), since a 128-token tile's products
 * cost the same whatever the row count.  Past 64 rows this entry runs the same
 * prompt-chunk kernel as pf_paged_attention_multi_query.
 *
 * Supported: head_dim == 128 (else PF_ERR_UNSUPPORTED); the other shapes,
 * arguments and errors as pf_paged_attention_multi_query.
 */
PF_API pf_status pf_paged_attention_multi_query_tcgen05(const void* q, const void* k_cache, const void* v_cache,
                                                        const int32_t* block_tables, const int32_t* context_lens,
                                                        int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                                        int head_dim, int block_size, int max_blocks_per_seq,
                                                        int64_t num_blocks, float scale, float* out,
                                                        pf_stream_t stream);

/*
 * Split over context partitions ("flash-decoding") for long contexts.
 *
 * Source: no passage of the source pages describes a split of one sequence's
 * context; the pages stop at decode-only block-table attention with online
 * softmax (ForgeLLM README, feature list).  The pair below is defined by the
 * identity that makes it exact: the softmax over a sequence's tokens, split into
 * disjoint partitions, equals the combination of each partition's normalised
 * result o_k weighted by l_k exp(m_k - M) (the merge formula further down), so
 * partition pass + merge compute the same attention as pf_paged_attention_decode.
 *
 * The workspace holds, for NP = ceil(max_context_len / partition_size)
 * partitions, three fp32 arrays, each starting on a 256-byte boundary:
 *   tmp_out [num_seqs][num_q_heads][NP][head_dim]  o_k = sum e_t V_t / l_k
 *   tmp_m   [num_seqs][num_q_heads][NP]            m_k = max_t scale*q.K_t
 *   tmp_l   [num_seqs][num_q_heads][NP]            l_k = sum_t exp(s_t - m_k)
 * over the tokens [k*P, (k+1)*P) of each sequence.  Only the partitions
 * k < ceil(context_lens[i] / P) are written.
 *
 * pf_paged_attention_partition_workspace_layout() returns the byte offsets of
 * the three arrays and the total size (0 on invalid arguments); the size query
 * returns just the total.  partition_size must be a positive multiple of 16
 * (tiles of 16 tokens never straddle two partitions).
 */
PF_API size_t pf_paged_attention_partition_workspace_layout(int num_seqs, int num_q_heads, int head_dim,
                                                     int max_context_len, int partition_size,
                                                     size_t* tmp_out_offset, size_t* tmp_m_offset,
                                                     size_t* tmp_l_offset);
PF_API size_t pf_paged_attention_partition_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                                   int max_context_len, int partition_size);

/*
 * Partition pass: the decode computation restricted to each context
 * partition, writing (o_k, m_k, l_k) into the workspace.  Same arguments and
 * supported shapes as pf_paged_attention_decode plus partition_size, the
 * max_context_len the workspace was sized for (every context_lens[i] must be
 * <= it; a longer one flags PF_ERR_DEVICE_BOUNDS and NaN-fills its partials),
 * the workspace and its size in bytes (checked against the layout).
 */
PF_API pf_status pf_paged_attention_decode_partition(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* block_tables, const int32_t* context_lens,
                                              int num_seqs, int num_q_heads, int num_kv_heads,
                                              int head_dim, int block_size, int max_blocks_per_seq,
                                              int64_t num_blocks, float scale, int partition_size,
                                              int max_context_len, void* workspace,
                                              size_t workspace_bytes, pf_stream_t stream);

/*
 * Log-sum-exp merge of the partitions written by the partition pass (the
 * identity stated above the workspace layout; no page passage defines it):
 *   M = max_k m_k,  w_k = l_k exp(m_k - M),  out = sum_k w_k o_k / sum_k w_k
 * over k < ceil(context_lens[i] / partition_size); zero rows for empty
 * sequences.  The arguments must match the partition pass that filled the
 * workspace.  head_dim in {64, 128}.
 */
PF_API pf_status pf_paged_attention_merge(const void* workspace, const int32_t* context_lens, int num_seqs,
                                   int num_q_heads, int head_dim, int partition_size,
                                   int max_context_len, float* out, pf_stream_t stream);

/*
 * Decode attention that chooses its own decomposition from the sizes the host
 * knows (no device memory is read), one of three:
 *   - the single pass, when there are enough (sequence, kv head) items to fill
 *     the GPU or the contexts are short;
 *   - the cluster split, when the items are few (fewer than half the SMs would
 *     get one) and a cluster of at most 8 CTAs covers max_context_len in chunks
 *     of at most 1,024 tokens: each item's CTAs take consecutive chunks, and the
 *     chunks' partials are merged through distributed shared memory within the
 *     cluster in the same launch -- no workspace, one kernel;
 *   - otherwise the split over context partitions + merge, with a partition size
 *     that gives a long sequence enough partitions (workspace needed).
 * The result is the same attention (within fp32 rounding).
 *
 * pf_paged_attention_decode_auto_plan() returns the partition size the call
 * will use -- 0 for the single pass, the chunk of each CTA for the cluster split
 * -- and writes the workspace bytes it needs to *workspace_bytes (0 for the
 * single pass and the cluster split, which a positive return with 0 bytes
 * identifies); it needs the current device (SM count).
 * pf_paged_attention_decode_auto takes the decode arguments plus
 * max_context_len (>= every context length: a longer one flags
 * PF_ERR_DEVICE_BOUNDS and NaN-fills its rows) and a workspace of at least that
 * size (256-byte aligned; may be NULL when the plan needs none).
 */
PF_API int pf_paged_attention_decode_auto_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                               int max_context_len, size_t* workspace_bytes);
PF_API pf_status pf_paged_attention_decode_auto(const void* q, const void* k_cache, const void* v_cache,
                                                const int32_t* block_tables, const int32_t* context_lens,
                                                int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                                int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                                float scale, int max_context_len, void* workspace,
                                                size_t workspace_bytes, float* out, pf_stream_t stream);

/*
 * Device error word of the current device.  Synchronises `stream`, reads the
 * word, clears it and returns PF_ERR_DEVICE_TIMEOUT or PF_ERR_DEVICE_BOUNDS if
 * the corresponding bit was set (timeout first), PF_ERR_CUDA if the
 * synchronisation or the read failed, PF_OK otherwise.  The word collects the
 * errors of every call on the device since it was last read.
 */
PF_API pf_status pf_get_device_error(pf_stream_t stream);

/* Static, human-readable name of a status. */
PF_API const char* pf_status_string(pf_status status);

/*
 * Failure-detection check (not part of the attention method): launches one
 * block whose thread waits on a shared-memory barrier that nothing completes,
 * through the same bounded wait the attention kernels use, giving up after
 * about limit_ns nanoseconds (1e3 .. 1e10).  The kernel then returns normally,
 * with PF_ERR_DEVICE_TIMEOUT set in the error word.  It exists so that tests
 * can exercise the timeout path without disturbing the GPU.
 */
PF_API pf_status pf_debug_bounded_wait(int64_t limit_ns, pf_stream_t stream);

/*
 * Split-K decode that allocates nothing.  The source pages have no counterpart; this
 * exists for callers that cannot hand the library a workspace: a plugin or
 * custom op inside a host runtime that owns all device memory and offers no
 * allocator on the decode path, a decode loop that must not call cudaMalloc
 * (it can synchronise the whole device and stall other streams), or a process
 * whose memory is already fully reserved by another allocator.
 *
 * It computes the same result as pf_paged_attention_decode_partition followed
 * by pf_paged_attention_merge (same arguments, same supported shapes), with
 * the partials kept in a scratch array compiled into the library: a
 * file-scope __device__ array of PF_SPLIT_NOALLOC_SCRATCH_BYTES bytes that a
 * device keeps from the first use until the process exits.  When the workspace
 * layout for these arguments (pf_paged_attention_partition_workspace_size) is
 * larger than that, the call returns PF_ERR_UNSUPPORTED and launches nothing.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call outside any stream
 * capture.  The call performs no allocation (no cudaMalloc, cudaFree or
 * allocating library routine).  Every call on a device shares the one array
 * and leaves its partials there; nothing in it has to start at zero, because
 * the partition pass writes every partial the merge then reads.  Calls whose
 * executions overlap on the GPU (for example on two streams of one device)
 * race on the array and must be ordered by the caller.
 */
#define PF_SPLIT_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
PF_API pf_status pf_paged_attention_split_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                  const int32_t* block_tables, const int32_t* context_lens,
                                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                                  int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                                  float scale, int partition_size, int max_context_len,
                                                  float* out, pf_stream_t stream);

/* Library version, e.g. "0.1.0". */
PF_API const char* pf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PF_H */

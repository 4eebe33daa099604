// C ABI of libpf.so (declared in include/pf.h): argument validation, launch
// configuration, the per-device error word, and the small kernels that are not
// the decode loop itself -- the KV-append scatter, the log-sum-exp merge of
// context partitions and the bounded-wait check.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>

#include "pf.h"
#include "pf_device.cuh"
#include "pf_internal.h"

namespace pf {

// ------------------------------------------------------------- error word

// One word per device (each context holds its own copy of this variable).
__device__ unsigned int g_error_word;

static std::atomic<unsigned*> g_error_ptr[64];
static std::atomic<int> g_sm_count[64];

static cudaError_t current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    return (*dev >= 0 && *dev < 64) ? cudaSuccess : cudaErrorInvalidDevice;
}

// Device address of the error word of the current device, looked up once per device.
cudaError_t error_word(unsigned** out) {
    int dev = 0;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return e;
    unsigned* p = g_error_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_error_word);
        if (e != cudaSuccess) return e;
        g_error_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

cudaError_t sm_count(int* out) {
    int dev = 0;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return e;
    int n = g_sm_count[dev].load(std::memory_order_acquire);
    if (n <= 0) {
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_sm_count[dev].store(n, std::memory_order_release);
    }
    *out = n;
    return cudaSuccess;
}

// ------------------------------------------------------------------ append

// One thread per 16-byte chunk of a (token, kv head) row; copies the K and the V chunk.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const uint4* __restrict__ k,
                                                                const uint4* __restrict__ v,
                                                                const int64_t* __restrict__ slots,
                                                                uint4* __restrict__ k_cache,
                                                                uint4* __restrict__ v_cache, long long total,
                                                                int num_kv_heads, int chunks_per_row,
                                                                int block_size, long long num_slots,
                                                                unsigned* err) {
    const int row_chunks = num_kv_heads * chunks_per_row;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long i = idx / row_chunks;
        const int rem = int(idx - i * row_chunks);
        const long long s = __ldg(slots + i);
        if (s == -1) continue;  // padding token
        if (s < 0 || s >= num_slots) {
            if (rem == 0) set_error(err, ERR_BOUNDS);
            continue;
        }
        const int h = rem / chunks_per_row, c = rem - h * chunks_per_row;
        const long long blk = s / block_size;
        const int off = int(s - blk * block_size);
        const long long dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + c;
        k_cache[dst] = __ldg(k + idx);
        v_cache[dst] = __ldg(v + idx);
    }
}

// ------------------------------------------------------------------- merge

// Log-sum-exp merge.  A CTA of 8 warps serves 8 / WPR rows (sequence, query
// head); the WPR warps of a row each take every WPR-th partition, with lanes
// owning D/32 dims and up to 8 partitions in flight per warp, and add their sums
// in shared memory.  Every warp of a row first reduces the maximum m_k and the
// weight sum over all partitions itself (lane-parallel), so no barrier is needed
// before the accumulation.  WPR grows with the partition count (host side).
constexpr int MERGE_WARPS = 8;
#ifndef PF_MERGE_WPR16_FROM
#define PF_MERGE_WPR16_FROM 256  // partitions per row from which a row takes 16 warps
#endif

// Loads of the partials the partition pass wrote just before: each is read once.
__device__ __forceinline__ float ld_stream(const float* p) {
    float v;
    asm volatile("ld.global.cs.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
template <int DPL>
__device__ __forceinline__ void ld_stream_row(const float* src, bool in, float (&x)[DPL]) {
    if constexpr (DPL == 4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (in)
            asm volatile("ld.global.cs.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(src));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
        float2 v = make_float2(0.f, 0.f);
        if (in) asm volatile("ld.global.cs.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(src));
        x[0] = v.x; x[1] = v.y;
    }
}

// warps of a merge CTA: MERGE_WARPS, or WPR when one row takes more
template <int WPR>
constexpr int merge_warps() { return WPR > MERGE_WARPS ? WPR : MERGE_WARPS; }

template <int D, int WPR>
__global__ void __launch_bounds__(merge_warps<WPR>() * 32) lse_merge_kernel(const float* __restrict__ tmp_out,
                                                                     const float* __restrict__ tmp_m,
                                                                     const float* __restrict__ tmp_l,
                                                                     const int32_t* __restrict__ context_lens,
                                                                     int num_seqs, int num_q_heads,
                                                                     int partition_size, int num_partitions,
                                                                     int max_context_len, float* __restrict__ out,
                                                                     unsigned* err) {
    constexpr int DPL = D / 32;
    constexpr int NWM = merge_warps<WPR>();
    constexpr int ROWS = NWM / WPR;
    constexpr float kLog2e = 1.4426950408889634f;
    __shared__ __align__(16) float accs[NWM][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rloc = warp / WPR, sub = warp % WPR;
    const long long row = (long long)blockIdx.x * ROWS + rloc;   // (seq, q head)
    const bool active = row < (long long)num_seqs * num_q_heads;
    const int L = active ? __ldg(context_lens + row / num_q_heads) : 0;
    const bool bad = active && (L < 0 || L > max_context_len);
    if (bad && sub == 0 && lane == 0) set_error(err, ERR_BOUNDS);
    const int np = (active && !bad) ? (L + partition_size - 1) / partition_size : 0;
    const size_t base = active ? size_t(row) * num_partitions : 0;

    // The partials come from the partition pass launched just before on this stream;
    // with programmatic launch this CTA may start early and waits here for that grid.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // maximum M and weight sum W = sum_k l_k exp(m_k - M), online per lane over batches
    // of SB partitions whose loads are all in flight together ...
    constexpr int SB = 8;
    float M = -INFINITY, W = 0.f;
    for (int k0 = 0; k0 < np; k0 += 32 * SB) {
        float mk[SB], lk[SB];
#pragma unroll
        for (int u = 0; u < SB; ++u) {
            const int k = k0 + lane + 32 * u;
            mk[u] = k < np ? ld_stream(tmp_m + base + k) : -INFINITY;
            lk[u] = k < np ? ld_stream(tmp_l + base + k) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < SB; ++u) {
            const float Mn = fmaxf(M, mk[u]);
            if (Mn != -INFINITY) W = W * exp2_approx((M - Mn) * kLog2e) + lk[u] * exp2_approx((mk[u] - Mn) * kLog2e);
            M = Mn;
        }
    }
    // ... then across the warp
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const float M2 = __shfl_xor_sync(FULL_MASK, M, s), W2 = __shfl_xor_sync(FULL_MASK, W, s);
        const float Mn = fmaxf(M, M2);
        if (Mn != -INFINITY) W = W * exp2_approx((M - Mn) * kLog2e) + W2 * exp2_approx((M2 - Mn) * kLog2e);
        M = Mn;
    }

    // weighted sum of this warp's partitions sub, sub + WPR, ..., AB at a time
    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
    constexpr int AB = 16;
    for (int k0 = sub; k0 < np; k0 += AB * WPR) {
        float wk[AB], x[AB][DPL];
#pragma unroll
        for (int u = 0; u < AB; ++u) {
            const int k = k0 + u * WPR;
            const bool in = k < np;
            const float m = in ? ld_stream(tmp_m + base + k) : -INFINITY;
            const float l = in ? ld_stream(tmp_l + base + k) : 0.f;
            wk[u] = in ? l * exp2_approx((m - M) * kLog2e) : 0.f;
            ld_stream_row(tmp_out + (base + (in ? k : 0)) * D + lane * DPL, in, x[u]);
        }
#pragma unroll
        for (int u = 0; u < AB; ++u)
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[e] += wk[u] * x[u][e];
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) accs[warp][lane * DPL + e] = acc[e];
    __syncthreads();
    if (!active) return;
    float* o = out + row * D;
    for (int d = sub * 32 + lane; d < D; d += WPR * 32) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < WPR; ++j) s += accs[rloc * WPR + j][d];
        o[d] = bad ? NAN : (np == 0 ? 0.f : s / W);
    }
}

// Launched with programmatic stream serialization: the merge's CTAs may be
// scheduled while the partition pass finishes, and wait in griddepcontrol.wait.
template <int D, int WPR>
static cudaError_t launch_merge_wpr(unsigned blocks, cudaStream_t s, const float* to, const float* tm,
                                    const float* tl, const int32_t* context_lens, int num_seqs, int num_q_heads,
                                    int partition_size, int np, int max_context_len, float* out, unsigned* err) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(merge_warps<WPR>() * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lse_merge_kernel<D, WPR>, to, tm, tl, context_lens, num_seqs, num_q_heads,
                              partition_size, np, max_context_len, out, err);
}

template <int D>
static cudaError_t launch_merge(int wpr, unsigned blocks, cudaStream_t s, const float* to, const float* tm,
                                const float* tl, const int32_t* context_lens, int num_seqs, int num_q_heads,
                                int partition_size, int np, int max_context_len, float* out, unsigned* err) {
    switch (wpr) {
        case 1: return launch_merge_wpr<D, 1>(blocks, s, to, tm, tl, context_lens, num_seqs, num_q_heads,
                                              partition_size, np, max_context_len, out, err);
        case 2: return launch_merge_wpr<D, 2>(blocks, s, to, tm, tl, context_lens, num_seqs, num_q_heads,
                                              partition_size, np, max_context_len, out, err);
        case 4: return launch_merge_wpr<D, 4>(blocks, s, to, tm, tl, context_lens, num_seqs, num_q_heads,
                                              partition_size, np, max_context_len, out, err);
        case 16: return launch_merge_wpr<D, 16>(blocks, s, to, tm, tl, context_lens, num_seqs, num_q_heads,
                                                 partition_size, np, max_context_len, out, err);
        default: return launch_merge_wpr<D, 8>(blocks, s, to, tm, tl, context_lens, num_seqs, num_q_heads,
                                               partition_size, np, max_context_len, out, err);
    }
}

// ------------------------------------------------------ bounded-wait check

// Waits on a barrier that nothing completes, through the same bounded wait as
// the attention kernels; there are no copies in flight, so giving up is clean.
__global__ void bounded_wait_kernel(unsigned* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(b, 0, limit_ns)) set_error(err, ERR_TIMEOUT);
}

// ------------------------------------------------------------------ helpers

static bool aligned(const void* p, size_t a) { return p != nullptr && reinterpret_cast<uintptr_t>(p) % a == 0; }
static bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
static int log2_int(int x) {
    int s = 0;
    while ((1 << s) < x) ++s;
    return s;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// a * b * c * d without overflow of size_t, or SIZE_MAX
static size_t mul_sat(size_t a, size_t b) { return (b != 0 && a > SIZE_MAX / b) ? SIZE_MAX : a * b; }

struct AttnArgs {
    const void* q; const void* k_cache; const void* v_cache;
    const int32_t* block_tables; const int32_t* context_lens;
    int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq;
    int64_t num_blocks;
    float scale;
};

static pf_status check_attention(const AttnArgs& a) {
    if (a.num_seqs < 0 || a.num_q_heads <= 0 || a.num_kv_heads <= 0 || a.head_dim <= 0 || a.block_size <= 0 ||
        a.max_blocks_per_seq <= 0 || a.num_blocks <= 0 || !std::isfinite(a.scale))
        return PF_ERR_INVALID_ARG;
    if (a.num_q_heads % a.num_kv_heads != 0) return PF_ERR_INVALID_ARG;
    if (a.num_blocks > INT32_MAX) return PF_ERR_INVALID_ARG;  // table entries are int32
    const size_t cache_elems =
        mul_sat(mul_sat(mul_sat(size_t(a.num_blocks), size_t(a.num_kv_heads)), size_t(a.block_size)),
                size_t(a.head_dim));
    if (cache_elems >= (SIZE_MAX >> 2)) return PF_ERR_INVALID_ARG;
    if ((long long)a.num_seqs * a.num_kv_heads > INT32_MAX) return PF_ERR_INVALID_ARG;
    if (a.num_seqs > 0 && (!aligned(a.q, 16) || !aligned(a.k_cache, 16) || !aligned(a.v_cache, 16) ||
                           !aligned(a.block_tables, 4) || !aligned(a.context_lens, 4)))
        return PF_ERR_INVALID_ARG;
    const int g = a.num_q_heads / a.num_kv_heads;
    if (a.head_dim != 64 && a.head_dim != 128) return PF_ERR_UNSUPPORTED;
    if (g != 1 && g != 2 && g != 4 && g != 8) return PF_ERR_UNSUPPORTED;
    if (a.block_size % kTileTokens != 0) return PF_ERR_UNSUPPORTED;
    return PF_OK;
}

static DecodeParams make_params(const AttnArgs& a, unsigned* err) {
    DecodeParams p{};
    p.q = static_cast<const uint16_t*>(a.q);
    p.k_cache = static_cast<const uint16_t*>(a.k_cache);
    p.v_cache = static_cast<const uint16_t*>(a.v_cache);
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    p.err = err;
    p.num_blocks = a.num_blocks;
    p.wait_limit_ns = kDefaultWaitLimitNs;
    p.scale_log2 = float(double(a.scale) * 1.4426950408889634);
    p.num_seqs = a.num_seqs;
    p.num_q_heads = a.num_q_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.block_size = a.block_size;
    p.block_shift = is_pow2(a.block_size) ? log2_int(a.block_size) : -1;
    p.max_blocks_per_seq = a.max_blocks_per_seq;
    return p;
}

// CTA order of the single pass: longest first when the items outnumber the CTAs that are resident
// at once (three per SM) -- the hardware's in-order dispatch then starts the long items first --
// and natural otherwise, where every item starts at once and the order cannot matter.
static int decode_order(int num_seqs, int num_kv_heads) {
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) sms = 0;
    const long long items = (long long)num_seqs * num_kv_heads;
    const bool queued = sms <= 0 || items > 3LL * sms;
    return (queued && num_seqs > 1 && num_seqs <= kMaxSortedSeqsDecode) ? ORDER_SORTED : ORDER_NATURAL;
}

static cudaError_t launch_decode(const DecodeParams& p, int head_dim, int group, int mode, cudaStream_t stream) {
    return head_dim == 64 ? launch_decode_d64(p, group, mode, stream) : launch_decode_d128(p, group, mode, stream);
}

pf_status check_split_arguments(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int max_blocks_per_seq, int64_t num_blocks, float scale, int partition_size,
                                int max_context_len) {
    const AttnArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, max_blocks_per_seq, num_blocks, scale};
    pf_status st = check_attention(a);
    if (st != PF_OK) return st;
    if (partition_size <= 0 || max_context_len < 0) return PF_ERR_INVALID_ARG;
    if (partition_size % kTileTokens != 0) return PF_ERR_UNSUPPORTED;
    return PF_OK;
}

}  // namespace pf

using namespace pf;

// ======================================================================= ABI

extern "C" {

const char* pf_version(void) { return "0.1.0"; }

const char* pf_status_string(pf_status s) {
    switch (s) {
        case PF_OK: return "PF_OK";
        case PF_ERR_INVALID_ARG: return "PF_ERR_INVALID_ARG";
        case PF_ERR_UNSUPPORTED: return "PF_ERR_UNSUPPORTED";
        case PF_ERR_CUDA: return "PF_ERR_CUDA";
        case PF_ERR_DEVICE_BOUNDS: return "PF_ERR_DEVICE_BOUNDS";
        case PF_ERR_DEVICE_TIMEOUT: return "PF_ERR_DEVICE_TIMEOUT";
        default: return "PF_UNKNOWN_STATUS";
    }
}

pf_status pf_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping, void* k_cache,
                               void* v_cache, int64_t num_tokens, int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, pf_stream_t stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PF_ERR_INVALID_ARG;
    if (head_dim % 8 != 0) return PF_ERR_UNSUPPORTED;
    const size_t cache_elems =
        mul_sat(mul_sat(mul_sat(size_t(num_blocks), size_t(num_kv_heads)), size_t(block_size)), size_t(head_dim));
    const size_t in_elems = mul_sat(mul_sat(size_t(num_tokens), size_t(num_kv_heads)), size_t(head_dim));
    if (cache_elems >= (SIZE_MAX >> 2) || in_elems >= (SIZE_MAX >> 2) ||
        (long long)num_kv_heads * (head_dim / 8) > INT32_MAX)
        return PF_ERR_INVALID_ARG;
    if (num_tokens == 0) return PF_OK;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PF_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    int sms = 0;
    if (error_word(&err) != cudaSuccess || sm_count(&sms) != cudaSuccess) return PF_ERR_CUDA;
    const long long total = (long long)num_tokens * num_kv_heads * (head_dim / 8);
    const long long want = (total + 255) / 256;
    const unsigned blocks = unsigned(want < (long long)sms * 16 ? want : (long long)sms * 16);
    reshape_and_cache_kernel<<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, static_cast<uint4*>(k_cache),
        static_cast<uint4*>(v_cache), total, num_kv_heads, head_dim / 8, block_size,
        (long long)num_blocks * block_size, err);
    return cudaGetLastError() == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

pf_status pf_paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                    int max_blocks_per_seq, int64_t num_blocks, float scale, float* out,
                                    pf_stream_t stream) {
    const AttnArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, max_blocks_per_seq, num_blocks, scale};
    pf_status st = check_attention(a);
    if (st != PF_OK) return st;
    if (num_seqs == 0) return PF_OK;
    if (!aligned(out, 16)) return PF_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    if (error_word(&err) != cudaSuccess) return PF_ERR_CUDA;
    DecodeParams p = make_params(a, err);
    p.out = out;
    p.order_mode = decode_order(num_seqs, num_kv_heads);
    const cudaError_t e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, MODE_DECODE,
                                        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

pf_status pf_paged_attention_decode_bf16(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                         int max_blocks_per_seq, int64_t num_blocks, float scale, void* out,
                                         pf_stream_t stream) {
    const AttnArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, max_blocks_per_seq, num_blocks, scale};
    pf_status st = check_attention(a);
    if (st != PF_OK) return st;
    if (num_seqs == 0) return PF_OK;
    if (!aligned(out, 16)) return PF_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    if (error_word(&err) != cudaSuccess) return PF_ERR_CUDA;
    DecodeParams p = make_params(a, err);
    p.out_bf16 = static_cast<uint16_t*>(out);
    p.order_mode = decode_order(num_seqs, num_kv_heads);
    const cudaError_t e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, MODE_DECODE,
                                        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

pf_status pf_paged_attention_decode_append(const void* q, const void* k_new, const void* v_new,
                                           const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                           const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                           int max_blocks_per_seq, int64_t num_blocks, float scale, float* out,
                                           pf_stream_t stream) {
    const AttnArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, max_blocks_per_seq, num_blocks, scale};
    pf_status st = check_attention(a);
    if (st != PF_OK) return st;
    if (num_seqs == 0) return PF_OK;
    if (!aligned(out, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8))
        return PF_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    if (error_word(&err) != cudaSuccess) return PF_ERR_CUDA;
    DecodeParams p = make_params(a, err);
    p.out = out;
    p.order_mode = decode_order(num_seqs, num_kv_heads);
    p.k_new = static_cast<const uint16_t*>(k_new);
    p.v_new = static_cast<const uint16_t*>(v_new);
    p.slot_mapping = slot_mapping;
    p.k_cache_w = static_cast<uint16_t*>(k_cache);
    p.v_cache_w = static_cast<uint16_t*>(v_cache);
    const cudaError_t e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, MODE_DECODE_APPEND,
                                        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

size_t pf_paged_attention_partition_workspace_layout(int num_seqs, int num_q_heads, int head_dim,
                                                     int max_context_len, int partition_size,
                                                     size_t* tmp_out_offset, size_t* tmp_m_offset,
                                                     size_t* tmp_l_offset) {
    if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 || partition_size <= 0)
        return 0;
    const size_t np = max_context_len > 0 ? (size_t(max_context_len) + partition_size - 1) / partition_size : 1;
    const size_t n = mul_sat(mul_sat(size_t(num_seqs), size_t(num_q_heads)), np);
    const size_t out_elems = mul_sat(n, size_t(head_dim));
    if (out_elems >= (SIZE_MAX >> 4)) return 0;
    const size_t out_bytes = round_up(out_elems * 4, 256);
    const size_t ml_bytes = round_up(n * 4, 256);
    if (tmp_out_offset) *tmp_out_offset = 0;
    if (tmp_m_offset) *tmp_m_offset = out_bytes;
    if (tmp_l_offset) *tmp_l_offset = out_bytes + ml_bytes;
    return out_bytes + 2 * ml_bytes;
}

size_t pf_paged_attention_partition_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                                   int max_context_len, int partition_size) {
    return pf_paged_attention_partition_workspace_layout(num_seqs, num_q_heads, head_dim, max_context_len,
                                                         partition_size, nullptr, nullptr, nullptr);
}

pf_status pf_paged_attention_decode_partition(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* block_tables, const int32_t* context_lens,
                                              int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                              int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                              float scale, int partition_size, int max_context_len,
                                              void* workspace, size_t workspace_bytes, pf_stream_t stream) {
    const AttnArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, max_blocks_per_seq, num_blocks, scale};
    pf_status st = check_split_arguments(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                                         num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                                         partition_size, max_context_len);
    if (st != PF_OK) return st;
    if (num_seqs == 0) return PF_OK;
    size_t off_o = 0, off_m = 0, off_l = 0;
    const size_t need = pf_paged_attention_partition_workspace_layout(num_seqs, num_q_heads, head_dim,
                                                                      max_context_len, partition_size, &off_o,
                                                                      &off_m, &off_l);
    if (need == 0 || workspace_bytes < need || !aligned(workspace, 256)) return PF_ERR_INVALID_ARG;
    const long long np = max_context_len > 0 ? ((long long)max_context_len + partition_size - 1) / partition_size : 1;
    if (np * num_kv_heads * num_seqs > INT32_MAX) return PF_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    if (error_word(&err) != cudaSuccess) return PF_ERR_CUDA;
    DecodeParams p = make_params(a, err);
    char* ws = static_cast<char*>(workspace);
    p.out = reinterpret_cast<float*>(ws + off_o);
    p.part_m = reinterpret_cast<float*>(ws + off_m);
    p.part_l = reinterpret_cast<float*>(ws + off_l);
    p.partition_size = partition_size;
    p.num_partitions = int(np);
    p.max_context_len = max_context_len;
    p.order_mode = num_seqs <= kMaxSortedSeqsPartition ? ORDER_SORTED : ORDER_NATURAL;
    const cudaError_t e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, MODE_PARTITION,
                                        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

pf_status pf_paged_attention_merge(const void* workspace, const int32_t* context_lens, int num_seqs,
                                   int num_q_heads, int head_dim, int partition_size, int max_context_len,
                                   float* out, pf_stream_t stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || partition_size <= 0 || max_context_len < 0)
        return PF_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PF_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PF_OK;
    if (!aligned(workspace, 256) || !aligned(context_lens, 4) || !aligned(out, 16)) return PF_ERR_INVALID_ARG;
    size_t off_o = 0, off_m = 0, off_l = 0;
    if (pf_paged_attention_partition_workspace_layout(num_seqs, num_q_heads, head_dim, max_context_len,
                                                      partition_size, &off_o, &off_m, &off_l) == 0)
        return PF_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    if (error_word(&err) != cudaSuccess) return PF_ERR_CUDA;
    const int np = max_context_len > 0 ? int(((long long)max_context_len + partition_size - 1) / partition_size) : 1;
    const char* ws = static_cast<const char*>(workspace);
    const long long rows = (long long)num_seqs * num_q_heads;
    // warps per row: enough that each warp has about 16 partitions or fewer to add
    const int wpr = np >= PF_MERGE_WPR16_FROM ? 16 : np >= 128 ? 8 : np >= 64 ? 4 : np >= 32 ? 2 : 1;
    const int rows_per_cta = (wpr > MERGE_WARPS ? wpr : MERGE_WARPS) / wpr;
    const long long blocks = (rows + rows_per_cta - 1) / rows_per_cta;
    if (blocks > INT32_MAX) return PF_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float* to = reinterpret_cast<const float*>(ws + off_o);
    const float* tm = reinterpret_cast<const float*>(ws + off_m);
    const float* tl = reinterpret_cast<const float*>(ws + off_l);
    const cudaError_t e =
        head_dim == 64 ? launch_merge<64>(wpr, unsigned(blocks), s, to, tm, tl, context_lens, num_seqs, num_q_heads,
                                          partition_size, np, max_context_len, out, err)
                       : launch_merge<128>(wpr, unsigned(blocks), s, to, tm, tl, context_lens, num_seqs, num_q_heads,
                                           partition_size, np, max_context_len, out, err);
    return e == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

pf_status pf_get_device_error(pf_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned* err = nullptr;
    if (error_word(&err) != cudaSuccess) return PF_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PF_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, err, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess) return PF_ERR_CUDA;
    if (cudaMemsetAsync(err, 0, sizeof word, s) != cudaSuccess) return PF_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PF_ERR_CUDA;
    if (word & ERR_TIMEOUT) return PF_ERR_DEVICE_TIMEOUT;
    if (word & ERR_BOUNDS) return PF_ERR_DEVICE_BOUNDS;
    return PF_OK;
}

pf_status pf_debug_bounded_wait(int64_t limit_ns, pf_stream_t stream) {
    if (limit_ns < 1000 || limit_ns > 10000000000LL) return PF_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    if (error_word(&err) != cudaSuccess) return PF_ERR_CUDA;
    bounded_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err, (unsigned long long)limit_ns);
    return cudaGetLastError() == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

}  // extern "C"

// ======================================================== auto decomposition

namespace pf {
// Decode CTAs resident per SM at the compiled configuration (shared memory bound).
constexpr int kDecodeCtasPerSm = 3;
// Cluster split: at most this many CTAs per item (the portable cluster size) and tokens per CTA.
constexpr int kClusterMax = kClusterMaxSize;
constexpr int kClusterMaxChunk = 1024;

// The cluster split applies when the single pass would leave more than half the SMs without
// an item and a cluster of at most kClusterMax CTAs covers the longest context in chunks of at
// most kClusterMaxChunk tokens.  C: the largest power of two with items * C <= the resident CTA
// slots, at most one chunk of 16 tokens per CTA; chunk: tokens per CTA, a multiple of 16.
static bool cluster_plan(long long items, int sms, int max_context_len, int* C_out, int* chunk_out) {
    if (items <= 0 || items * 2 > sms || max_context_len < 2 * kTileTokens) return false;
    const long long slots = (long long)sms * kDecodeCtasPerSm;
    const int tiles = (max_context_len + kTileTokens - 1) / kTileTokens;
    int C = 1;
    while (C * 2 <= kClusterMax && items * C * 2 <= slots && C * 2 <= tiles) C *= 2;
    if (C < 2) return false;
    const int chunk = (tiles + C - 1) / C * kTileTokens;
    if (chunk > kClusterMaxChunk) return false;
    *C_out = C;
    *chunk_out = chunk;
    return true;
}
}  // namespace pf

extern "C" {

int pf_paged_attention_decode_auto_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                        int max_context_len, size_t* workspace_bytes) {
    if (workspace_bytes) *workspace_bytes = 0;
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess || sms <= 0) return 0;
    const long long slots = (long long)sms * kDecodeCtasPerSm;
    const long long items = (long long)num_seqs * num_kv_heads;
    // Few items and short contexts: the cluster split (no workspace) -- C CTAs per item, each
    // a chunk of at most kClusterMaxChunk tokens, merged through distributed shared memory.
    int C = 0, chunk = 0;
    if (cluster_plan(items, sms, max_context_len, &C, &chunk)) return chunk;
    // Enough (sequence, kv head) items, or short contexts: one pass, ordered longest first.
    if (items >= 2 * slots || max_context_len <= 1024) return 0;
    // Otherwise split so that one sequence of the longest length alone spreads over about
    // two CTAs per slot: P = the largest power of two <= max_len * Hkv / (2 * slots), >= 256.
    const long long target = (long long)max_context_len * num_kv_heads / (2 * slots);
    int P = 256;
    while ((long long)P * 2 <= target && P < (1 << 16)) P *= 2;
    const size_t need =
        pf_paged_attention_partition_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len, P);
    if (need == 0) return 0;
    if (workspace_bytes) *workspace_bytes = need;
    return P;
}

pf_status pf_paged_attention_decode_auto(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                         int max_blocks_per_seq, int64_t num_blocks, float scale,
                                         int max_context_len, void* workspace, size_t workspace_bytes, float* out,
                                         pf_stream_t stream) {
    if (max_context_len < 0) return PF_ERR_INVALID_ARG;
    size_t need = 0;
    const int P = pf_paged_attention_decode_auto_plan(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                      max_context_len, &need);
    if (P > 0 && need == 0) {
        // the cluster split: no workspace
        const AttnArgs a{q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                         head_dim, block_size, max_blocks_per_seq, num_blocks, scale};
        pf_status st = check_attention(a);
        if (st != PF_OK) return st;
        if (!aligned(out, 16)) return PF_ERR_INVALID_ARG;
        int sms = 0, C = 0, chunk = 0;
        if (sm_count(&sms) != cudaSuccess) return PF_ERR_CUDA;
        if (!cluster_plan((long long)num_seqs * num_kv_heads, sms, max_context_len, &C, &chunk) || chunk != P)
            return PF_ERR_CUDA;
        unsigned* err = nullptr;
        if (error_word(&err) != cudaSuccess) return PF_ERR_CUDA;
        DecodeParams p = make_params(a, err);
        p.out = out;
        p.order_mode = ORDER_NATURAL;
        p.partition_size = chunk;
        p.cluster_size = C;
        p.max_context_len = max_context_len;
        const cudaError_t e = launch_decode(p, head_dim, num_q_heads / num_kv_heads, MODE_CLUSTER,
                                            reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? PF_OK : PF_ERR_CUDA;
    }
    if (P == 0)
        return pf_paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                                         num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                                         out, stream);
    if (workspace_bytes < need || !aligned(workspace, 256)) return PF_ERR_INVALID_ARG;
    pf_status st = pf_paged_attention_decode_partition(q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                                       num_q_heads, num_kv_heads, head_dim, block_size,
                                                       max_blocks_per_seq, num_blocks, scale, P, max_context_len,
                                                       workspace, workspace_bytes, stream);
    if (st != PF_OK) return st;
    return pf_paged_attention_merge(workspace, context_lens, num_seqs, num_q_heads, head_dim, P, max_context_len,
                                    out, stream);
}

}  // extern "C"

// Paged-KV decode attention kernel (single pass and context-partition pass).
//
// Method: decode-phase attention that reads K/V straight out of physical KV
// blocks through a per-sequence block table with an online softmax and
// grouped-query heads (ForgeLLM README, feature list: "Physical KV blocks with
// logical per-request block tables", "Decode-only block-table attention reads
// physical KV blocks directly ... online softmax without constructing padded
// batch-wide K/V", "grouped-query attention"), with warp-shuffle max / sum
// reductions (LLM-Inference-Engine README, "Flash Attention CUDA Kernel ...
// warp-level shuffle reductions").  The split over context partitions with a
// log-sum-exp merge is the flash-decoding decomposition of the same sums.
//
// GB300 design:
//  * One CTA owns one (sequence, kv head [, partition]) item and all G query
//    heads that share the kv head, so each K/V byte is read from HBM once.
//  * The cache layout [block, kv head, token, dim] makes every (block, kv head)
//    tile contiguous; a tile of 16 tokens (2 KiB for D=64, 4 KiB for D=128, for
//    each of K and V) moves with one cp.async.bulk per operand into shared
//    memory, completing on an mbarrier.  Only the valid rows of a sequence's
//    last tile are copied.
//  * Each warp is an independent streamer: it takes every NW-th tile of the
//    item, keeps NST tiles in flight in a private ring, and lane 0 issues the
//    copies, prefetching block-table entries NST+2 tiles ahead.
//  * Scores: lanes split each 16-token tile as (token, 16-byte chunk); a lane
//    holds its chunk of all G query rows in fp32 registers (64 values), so the
//    G dot products cost one shared-memory read per chunk.  Chunk order is
//    rotated per token so the 8 lanes of a shared-memory phase hit distinct
//    banks.  A reduce-scatter over the lanes of a token leaves one finished
//    score per lane.
//  * fp32 online softmax in base 2 (scale*log2(e) folded in), warp-shuffle max
//    and sum; probabilities go through a warp-private shared buffer to the
//    P.V step, where each lane owns D/32 output dims of all G heads.
//  * The NW warps of a CTA merge their (m, l, acc) in shared memory at the end.
//  * No trap, no unbounded spin: every mbarrier wait is bounded; a bad table
//    entry or length sets the device error word and NaN-fills the item's rows.
#pragma once

#include <atomic>
#include <cmath>

#include "pf_device.cuh"
#include "pf_internal.h"

namespace pf {

template <int D, int G>
struct DecodeGeometry {
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group");
    static constexpr int TT = kTileTokens;
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int TILE_BYTES = TT * ROW_BYTES;        // one K (or V) tile
    static constexpr int CHUNKS_PER_ROW = D / 8;             // 16-byte chunks in a token row
    static constexpr int LPT = (G * D / 64) > 2 ? (G * D / 64) : 2;  // lanes per token (scores)
    static constexpr int TPP = 32 / LPT;                     // tokens per score pass
    static constexpr int NPASS = TT / TPP;                   // score passes per tile
    static constexpr int CPL = CHUNKS_PER_ROW / LPT;         // chunks per lane per row
    static constexpr int DUP = LPT / G;                      // lanes left holding the same score
    static constexpr int DPL = D / 32;                       // output dims per lane (P.V)
    static constexpr int ROT_MOD = LPT < 8 ? 8 / LPT : 1;    // tokens sharing a smem phase
    static constexpr int PSM = TT * G + G;                   // probabilities + per-head alpha
    static constexpr int PSM_PAD = (PSM + 3) & ~3;
    static_assert(CPL * LPT == CHUNKS_PER_ROW && NPASS * TPP == TT, "geometry");
};

// Bytes of the per-warp failure flags, padded so the mbarriers that follow stay aligned.
template <int NW>
constexpr int flag_bytes() { return (NW * 4 + 15) / 16 * 16; }

// Offset, from the first mbarrier, of the int array used to order work items.
template <int NW, int NST>
constexpr int sorted_keys_offset() { return (NW * NST * 8 + 15) / 16 * 16; }

template <int D, int G, int NW, int NST>
constexpr size_t decode_smem_bytes() {
    using Geo = DecodeGeometry<D, G>;
    return size_t(NW) * NST * 2 * Geo::TILE_BYTES      // K/V stages
           + size_t(NW) * Geo::PSM_PAD * 4             // probabilities, alpha; then m, l
           + flag_bytes<NW>()                          // per-warp failure flags
           + sorted_keys_offset<NW, NST>();            // mbarriers (+ padding)
    // followed, in ORDER_SORTED launches, by round_up(num_seqs, 4) ints of keys
}

// ORDER_SORTED item selection (see pf_internal.h).  `keys` holds round_up(S, 4)
// ints of shared memory.  Returns false when this CTA has no item.
template <int NW, bool PART>
__device__ __forceinline__ bool select_sorted_item(const DecodeParams& p, int* keys, int* seq, int* kvh,
                                                   int* part) {
    __shared__ int s_item;
    __shared__ int s_warp_sum[NW];
    constexpr int NT = NW * 32;
    const int S = p.num_seqs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    *kvh = blockIdx.x % p.num_kv_heads;
    const int r = blockIdx.x / p.num_kv_heads;
    if constexpr (!PART) {
        // key = (length, reversed index): unique, so the ranks are a permutation
        const int Sp = (S + 3) & ~3;
        for (int i = tid; i < Sp; i += NT) {
            int key = -1;
            if (i < S) {
                const int Li = min(max(__ldg(p.context_lens + i), 0), (1 << 20) - 1);
                key = (Li << 10) | (1023 - i);
            }
            keys[i] = key;
        }
        __syncthreads();
        for (int i = tid; i < S; i += NT) {
            const int ki = keys[i];
            int rank = 0;
            for (int j = 0; j < Sp; j += 4) {
                const int4 kj = *reinterpret_cast<const int4*>(keys + j);
                rank += int(kj.x > ki) + int(kj.y > ki) + int(kj.z > ki) + int(kj.w > ki);
            }
            if (rank == r) s_item = i;
        }
        __syncthreads();
        *seq = s_item;
        *part = 0;
        return true;
    } else {
        // non-empty partitions per sequence, then an inclusive prefix over sequences
        const int P = p.partition_size;
        bool bad = false;
        for (int i = tid; i < S; i += NT) {
            const int Li = __ldg(p.context_lens + i);
            const bool b = Li < 0 || Li > p.max_context_len;
            bad = bad || b;
            keys[i] = b ? 0 : (Li + P - 1) / P;
        }
        if (bad && blockIdx.x == 0) set_error(p.err, ERR_BOUNDS);  // the merge NaN-fills those rows
        __syncthreads();
        const int per = (S + NT - 1) / NT;
        const int i0 = tid * per;
        int sum = 0;
        for (int k = 0; k < per; ++k)
            if (i0 + k < S) sum += keys[i0 + k];
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL_MASK, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_warp_sum[warp] = incl;
        __syncthreads();
        int run = incl - sum;
        for (int w = 0; w < warp; ++w) run += s_warp_sum[w];
        for (int k = 0; k < per; ++k)
            if (i0 + k < S) {
                run += keys[i0 + k];
                keys[i0 + k] = run;
            }
        __syncthreads();
        if (r >= keys[S - 1]) return false;
        int lo = 0, hi = S - 1;  // first sequence whose inclusive prefix exceeds r
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (keys[mid] > r) hi = mid; else lo = mid + 1;
        }
        *seq = lo;
        *part = r - (lo > 0 ? keys[lo - 1] : 0);
        return true;
    }
}

// Sum of v[0..G-1] over the LPT lanes of one token, spread so that afterwards
// lane slice `sl` holds the full sum of head sl / DUP in v[0].
template <int G, int LPT>
__device__ __forceinline__ float reduce_scatter_heads(float (&v)[G], int sl) {
#pragma unroll
    for (int n = G, m = LPT / 2; n > 1; n >>= 1, m >>= 1) {
        const bool upper = (sl & m) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(FULL_MASK, send, m);
        }
    }
#pragma unroll
    for (int m = (LPT / G) / 2; m >= 1; m >>= 1) v[0] += __shfl_xor_sync(FULL_MASK, v[0], m);
    return v[0];
}

template <int G>
__device__ __forceinline__ void load_probs(const float* src, float (&pw)[G]) {
    if constexpr (G == 1) {
        pw[0] = src[0];
    } else if constexpr (G == 2) {
        const float2 a = *reinterpret_cast<const float2*>(src);
        pw[0] = a.x; pw[1] = a.y;
    } else {
#pragma unroll
        for (int i = 0; i < G; i += 4) {
            const float4 a = *reinterpret_cast<const float4*>(src + i);
            pw[i] = a.x; pw[i + 1] = a.y; pw[i + 2] = a.z; pw[i + 3] = a.w;
        }
    }
}

// One warp's share of an item: the lane's slice of the G query rows in fp32
// registers, the online-softmax state of the head whose scores the lane holds,
// and the P.V accumulator for D/32 output dims of all G heads.  tile() consumes
// one 16-token K/V tile from shared memory (nvalid of its rows are tokens).
template <int D, int G>
struct WarpAttention {
    using Geo = DecodeGeometry<D, G>;
    static constexpr int TT = Geo::TT, LPT = Geo::LPT, TPP = Geo::TPP, NPASS = Geo::NPASS, CPL = Geo::CPL;
    static constexpr int DUP = Geo::DUP, DPL = Geo::DPL, ROW = Geo::ROW_BYTES;

    int lane, tp, sl, hh, rot;
    bool writer;  // one lane per (head, token) writes shared state
    int kofs[CPL];
    float2 qf[G][CPL][4];
    float m_run, l_run;
    float2 acc[G][DPL / 2];

    __device__ __forceinline__ void init(int lane_) {
        lane = lane_;
        tp = lane / LPT;
        sl = lane % LPT;
        hh = sl / DUP;
        rot = tp % Geo::ROT_MOD;
        writer = (sl % DUP) == 0;
#pragma unroll
        for (int j = 0; j < CPL; ++j) kofs[j] = tp * ROW + (sl + LPT * ((j + rot) % CPL)) * 16;
    }

    // q rows of the group's G heads, consecutive [G][D] bf16
    __device__ __forceinline__ void load_q(const uint16_t* qrows) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int chunk = sl + LPT * ((j + rot) % CPL);
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(qrows + h * D + chunk * 8));
                qf[h][j][0] = bf16x2_to_float2(w.x);
                qf[h][j][1] = bf16x2_to_float2(w.y);
                qf[h][j][2] = bf16x2_to_float2(w.z);
                qf[h][j][3] = bf16x2_to_float2(w.w);
            }
        }
    }

    __device__ __forceinline__ void reset() {
        m_run = -INFINITY;
        l_run = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < DPL / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);
    }

    __device__ __forceinline__ void tile(const unsigned char* Ks, const unsigned char* Vs, int nvalid, float* psm,
                                         float scale_log2) {
        // -- scores of this lane's tokens for head hh, base-2 units
        float sc[NPASS];
#pragma unroll
        for (int pass = 0; pass < NPASS; ++pass) {
            const unsigned char* rowp = Ks + pass * TPP * ROW;
            float2 a[G];
#pragma unroll
            for (int h = 0; h < G; ++h) a[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const uint4 w = *reinterpret_cast<const uint4*>(rowp + kofs[j]);
                const float2 k0 = bf16x2_to_float2(w.x), k1 = bf16x2_to_float2(w.y);
                const float2 k2 = bf16x2_to_float2(w.z), k3 = bf16x2_to_float2(w.w);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    a[h] = ffma2(qf[h][j][0], k0, a[h]);
                    a[h] = ffma2(qf[h][j][1], k1, a[h]);
                    a[h] = ffma2(qf[h][j][2], k2, a[h]);
                    a[h] = ffma2(qf[h][j][3], k3, a[h]);
                }
            }
            float v[G];
#pragma unroll
            for (int h = 0; h < G; ++h) v[h] = a[h].x + a[h].y;
            const float dot = reduce_scatter_heads<G, LPT>(v, sl);
            sc[pass] = (pass * TPP + tp < nvalid) ? dot * scale_log2 : -INFINITY;
        }

        // -- online softmax for head hh
        float mx = sc[0];
#pragma unroll
        for (int pass = 1; pass < NPASS; ++pass) mx = fmaxf(mx, sc[pass]);
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, o));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = exp2_approx(m_run - m_new);
        float psum = 0.f;
#pragma unroll
        for (int pass = 0; pass < NPASS; ++pass) {
            const float pv = exp2_approx(sc[pass] - m_new);
            psum += pv;
            if (writer) psm[(pass * TPP + tp) * G + hh] = pv;
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        if (writer && tp == 0) psm[TT * G + hh] = alpha;
        __syncwarp();

        // -- acc = alpha * acc + sum_t p_t V_t, lane owns dims [lane*DPL, lane*DPL + DPL)
        {
            float al[G];
            load_probs<G>(psm + TT * G, al);
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < DPL / 2; ++e) {
                    acc[h][e].x *= al[h];
                    acc[h][e].y *= al[h];
                }
        }
        auto pv_step = [&](int t) {
            float pw[G];
            load_probs<G>(psm + t * G, pw);
            float2 vv[DPL / 2];
            if constexpr (DPL == 4) {
                const uint2 w = *reinterpret_cast<const uint2*>(Vs + t * ROW + lane * 8);
                vv[0] = bf16x2_to_float2(w.x);
                vv[1] = bf16x2_to_float2(w.y);
            } else {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(Vs + t * ROW + lane * 4);
                vv[0] = bf16x2_to_float2(w);
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < DPL / 2; ++e) acc[h][e] = ffma2(make_float2(pw[h], pw[h]), vv[e], acc[h][e]);
        };
        if (nvalid == TT) {
#pragma unroll
            for (int t = 0; t < TT; ++t) pv_step(t);
        } else {
            for (int t = 0; t < nvalid; ++t) pv_step(t);  // rows past the length are never read
        }
        __syncwarp();
    }

    // Per-head l over the lanes holding that head, then (m, l) of the G heads to
    // ml[0 .. 2G) and acc to accs [G][D] (fp32).
    __device__ __forceinline__ void stash(float* ml, float* accs) {
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) l_run += __shfl_xor_sync(FULL_MASK, l_run, o);
        __syncwarp();
        if (writer && tp == 0) {
            ml[hh] = m_run;
            ml[G + hh] = l_run;
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < DPL / 2; ++e)
                *reinterpret_cast<float2*>(accs + h * D + lane * DPL + 2 * e) = acc[h][e];
    }
};

// fp32 -> bf16 bits, rounded to nearest with ties to even (a NaN stays a NaN).
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
    return r;
}

// Merge the NW warps' stashes of one item and write it: element e = h * D + d of the
// group; ml(w) / accs(w) locate warp w's (m, l) pairs and [G][D] accumulator.  Writes
// out_rows[h * D + d] (normalised) -- or, when out_bf16 is set, its bf16 rounding to
// out_bf16[h * D + d] -- and for a partition its natural-log max and sum.
template <int D, int G, int NW, typename MlFn, typename AccFn>
__device__ __forceinline__ void merge_warps_and_store(MlFn ml, AccFn accs, bool failed, float* out_rows,
                                                      float* part_m, float* part_l, size_t part_stride,
                                                      uint16_t* out_bf16 = nullptr) {
    for (int e = threadIdx.x; e < G * D; e += NW * 32) {
        const int h = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, ml(w)[h]);
        float wsum = 0.f, o = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float f = exp2_approx(ml(w)[h] - M);
                wsum += f * ml(w)[G + h];
                o += f * accs(w)[h * D + d];
            }
        }
        float res = wsum == 0.f ? 0.f : o / wsum;  // no token: 0; a NaN input stays NaN
        if (failed) res = NAN;
        if (out_bf16 != nullptr) out_bf16[h * part_stride * D + d] = f32_to_bf16_rn(res);
        else out_rows[h * part_stride * D + d] = res;
        if (part_m != nullptr && d == 0) {
            part_m[h * part_stride] = failed ? NAN : M * 0.6931471805599453f;
            part_l[h * part_stride] = failed ? NAN : wsum;
        }
    }
}

template <int D, int G, int NW, int NST, int MODE>
__global__ void __launch_bounds__(NW * 32) paged_decode_kernel(const DecodeParams p) {
    constexpr bool PART = MODE == MODE_PARTITION;
    constexpr bool APPEND = MODE == MODE_DECODE_APPEND;
    constexpr bool CLUS = MODE == MODE_CLUSTER;
    using Geo = DecodeGeometry<D, G>;
    constexpr int TT = Geo::TT, ROW = Geo::ROW_BYTES, TILE = Geo::TILE_BYTES;
    constexpr int PSM_PAD = Geo::PSM_PAD;
    constexpr int R = NST + 2;  // table entries lane 0 holds ahead of the copies

    extern __shared__ __align__(128) unsigned char smem[];
    float* psm_all = reinterpret_cast<float*>(smem + size_t(NW) * NST * 2 * TILE);
    int* flags = reinterpret_cast<int*>(psm_all + NW * PSM_PAD);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(flags) + flag_bytes<NW>());

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if constexpr (PART) asm volatile("griddepcontrol.launch_dependents;");  // the merge waits for completion

    // cluster split: every CTA announces it has started; the wait before the first write into
    // another CTA's shared memory (below) ensures that CTA is running
    if constexpr (CLUS) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    // ---- which item
    int seq, kvh, part = 0;
    if constexpr (CLUS) {
        // CTA `part` of its cluster takes chunk `part` of the item's tokens
        part = int(cluster_ctarank());
        const int item = blockIdx.x / p.cluster_size;
        kvh = item % p.num_kv_heads;
        seq = item / p.num_kv_heads;
    } else if (p.order_mode == ORDER_SORTED) {
        int* keys = reinterpret_cast<int*>(bars + sorted_keys_offset<NW, NST>() / 8);
        if (!select_sorted_item<NW, PART>(p, keys, &seq, &kvh, &part)) return;
    } else if constexpr (PART) {
        part = blockIdx.x % p.num_partitions;
        const int rest = blockIdx.x / p.num_partitions;
        kvh = rest % p.num_kv_heads;
        seq = rest / p.num_kv_heads;
    } else {
        kvh = blockIdx.x % p.num_kv_heads;
        seq = blockIdx.x / p.num_kv_heads;
    }
    const int Hq = p.num_q_heads;
    const int qh0 = kvh * G;
    // When the item follows from the block index (natural order, cluster split), lane 0 loads the
    // table entries of this warp's first R tiles alongside the length instead of after it; entries
    // at or past the length are loaded but never used.
    const bool spec = CLUS || (!PART && p.order_mode == ORDER_NATURAL);
    int spec_ent[R];
    if (spec && (threadIdx.x & 31) == 0) {
        const int32_t* srow = p.block_tables + size_t(seq) * p.max_blocks_per_seq;
        const int st0 = CLUS ? part * p.partition_size : 0;
        const long long cap = min((long long)p.max_blocks_per_seq * p.block_size,
                                  CLUS ? (long long)st0 + p.partition_size : (long long)INT32_MAX);
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int tok = (st0 / TT + (threadIdx.x >> 5) + j * NW) * TT;
            spec_ent[j] = tok < cap ? __ldg(srow + tok / p.block_size) : 0;
        }
    }
    const int L = __ldg(p.context_lens + seq);
    bool len_bad = L < 0 || (long long)L > (long long)p.max_blocks_per_seq * p.block_size;
    int t0 = 0, t1 = L;
    if constexpr (PART) {
        len_bad = len_bad || L > p.max_context_len;
        t0 = part * p.partition_size;
        if (!len_bad && t0 >= L) return;  // empty partition: the merge never reads it
        t1 = min(L, t0 + p.partition_size);
    }
    if constexpr (CLUS) {
        // every CTA of the cluster runs to the cluster barriers: an empty or failed chunk
        // streams nothing and contributes an empty partial
        len_bad = len_bad || L > p.max_context_len || (long long)L > (long long)p.partition_size * p.cluster_size;
        t0 = part * p.partition_size;
        t1 = len_bad ? t0 : max(t0, min(L, t0 + p.partition_size));
    }
    // Decode with append: the new token of this sequence is its position L-1, and its
    // slot must be that position's slot (or -1: nothing to append).  The slot and the
    // last table entry are loaded here but checked only after the first copies are
    // issued, so their latency does not delay them.  A mismatch writes nothing and
    // NaN-fills the rows.
    long long app_slot = -1;
    int app_blk = -1;
    if constexpr (APPEND) {
        app_slot = __ldg(p.slot_mapping + seq);
        if (!len_bad && L >= 1)
            app_blk = __ldg(p.block_tables + size_t(seq) * p.max_blocks_per_seq + (L - 1) / p.block_size);
    }
    auto append_row = [&]() -> long long {  // the new token's cache row [block][kv head][offset], -1, or -2 (bad)
        if (app_slot == -1) return -1;
        const bool ok = L >= 1 && app_blk >= 0 && (long long)app_blk < p.num_blocks &&
                        app_slot == (long long)app_blk * p.block_size + (L - 1) % p.block_size;
        return ok ? ((app_slot / p.block_size) * p.num_kv_heads + kvh) * p.block_size + app_slot % p.block_size
                  : -2;
    };
    if (!CLUS && len_bad) {
        if (threadIdx.x == 0) set_error(p.err, ERR_BOUNDS);
        for (int e = threadIdx.x; e < G * D; e += NW * 32) {
            const int h = e / D, d = e % D;
            if constexpr (PART) {
                const size_t slot = (size_t(seq) * Hq + qh0 + h) * p.num_partitions + part;
                p.out[slot * D + d] = NAN;
                if (d == 0) { p.part_m[slot] = NAN; p.part_l[slot] = NAN; }
            } else {
                p.out[(size_t(seq) * Hq + qh0) * D + e] = NAN;
            }
        }
        return;
    }

    // ---- this warp's tiles: ti0 + warp + k*NW, k < nk
    const int ti0 = t0 / TT;
    const int ntiles = (t1 - t0 + TT - 1) / TT;
    const int nk = ntiles > warp ? (ntiles - warp + NW - 1) / NW : 0;

    unsigned char* my_stages = smem + size_t(warp) * NST * 2 * TILE;
    const uint32_t stage0 = smem_u32(my_stages);
    const uint32_t bar0 = smem_u32(bars + warp * NST);
    float* psm = psm_all + warp * PSM_PAD;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < NST; ++s) mbar_init(bar0 + 8 * s, 1);
        mbar_init_fence();
    }
    __syncwarp();

    // ---- producer state (lane 0)
    const int32_t* trow = p.block_tables + size_t(seq) * p.max_blocks_per_seq;
    const int bs = p.block_size, bshift = p.block_shift;
    auto block_index = [&](int tok) { return bshift >= 0 ? (tok >> bshift) : (tok / bs); };
    auto block_offset = [&](int tok) { return bshift >= 0 ? (tok & (bs - 1)) : (tok % bs); };
    auto tile_token = [&](int k) { return (ti0 + warp + k * NW) * TT; };
    int ent[R];
    bool bad_block = false;
    const uint64_t policy = l2_policy_evict_first();

    auto issue = [&](int k, int pb) {
        const int s = k % NST;
        const uint32_t bar = bar0 + 8 * s;
        const int tok = tile_token(k);
        if (pb >= 0 && (long long)pb < p.num_blocks) {
            const uint32_t bytes = uint32_t(min(TT, t1 - tok)) * ROW;
            const size_t row = (size_t(pb) * p.num_kv_heads + kvh) * size_t(bs) + block_offset(tok);
            const uint32_t dst = stage0 + uint32_t(s) * 2 * TILE;
            mbar_arrive_expect_tx(bar, 2 * bytes);
            bulk_copy_g2s(dst, p.k_cache + row * D, bytes, bar, policy);
            bulk_copy_g2s(dst + TILE, p.v_cache + row * D, bytes, bar, policy);
        } else {
            bad_block = true;   // no copy: the stage keeps stale data, the rows end up NaN
            mbar_arrive(bar);
        }
    };
    auto advance = [&](int k_next_load) {  // shift the table window after an issue
#pragma unroll
        for (int j = 0; j < R - 1; ++j) ent[j] = ent[j + 1];
        ent[R - 1] = k_next_load < nk ? __ldg(trow + block_index(tile_token(k_next_load))) : 0;
    };
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < R; ++j) ent[j] = j < nk ? (spec ? spec_ent[j] : __ldg(trow + block_index(tile_token(j)))) : 0;
#pragma unroll
        for (int k = 0; k < NST; ++k) {
            if (k < nk) {
                issue(k, ent[0]);
                advance(k + R);
            }
        }
    }

    // ---- this lane's slice of the G query rows and the softmax / P.V state
    WarpAttention<D, G> wa;
    wa.init(lane);
    wa.load_q(p.q + (size_t(seq) * Hq + qh0) * D);
    wa.reset();
    // decode with append: the new token's cache row, settled once the first copies are in
    // flight (its inputs were loaded at the start), not re-derived per tile
    long long app_row = -1;
    if constexpr (APPEND) app_row = append_row();

    bool timed_out = false;
    int k = 0;
    for (; k < nk; ++k) {
        const int s = k % NST;
        const bool ok = mbar_wait_bounded(bar0 + 8 * s, (k / NST) & 1, p.wait_limit_ns);
        if (__any_sync(FULL_MASK, !ok)) { timed_out = true; break; }
        const unsigned char* Ks = my_stages + size_t(s) * 2 * TILE;
        const unsigned char* Vs = Ks + TILE;
        const int nvalid = min(TT, t1 - tile_token(k));
        if constexpr (APPEND) {
            const int r = (L - 1) - tile_token(k);
            if (app_row >= 0 && r >= 0 && r < TT) {
                // The tile holding the new token: its copy brought the slot's old bytes.
                // Put the new K/V row in their place, and write it to the cache.
                constexpr int LB = ROW / 32;  // bytes of the row per lane
                const size_t src = (size_t(seq) * p.num_kv_heads + kvh) * D + lane * (LB / 2);
                const size_t dst = size_t(app_row) * D + lane * (LB / 2);
                unsigned char* kr = my_stages + size_t(s) * 2 * TILE + r * ROW + lane * LB;
                if constexpr (LB == 8) {
                    const uint2 kv = __ldg(reinterpret_cast<const uint2*>(p.k_new + src));
                    const uint2 vv = __ldg(reinterpret_cast<const uint2*>(p.v_new + src));
                    *reinterpret_cast<uint2*>(kr) = kv;
                    *reinterpret_cast<uint2*>(kr + TILE) = vv;
                    *reinterpret_cast<uint2*>(p.k_cache_w + dst) = kv;
                    *reinterpret_cast<uint2*>(p.v_cache_w + dst) = vv;
                } else {
                    const uint32_t kv = __ldg(reinterpret_cast<const uint32_t*>(p.k_new + src));
                    const uint32_t vv = __ldg(reinterpret_cast<const uint32_t*>(p.v_new + src));
                    *reinterpret_cast<uint32_t*>(kr) = kv;
                    *reinterpret_cast<uint32_t*>(kr + TILE) = vv;
                    *reinterpret_cast<uint32_t*>(p.k_cache_w + dst) = kv;
                    *reinterpret_cast<uint32_t*>(p.v_cache_w + dst) = vv;
                }
                __syncwarp();
            }
        }

        wa.tile(Ks, Vs, nvalid, psm, p.scale_log2);

        // -- refill the stage just drained
        if (lane == 0 && k + NST < nk) {
            issue(k + NST, ent[0]);
            advance(k + NST + R);
        }
    }

    if (timed_out) {
        // give the copies still in flight a bounded chance to land before the
        // shared memory is reused, then report
        if (lane == 0) set_error(p.err, ERR_TIMEOUT);
        const int last = min(k + NST, nk);
        for (int kk = k; kk < last; ++kk) mbar_wait_bounded(bar0 + 8 * (kk % NST), (kk / NST) & 1, p.wait_limit_ns);
    }
    if constexpr (APPEND) {
        if (app_row == -2) bad_block = true;  // the slot is not position L-1's: nothing was written
    }
    if (lane == 0 && bad_block) set_error(p.err, ERR_BOUNDS);
    const bool warp_failed = __any_sync(FULL_MASK, bad_block || timed_out);

    // ---- stash (m, l, acc) of this warp; its stage memory and psm are free now
    wa.stash(psm, reinterpret_cast<float*>(my_stages));
    if (lane == 0) flags[warp] = warp_failed ? 1 : 0;
    __syncthreads();

    // ---- merge the NW warps and write out
    bool failed = false;
#pragma unroll
    for (int w = 0; w < NW; ++w) failed = failed || flags[w] != 0;
    auto ml_of = [&](int w) { return psm_all + w * PSM_PAD; };
    auto acc_of = [&](int w) { return reinterpret_cast<const float*>(smem + size_t(w) * NST * 2 * TILE); };
    if constexpr (PART) {
        const size_t slot0 = (size_t(seq) * Hq + qh0) * p.num_partitions + part;
        merge_warps_and_store<D, G, NW>(ml_of, acc_of, failed, p.out + slot0 * D, p.part_m + slot0,
                                        p.part_l + slot0, size_t(p.num_partitions));
    } else if constexpr (CLUS) {
        // This chunk's partial -- per element its normalised value, per head its maximum (log2
        // units) and sum, and a failure flag -- goes straight into the shared memory of the CTA
        // that finishes the element: CTA r of the cluster merges elements [r SL, (r + 1) SL) of
        // the G x D output from every chunk's values, after one cluster barrier.
        constexpr int GD = G * D;
        const int C = p.cluster_size, SL = GD / C;
        float* go = reinterpret_cast<float*>(bars + sorted_keys_offset<NW, NST>() / 8);  // [C][SL] values
        float* gm = go + GD;                                                             // [C][G] maxima
        float* gl = gm + kClusterMaxSize * G;                                            // [C][G] sums
        float* gf = gl + kClusterMaxSize * G;                                            // [C] failures
        const bool bad_here = failed || len_bad;
        if (len_bad && threadIdx.x == 0 && part == 0) set_error(p.err, ERR_BOUNDS);
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA of the cluster has started
        for (int e = threadIdx.x; e < GD; e += NW * 32) {
            const int h = e / D, d = e % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NW; ++w) M = fmaxf(M, ml_of(w)[h]);
            float wsum = 0.f, o = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float f = exp2_approx(ml_of(w)[h] - M);
                    wsum += f * ml_of(w)[G + h];
                    o += f * acc_of(w)[h * D + d];
                }
            }
            const float res = bad_here ? NAN : (wsum == 0.f ? 0.f : o / wsum);
            st_shared_remote(go + part * SL + e % SL, uint32_t(e / SL), res);
            if (d == 0)
                for (int r = 0; r < C; ++r) {
                    st_shared_remote(gm + part * G + h, uint32_t(r), M);
                    st_shared_remote(gl + part * G + h, uint32_t(r), wsum);
                }
        }
        if (threadIdx.x == 0)
            for (int r = 0; r < C; ++r) st_shared_remote(gf + part, uint32_t(r), bad_here ? 1.f : 0.f);
        cluster_sync_all();
        float* orow = p.out + (size_t(seq) * Hq + qh0) * D;
        for (int el = threadIdx.x; el < SL; el += NW * 32) {
            const int e = part * SL + el, h = e / D;
            float M = -INFINITY;
            bool bad_any = false;
            for (int r = 0; r < C; ++r) {
                M = fmaxf(M, gm[r * G + h]);
                bad_any = bad_any || gf[r] != 0.f;
            }
            float W = 0.f, o = 0.f;
            if (M != -INFINITY)
                for (int r = 0; r < C; ++r) {
                    const float w = gl[r * G + h] * exp2_approx(gm[r * G + h] - M);
                    W += w;
                    o += w * go[r * SL + el];
                }
            float res = W == 0.f ? 0.f : o / W;  // no token: 0; a NaN input stays NaN
            if (bad_any) res = NAN;
            orow[e] = res;
        }
    } else {
        const size_t row0 = (size_t(seq) * Hq + qh0) * D;
        if (p.out_bf16 != nullptr)
            merge_warps_and_store<D, G, NW>(ml_of, acc_of, failed, nullptr, nullptr, nullptr, 1, p.out_bf16 + row0);
        else
            merge_warps_and_store<D, G, NW>(ml_of, acc_of, failed, p.out + row0, nullptr, nullptr, 1);
    }
}

// Shared memory past the mbarriers that the cluster split gathers the chunks' partials in:
// G x D values, and per chunk G maxima, G sums and a flag.
template <int D, int G>
constexpr size_t cluster_partial_bytes() { return (size_t(G) * D + size_t(kClusterMaxSize) * (2 * G + 1)) * 4; }

template <int D, int G, int NW, int NST>
cudaError_t launch_decode_cluster(const DecodeParams& p, cudaStream_t stream) {
    constexpr size_t smem = decode_smem_bytes<D, G, NW, NST>() + cluster_partial_bytes<D, G>();
    auto kern = paged_decode_kernel<D, G, NW, NST, MODE_CLUSTER>;
    static std::atomic<unsigned long long> configured{0};  // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const long long grid = (long long)p.num_seqs * p.num_kv_heads * p.cluster_size;
    if (grid <= 0) return cudaSuccess;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(p.cluster_size);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int D, int G, int NW, int NST, int MODE>
cudaError_t launch_decode_variant(const DecodeParams& p, cudaStream_t stream) {
    constexpr bool PART = MODE == MODE_PARTITION;
    constexpr size_t smem_base = decode_smem_bytes<D, G, NW, NST>();
    constexpr size_t smem_max = smem_base + size_t(kMaxSortedSeqsPartition) * 4;
    const size_t smem = smem_base + (p.order_mode == ORDER_SORTED ? size_t((p.num_seqs + 3) & ~3) * 4 : 0);
    auto kern = paged_decode_kernel<D, G, NW, NST, MODE>;
    static std::atomic<unsigned long long> configured{0};  // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_max));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const long long grid = PART ? (long long)p.num_partitions * p.num_kv_heads * p.num_seqs
                                : (long long)p.num_seqs * p.num_kv_heads;
    if (grid <= 0) return cudaSuccess;
    kern<<<unsigned(grid), NW * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pf

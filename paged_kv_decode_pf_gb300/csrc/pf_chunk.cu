// Prompt-chunk query: the multi-token query of pf_paged_attention_multi_query for more
// than 64 query rows per kv head.
//
// A long prompt is fed to the model in bounded chunks interleaved with decode (ForgeLLM
// README: "long prompts are split into bounded chunks and interleaved with decode"): the
// chunk's q_len tokens are already appended to the paged cache and each attends to every
// earlier token and to the chunk's tokens up to itself.  With g query heads per kv head a
// (sequence, kv head) has R = g * q_len query rows, so for chunks of tens to hundreds of
// tokens both products are real matrix products.  Here the query rows are the M side of
// single-CTA tcgen05.mma:
//     S(j)  = Q K(j)^T        M = 128 rows, N = 128 tokens, K = D
//     O    += P(j) V(j)       M = 128 rows, N = D,          K = 128 tokens
// with the K / V tiles in shared memory (TMA tiles with the 128-byte swizzle) and S, P and
// O in tensor memory (P as the A operand).  P enters the product as its bf16 high part and
// the bf16 remainder (two MMAs against the same V tile), so the probabilities keep about 16
// significant bits, as in the other multi-token kernels.
//
// One CTA per (sequence, kv head, tile of 128 rows).  Q lives in tensor memory and S is
// double-buffered: S(j + 1) runs while the softmax works on S(j).
// Seven warps:
//  * warps 0-3 (the softmax warpgroup): thread 32 w + l holds query row 32 w + l of a tile,
//    which is lane 32 w + l of tensor memory, so a row's maximum and sum never leave its
//    thread.  Per tile it reads its 128 scores, masks the tokens its row may not see, and
//    moves its reference maximum only when a score exceeds it by more than 2^8; it writes
//    the probabilities' hi and lo parts over the scores it read, as the A operand of P.V.
//    Only a move of the reference makes it wait for the previous P.V (to rescale its O row);
//  * warp 4 issues the MMAs from one lane, each as soon as its operands are ready;
//  * warp 5 copies K tiles into a ring of stages and warp 6 V tiles into another: a tile is
//    eight 16-token boxes, and each box and dim half is one TMA copy issued by its own lane.
// The row tiles of one (sequence, kv head) are adjacent in the grid, so that the CTAs that
// share K/V tiles stream them at about the same time and all but the first read them from L2.
// Every wait is bounded; one that gives up raises an abort flag that ends the others, and
// every role still runs to its end, so tensor memory is always released.
#include <atomic>
#include <cmath>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "pf.h"
#include "pf_device.cuh"
#include "pf_internal.h"
#include "pf_multi.cuh"
#include "pf_tcgen05.cuh"

namespace pf {

constexpr int kChTok = 128;        // tokens per K/V tile: the N of S, the K of P.V
constexpr int kChRows = 128;       // query rows per row tile: the M of both products
constexpr int kChMath = 4;         // softmax warps (warp w: TMEM lanes 32 w .. 32 w + 31)
constexpr int kChMmaWarp = kChMath;
constexpr int kChProducers = 2;    // one warp copies K, one copies V
constexpr int kChThreads = 32 * (kChMath + 1 + kChProducers);
constexpr float kChRescale = 8.f;  // the reference maximum moves when a score exceeds it by more (log2 units)
constexpr int kChCols = 512;       // tensor memory columns
// two score buffers (each later holds its tile's P: hi in its first 64 columns, lo in the next
// 64), O (D columns), Q (D / 2 columns: two bf16 per column)
constexpr uint32_t kChTS0 = 0, kChTS1 = 128, kChTO = 256, kChTQ = 384;

template <int D>
struct ChunkLayout {
    static constexpr int HALVES = D / 64;              // 128-byte swizzle rows per token (or query) row
    static constexpr int HALF = kChTok * 128;          // 128 rows of 128 bytes: 16 KiB
    static constexpr int TILE = HALVES * HALF;         // one K or V tile
    static constexpr int KST = D == 128 ? 3 : 6;       // K ring depth
    static constexpr int VST = D == 128 ? 3 : 6;       // V ring depth
    static constexpr int KRING = 0;
    static constexpr int VRING = KRING + KST * TILE;
    static constexpr int NBARS = 2 * KST + 2 * VST + 8;
    static constexpr int BARS = VRING + VST * TILE;
    static constexpr int MISC = BARS + ((NBARS * 8 + 15) / 16) * 16;  // TMEM base, bad-block flag, abort flag
    static constexpr int BYTES = MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the operands to 1 KiB
};
static_assert(ChunkLayout<128>::ALLOC + (kMultiSortMax + 4) * 4 <= 227 * 1024, "shared memory, D = 128");
static_assert(ChunkLayout<64>::ALLOC + (kMultiSortMax + 4) * 4 <= 227 * 1024, "shared memory, D = 64");

// Barriers of a CTA and its bounded waits: a wait gives up after the call's limit, raising the
// shared abort flag (and the device error word) so that every other role gives up at once.
struct ChunkSync {
    uint32_t bar0;             // shared-memory address of mbarrier 0
    volatile int* abort_flag;
    unsigned* err;
    unsigned long long limit_ns;

    __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + uint32_t(8 * i); }
    __device__ __forceinline__ void give_up() const {
        *abort_flag = 1;
        set_error(err, ERR_TIMEOUT);
    }
    // false once this or another role has given up
    __device__ __forceinline__ bool wait(int i, uint32_t parity) const {
        const uint32_t b = bar(i);
        if (mbar_try_wait(b, parity)) return true;
        if (*abort_flag) return false;
        const uint64_t start = global_timer_ns();
        for (uint32_t it = 1;; ++it) {
            if (mbar_try_wait(b, parity)) return true;
            if ((it & 63u) == 0u) {
                if (*abort_flag) return false;
                if (global_timer_ns() - start > limit_ns) {
                    give_up();
                    return false;
                }
            }
        }
    }
};

// One producer warp: copies the nt K (or V) tiles of the CTA's sequence into an ns-stage ring
// (stage s at ring + s * tile_bytes).  A tile is eight 16-token boxes.  With BLK false, lane
// l < 8 * HALVES copies dim half l % HALVES of box l / HALVES to + h * half_bytes + box * 2 KiB
// (a stage is [dim half][128 rows][128 bytes]); with BLK true (the 3D block map), lane l < 8
// copies box l whole to + l * HALVES * 2 KiB (a stage is [box][dim half][16 rows][128 bytes]).
// Table entries come 32 boxes (4 tiles) a batch ahead: lane l holds box 32 b + l.  Boxes at or
// past tmax are not copied.  Before returning it waits for the last fill of every stage, so
// the CTA never ends with copies in flight.
template <int HALVES, bool BLK>
__device__ __forceinline__ void chunk_produce(const ChunkSync& sy, const MultiParams& p, const CUtensorMap* map,
                                              uint32_t ring, int tile_bytes, int half_bytes, int ns, int fullb,
                                              int emptyb, int seq, int kvh, int tmax, int nt, volatile int* bad,
                                              int lane) {
    constexpr int BOXES = kChTok / kTileTokens;
    constexpr int TPB = 32 / BOXES;  // tiles per batch of table entries
    const int32_t* trow = p.block_tables + size_t(seq) * p.max_blocks_per_seq;
    const int bs = p.block_size, bshift = p.block_shift, Hkv = p.num_kv_heads;
    auto block_index = [&](int tok) { return bshift >= 0 ? (tok >> bshift) : (tok / bs); };
    auto block_offset = [&](int tok) { return bshift >= 0 ? (tok & (bs - 1)) : (tok % bs); };
    auto batch = [&](int b) {  // entry of box 32 b + lane (0 past the tokens the CTA reads)
        const int tok = (32 * b + lane) * kTileTokens;
        return tok < tmax ? __ldg(trow + block_index(tok)) : 0;
    };
    const uint64_t policy = l2_policy_evict_first();
    int ent_cur = batch(0), ent_nxt = nt > TPB ? batch(1) : 0;
    int issued = 0;
    constexpr int LPB = BLK ? 1 : HALVES;                                   // lanes per box
    constexpr uint32_t LANE_BYTES = kTileTokens * 128u * (BLK ? HALVES : 1);  // bytes per lane's copy
    const int bi = lane / LPB, hf = lane % LPB;
    for (int j = 0; j < nt; ++j) {
        if (j > 0 && j % TPB == 0) {
            ent_cur = ent_nxt;
            ent_nxt = batch(j / TPB + 1);
        }
        const int el = __shfl_sync(FULL_MASK, ent_cur, ((j % TPB) * BOXES + bi) & 31);
        const int tok = j * kChTok + bi * kTileTokens;
        const bool live = lane < BOXES * LPB && tok < tmax;
        const bool good = live && el >= 0 && (long long)el < p.num_blocks;
        if (live && !good) {
            *bad = 1;
            set_error(p.err, ERR_BOUNDS);
        }
        const int s = j % ns;
        bool ok = true;
        if (lane == 0 && j >= ns) ok = sy.wait(emptyb + s, ((j / ns) - 1) & 1);
        if (!__shfl_sync(FULL_MASK, ok ? 1 : 0, 0)) break;
        const uint32_t bytes = uint32_t(__popc(__ballot_sync(FULL_MASK, good))) * LANE_BYTES;
        if (lane == 0) mbar_arrive_expect_tx(sy.bar(fullb + s), bytes);
        __syncwarp();  // the byte count is set before any copy can complete
        const int row = (el * Hkv + kvh) * bs + block_offset(tok);
        if (good && BLK)
            tma_load_3d(ring + uint32_t(s * tile_bytes) + uint32_t(bi) * LANE_BYTES, map, 0, row, 0,
                        sy.bar(fullb + s), policy);
        else if (good)
            tma_load_2d(ring + uint32_t(s * tile_bytes + bi * kTileTokens * 128 + hf * half_bytes), map, 64 * hf,
                        row, sy.bar(fullb + s), policy);
        ++issued;
    }
    if (lane == 0)
        for (int s = 0; s < ns && s < issued; ++s) {
            const int jl = s + ns * ((issued - 1 - s) / ns);
            mbar_wait_bounded(sy.bar(fullb + s), (jl / ns) & 1, p.wait_limit_ns);
        }
    __syncwarp();
}

// Zero the rows [nvalid, 128) of a V stage (both dim halves): they hold other data or poison,
// or were not copied, and 0 * V must stay 0.  Called by a whole warp.  Row r's 128 bytes of
// dim half h: + h * half_bytes + r * 128 (BLK false), or + (r / 16) * HALVES * 2 KiB + h * 2 KiB
// + (r % 16) * 128 (BLK true); the swizzle moves 16-byte chunks only within their row.
template <int HALVES, bool BLK>
__device__ __forceinline__ void chunk_zero_v_rows(unsigned char* stage, int half_bytes, int nvalid, int lane) {
    for (int e = lane; e < (kChTok - nvalid) * 8 * HALVES; e += 32) {
        const int r = nvalid + e / (8 * HALVES), c = e % (8 * HALVES);
        const int off = BLK ? (r / kTileTokens) * HALVES * 2048 + (c >> 3) * 2048 + (r % kTileTokens) * 128
                            : (c >> 3) * half_bytes + r * 128;
        *reinterpret_cast<uint4*>(stage + off + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncwarp();
    tc_fence_after_sync();
}

// Online-softmax state of one query row of one row tile.
struct ChunkRow {
    float m_ref;  // reference maximum (log2 units)
    float l_sum;  // sum of the probabilities, relative to m_ref
};

// The softmax of one row tile for K/V tile j, by the softmax warpgroup (thread = row):
// waits for its scores (barrier sfull, parity sp), reads them (buffer ts of this warp's lane
// quarter), masks the tokens t >= lim, updates the row state, rescales the O row (columns to)
// after waiting for the previous P.V (barrier pfree, parity fp) when the reference moved,
// writes P over the scores (hi in columns 0-63, lo in 64-127) and arrives on pfull.
template <int D>
__device__ __forceinline__ void chunk_softmax_tile(const ChunkSync& sy, uint32_t ts, uint32_t to, int sfull,
                                                   uint32_t sp, int pfree, uint32_t fp, int pfull, int j, int lim,
                                                   float sc, ChunkRow& row, int lane) {
    sy.wait(sfull, sp);
    __syncwarp();
    tc_fence_after_sync();
    // a positive scale commutes with the maximum: the row maximum of the raw scores, and one
    // FFMA per score inside the exponent; otherwise (zero or negative scale) scores scale first
    const bool pos = sc > 0.f;
    float y[kChTok];
    {
        uint32_t v[kChTok];
        tmem_ld_x128(ts, v);
#pragma unroll
        for (int c = 0; c < kChTok; ++c) y[c] = __uint_as_float(v[c]);
    }
    if (!pos) {
#pragma unroll
        for (int c = 0; c < kChTok; ++c) y[c] *= sc;
    }
    const int t0 = j * kChTok;
    if (t0 + kChTok > lim) {  // tokens this row may not see (or past the sequence)
#pragma unroll
        for (int c = 0; c < kChTok; ++c)
            if (t0 + c >= lim) y[c] = -INFINITY;
    }
    // row maximum in log2 units, as a tree (8 independent chains)
    float mx;
    {
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = y[i];
#pragma unroll
        for (int c = 8; c < kChTok; ++c) m8[c & 7] = fmaxf(m8[c & 7], y[c]);
        mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        if (pos) mx *= sc;  // -inf stays -inf
    }
    // move the reference only when a score exceeds it by more than the margin (any visible score
    // when there is none yet); the probabilities stay below 2^8
    float alpha = 1.f;
    bool rescale = false;
    if (mx > row.m_ref + kChRescale) {
        alpha = exp2_approx(row.m_ref - mx);  // no reference yet: 0
        rescale = j > 0;
        row.l_sum *= alpha;
        row.m_ref = mx;
    }
    const float ref = row.m_ref == -INFINITY ? 0.f : row.m_ref;
    const float ysc = pos ? sc : 1.f;  // exponent: y * ysc - ref
    // probabilities as a bf16 high part (truncation: the top 16 bits) and the bf16 rounding of
    // the exact remainder, so that hi + lo carries about 16 significant bits
    uint32_t ph[kChTok / 2], pl[kChTok / 2];
    float s8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s8[i] = 0.f;
#pragma unroll
    for (int e = 0; e < kChTok / 2; ++e) {
        const float a = exp2_approx(fmaf(y[2 * e], ysc, -ref));
        const float c = exp2_approx(fmaf(y[2 * e + 1], ysc, -ref));
        s8[(2 * e) & 7] += a;
        s8[(2 * e + 1) & 7] += c;
        const uint32_t ua = __float_as_uint(a), uc = __float_as_uint(c);
        ph[e] = __byte_perm(ua, uc, 0x7632);  // high halves: element 2e low, 2e + 1 high
        pl[e] = pack_bf16x2(a - __uint_as_float(ua & 0xffff0000u), c - __uint_as_float(uc & 0xffff0000u));
    }
    row.l_sum += ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
    if (__any_sync(FULL_MASK, rescale)) {
        // O is complete up to the previous P.V before its rows are rescaled
        sy.wait(pfree, fp);
        __syncwarp();
        tc_fence_after_sync();
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
            uint32_t v[32];
            tmem_ld_x32(to + uint32_t(32 * q), v);
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
            tmem_st_x32(to + uint32_t(32 * q), v);
        }
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) w[c] = ph[32 * q + c];
        tmem_st_x32(ts + uint32_t(32 * q), w);
#pragma unroll
        for (int c = 0; c < 32; ++c) w[c] = pl[32 * q + c];
        tmem_st_x32(ts + uint32_t(64 + 32 * q), w);
    }
    tmem_st_wait();
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(sy.bar(pfull));
}

// O / l of one row (TMEM columns to of this warp's lane quarter) into dst (null: not a row).
template <int D>
__device__ __forceinline__ void chunk_store_row(uint32_t to, float* dst, float l_sum, bool any_tile, bool failed) {
    const float inv = l_sum == 0.f ? 0.f : 1.f / l_sum;  // no token: 0; a NaN input stays NaN
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
        uint32_t v[32];
        if (any_tile) {
            tmem_ld_x32(to + uint32_t(32 * q), v);
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = 0u;
        }
        if (dst != nullptr) {
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                float4 o = make_float4(__uint_as_float(v[c]) * inv, __uint_as_float(v[c + 1]) * inv,
                                       __uint_as_float(v[c + 2]) * inv, __uint_as_float(v[c + 3]) * inv);
                if (!any_tile) o = make_float4(0.f, 0.f, 0.f, 0.f);
                if (failed) o = make_float4(NAN, NAN, NAN, NAN);
                *reinterpret_cast<float4*>(dst + 32 * q + c) = o;
            }
        }
    }
}

// ------------------------------------------------------------ single row tile

template <int D>
__global__ void __launch_bounds__(kChThreads, 1) paged_chunk_query_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                           const __grid_constant__ CUtensorMap tmap_v,
                                                                           const MultiParams p) {
    using Lay = ChunkLayout<D>;
    constexpr int NT = kChThreads, TOK = kChTok, NK = Lay::KST, NV = Lay::VST, HALVES = Lay::HALVES;
    constexpr bool VBLK = kVBlockCopies && HALVES == 2;  // V by whole 16-token blocks (4 KiB copies)
    // mbarriers: K and V rings full / empty; per score buffer: S written, P written, P.V
    // complete (the buffer free again); Q stored; every MMA complete
    enum { KFULL = 0, KEMPTY = NK, VFULL = 2 * NK, VEMPTY = 2 * NK + NV, SFULL = 2 * NK + 2 * NV, PFULL = SFULL + 2,
           PFREE = PFULL + 2, QREADY = PFREE + 2, DONE = QREADY + 1 };
    static_assert(DONE + 1 == Lay::NBARS, "barrier count");

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // swizzled operands need 1 KiB alignment
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::MISC);
    volatile int* bad = reinterpret_cast<volatile int*>(smem + Lay::MISC + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::MISC + 8);
    const ChunkSync sy{sbase + uint32_t(Lay::BARS), abort_flag, p.err, p.wait_limit_ns};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = p.num_kv_heads, G = p.group, Q = p.q_len, RR = p.rows, Hq = p.num_q_heads;
    const int nrt = (RR + kChRows - 1) / kChRows;  // row tiles per (sequence, kv head)
    const int rt = blockIdx.x % nrt;
    const int item = blockIdx.x / nrt;
    const int kvh = item % Hkv;
    const int seq = p.sorted ? multi_sorted_seq<NT>(p, item / Hkv) : item / Hkv;
    const int L = __ldg(p.context_lens + seq);
    const int r0 = rt * kChRows;                     // the CTA's first query row
    const int nrows = min(kChRows, RR - r0);          // its rows
    auto out_row = [&](int r) -> float* {             // query row r = j * G + h
        const int j = r / G, h = r - (r / G) * G;
        return p.out + ((size_t(seq) * Q + j) * Hq + kvh * G + h) * D;
    };
    if (L < 0 || (long long)L > (long long)p.max_blocks_per_seq * p.block_size) {
        if (threadIdx.x == 0) set_error(p.err, ERR_BOUNDS);
        for (int e = threadIdx.x; e < nrows * D; e += NT) out_row(r0 + e / D)[e % D] = NAN;
        return;
    }
    const int lim0 = L - Q + 1;  // row r sees the tokens t < lim0 + r / G (none when that is <= 0)
    const int tmax = max(0, lim0 + (r0 + nrows - 1) / G);  // tokens some row of the CTA sees
    const int nt = (tmax + TOK - 1) / TOK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Lay::NBARS; ++i) {
            int count = 1;                                                     // commits, producers
            if (i == PFULL || i == PFULL + 1 || i == QREADY) count = kChMath;  // the softmax warps
            mbar_init(sy.bar(i), count);
        }
        *bad = 0;
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == kChMmaWarp) tmem_alloc(smem_u32(tmem_slot), kChCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp > kChMmaWarp) {
        // ---- producer warps: warp 5 copies K, warp 6 V
        const bool is_v = warp - kChMmaWarp - 1 == 1;
        if (is_v)
            chunk_produce<HALVES, VBLK>(sy, p, &tmap_v, sbase + uint32_t(Lay::VRING), Lay::TILE, Lay::HALF, NV,
                                        VFULL, VEMPTY, seq, kvh, tmax, nt, bad, lane);
        else
            chunk_produce<HALVES, false>(sy, p, &tmap_k, sbase + uint32_t(Lay::KRING), Lay::TILE, Lay::HALF, NK,
                                         KFULL, KEMPTY, seq, kvh, tmax, nt, bad, lane);
    } else if (warp == kChMmaWarp) {
        // ---- MMA issuer: P(jp) V(jp) when ready, else S(js) (at most two ahead: two score buffers)
        constexpr uint32_t IDESC_S = umma_idesc_bf16(kChRows, TOK, 0, 0);
        constexpr uint32_t IDESC_O = umma_idesc_bf16(kChRows, D, 0, 1);
        __syncwarp();
        if (nt > 0) {
            const bool qok = __all_sync(FULL_MASK, sy.wait(QREADY, 0));
            (void)qok;
        }
        tc_fence_after_sync();
        int js = 0, jp = 0;
        uint64_t idle_since = 0;
        bool idle = false;
        while (jp < nt) {
            int act = 0;  // 1: P.V(jp), 2: S(js), -1: give up
            if (lane == 0) {
                if (jp < js && mbar_test_wait(sy.bar(PFULL + (jp & 1)), (jp >> 1) & 1) &&
                    mbar_test_wait(sy.bar(VFULL + jp % NV), (jp / NV) & 1))
                    act = 1;
                // S(js): K landed, and P(js - 2) V(js - 2) -- the last reader of the buffer -- is complete
                else if (js < nt && mbar_test_wait(sy.bar(KFULL + js % NK), (js / NK) & 1) &&
                         (js < 2 || mbar_test_wait(sy.bar(PFREE + (js & 1)), ((js >> 1) - 1) & 1)))
                    act = 2;
                else if (*abort_flag) act = -1;
                else if (!idle) {
                    idle = true;
                    idle_since = global_timer_ns();
                } else if (global_timer_ns() - idle_since > p.wait_limit_ns) {
                    sy.give_up();
                    act = -1;
                }
                if (act != 0) idle = false;
            }
            act = __shfl_sync(FULL_MASK, act, 0);
            if (act < 0) break;
            if (act == 0) continue;
            tc_fence_after_sync();
            if (act == 2) {
                if (lane == 0) {
                    const uint32_t ka = sbase + uint32_t(Lay::KRING + (js % NK) * Lay::TILE);
                    const uint32_t ts = tmem + ((js & 1) ? kChTS1 : kChTS0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)  // 16 dims: 8 TMEM columns of Q, 32 bytes into K's rows
                        umma_bf16_tmem_a(ts, tmem + kChTQ + uint32_t(8 * kk),
                                         umma_desc_sw128(ka + uint32_t((kk >> 2) * Lay::HALF + (kk & 3) * 32), 16, 1024),
                                         IDESC_S, kk > 0);
                    umma_commit(sy.bar(SFULL + (js & 1)));
                    umma_commit(sy.bar(KEMPTY + js % NK));
                }
                ++js;
            } else {
                const uint32_t voff = uint32_t(Lay::VRING + (jp % NV) * Lay::TILE);
                // rows past the sequence, and boxes past the CTA's last token, hold no V row
                const int vend = min(L, (tmax + kTileTokens - 1) / kTileTokens * kTileTokens);
                const int nvalid = min(TOK, vend - jp * TOK);
                if (nvalid < TOK) chunk_zero_v_rows<HALVES, VBLK>(smem + voff, Lay::HALF, nvalid, lane);
                if (lane == 0) {
                    const uint32_t va = sbase + voff;
                    const uint32_t tp = tmem + ((jp & 1) ? kChTS1 : kChTS0);
#pragma unroll
                    for (int part = 0; part < 2; ++part)      // P hi, then P lo, against the same V
#pragma unroll
                        for (int kk = 0; kk < TOK / 16; ++kk)  // 16 tokens: 8 TMEM columns of P, 2 KiB of V
                            umma_bf16_tmem_a(tmem + kChTO, tp + uint32_t(64 * part + 8 * kk),
                                             VBLK ? umma_desc_sw128(va + kk * 4096, 2048, 1024)
                                                  : umma_desc_sw128(va + kk * 2048, Lay::HALF, 1024),
                                             IDESC_O,
                                             (jp | part | kk) != 0);
                    umma_commit(sy.bar(PFREE + (jp & 1)));
                    umma_commit(sy.bar(VEMPTY + jp % NV));
                }
                ++jp;
            }
            __syncwarp();
        }
        // every MMA of the CTA is complete before O is read and tensor memory released
        if (lane == 0) {
            umma_commit(sy.bar(DONE));
            mbar_wait_bounded(sy.bar(DONE), 0, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ---- softmax warpgroup: thread rl = 32 warp + lane holds query row r0 + rl
        const int rl = threadIdx.x;
        const int r = r0 + rl;
        const bool is_row = rl < nrows;
        const uint32_t tl = tmem + (uint32_t(warp * 32) << 16);  // this warp's TMEM lane quarter

        // this row of Q into tensor memory (two bf16 per column; zero past the CTA's rows)
        {
            constexpr int CH = D / 8;  // 16-byte chunks per row
            uint32_t w[D / 2];
            if (is_row) {
                const int j = r / G, h = r - (r / G) * G;
                const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t(seq) * Q + j) * Hq + kvh * G + h) * D);
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    const uint4 v = __ldg(src + c);
                    w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int c = 0; c < D / 2; ++c) w[c] = 0u;
            }
#pragma unroll
            for (int q = 0; q < D / 64; ++q) {
                uint32_t x[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] = w[32 * q + c];
                tmem_st_x32(tl + kChTQ + uint32_t(32 * q), x);
            }
            tmem_st_wait();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(sy.bar(QREADY));

        const int lim = is_row ? lim0 + r / G : 0;  // tokens t < lim are visible to this row
        ChunkRow row{-INFINITY, 0.f};
        for (int j = 0; j < nt; ++j) {
            const int b = j & 1;
            chunk_softmax_tile<D>(sy, tl + (b ? kChTS1 : kChTS0), tl + kChTO, SFULL + b, (j >> 1) & 1,
                                  PFREE + ((j - 1) & 1), ((j - 1) >> 1) & 1, PFULL + b, j, lim, p.scale_log2, row,
                                  lane);
        }

        // ---- epilogue: O / l once every MMA is complete
        if (nt > 0) sy.wait(DONE, 0);
        __syncwarp();
        tc_fence_after_sync();
        const bool failed = *bad != 0 || *abort_flag != 0;
        chunk_store_row<D>(tl + kChTO, is_row ? out_row(r) : nullptr, row.l_sum, nt > 0, failed);
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == kChMmaWarp) tmem_dealloc(tmem, kChCols);
}

// ------------------------------------------------------------------ launches

template <typename Kern>
static cudaError_t configure_once(Kern kern, int smem_bytes, std::atomic<unsigned long long>& configured) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    return cudaSuccess;
}

template <int D>
static cudaError_t launch_chunk_d(const CUtensorMap& mk, const CUtensorMap& mv, const MultiParams& p,
                                  cudaStream_t stream) {
    static std::atomic<unsigned long long> configured{0};
    auto kern = paged_chunk_query_kernel<D>;
    cudaError_t e = configure_once(kern, ChunkLayout<D>::ALLOC, configured);
    if (e != cudaSuccess) return e;
    const long long nrt = (p.rows + kChRows - 1) / kChRows;
    const long long grid = (long long)p.num_seqs * p.num_kv_heads * nrt;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    kern<<<unsigned(grid), kChThreads, ChunkLayout<D>::ALLOC, stream>>>(mk, mv, p);
    return cudaGetLastError();
}

cudaError_t launch_chunk(const CUtensorMap& mk, const CUtensorMap& mv, const MultiParams& p, int head_dim,
                         cudaStream_t stream) {
    if (head_dim == 128) return launch_chunk_d<128>(mk, mv, p, stream);
    if (head_dim == 64) return launch_chunk_d<64>(mk, mv, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pf

// Multi-token paged query: pf_paged_attention_multi_query.
//
// Several new tokens per sequence attend over the paged cache at once -- the
// draft tokens a speculative step verifies (TokenForge post: "paired the main
// model with a tiny draft model to guess tokens ahead of time") or a short chunk
// of a prompt interleaved with decode (ForgeLLM README: "long prompts are split
// into bounded chunks and interleaved with decode").  Sequence i has q_len new
// tokens at positions L_i - q_len + j, already in the cache; query row (j, h)
// sees the tokens t <= L_i - q_len + j.
//
// With R = g * q_len query rows per kv head the scores are a real (small)
// contraction, [R x D] . [D x 16] per tile, so this kernel runs both products on
// the tensor cores:
//  * One CTA per (sequence, kv head); 4 warps split the 16-token tiles as in the
//    decode kernel, each with its own 2-stage ring; lane 0 issues TMA tensor
//    copies (cp.async.bulk.tensor) of the K and V tiles with the 128-byte swizzle,
//    so the ldmatrix reads below are free of bank conflicts.
//  * S = Q K^T with mma.sync m16n8k16 (bf16 in, fp32 accumulate): Q (R <= 16 rows,
//    zero-padded) lives in registers as A fragments, K^T comes from ldmatrix.
//  * Per-row causal limits, an fp32 online softmax on the accumulator fragments
//    (quad shuffles), then P.V: P is split into bf16 hi + lo parts (two MMAs
//    against the same V fragments, ldmatrix.trans) so the probabilities keep
//    about 16 significant bits.
//  * The 4 warps merge (m, l, O) in shared memory at the end.
// Above 16 rows (up to 64) a second kernel gives each 16-row tile its own warp and
// shares the K/V stages among them (below).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include <cuda.h>  // CUtensorMap and its enums only; the encoder is fetched from the runtime
#include <cuda_runtime.h>

#include "pf.h"
#include "pf_device.cuh"
#include "pf_tcgen05.cuh"
#include "pf_internal.h"
#include "pf_multi.cuh"

namespace pf {

constexpr int kMultiMaxRows = 16;  // g * q_len: one m16 tile of query rows

template <int D, int NW, int NST>
struct MultiLayout {
    static constexpr int TT = kTileTokens;
    static constexpr int HALVES = D / 64;                // 128-byte swizzle rows per token row
    static constexpr int HALF_BYTES = TT * 128;          // one TMA box: 16 rows x 128 B
    static constexpr int TILE = HALVES * HALF_BYTES;     // K or V tile, 16 x D bf16
    static constexpr int STAGE = 2 * TILE;
    static constexpr size_t STAGES_BYTES = size_t(NW) * NST * STAGE;
    static constexpr size_t BARS = STAGES_BYTES;                          // NW*NST mbarriers
    static constexpr size_t FLAGS = BARS + size_t(NW) * NST * 8;           // NW ints
    static constexpr size_t ML = FLAGS + ((NW * 4 + 15) / 16) * 16;        // [NW][2][16] floats
    static constexpr size_t BYTES = ML + size_t(NW) * 2 * kMultiMaxRows * 4;
    static constexpr size_t ALLOC = BYTES + 1024;                          // room to align to 1024
    static_assert(NST * STAGE >= kMultiMaxRows * D * 4, "stage area holds a warp's O for the merge");
};

template <int D, int NW, int NST>
__global__ void __launch_bounds__(NW * 32) paged_multi_query_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                     const __grid_constant__ CUtensorMap tmap_v,
                                                                     const MultiParams p) {
    using Lay = MultiLayout<D, NW, NST>;
    constexpr int TT = Lay::TT, HALVES = Lay::HALVES, HALF = Lay::HALF_BYTES, TILE = Lay::TILE;
    constexpr int STAGE = Lay::STAGE;
    constexpr int KSTEPS = D / 16;  // k-steps of S = Q K^T
    constexpr int NTD = D / 8;      // n-tiles of O = P V
    constexpr int R = NST + 2;      // table entries lane 0 holds ahead of the copies

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // swizzled boxes need 1 KiB alignment
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::BARS);
    int* flags = reinterpret_cast<int*>(smem + Lay::FLAGS);
    float* ml = reinterpret_cast<float*>(smem + Lay::ML);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int Hkv = p.num_kv_heads, G = p.group, Q = p.q_len, RR = p.rows, Hq = p.num_q_heads;
    const int kvh = blockIdx.x % Hkv;
    const int seq = p.sorted ? multi_sorted_seq<NW * 32>(p, blockIdx.x / Hkv) : blockIdx.x / Hkv;
    const int L = __ldg(p.context_lens + seq);
    const bool len_bad = L < 0 || (long long)L > (long long)p.max_blocks_per_seq * p.block_size;
    auto out_row = [&](int r) -> float* {  // query row r = j * G + h
        const int j = r / G, h = r - (r / G) * G;
        return p.out + ((size_t(seq) * Q + j) * Hq + kvh * G + h) * D;
    };
    if (len_bad) {
        if (threadIdx.x == 0) set_error(p.err, ERR_BOUNDS);
        for (int e = threadIdx.x; e < RR * D; e += NW * 32) out_row(e / D)[e % D] = NAN;
        return;
    }

    const int ntiles = (L + TT - 1) / TT;
    const int nk = ntiles > warp ? (ntiles - warp + NW - 1) / NW : 0;
    unsigned char* my_stages = smem + size_t(warp) * NST * STAGE;
    const uint32_t stage0 = smem_u32(my_stages);
    const uint32_t bar0 = smem_u32(bars + warp * NST);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < NST; ++s) mbar_init(bar0 + 8 * s, 1);
        mbar_init_fence();
    }
    __syncwarp();

    // ---- producer (lane 0): TMA boxes of the warp's tiles, table entries NST+2 ahead
    const int32_t* trow = p.block_tables + size_t(seq) * p.max_blocks_per_seq;
    const int bs = p.block_size, bshift = p.block_shift;
    auto block_index = [&](int tok) { return bshift >= 0 ? (tok >> bshift) : (tok / bs); };
    auto block_offset = [&](int tok) { return bshift >= 0 ? (tok & (bs - 1)) : (tok % bs); };
    auto tile_token = [&](int k) { return (warp + k * NW) * TT; };
    int ent[R];
    bool bad_block = false;
    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int k, int pb) {
        const int s = k % NST;
        const uint32_t bar = bar0 + 8 * s;
        if (pb >= 0 && (long long)pb < p.num_blocks) {
            const int tok = tile_token(k);
            const int y = (pb * Hkv + kvh) * bs + block_offset(tok);
            const uint32_t dst = stage0 + uint32_t(s) * STAGE;
            mbar_arrive_expect_tx(bar, STAGE);
#pragma unroll
            for (int hh = 0; hh < HALVES; ++hh) {
                tma_load_2d(dst + hh * HALF, &tmap_k, hh * 64, y, bar, policy);
                tma_load_2d(dst + TILE + hh * HALF, &tmap_v, hh * 64, y, bar, policy);
            }
        } else {
            bad_block = true;
            mbar_arrive(bar);
        }
    };
    auto advance = [&](int k_next_load) {
#pragma unroll
        for (int j = 0; j < R - 1; ++j) ent[j] = ent[j + 1];
        ent[R - 1] = k_next_load < nk ? __ldg(trow + block_index(tile_token(k_next_load))) : 0;
    };
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < R; ++j) ent[j] = j < nk ? __ldg(trow + block_index(tile_token(j))) : 0;
#pragma unroll
        for (int k = 0; k < NST; ++k)
            if (k < nk) {
                issue(k, ent[0]);
                advance(k + R);
            }
    }

    // ---- query rows g and g+8 of the m16 tile as A fragments (zero rows past RR)
    const int r0 = g, r1 = g + 8;
    auto qrow = [&](int r) -> const uint16_t* {
        const int j = r / G, h = r - (r / G) * G;
        return p.q + ((size_t(seq) * Q + j) * Hq + kvh * G + h) * D;
    };
    uint32_t qa[KSTEPS][4];
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
        const int c = ks * 16 + 2 * t;
        qa[ks][0] = r0 < RR ? __ldg(reinterpret_cast<const uint32_t*>(qrow(r0) + c)) : 0u;
        qa[ks][1] = r1 < RR ? __ldg(reinterpret_cast<const uint32_t*>(qrow(r1) + c)) : 0u;
        qa[ks][2] = r0 < RR ? __ldg(reinterpret_cast<const uint32_t*>(qrow(r0) + c + 8)) : 0u;
        qa[ks][3] = r1 < RR ? __ldg(reinterpret_cast<const uint32_t*>(qrow(r1) + c + 8)) : 0u;
    }
    // tokens t < lim are visible to a row; padding rows see nothing
    const int lim0 = r0 < RR ? L - Q + r0 / G + 1 : 0;
    const int lim1 = r1 < RR ? L - Q + r1 / G + 1 : 0;

    float o[NTD][4];
#pragma unroll
    for (int n = 0; n < NTD; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    // swizzled byte offset of 16-byte chunk c (0 .. D/8-1) of token row `tok` in a tile
    auto swz = [](int tok, int c) { return (c >> 3) * HALF + tok * 128 + (((c & 7) ^ (tok & 7)) << 4); };

    bool timed_out = false;
    int k = 0;
    for (; k < nk; ++k) {
        const int s = k % NST;
        const bool ok = mbar_wait_bounded(bar0 + 8 * s, (k / NST) & 1, p.wait_limit_ns);
        if (__any_sync(FULL_MASK, !ok)) { timed_out = true; break; }
        unsigned char* Ks = my_stages + size_t(s) * STAGE;
        unsigned char* Vs = Ks + TILE;
        const uint32_t ks_addr = smem_u32(Ks), vs_addr = smem_u32(Vs);
        const int tok0 = tile_token(k);
        const int nvalid = min(TT, L - tok0);
        if (nvalid < TT) {
            // rows past the sequence hold other data (or poison): zero V there so 0 * V stays 0
            for (int b = lane; b < (TT - nvalid) * HALVES * 8; b += 32) {
                const int row = nvalid + b / (HALVES * 8), rest = b % (HALVES * 8);
                *reinterpret_cast<uint4*>(Vs + (rest >> 3) * HALF + row * 128 + (rest & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }

        // -- S = Q K^T for the 16 tokens: two n-tiles of 8
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kp = 0; kp < KSTEPS / 2; ++kp) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tok = nt * 8 + (lane & 7);
                const int c = kp * 4 + (lane >> 3);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(ks_addr + swz(tok, c), b0, b1, b2, b3);
                mma_bf16_16816(sc[nt], qa[2 * kp], b0, b1);
                mma_bf16_16816(sc[nt], qa[2 * kp + 1], b2, b3);
            }
        }
        // -- mask, scale to base 2, online softmax per row (the 4 lanes of a quad share a row)
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = tok0 + nt * 8 + 2 * t + (e & 1);
                const bool vis = tok < (e < 2 ? lim0 : lim1);
                sc[nt][e] = vis ? sc[nt][e] * p.scale_log2 : -INFINITY;
                if (e < 2) mx0 = fmaxf(mx0, sc[nt][e]); else mx1 = fmaxf(mx1, sc[nt][e]);
            }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float sf0 = mn0 == -INFINITY ? 0.f : mn0, sf1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = exp2_approx(m0 - sf0), al1 = exp2_approx(m1 - sf1);
        m0 = mn0;
        m1 = mn1;
        float pr[2][4];
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                pr[nt][e] = exp2_approx(sc[nt][e] - (e < 2 ? sf0 : sf1));
                if (e < 2) ps0 += pr[nt][e]; else ps1 += pr[nt][e];
            }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int n = 0; n < NTD; ++n) {
            o[n][0] *= al0; o[n][1] *= al0;
            o[n][2] *= al1; o[n][3] *= al1;
        }
        // -- P as A fragments, split into bf16 hi + lo
        uint32_t ph[4], pl[4];
        {
            const float* v[4] = {&pr[0][0], &pr[0][2], &pr[1][0], &pr[1][2]};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float a = v[i][0], b = v[i][1];
                ph[i] = pack_bf16x2(a, b);
                const float ah = __uint_as_float(ph[i] << 16), bh = __uint_as_float(ph[i] & 0xffff0000u);
                pl[i] = pack_bf16x2(a - ah, b - bh);
            }
        }
        // -- O += P V: V fragments via ldmatrix.trans, two n-tiles of 8 dims per load
#pragma unroll
        for (int dp = 0; dp < NTD / 2; ++dp) {
            const int mi = lane >> 3;
            const int tok = ((mi & 1) << 3) + (lane & 7);
            const int c = 2 * dp + (mi >> 1);
            uint32_t v0, v1, v2, v3;
            ldmatrix_x4_trans(vs_addr + swz(tok, c), v0, v1, v2, v3);
            mma_bf16_16816(o[2 * dp], ph, v0, v1);
            mma_bf16_16816(o[2 * dp], pl, v0, v1);
            mma_bf16_16816(o[2 * dp + 1], ph, v2, v3);
            mma_bf16_16816(o[2 * dp + 1], pl, v2, v3);
        }
        __syncwarp();
        if (lane == 0 && k + NST < nk) {
            issue(k + NST, ent[0]);
            advance(k + NST + R);
        }
    }

    if (timed_out) {
        if (lane == 0) set_error(p.err, ERR_TIMEOUT);
        const int last = min(k + NST, nk);
        for (int kk = k; kk < last; ++kk) mbar_wait_bounded(bar0 + 8 * (kk % NST), (kk / NST) & 1, p.wait_limit_ns);
    }
    if (lane == 0 && bad_block) set_error(p.err, ERR_BOUNDS);
    const bool warp_failed = __any_sync(FULL_MASK, bad_block || timed_out);

    // ---- row sums over the quad, then stash (m, l, O) of this warp
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
        l0 += __shfl_xor_sync(FULL_MASK, l0, off);
        l1 += __shfl_xor_sync(FULL_MASK, l1, off);
    }
    __syncwarp();
    float* mlw = ml + warp * 2 * kMultiMaxRows;
    if (t == 0) {
        mlw[r0] = m0; mlw[r1] = m1;
        mlw[kMultiMaxRows + r0] = l0; mlw[kMultiMaxRows + r1] = l1;
    }
    float* ow = reinterpret_cast<float*>(my_stages);  // [16 rows][D]
#pragma unroll
    for (int n = 0; n < NTD; ++n) {
        *reinterpret_cast<float2*>(ow + r0 * D + n * 8 + 2 * t) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(ow + r1 * D + n * 8 + 2 * t) = make_float2(o[n][2], o[n][3]);
    }
    if (lane == 0) flags[warp] = warp_failed ? 1 : 0;
    __syncthreads();

    // ---- merge the warps and write the RR real rows
    bool failed = false;
#pragma unroll
    for (int w = 0; w < NW; ++w) failed = failed || flags[w] != 0;
    for (int e = threadIdx.x; e < RR * D; e += NW * 32) {
        const int r = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, ml[w * 2 * kMultiMaxRows + r]);
        float wsum = 0.f, acc = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float f = exp2_approx(ml[w * 2 * kMultiMaxRows + r] - M);
                wsum += f * ml[w * 2 * kMultiMaxRows + kMultiMaxRows + r];
                acc += f * reinterpret_cast<const float*>(smem + size_t(w) * NST * STAGE)[r * D + d];
            }
        }
        out_row(r)[d] = failed ? NAN : (wsum == 0.f ? 0.f : acc / wsum);  // a NaN input stays NaN
    }
}

// ---------------------------------------------------------------- wide variant
//
// More than 16 query rows per kv head (g * q_len up to 64: e.g. 16 draft tokens at
// g = 4, or a 64-token prompt chunk of a multi-head model).  One CTA per
// (sequence, kv head) with MT x NG consumer warps -- warp w owns query rows
// [16 mt, 16 mt + 16), mt = w % MT, as one m16 tile, and takes the stages
// k = grp, grp + NG, ... of its group grp = w / MT -- and two producer warps.  With
// 32 rows or fewer two groups split the stages (four consumer warps, like the
// 16-row kernel's token split) and merge their (m, l, O) at the end.  The producer's lane 0
// streams the sequence in stages of 64 tokens (four 16-token tiles, K and V, by TMA
// tensor copies with the 128-byte swizzle) through an NST-deep ring shared by all
// consumers: a "full" mbarrier per stage completes when its bytes land, an "empty"
// one when every consumer has read it.  Each consumer runs the same per-tile
// arithmetic as the 16-row kernel on its rows and writes them itself.
constexpr int kWideMaxRows = 64;
// per variant (2, 3 or 4 m-tiles): ring depth, and the options of the kernel (OPT bits
// below: query rows in shared memory, two tiles per softmax step, two score chains)
#ifndef PF_WIDE_NST_2
#define PF_WIDE_NST_2 3
#endif
#ifndef PF_WIDE_OPT_2
#define PF_WIDE_OPT_2 2
#endif
#ifndef PF_WIDE_NST_3
#define PF_WIDE_NST_3 2
#endif
#ifndef PF_WIDE_OPT_3
#define PF_WIDE_OPT_3 3
#endif
#ifndef PF_WIDE_NST_4
#define PF_WIDE_NST_4 2
#endif
#ifndef PF_WIDE_OPT_4
#define PF_WIDE_OPT_4 3
#endif
constexpr int kWideSub = 4;      // 16-token tiles per stage
constexpr int kWideMaxProd = 2;  // producer warps at most (kWideSub / NPW tiles of each stage apiece)

template <int D, int NST, int NC = 0>
struct WideLayout {
    static constexpr int TT = kTileTokens;
    static constexpr int HALVES = D / 64;
    static constexpr int HALF_BYTES = TT * 128;             // one TMA box: 16 rows x 128 B
    static constexpr int SUBTILE = HALVES * HALF_BYTES;     // one 16-token tile of K or V
    static constexpr int KV = kWideSub * SUBTILE;           // the K (or V) part of a stage
    static constexpr int STAGE = 2 * KV;
    static constexpr size_t FULL = size_t(NST) * STAGE;     // NST mbarriers
    static constexpr size_t EMPTY = FULL + size_t(NST) * 8;  // NST mbarriers
    static constexpr size_t BAD = EMPTY + size_t(NST) * 8;   // [NST][producer] ints: bit u = tile u had no copy
    // query rows in shared memory (when the registers are short): per consumer warp 16 rows
    // of D bf16, rows padded by 16 bytes so the ldmatrix reads are free of bank conflicts
    static constexpr int QSTRIDE = D * 2 + 16;
    static constexpr size_t QAREA = BAD + ((NST * 4 * kWideMaxProd + 15) / 16) * 16;
    static constexpr size_t BYTES = QAREA + size_t(NC) * 16 * QSTRIDE;
    static constexpr size_t ALLOC = BYTES + 1024;           // room to align to 1024
};

// OPT bits: kWideQs (query rows in shared memory), kWidePairs (two tiles per softmax
// step), kWideSplit (two score accumulator chains)
constexpr int kWideQs = 1, kWidePairs = 2, kWideSplit = 4;

template <int D, int MT, int NG, int NST, int OPT, int NPW>
__global__ void __launch_bounds__((MT * NG + NPW) * 32, 2) paged_multi_query_wide_kernel(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v, const MultiParams p) {
    constexpr bool QS = (OPT & kWideQs) != 0;
    using Lay = WideLayout<D, NST, QS ? MT * NG : 0>;
    constexpr int TT = Lay::TT, HALVES = Lay::HALVES, HALF = Lay::HALF_BYTES, SUBTILE = Lay::SUBTILE;
    constexpr int KV = Lay::KV, STAGE = Lay::STAGE;
    constexpr int SUBTOK = kWideSub * TT;  // tokens per stage
    constexpr int KSTEPS = D / 16;         // k-steps of S = Q K^T
    constexpr int NTD = D / 8;             // n-tiles of O = P V
    constexpr int NC = MT * NG;            // consumer warps; warp NC is the producer
    constexpr bool PAIRS = (OPT & kWidePairs) != 0;
    constexpr bool SPLIT = (OPT & kWideSplit) != 0;

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // swizzled boxes need 1 KiB alignment
    const uint32_t full0 = smem_u32(smem + Lay::FULL), empty0 = smem_u32(smem + Lay::EMPTY);
    volatile int* bad = reinterpret_cast<volatile int*>(smem + Lay::BAD);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = p.num_kv_heads, G = p.group, Q = p.q_len, RR = p.rows, Hq = p.num_q_heads;
    const int kvh = blockIdx.x % Hkv;
    const int seq = p.sorted ? multi_sorted_seq<(MT * NG + NPW) * 32>(p, blockIdx.x / Hkv) : blockIdx.x / Hkv;
    const int L = __ldg(p.context_lens + seq);
    const bool len_bad = L < 0 || (long long)L > (long long)p.max_blocks_per_seq * p.block_size;
    auto out_row = [&](int r) -> float* {  // query row r = j * G + h
        const int j = r / G, h = r - (r / G) * G;
        return p.out + ((size_t(seq) * Q + j) * Hq + kvh * G + h) * D;
    };
    if (len_bad) {
        if (threadIdx.x == 0) set_error(p.err, ERR_BOUNDS);
        for (int e = threadIdx.x; e < RR * D; e += (NC + NPW) * 32) out_row(e / D)[e % D] = NAN;
        return;
    }
    const int nstages = (L + SUBTOK - 1) / SUBTOK;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < NST; ++s) {
            mbar_init(full0 + 8 * s, NPW);
            mbar_init(empty0 + 8 * s, MT);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (NPW == 1 ? warp == NC : warp >= NC) {
        if constexpr (NPW == 1) {
            // ---- producer: lane 0 fills stage k % NST once its consumers have released it
            if (lane != 0) return;  // one producer: lane 0 alone
            const int32_t* trow = p.block_tables + size_t(seq) * p.max_blocks_per_seq;
            const int bs = p.block_size, bshift = p.block_shift;
            auto block_index = [&](int tok) { return bshift >= 0 ? (tok >> bshift) : (tok / bs); };
            auto block_offset = [&](int tok) { return bshift >= 0 ? (tok & (bs - 1)) : (tok % bs); };
            const uint64_t policy = l2_policy_evict_first();
            int cur[kWideSub], nxt[kWideSub];
            auto entries = [&](int k, int (&e)[kWideSub]) {  // table entries of stage k's tiles
#pragma unroll
                for (int u = 0; u < kWideSub; ++u) {
                    const int tok = k * SUBTOK + u * TT;
                    e[u] = tok < L ? __ldg(trow + block_index(tok)) : 0;
                }
            };
            if (nstages > 0) entries(0, cur);
            for (int k = 0; k < nstages; ++k) {
                if (k + 1 < nstages) entries(k + 1, nxt);  // a stage ahead
                const int s = k % NST;
                if (k >= NST && !mbar_wait_bounded(empty0 + 8 * s, ((k / NST) - 1) & 1, p.wait_limit_ns)) {
                    set_error(p.err, ERR_TIMEOUT);  // the consumers' own waits give up in turn
                    return;
                }
                uint32_t bytes = 0;
                int badmask = 0;
#pragma unroll
                for (int u = 0; u < kWideSub; ++u) {
                    if (k * SUBTOK + u * TT >= L) continue;
                    if (cur[u] >= 0 && (long long)cur[u] < p.num_blocks) bytes += 2 * SUBTILE;
                    else badmask |= 1 << u;
                }
                bad[s] = badmask;
                if (badmask) set_error(p.err, ERR_BOUNDS);
                const uint32_t full = full0 + 8 * s;
                const uint32_t dst = smem_u32(smem) + uint32_t(s) * STAGE;
                mbar_arrive_expect_tx(full, bytes);
#pragma unroll
                for (int u = 0; u < kWideSub; ++u) {
                    const int tok = k * SUBTOK + u * TT;
                    if (tok >= L || (badmask >> u) & 1) continue;
                    const int y = (cur[u] * Hkv + kvh) * bs + block_offset(tok);
#pragma unroll
                    for (int hh = 0; hh < HALVES; ++hh) {
                        tma_load_2d(dst + u * SUBTILE + hh * HALF, &tmap_k, hh * 64, y, full, policy);
                        tma_load_2d(dst + KV + u * SUBTILE + hh * HALF, &tmap_v, hh * 64, y, full, policy);
                    }
                }
#pragma unroll
                for (int u = 0; u < kWideSub; ++u) cur[u] = nxt[u];
            }
        } else {
            // ---- producer warp pw of NPW: lane 0 fills its kWideSub / NPW tiles of stage k % NST once
            // the consumers have released it.  The blocks of a sequence lie anywhere in the pool and one
            // thread's copies to scattered pages are served one after another, so where the registers
            // allow, two warps issue.
            // The warp loads the table entries of 32 boxes (8 stages) a batch ahead: lane l holds
            // box 32 b + l.
            const int pw = warp - NC;
            const int32_t* trow = p.block_tables + size_t(seq) * p.max_blocks_per_seq;
            const int bs = p.block_size, bshift = p.block_shift;
            auto block_index = [&](int tok) { return bshift >= 0 ? (tok >> bshift) : (tok / bs); };
            auto block_offset = [&](int tok) { return bshift >= 0 ? (tok & (bs - 1)) : (tok % bs); };
            auto batch = [&](int b) {
                const int tok = (32 * b + lane) * TT;
                return tok < L ? __ldg(trow + block_index(tok)) : 0;
            };
            constexpr int SPB = 32 / kWideSub;  // stages per batch
            const uint64_t policy = l2_policy_evict_first();
            int ent_cur = batch(0), ent_nxt = batch(1);
            for (int k = 0; k < nstages; ++k) {
                if (k > 0 && k % SPB == 0) {
                    ent_cur = ent_nxt;
                    ent_nxt = batch(k / SPB + 1);
                }
                int e[kWideSub / NPW];
#pragma unroll
                for (int i = 0; i < kWideSub / NPW; ++i)
                    e[i] = __shfl_sync(FULL_MASK, ent_cur, (k % SPB) * kWideSub + pw * (kWideSub / NPW) + i);
                const int s = k % NST;
                bool ok = true;
                if (lane == 0 && k >= NST) ok = mbar_wait_bounded(empty0 + 8 * s, ((k / NST) - 1) & 1, p.wait_limit_ns);
                if (!__shfl_sync(FULL_MASK, ok ? 1 : 0, 0)) {
                    if (lane == 0) set_error(p.err, ERR_TIMEOUT);  // the consumers' own waits give up in turn
                    return;
                }
                if (lane == 0) {
                    uint32_t bytes = 0;
                    int badmask = 0;
#pragma unroll
                    for (int i = 0; i < kWideSub / NPW; ++i) {
                        const int u = pw * (kWideSub / NPW) + i;
                        if (k * SUBTOK + u * TT >= L) continue;
                        if (e[i] >= 0 && (long long)e[i] < p.num_blocks) bytes += 2 * SUBTILE;
                        else badmask |= 1 << u;
                    }
                    bad[NPW * s + pw] = badmask;
                    if (badmask) set_error(p.err, ERR_BOUNDS);
                    const uint32_t full = full0 + 8 * s;
                    const uint32_t dst = smem_u32(smem) + uint32_t(s) * STAGE;
                    mbar_arrive_expect_tx(full, bytes);
#pragma unroll
                    for (int i = 0; i < kWideSub / NPW; ++i) {
                        const int u = pw * (kWideSub / NPW) + i;
                        const int tok = k * SUBTOK + u * TT;
                        if (tok >= L || (badmask >> u) & 1) continue;
                        const int y = (e[i] * Hkv + kvh) * bs + block_offset(tok);
#pragma unroll
                        for (int hh = 0; hh < HALVES; ++hh) {
                            tma_load_2d(dst + u * SUBTILE + hh * HALF, &tmap_k, hh * 64, y, full, policy);
                            tma_load_2d(dst + KV + u * SUBTILE + hh * HALF, &tmap_v, hh * 64, y, full, policy);
                        }
                    }
                }
            }
        }
        return;
    }

    // ---- consumer warp: m-tile mt (query rows r0 = 16 mt + g and r1 = r0 + 8, zero rows past
    // RR) over the stages of its group, k = grp, grp + NG, ...
    const int mt = warp % MT, grp = warp / MT;
    const int g = lane >> 2, t = lane & 3;
    const int r0 = 16 * mt + g, r1 = r0 + 8;
    auto qrow = [&](int r) -> const uint16_t* {
        const int j = r / G, h = r - (r / G) * G;
        return p.q + ((size_t(seq) * Q + j) * Hq + kvh * G + h) * D;
    };
    // Q as mma A fragments of k-step ks: held in registers, or (QS) read from this warp's
    // 16 rows in shared memory by ldmatrix at each use
    uint32_t qa[QS ? 1 : KSTEPS][4];
    const uint32_t qbase = smem_u32(smem + Lay::QAREA) + uint32_t(warp) * 16 * Lay::QSTRIDE;
    if constexpr (QS) {
        unsigned char* qs = smem + Lay::QAREA + size_t(warp) * 16 * Lay::QSTRIDE;
        for (int e = lane; e < 16 * (D / 8); e += 32) {
            const int rr = e / (D / 8), ch = e % (D / 8), r = 16 * mt + rr;
            const uint4 v = r < RR ? __ldg(reinterpret_cast<const uint4*>(qrow(r)) + ch) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(qs + rr * Lay::QSTRIDE + ch * 16) = v;
        }
        __syncwarp();
    } else {
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
            const int c = ks * 16 + 2 * t;
            qa[ks][0] = r0 < RR ? __ldg(reinterpret_cast<const uint32_t*>(qrow(r0) + c)) : 0u;
            qa[ks][1] = r1 < RR ? __ldg(reinterpret_cast<const uint32_t*>(qrow(r1) + c)) : 0u;
            qa[ks][2] = r0 < RR ? __ldg(reinterpret_cast<const uint32_t*>(qrow(r0) + c + 8)) : 0u;
            qa[ks][3] = r1 < RR ? __ldg(reinterpret_cast<const uint32_t*>(qrow(r1) + c + 8)) : 0u;
        }
    }
    auto q_frag = [&](int ks, uint32_t (&a)[4]) {
        if constexpr (QS) {
            ldmatrix_x4(qbase + uint32_t((lane & 15) * Lay::QSTRIDE + (ks * 16 + (lane >> 4) * 8) * 2), a[0], a[1],
                        a[2], a[3]);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = qa[ks][i];
        }
    };
    // tokens t < lim are visible to a row; padding rows see nothing
    const int lim0 = r0 < RR ? L - Q + r0 / G + 1 : 0;
    const int lim1 = r1 < RR ? L - Q + r1 / G + 1 : 0;

    float o[NTD][4];
#pragma unroll
    for (int n = 0; n < NTD; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    // swizzled byte offset of 16-byte chunk c (0 .. D/8-1) of token row `tok` in a tile
    auto swz = [](int tok, int c) { return (c >> 3) * HALF + tok * 128 + (((c & 7) ^ (tok & 7)) << 4); };

    bool timed_out = false, failed = false;
    int k = grp;
    for (; k < nstages; k += NG) {
        const int s = k % NST;
        if constexpr (NST % NG != 0) {
            // stage s alternates between the groups, so this group does not wait on every phase of
            // its full barrier, and a parity names a phase only up to two fills.  Waiting first for
            // the release of the stage's previous fill (the other group's) pins the barrier to this
            // fill or the one before it, where the parity is unambiguous.
            if (k >= NST) {
                const bool okr = mbar_wait_bounded(empty0 + 8 * s, ((k / NST) - 1) & 1, p.wait_limit_ns);
                if (__any_sync(FULL_MASK, !okr)) { timed_out = true; break; }
            }
        }
        const bool ok = mbar_wait_bounded(full0 + 8 * s, (k / NST) & 1, p.wait_limit_ns);
        if (__any_sync(FULL_MASK, !ok)) { timed_out = true; break; }
        int badbits = bad[NPW * s];
        if constexpr (NPW > 1) badbits |= bad[NPW * s + 1];
        if (badbits) failed = true;  // a tile without its copy: the rows end up NaN
        unsigned char* Kst = smem + size_t(s) * STAGE;
        unsigned char* Vst = Kst + KV;
        const int tok_base = k * SUBTOK;
        const int nv = min(SUBTOK, L - tok_base);          // valid tokens of the stage
        const int nsub = (nv + TT - 1) / TT;
        if (nv < nsub * TT) {
            // rows past the sequence in its last tile hold other data (or poison): zero V
            // there so 0 * V stays 0.  Every consumer writes the same zeros before reading.
            unsigned char* Vl = Vst + (nsub - 1) * SUBTILE;
            const int r_first = nv - (nsub - 1) * TT;
            for (int b = lane; b < (TT - r_first) * HALVES * 8; b += 32) {
                const int row = r_first + b / (HALVES * 8), rest = b % (HALVES * 8);
                *reinterpret_cast<uint4*>(Vl + (rest >> 3) * HALF + row * 128 + (rest & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before the stage's next TMA fill
            __syncwarp();
        }
        // tiles u .. u + NS - 1 of the stage per softmax step: NS = 2 where the registers allow
        // it (two warp groups), else 1
        auto step = [&](auto ns_const, int u) {
            constexpr int NS = decltype(ns_const)::value;
            constexpr int NT = 2 * NS;  // n-tiles of 8 tokens
            const int tok0 = tok_base + u * TT;
            // -- S = Q K^T (with two warp groups the k-steps alternate between two accumulator
            // chains; the 64-row variant has no registers for the second chain)
            float sa[NT][4], sb[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
#pragma unroll
            for (int kp = 0; kp < KSTEPS / 2; ++kp) {
                uint32_t qlo[4], qhi[4];
                q_frag(2 * kp, qlo);
                q_frag(2 * kp + 1, qhi);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int tok = (nt & 1) * 8 + (lane & 7);
                    const int c = kp * 4 + (lane >> 3);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(smem_u32(Kst + (u + nt / 2) * SUBTILE) + swz(tok, c), b0, b1, b2, b3);
                    mma_bf16_16816(sa[nt], qlo, b0, b1);
                    if constexpr (SPLIT) mma_bf16_16816(sb[nt], qhi, b2, b3);
                    else mma_bf16_16816(sa[nt], qhi, b2, b3);
                }
            }
            // -- mask, scale to base 2, online softmax per row (the 4 lanes of a quad share a row)
            float sc[NT][4];
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = tok0 + nt * 8 + 2 * t + (e & 1);
                    const bool vis = tok < (e < 2 ? lim0 : lim1);
                    const float dot = SPLIT ? sa[nt][e] + sb[nt][e] : sa[nt][e];
                    sc[nt][e] = vis ? dot * p.scale_log2 : -INFINITY;
                    if (e < 2) mx0 = fmaxf(mx0, sc[nt][e]); else mx1 = fmaxf(mx1, sc[nt][e]);
                }
#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float sf0 = mn0 == -INFINITY ? 0.f : mn0, sf1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = exp2_approx(m0 - sf0), al1 = exp2_approx(m1 - sf1);
            m0 = mn0;
            m1 = mn1;
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sc[nt][e] = exp2_approx(sc[nt][e] - (e < 2 ? sf0 : sf1));  // now the probability
                    if (e < 2) ps0 += sc[nt][e]; else ps1 += sc[nt][e];
                }
            l0 = l0 * al0 + ps0;
            l1 = l1 * al1 + ps1;
#pragma unroll
            for (int n = 0; n < NTD; ++n) {
                o[n][0] *= al0; o[n][1] *= al0;
                o[n][2] *= al1; o[n][3] *= al1;
            }
            // -- P of each 16-token tile as A fragments, split into bf16 hi + lo
            uint32_t ph[NS][4], pl[NS][4];
#pragma unroll
            for (int s2 = 0; s2 < NS; ++s2) {
                const float* v[4] = {&sc[2 * s2][0], &sc[2 * s2][2], &sc[2 * s2 + 1][0], &sc[2 * s2 + 1][2]};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float a = v[i][0], b = v[i][1];
                    ph[s2][i] = pack_bf16x2(a, b);
                    const float ah = __uint_as_float(ph[s2][i] << 16), bh = __uint_as_float(ph[s2][i] & 0xffff0000u);
                    pl[s2][i] = pack_bf16x2(a - ah, b - bh);
                }
            }
            // -- O += P V: V fragments via ldmatrix.trans, two n-tiles of 8 dims per load
#pragma unroll
            for (int dp = 0; dp < NTD / 2; ++dp) {
#pragma unroll
                for (int s2 = 0; s2 < NS; ++s2) {
                    const int mi = lane >> 3;
                    const int tok = ((mi & 1) << 3) + (lane & 7);
                    const int c = 2 * dp + (mi >> 1);
                    uint32_t v0, v1, v2, v3;
                    ldmatrix_x4_trans(smem_u32(Vst + (u + s2) * SUBTILE) + swz(tok, c), v0, v1, v2, v3);
                    mma_bf16_16816(o[2 * dp], ph[s2], v0, v1);
                    mma_bf16_16816(o[2 * dp], pl[s2], v0, v1);
                    mma_bf16_16816(o[2 * dp + 1], ph[s2], v2, v3);
                    mma_bf16_16816(o[2 * dp + 1], pl[s2], v2, v3);
                }
            }
        };
        int u = 0;
        if constexpr (PAIRS) {
            for (; u + 1 < nsub; u += 2) step(std::integral_constant<int, 2>{}, u);
        }
        for (; u < nsub; ++u) step(std::integral_constant<int, 1>{}, u);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);  // this warp is done with the stage
    }
    if (timed_out) {
        // the producer may still have fills of the next stages in flight: give them a
        // bounded chance to land before the CTA's shared memory goes away
        if (lane == 0) set_error(p.err, ERR_TIMEOUT);
        const int last = min(k + NST, nstages);
        for (int kk = k; kk < last; ++kk) mbar_wait_bounded(full0 + 8 * (kk % NST), (kk / NST) & 1, p.wait_limit_ns);
        failed = true;
    }

    // ---- row sums over the quad
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
        l0 += __shfl_xor_sync(FULL_MASK, l0, off);
        l1 += __shfl_xor_sync(FULL_MASK, l1, off);
    }
    if constexpr (NG > 1) {
        // ---- the groups' partial (m, l, O) of an m-tile meet in the stage memory, free once
        // every consumer is past its last stage (named barrier of the consumers only)
        asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");
        constexpr int SLOT = 16 * D + 64;  // floats: O [16][D], then m, l of the 16 rows, failed
        float* mine = reinterpret_cast<float*>(smem) + size_t(warp) * SLOT;
        if (grp > 0) {
#pragma unroll
            for (int n = 0; n < NTD; ++n) {
                *reinterpret_cast<float2*>(mine + g * D + n * 8 + 2 * t) = make_float2(o[n][0], o[n][1]);
                *reinterpret_cast<float2*>(mine + (g + 8) * D + n * 8 + 2 * t) = make_float2(o[n][2], o[n][3]);
            }
            if (t == 0) {
                mine[16 * D + g] = m0; mine[16 * D + g + 8] = m1;
                mine[16 * D + 16 + g] = l0; mine[16 * D + 16 + g + 8] = l1;
            }
            if (lane == 0) mine[16 * D + 32] = failed ? 1.f : 0.f;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");
        if (grp > 0) return;
#pragma unroll
        for (int gi = 1; gi < NG; ++gi) {
            const float* other = reinterpret_cast<const float*>(smem) + size_t(gi * MT + mt) * SLOT;
            if (other[16 * D + 32] != 0.f) failed = true;
            const float mo0 = other[16 * D + g], mo1 = other[16 * D + g + 8];
            const float lo0 = other[16 * D + 16 + g], lo1 = other[16 * D + 16 + g + 8];
            const float M0 = fmaxf(m0, mo0), M1 = fmaxf(m1, mo1);
            const float s0 = M0 == -INFINITY ? 0.f : M0, s1 = M1 == -INFINITY ? 0.f : M1;
            const float a0 = exp2_approx(m0 - s0), b0 = exp2_approx(mo0 - s0);
            const float a1 = exp2_approx(m1 - s1), b1 = exp2_approx(mo1 - s1);
#pragma unroll
            for (int n = 0; n < NTD; ++n) {
                const float2 x0 = *reinterpret_cast<const float2*>(other + g * D + n * 8 + 2 * t);
                const float2 x1 = *reinterpret_cast<const float2*>(other + (g + 8) * D + n * 8 + 2 * t);
                o[n][0] = o[n][0] * a0 + x0.x * b0; o[n][1] = o[n][1] * a0 + x0.y * b0;
                o[n][2] = o[n][2] * a1 + x1.x * b1; o[n][3] = o[n][3] * a1 + x1.y * b1;
            }
            l0 = l0 * a0 + lo0 * b0;
            l1 = l1 * a1 + lo1 * b1;
            m0 = M0;
            m1 = M1;
        }
    }

    // ---- this warp's rows
    const float i0 = l0 == 0.f ? 0.f : 1.f / l0, i1 = l1 == 0.f ? 0.f : 1.f / l1;  // no token: 0
#pragma unroll
    for (int n = 0; n < NTD; ++n) {
        const int d = n * 8 + 2 * t;
        if (r0 < RR)
            *reinterpret_cast<float2*>(out_row(r0) + d) =
                failed ? make_float2(NAN, NAN) : make_float2(o[n][0] * i0, o[n][1] * i0);
        if (r1 < RR)
            *reinterpret_cast<float2*>(out_row(r1) + d) =
                failed ? make_float2(NAN, NAN) : make_float2(o[n][2] * i1, o[n][3] * i1);
    }
}

// ---------------------------------------------------------------- tcgen05 variant
//
// Up to 64 query rows per kv head at D = 128, with both products on the fifth-generation
// tensor cores (single-CTA tcgen05.mma, fp32 accumulators in tensor memory), computed
// transposed so that the 128-lane M side of every product is filled by the tile's tokens
// or by the head dimensions and the query rows are the N side:
//     S^T(j) = K(j) Q^T           M = 128 tokens, N = 64 rows, K = D
//     O^T   += V(j)^T P(j)^T      M = D = 128,    N = 64 rows x {hi, lo}, K = 128 tokens
// K(j) is the A operand straight from its swizzled stage (K-major), V(j) the A operand
// read MN-major from its stage, Q and P^T the B operands in shared memory.  P enters the
// product as its bf16 hi part and the bf16 remainder (N columns 0-63 and 64-127 of O^T),
// summed at the end.  One CTA per (sequence, kv head), thirteen warps, one CTA per SM
// (by its shared memory), 256 TMEM columns (two 64-column score buffers, O^T).
//  * warps 0-1 stream the sequence's K tiles through a 3-deep ring and warps 2-3 its V
//    tiles through a 2-deep one, each warp copying half of a tile's eight 16-token boxes
//    (TMA tensor copies with the 128-byte swizzle, one per box and dim half, issued by
//    eight lanes); the blocks of a sequence lie anywhere in the pool and one thread's
//    copies to scattered pages are served one after another, so four warps issue.  Table
//    entries are fetched 32 boxes at a time, a batch ahead;
//  * warp 4, lane 0 issues S^T(j) once K(j) has landed and its score buffer (j % 2) is
//    read, and O^T += V(j)^T P(j)^T once P(j) is written and V(j) has landed, the latter
//    first; S^T(j + 1) thus runs while the softmax of tile j does;
//  * warps 5-12: lane l of the warp with TMEM lane quarter u (warp % 4) holds token
//    32 u + l of the tile, and warps 5-8 / 9-12 take query rows 0-31 / 32-63.  A row's
//    reference maximum is shared by the whole tile (the product sums over its tokens):
//    the four warps of a row half tell each other through shared memory whether any score
//    exceeds its reference by more than 2^8, and only then take the tile's row maxima
//    (a shuffle transpose and shared memory), move the references and rescale those rows
//    of O^T in place once the previous product is complete.  Each thread writes its
//    token's P row into P^T (swizzled, MN-major) and keeps the row sums of its tokens;
//    at the end they are summed over the tile's lanes (a transposed shuffle) and O^T is
//    staged through P^T's buffer, so that each warp writes 8 whole normalised output rows.
// Every wait is bounded; one that gives up raises an abort flag that ends the others at
// once, and every role still runs all its iterations, so the CTA stays in step and
// releases its tensor memory.
constexpr int kTcTok = 128;       // tokens per tile
constexpr int kTcKStages = 3;     // K ring depth
constexpr int kTcVStages = 2;     // V ring depth
constexpr int kTcRows = 64;       // query rows per kv head (the N of the score product)
constexpr int kTcCols = 256;      // TMEM columns: score buffers [0, 64) and [64, 128), O^T [128, 256)
constexpr int kTcProducers = 4;   // issuing warps: two for K, two for V
constexpr int kTcMath = 8;        // softmax warps
constexpr int kTcThreads = 32 * (kTcProducers + 1 + kTcMath);
constexpr float kTcRescale = 8.f; // a reference maximum moves when a score exceeds it by more (log2 units)

struct TcLayout {
    static constexpr int HALF = kTcTok * 128;         // 128 rows of 128 bytes (64 bf16): 16 KiB
    static constexpr int STAGE = 2 * HALF;            // one tile of K or of V: dims [0, 64), [64, 128)
    static constexpr int KRING = 0;
    static constexpr int VRING = KRING + kTcKStages * STAGE;
    static constexpr int PT = VRING + kTcVStages * STAGE;  // P^T: N blocks hi, lo of [128 tokens][64 rows]
    static constexpr int QS = PT + 2 * HALF;                // Q: dim halves of [64 rows][64 dims]
    static constexpr int NBARS = 2 * kTcKStages + 2 * kTcVStages + 8;
    static constexpr int BARS = QS + 2 * kTcRows * 128;
    static constexpr int FLAGS = BARS + ((NBARS * 8 + 15) / 16) * 16;  // [2 row halves][2 tiles][4 quarters] int
    static constexpr int RMAX = FLAGS + 2 * 2 * 4 * 4;                 // [2 row halves][32 rows][4 quarters] float
    static constexpr int LSUM = RMAX + 2 * 32 * 4 * 4;                 // [4 quarters][64 rows] float
    static constexpr int MREF = LSUM + 4 * kTcRows * 4;                // [8 math warps][3][32 rows] float
    static constexpr int MISC = MREF + kTcMath * 3 * 32 * 4;           // TMEM base, bad-block flag, abort flag
    static constexpr int BYTES = MISC + 16;
    static constexpr int ALLOC = BYTES + 1024;                         // room to align to 1024
};
// one CTA per SM: the dynamic part plus the longest-first ranking's static arrays fit in a
// block's 227 KiB of shared memory
static_assert(TcLayout::ALLOC + (kMultiSortMax + 4) * 4 <= 227 * 1024, "shared memory of the tcgen05 kernel");

// Sum over the warp's 32 lanes of each of 32 values, transposed: lane l returns the sum
// of value l (31 shuffles instead of 160).  The values are consumed.
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32], int lane) {
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int c = 0; c < w; ++c) {
            const float send = up ? v[c] : v[c + w];
            const float keep = up ? v[c + w] : v[c];
            v[c] = keep + __shfl_xor_sync(FULL_MASK, send, w);
        }
    }
    return v[0];
}

// fp32 <-> int32 keys whose signed order is the order of the floats (-inf lowest), for
// the integer warp reduction.
__device__ __forceinline__ int float_to_ordered(float f) {
    const int i = __float_as_int(f);
    return i ^ ((i >> 31) & 0x7FFFFFFF);
}
__device__ __forceinline__ float ordered_to_float(int i) { return __int_as_float(i ^ ((i >> 31) & 0x7FFFFFFF)); }

__global__ void __launch_bounds__(kTcThreads, 1) paged_multi_query_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v, const MultiParams p) {
    constexpr int D = 128, NT = kTcThreads, TOK = kTcTok, NK = kTcKStages, NV = kTcVStages, NR = kTcRows;
    constexpr int BOXES = TOK / kTileTokens;  // 16-token boxes per tile
    constexpr int NMW = kTcMath, MMAW = kTcProducers;
    constexpr uint32_t TO = 128;              // O^T columns: rows 0-63 (hi), 64-127 (lo)
    auto TS = [](int b) { return uint32_t(64 * b); };
    using Lay = TcLayout;
    // mbarriers: K and V rings full / empty; per score buffer written / read; P^T written /
    // read (its product complete); Q stored; all MMAs done
    enum { KFULL = 0, KEMPTY = NK, VFULL = 2 * NK, VEMPTY = 2 * NK + NV, SFULL = 2 * NK + 2 * NV, SFREE = SFULL + 2,
           PFULL = SFREE + 2, PFREE = PFULL + 1, QREADY = PFREE + 1, DONE = QREADY + 1 };
    static_assert(DONE + 1 == Lay::NBARS, "barrier count");

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // swizzled operands need 1 KiB alignment
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + uint32_t(Lay::BARS + 8 * i); };
    volatile int* flags = reinterpret_cast<volatile int*>(smem + Lay::FLAGS);
    float* rmax = reinterpret_cast<float*>(smem + Lay::RMAX);
    float* lsum = reinterpret_cast<float*>(smem + Lay::LSUM);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::MISC);
    volatile int* bad = reinterpret_cast<volatile int*>(smem + Lay::MISC + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::MISC + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = p.num_kv_heads, G = p.group, Q = p.q_len, RR = p.rows, Hq = p.num_q_heads;
    const int kvh = blockIdx.x % Hkv;
    const int seq = p.sorted ? multi_sorted_seq<NT>(p, blockIdx.x / Hkv) : blockIdx.x / Hkv;
    const int L = __ldg(p.context_lens + seq);
    const bool len_bad = L < 0 || (long long)L > (long long)p.max_blocks_per_seq * p.block_size;
    auto out_row = [&](int r) -> float* {  // query row r = j * G + h
        const int j = r / G, h = r - (r / G) * G;
        return p.out + ((size_t(seq) * Q + j) * Hq + kvh * G + h) * D;
    };
    if (len_bad) {
        if (threadIdx.x == 0) set_error(p.err, ERR_BOUNDS);
        for (int e = threadIdx.x; e < RR * D; e += NT) out_row(e / D)[e % D] = NAN;
        return;
    }
    const int nt = (L + TOK - 1) / TOK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Lay::NBARS; ++i) {
            int count = 1;                                                 // commits
            if ((i >= KFULL && i < KFULL + NK) || (i >= VFULL && i < VFULL + NV)) count = 2;  // two issuing warps
            if (i == SFREE || i == SFREE + 1 || i == PFULL || i == QREADY) count = NMW;      // the math warps
            mbar_init(bar(i), count);
        }
        *bad = 0;
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kTcCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    // Bounded wait; false once this or another role has given up.
    auto give_up = [&]() {
        *abort_flag = 1;
        set_error(p.err, ERR_TIMEOUT);
    };
    auto wait = [&](int i, uint32_t parity) -> bool {
        const uint32_t b = bar(i);
        if (mbar_try_wait(b, parity)) return true;
        if (*abort_flag) return false;
        const uint64_t start = global_timer_ns();
        for (uint32_t it = 1;; ++it) {
            if (mbar_try_wait(b, parity)) return true;
            if ((it & 63u) == 0u) {
                if (*abort_flag) return false;
                if (global_timer_ns() - start > p.wait_limit_ns) {
                    give_up();
                    return false;
                }
            }
        }
    };

    if (warp < kTcProducers) {
        // ---- producer warp: warps 0-1 copy K, warps 2-3 V; warp w takes boxes w % 2, + 2, + 4,
        // + 6 of every tile.  The warp loads the table entries of 32 boxes (4 tiles) a batch
        // ahead: lane l holds box 32 b + l.
        const bool is_v = warp >= 2;
        const int pw = warp & 1;
        const int NS = is_v ? NV : NK;
        const int FULLB = is_v ? VFULL : KFULL, EMPTYB = is_v ? VEMPTY : KEMPTY;
        const uint32_t ring = sbase + uint32_t(is_v ? Lay::VRING : Lay::KRING);
        const CUtensorMap* map = is_v ? &tmap_v : &tmap_k;
        const int32_t* trow = p.block_tables + size_t(seq) * p.max_blocks_per_seq;
        const int bs = p.block_size, bshift = p.block_shift;
        auto block_index = [&](int tok) { return bshift >= 0 ? (tok >> bshift) : (tok / bs); };
        auto block_offset = [&](int tok) { return bshift >= 0 ? (tok & (bs - 1)) : (tok % bs); };
        auto batch = [&](int b) {  // entry of box 32 b + lane (0 past the sequence)
            const int tok = (32 * b + lane) * kTileTokens;
            return tok < L ? __ldg(trow + block_index(tok)) : 0;
        };
        constexpr int TPB = 32 / BOXES;  // tiles per batch
        const uint64_t policy = l2_policy_evict_first();
        int ent_cur = batch(0), ent_nxt = batch(1);
        int issued = 0;
        for (int j = 0; j < nt; ++j) {
            if (j > 0 && j % TPB == 0) {
                ent_cur = ent_nxt;
                ent_nxt = batch(j / TPB + 1);
            }
            int e[BOXES / 2];
#pragma unroll
            for (int i = 0; i < BOXES / 2; ++i) e[i] = __shfl_sync(FULL_MASK, ent_cur, (j % TPB) * BOXES + pw + 2 * i);
            const int s = j % NS;
            bool ok = true;
            if (lane == 0 && j >= NS) ok = wait(EMPTYB + s, ((j / NS) - 1) & 1);
            if (!__shfl_sync(FULL_MASK, ok ? 1 : 0, 0)) break;
            if (lane == 0) {
                bool good[BOXES / 2];
                uint32_t bytes = 0;
#pragma unroll
                for (int i = 0; i < BOXES / 2; ++i) {
                    const int tok = j * TOK + (pw + 2 * i) * kTileTokens;
                    const bool live = tok < L;
                    good[i] = live && e[i] >= 0 && (long long)e[i] < p.num_blocks;
                    if (live && !good[i]) {
                        *bad = 1;
                        set_error(p.err, ERR_BOUNDS);
                    }
                    bytes += good[i] ? 2u * kTileTokens * 128u : 0u;
                }
                mbar_arrive_expect_tx(bar(FULLB + s), bytes);
            }
            {
                // lanes 0-7 issue one copy each (box pw + 2 (lane / 2), dim half lane % 2), once lane 0
                // has set the byte count: copies from different threads to scattered pages go out side
                // by side rather than one after another
                __syncwarp();
                const int el = __shfl_sync(FULL_MASK, ent_cur, ((j % TPB) * BOXES + pw + 2 * (lane >> 1)) & 31);
                const int b = pw + 2 * (lane >> 1), hf = lane & 1, tok = j * TOK + b * kTileTokens;
                if (lane < BOXES && tok < L && el >= 0 && (long long)el < p.num_blocks)
                    tma_load_2d(ring + uint32_t(s * Lay::STAGE + b * kTileTokens * 128 + hf * Lay::HALF), map,
                                64 * hf, (el * Hkv + kvh) * bs + block_offset(tok), bar(FULLB + s), policy);
            }
            ++issued;
        }
        // the CTA may not end with copies in flight: wait for the last fill of each stage
        if (lane == 0)
            for (int s = 0; s < NS && s < issued; ++s) {
                const int jl = s + NS * ((issued - 1 - s) / NS);
                mbar_wait_bounded(bar(FULLB + s), (jl / NS) & 1, p.wait_limit_ns);
            }
        __syncwarp();
    } else if (warp == MMAW) {
        // ---- MMA issuer: whichever of O^T += V(jp)^T P(jp)^T and S^T(js) is ready, the former first
        constexpr uint32_t IDESC_S = umma_idesc_bf16(TOK, NR, 0, 0);
        constexpr uint32_t IDESC_O = umma_idesc_bf16(D, 2 * NR, 1, 1);
        __syncwarp();
        const bool qok = __all_sync(FULL_MASK, wait(QREADY, 0));
        (void)qok;
        tc_fence_after_sync();
        int js = 0, jp = 0;
        uint64_t idle_since = 0;
        bool idle = false;
        while (jp < nt) {
            int act = 0;  // 1: P.V(jp), 2: S(js), -1: give up
            if (lane == 0) {
                if (jp < js && mbar_test_wait(bar(PFULL), jp & 1) &&
                    mbar_test_wait(bar(VFULL + jp % NV), (jp / NV) & 1))
                    act = 1;
                // S(js): K landed, and the softmax of tile js - 2 has read the score buffer
                else if (js < nt && mbar_test_wait(bar(KFULL + js % NK), (js / NK) & 1) &&
                         (js < 2 || mbar_test_wait(bar(SFREE + (js & 1)), ((js >> 1) - 1) & 1)))
                    act = 2;
                else if (*abort_flag) act = -1;
                else if (!idle) {
                    idle = true;
                    idle_since = global_timer_ns();
                } else if (global_timer_ns() - idle_since > p.wait_limit_ns) {
                    give_up();
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
                    const uint32_t ka = sbase + uint32_t(Lay::KRING + (js % NK) * Lay::STAGE);
                    const uint32_t qa = sbase + uint32_t(Lay::QS);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)  // 16 dims: 32 bytes into the swizzled rows of K and Q
                        umma_bf16(tmem + TS(js & 1),
                                  umma_desc_sw128(ka + (kk >> 2) * Lay::HALF + (kk & 3) * 32, 16, 1024),
                                  umma_desc_sw128(qa + (kk >> 2) * (NR * 128) + (kk & 3) * 32, 16, 1024), IDESC_S,
                                  kk > 0);
                    umma_commit(bar(SFULL + (js & 1)));
                    umma_commit(bar(KEMPTY + js % NK));
                }
                ++js;
            } else {
                const uint32_t voff = uint32_t(Lay::VRING + (jp % NV) * Lay::STAGE);
                const int nvalid = min(TOK, L - jp * TOK);
                if (nvalid < TOK) {
                    // tokens past the sequence hold other data (or poison): zero V there so 0 * V stays 0
                    for (int e = lane; e < (TOK - nvalid) * 16; e += 32) {
                        const int r = nvalid + (e >> 4), c = e & 15;
                        *reinterpret_cast<uint4*>(smem + voff + (c >> 3) * Lay::HALF + r * 128 + (c & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    const uint32_t va = sbase + voff, pa = sbase + uint32_t(Lay::PT);
#pragma unroll
                    for (int kk = 0; kk < TOK / 16; ++kk)  // 16 tokens: 2 KiB into V and into P^T
                        umma_bf16(tmem + TO, umma_desc_sw128(va + kk * 2048, Lay::HALF, 1024),
                                  umma_desc_sw128(pa + kk * 2048, Lay::HALF, 1024), IDESC_O, jp > 0 || kk > 0);
                    umma_commit(bar(VEMPTY + jp % NV));
                    umma_commit(bar(PFREE));
                }
                ++jp;
            }
            __syncwarp();
        }
        // every MMA of the CTA is complete before O^T is read and tensor memory released
        if (lane == 0) {
            umma_commit(bar(DONE));
            mbar_wait_bounded(bar(DONE), 0, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ---- math warps
        const int mw = warp - MMAW - 1;                        // 0 .. 7
        const int q4 = warp & 3, hh = mw >> 2;                 // TMEM lane quarter; row half
        const int tk = 32 * q4 + lane;                         // this thread's token of a tile, and its O^T dim
        const uint32_t tl = tmem + (uint32_t(q4 * 32) << 16);  // this warp's TMEM lane quarter
        const int barid = 1 + hh;                              // named barrier of the row half's four warps

        // Q (rows past RR zero) into its swizzled K-major tile: 1024 chunks of 16 bytes, four per
        // thread, all loads in flight before the first store
        {
            constexpr int PER = NR * 16 / (NMW * 32);
            uint4 v[PER];
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int i = mw * 32 + lane + k * NMW * 32, r = i >> 4, c16 = i & 15;
                v[k] = make_uint4(0, 0, 0, 0);
                if (r < RR) {
                    const int j = r / G, h = r - (r / G) * G;
                    v[k] = __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t(seq) * Q + j) * Hq + kvh * G + h) * D) + c16);
                }
            }
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int i = mw * 32 + lane + k * NMW * 32, r = i >> 4, c16 = i & 15;
                *reinterpret_cast<uint4*>(smem + Lay::QS + (c16 >> 3) * (NR * 128) + r * 128 +
                                          (((c16 & 7) ^ (r & 7)) << 4)) = v[k];
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(QREADY));

        const int lim0 = L - Q + 1;  // row r sees the tokens t < min(L, lim0 + r / G)
        // this warp's copy of rows 32 hh + c's reference maxima (the same in the half's four warps),
        // and per tile the factor and the shift that moving them applies
        float* mref = reinterpret_cast<float*>(smem + Lay::MREF) + mw * 3 * 32;
        float* alph = mref + 32;
        float* shft = mref + 64;
        mref[lane] = -INFINITY;
        __syncwarp();
        float l_part[32];  // this token's share of the rows' sums
#pragma unroll
        for (int c = 0; c < 32; ++c) l_part[c] = 0.f;
        unsigned char* prow = smem + Lay::PT + tk * 128;  // this token's 128-byte row in both N blocks of P^T

        for (int j = 0; j < nt; ++j) {
            const int b = j & 1;
            wait(SFULL + b, (j >> 1) & 1);
            __syncwarp();
            tc_fence_after_sync();
            float y[32];  // log2-scaled scores of rows 32 hh + c, then relative to the reference
            {
                uint32_t v[32];
                tmem_ld_x32(tl + TS(b) + uint32_t(32 * hh), v);
#pragma unroll
                for (int c = 0; c < 32; ++c) y[c] = __uint_as_float(v[c]) * p.scale_log2;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(SFREE + b));

            const int t = j * TOK + tk;
            if (j * TOK + TOK > lim0) {  // some row does not see some token of this tile
                // row r sees t iff t < L and r / G >= t - lim0 + 1, i.e. r >= (t - lim0 + 1) G
                const int rmin = t >= L ? NR : (t < lim0 ? 0 : min(NR, (t - lim0 + 1) * G));
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (32 * hh + c < rmin) y[c] = -INFINITY;
            }
            // does any score exceed its row's reference by more than the margin?  (-inf reference: any
            // finite score); then scores relative to the reference (-inf reference: 0)
            bool over = false;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float4 m4 = *reinterpret_cast<const float4*>(mref + 4 * c4);
                const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = 4 * c4 + i;
                    over |= y[c] > mm[i] + kTcRescale;
                    y[c] -= mm[i] == -INFINITY ? 0.f : mm[i];
                }
            }
            const bool wover = __any_sync(FULL_MASK, over);
            if (lane == 0) flags[(hh * 2 + b) * 4 + q4] = wover ? 1 : 0;
            asm volatile("bar.sync %0, 128;" ::"r"(barid) : "memory");
            const bool any_over = (flags[(hh * 2 + b) * 4 + 0] | flags[(hh * 2 + b) * 4 + 1] |
                                   flags[(hh * 2 + b) * 4 + 2] | flags[(hh * 2 + b) * 4 + 3]) != 0;
            bool do_rescale = false;  // rows of O^T to scale by alph once the previous product is complete
            if (any_over) {
                // the tile's row maxima: this warp's 32 tokens by integer warp reductions (lane c: row
                // 32 hh + c), then over the half's four warps through shared memory
                {
                    float mr = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int m = __reduce_max_sync(FULL_MASK, float_to_ordered(y[c]));
                        if (lane == c) mr = ordered_to_float(m);
                    }
                    const float old = mref[lane];
                    rmax[((hh * 32) + lane) * 4 + q4] = mr + (old == -INFINITY ? 0.f : old);
                }
                asm volatile("bar.sync %0, 128;" ::"r"(barid) : "memory");
                {
                    const float4 m4 = *reinterpret_cast<const float4*>(rmax + ((hh * 32) + lane) * 4);
                    const float mx = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
                    const float old = mref[lane];
                    const bool move = mx > old + kTcRescale;
                    const float now = move ? mx : old;
                    alph[lane] = move ? exp2_approx(old - mx) : 1.f;  // -inf reference: 0
                    shft[lane] = (old == -INFINITY ? 0.f : old) - (now == -INFINITY ? 0.f : now);
                    // the same decision in the half's four warps: their references agree
                    do_rescale = j > 0 && __any_sync(FULL_MASK, move && old != -INFINITY);
                    __syncwarp();
                    mref[lane] = now;
                    __syncwarp();
                }
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(alph + 4 * c4);
                    const float4 s4 = *reinterpret_cast<const float4*>(shft + 4 * c4);
                    const float aa[4] = {a4.x, a4.y, a4.z, a4.w}, ss[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        l_part[4 * c4 + i] *= aa[i];
                        y[4 * c4 + i] += ss[i];
                    }
                }
            }
            // the previous product (the last reader of P^T and writer of O^T) is complete
            if (j > 0) wait(PFREE, (j - 1) & 1);
            // probabilities of this token for the half's 32 rows, as bf16 hi and lo parts: chunk k
            // (rows 32 hh + 8 k ..) of each goes to 16-byte slot (4 hh + k) ^ (tk % 8) of the token's row
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t ph[4], pl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c0 = 8 * k + 2 * e;
                    const float a = exp2_approx(y[c0]), c = exp2_approx(y[c0 + 1]);
                    l_part[c0] += a;
                    l_part[c0 + 1] += c;
                    ph[e] = pack_bf16x2(a, c);
                    pl[e] = pack_bf16x2(a - __uint_as_float(ph[e] << 16), c - __uint_as_float(ph[e] & 0xffff0000u));
                }
                const int slot = ((4 * hh + k) ^ (tk & 7)) << 4;
                *reinterpret_cast<uint4*>(prow + slot) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                *reinterpret_cast<uint4*>(prow + Lay::HALF + slot) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            }
            if (do_rescale) {
                __syncwarp();
                tc_fence_after_sync();
#pragma unroll
                for (int part = 0; part < 4; ++part) {  // hi, lo columns of this half's rows, dim tk; 16 at a time
                    uint32_t v[16];
                    const uint32_t ta = tl + TO + uint32_t(64 * (part >> 1) + 32 * hh + 16 * (part & 1));
                    tmem_ld_x16(ta, v);
#pragma unroll
                    for (int c = 0; c < 16; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alph[16 * (part & 1) + c]);
                    tmem_st_x16(ta, v);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(PFULL));
        }

        // ---- epilogue.  Row sums over the tile's 128 token lanes (lane c of each warp: row
        // 32 hh + c) while the last products run; then, once every MMA is complete, each half's
        // O^T block goes through P^T's buffer (no product reads it any more) so that a warp
        // writes 8 whole output rows with 16-byte stores
        lsum[q4 * NR + 32 * hh + lane] = warp_transpose_sum(l_part, lane);
        wait(DONE, 0);
        __syncwarp();
        tc_fence_after_sync();
        float* blk = reinterpret_cast<float*>(smem + Lay::PT) + hh * 32 * D;  // [32 rows][D] fp32 of this half
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // 16 rows at a time: dim tk of rows 32 hh + 16 half + c
            uint32_t ohi[16], olo[16];
            tmem_ld_x16(tl + TO + uint32_t(32 * hh + 16 * half), ohi);
            tmem_ld_x16(tl + TO + uint32_t(64 + 32 * hh + 16 * half), olo);
#pragma unroll
            for (int c = 0; c < 16; ++c)
                blk[(16 * half + c) * D + tk] = __uint_as_float(ohi[c]) + __uint_as_float(olo[c]);
        }
        asm volatile("bar.sync 3, %0;" ::"r"(NMW * 32) : "memory");
        const bool failed = *bad != 0 || *abort_flag != 0;
#pragma unroll 2
        for (int i = 0; i < 8; ++i) {  // rows 32 hh + 8 q4 + i; lane l: dims 4 l .. 4 l + 3
            const int rl = 8 * q4 + i, r = 32 * hh + rl;
            if (r >= RR) break;
            const float l = lsum[r] + lsum[NR + r] + lsum[2 * NR + r] + lsum[3 * NR + r];
            const float inv = l == 0.f ? 0.f : 1.f / l;  // no token: 0; a NaN input stays NaN
            const float4 v = *reinterpret_cast<const float4*>(blk + rl * D + 4 * lane);
            float4 o = make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
            if (nt == 0) o = make_float4(0.f, 0.f, 0.f, 0.f);
            if (failed) o = make_float4(NAN, NAN, NAN, NAN);
            *reinterpret_cast<float4*>(out_row(r) + 4 * lane) = o;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kTcCols);
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn tensor_map_encoder() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || ptr == nullptr)
            return nullptr;
        f = reinterpret_cast<EncodeTiledFn>(ptr);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

// The cache as a 2D tensor [rows = NB * Hkv * bs][D] bf16, read in boxes of 16 rows x 64
// elements (128 bytes) with the 128-byte swizzle.
static bool encode_cache_map(CUtensorMap* map, const void* cache, long long rows, int D) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(D) * 2};
    const cuuint32_t box[2] = {64, cuuint32_t(kTileTokens)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_cache_map_vblocks(CUtensorMap* map, const void* cache, long long rows) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {64, cuuint64_t(rows), 2};
    const cuuint64_t strides[2] = {256, 128};  // a row of 128 bf16; the second dim half
    const cuuint32_t box[3] = {64, cuuint32_t(kTileTokens), 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(cache), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMultiWarps = 4;
constexpr int kMultiStages = 2;

template <int D>
static cudaError_t launch_multi(const CUtensorMap& mk, const CUtensorMap& mv, const MultiParams& p,
                                cudaStream_t stream) {
    using Lay = MultiLayout<D, kMultiWarps, kMultiStages>;
    auto kern = paged_multi_query_kernel<D, kMultiWarps, kMultiStages>;
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Lay::ALLOC));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const long long grid = (long long)p.num_seqs * p.num_kv_heads;
    kern<<<unsigned(grid), kMultiWarps * 32, Lay::ALLOC, stream>>>(mk, mv, p);
    return cudaGetLastError();
}

template <int D, int MT, int NG, int NST, int OPT, int NPW>
static cudaError_t launch_multi_wide(const CUtensorMap& mk, const CUtensorMap& mv, const MultiParams& p,
                                     cudaStream_t stream) {
    using Lay = WideLayout<D, NST, (OPT & kWideQs) ? MT * NG : 0>;
    auto kern = paged_multi_query_wide_kernel<D, MT, NG, NST, OPT, NPW>;
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Lay::ALLOC));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const long long grid = (long long)p.num_seqs * p.num_kv_heads;
    kern<<<unsigned(grid), (MT * NG + NPW) * 32, Lay::ALLOC, stream>>>(mk, mv, p);
    return cudaGetLastError();
}

static cudaError_t launch_multi_tc(const CUtensorMap& mk, const CUtensorMap& mv, const MultiParams& p,
                                   cudaStream_t stream) {
    auto kern = paged_multi_query_tc_kernel;
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcLayout::ALLOC);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const long long grid = (long long)p.num_seqs * p.num_kv_heads;
    kern<<<unsigned(grid), kTcThreads, TcLayout::ALLOC, stream>>>(mk, mv, p);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_multi_any(const CUtensorMap& mk, const CUtensorMap& mv, const MultiParams& p,
                                    cudaStream_t stream) {
    if (p.rows <= kMultiMaxRows) return launch_multi<D>(mk, mv, p, stream);
    // producer warps: two where the consumers' registers allow (the 32-row variant), else one.
    // At D = 128 rows past 32 go to the tcgen05 kernel instead.
    if (p.rows <= 32) return launch_multi_wide<D, 2, 2, PF_WIDE_NST_2, PF_WIDE_OPT_2, 2>(mk, mv, p, stream);  // two groups
    if constexpr (D == 64) {
        if (p.rows <= 48) return launch_multi_wide<D, 3, 1, PF_WIDE_NST_3, PF_WIDE_OPT_3, 1>(mk, mv, p, stream);
        return launch_multi_wide<D, 4, 1, PF_WIDE_NST_4, PF_WIDE_OPT_4, 1>(mk, mv, p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pf

using namespace pf;

// Host checks and parameters shared by both multi-query entry points; on success the two
// tensor maps and the parameter block are ready to launch.
static pf_status multi_query_setup(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int q_len,
                                   int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                   int max_blocks_per_seq, int64_t num_blocks, float scale, float* out,
                                   CUtensorMap* mk, CUtensorMap* mv, MultiParams* pp) {
    if (num_seqs < 0 || q_len <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        max_blocks_per_seq <= 0 || num_blocks <= 0 || !std::isfinite(scale) || num_q_heads % num_kv_heads != 0 ||
        num_blocks > INT32_MAX)
        return PF_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    if (head_dim != 64 && head_dim != 128) return PF_ERR_UNSUPPORTED;
    if (block_size % kTileTokens != 0) return PF_ERR_UNSUPPORTED;
    if ((long long)group * q_len > kChunkMaxRows) return PF_ERR_UNSUPPORTED;
    const long long rows = num_blocks * num_kv_heads * (long long)block_size;
    if (rows > INT32_MAX || (long long)num_seqs * num_kv_heads > INT32_MAX) return PF_ERR_UNSUPPORTED;
    auto al = [](const void* ptr, size_t a) { return ptr != nullptr && reinterpret_cast<uintptr_t>(ptr) % a == 0; };
    if (num_seqs > 0 && (!al(q, 16) || !al(k_cache, 16) || !al(v_cache, 16) || !al(block_tables, 4) ||
                         !al(context_lens, 4) || !al(out, 16)))
        return PF_ERR_INVALID_ARG;
    if (num_seqs == 0) return PF_OK;
    unsigned* err = nullptr;
    if (error_word(&err) != cudaSuccess) return PF_ERR_CUDA;
    if (!encode_cache_map(mk, k_cache, rows, head_dim) || !encode_cache_map(mv, v_cache, rows, head_dim))
        return PF_ERR_CUDA;
    MultiParams& p = *pp;
    p = MultiParams{};
    p.q = static_cast<const uint16_t*>(q);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = out;
    p.err = err;
    p.num_blocks = num_blocks;
    p.wait_limit_ns = kDefaultWaitLimitNs;
    p.scale_log2 = float(double(scale) * 1.4426950408889634);
    p.num_seqs = num_seqs;
    p.q_len = q_len;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.rows = group * q_len;
    p.block_size = block_size;
    p.block_shift = (block_size & (block_size - 1)) == 0 ? __builtin_ctz(unsigned(block_size)) : -1;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.sorted = num_seqs > 1 && num_seqs <= kMultiSortMax;
    return PF_OK;
}

extern "C" pf_status pf_paged_attention_multi_query(const void* q, const void* k_cache, const void* v_cache,
                                                    const int32_t* block_tables, const int32_t* context_lens,
                                                    int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                                    int head_dim, int block_size, int max_blocks_per_seq,
                                                    int64_t num_blocks, float scale, float* out,
                                                    pf_stream_t stream) {
    CUtensorMap mk, mv;
    MultiParams p;
    const pf_status st = multi_query_setup(q, k_cache, v_cache, block_tables, context_lens, num_seqs, q_len,
                                           num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                           num_blocks, scale, out, &mk, &mv, &p);
    if (st != PF_OK || num_seqs == 0) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const long long cache_rows = num_blocks * num_kv_heads * (long long)block_size;
    if (p.rows >= kChunkMinRows && head_dim == 128 && kVBlockCopies &&
        !encode_cache_map_vblocks(&mv, v_cache, cache_rows))
        return PF_ERR_CUDA;  // the prompt-chunk kernel reads V by whole blocks
    cudaError_t e;
    if (p.rows >= kChunkMinRows)
        e = launch_chunk(mk, mv, p, head_dim, s);  // prompt chunks: query rows on the tcgen05 M side
    else if (head_dim == 64)
        e = launch_multi_any<64>(mk, mv, p, s);
    else if (p.rows <= 32)
        e = launch_multi_any<128>(mk, mv, p, s);
    else
        e = launch_multi_tc(mk, mv, p, s);  // 33 to 64 rows at D = 128: the tcgen05 kernel
    return e == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

extern "C" pf_status pf_paged_attention_multi_query_tcgen05(const void* q, const void* k_cache, const void* v_cache,
                                                            const int32_t* block_tables, const int32_t* context_lens,
                                                            int num_seqs, int q_len, int num_q_heads,
                                                            int num_kv_heads, int head_dim, int block_size,
                                                            int max_blocks_per_seq, int64_t num_blocks, float scale,
                                                            float* out, pf_stream_t stream) {
    CUtensorMap mk, mv;
    MultiParams p;
    const pf_status st = multi_query_setup(q, k_cache, v_cache, block_tables, context_lens, num_seqs, q_len,
                                           num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                           num_blocks, scale, out, &mk, &mv, &p);
    if (st != PF_OK) return st;
    if (head_dim != 128) return PF_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PF_OK;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const long long cache_rows = num_blocks * num_kv_heads * (long long)block_size;
    if (p.rows >= kChunkMinRows && kVBlockCopies && !encode_cache_map_vblocks(&mv, v_cache, cache_rows))
        return PF_ERR_CUDA;  // the prompt-chunk kernel reads V by whole blocks
    const cudaError_t e = p.rows >= kChunkMinRows ? launch_chunk(mk, mv, p, head_dim, s) : launch_multi_tc(mk, mv, p, s);
    return e == cudaSuccess ? PF_OK : PF_ERR_CUDA;
}

// Persistent partition pass of the split over context partitions.
//
// The partition pass has many short work units -- (sequence, partition, kv head),
// e.g. 2,072 units of 512 tokens for one 131072-token sequence and three short
// ones -- and a kernel with one CTA per unit pays each CTA's start-up (lengths,
// table entries, first tiles: a few microseconds) over and over.  Here a grid of
// resident CTAs walks the units round-robin (CTA c takes units c, c + grid, ...),
// and each warp's copy ring runs on across unit boundaries: lane 0 keeps a
// look-ahead cursor over the warp's future (unit, tile) positions and a small
// FIFO of their table entries, so the next unit's tiles are already in flight
// while the current one finishes.  Each unit ends with the CTA merging its warps'
// (m, l, acc) in a dedicated shared-memory area and writing the partial.
#pragma once

#include "pf_decode.cuh"

namespace pf {

template <int D, int G, int NW, int NST>
struct PersistentLayout {
    using Geo = DecodeGeometry<D, G>;
    static constexpr size_t STAGES = size_t(NW) * NST * 2 * Geo::TILE_BYTES;
    static constexpr size_t PSM = STAGES;                                           // [NW][PSM_PAD]
    static constexpr size_t MACC = PSM + size_t(NW) * Geo::PSM_PAD * 4;             // [NW][G][D]
    static constexpr size_t MML = MACC + size_t(NW) * G * D * 4;                    // [NW][2G]
    static constexpr size_t BAD = MML + (size_t(NW) * 2 * G * 4 + 15) / 16 * 16;    // [NW][NST] stage flags
    static constexpr size_t BARS = BAD + (size_t(NW) * NST * 4 + 15) / 16 * 16;     // [NW][NST] mbarriers
    static constexpr size_t KEYS = BARS + (size_t(NW) * NST * 8 + 15) / 16 * 16;    // prefix, round_up(S,4)
    static size_t bytes(int num_seqs) { return KEYS + size_t((num_seqs + 3) & ~3) * 4; }
    static constexpr size_t max_bytes() { return KEYS + size_t(kMaxSortedSeqsPartition) * 4; }
};

// Inclusive prefix over sequences of their non-empty partition counts, into
// keys[0..S); lengths outside [0, max_context_len] count as 0 (the merge NaN-fills
// those rows) and CTA 0 flags them.  Returns the number of (sequence, partition) pairs.
template <int NW>
__device__ __forceinline__ int partition_prefix(const DecodeParams& p, int* keys) {
    __shared__ int s_warp_sum[NW];
    constexpr int NT = NW * 32;
    const int S = p.num_seqs, P = p.partition_size;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    bool bad = false;
    for (int i = tid; i < S; i += NT) {
        const int Li = __ldg(p.context_lens + i);
        const bool b = Li < 0 || Li > p.max_context_len;
        bad = bad || b;
        keys[i] = b ? 0 : (Li + P - 1) / P;
    }
    if (bad && blockIdx.x == 0) set_error(p.err, ERR_BOUNDS);
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
    return keys[S - 1];
}

// A unit and this warp's share of its tiles.
struct PartUnit {
    int seq, kvh, part;
    int t0, t1;       // token range
    int nkw;          // this warp's tiles: t0/16 + warp + NW*i, i < nkw
    bool bad;         // context length beyond the table: NaN partial
    const int32_t* trow;
};

template <int NW>
__device__ __forceinline__ PartUnit decode_unit(const DecodeParams& p, const int* keys, int u, int warp) {
    PartUnit x;
    const int pair = u / p.num_kv_heads;
    x.kvh = u - pair * p.num_kv_heads;
    int lo = 0, hi = p.num_seqs - 1;  // first sequence whose inclusive prefix exceeds pair
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (keys[mid] > pair) hi = mid; else lo = mid + 1;
    }
    x.seq = lo;
    x.part = pair - (lo > 0 ? keys[lo - 1] : 0);
    const int L = __ldg(p.context_lens + x.seq);
    x.bad = (long long)L > (long long)p.max_blocks_per_seq * p.block_size;
    x.t0 = x.part * p.partition_size;
    x.t1 = min(L, x.t0 + p.partition_size);
    const int ntiles = x.bad ? 0 : (x.t1 - x.t0 + kTileTokens - 1) / kTileTokens;
    x.nkw = ntiles > warp ? (ntiles - warp + NW - 1) / NW : 0;
    x.trow = p.block_tables + size_t(x.seq) * p.max_blocks_per_seq;
    return x;
}

template <int D, int G, int NW, int NST>
__global__ void __launch_bounds__(NW * 32) paged_partition_persistent_kernel(const DecodeParams p) {
    using Geo = DecodeGeometry<D, G>;
    using Lay = PersistentLayout<D, G, NW, NST>;
    constexpr int TT = Geo::TT, ROW = Geo::ROW_BYTES, TILE = Geo::TILE_BYTES, PSM_PAD = Geo::PSM_PAD;
    constexpr int R = NST + 2;  // look-ahead depth of lane 0's table FIFO

    extern __shared__ __align__(128) unsigned char smem[];
    float* psm_all = reinterpret_cast<float*>(smem + Lay::PSM);
    float* macc = reinterpret_cast<float*>(smem + Lay::MACC);
    float* mml = reinterpret_cast<float*>(smem + Lay::MML);
    int* stage_bad = reinterpret_cast<int*>(smem + Lay::BAD);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::BARS);
    int* keys = reinterpret_cast<int*>(smem + Lay::KEYS);

    // The merge that follows may be scheduled as SMs drain; it waits for this grid to complete.
    asm volatile("griddepcontrol.launch_dependents;");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = p.num_q_heads, Hkv = p.num_kv_heads;
    const int U = partition_prefix<NW>(p, keys) * Hkv;
    if (int(blockIdx.x) >= U) return;

    unsigned char* my_stages = smem + size_t(warp) * NST * 2 * TILE;
    const uint32_t stage0 = smem_u32(my_stages);
    const uint32_t bar0 = smem_u32(bars + warp * NST);
    int* my_bad = stage_bad + warp * NST;
    float* psm = psm_all + warp * PSM_PAD;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < NST; ++s) mbar_init(bar0 + 8 * s, 1);
        mbar_init_fence();
    }
    __syncwarp();

    const int bs = p.block_size, bshift = p.block_shift;
    auto block_index = [&](int tok) { return bshift >= 0 ? (tok >> bshift) : (tok / bs); };
    auto block_offset = [&](int tok) { return bshift >= 0 ? (tok & (bs - 1)) : (tok % bs); };
    const uint64_t policy = l2_policy_evict_first();

    // ---- lane 0: look-ahead cursor over (unit, tile) and a FIFO of the next R positions
    int look_j = 0, look_i = 0;
    PartUnit look{};
    bool look_done = false;
    auto look_unit = [&]() {  // settle on the first unit (from look_j on) where this warp has tiles
        for (;;) {
            const int u = int(blockIdx.x) + look_j * int(gridDim.x);
            if (u >= U) { look_done = true; return; }
            look = decode_unit<NW>(p, keys, u, warp);
            if (look.nkw > 0) { look_i = 0; return; }
            ++look_j;
        }
    };
    int f_pb[R], f_row[R], f_n[R];  // FIFO: table entry, first cache row of the tile (kvh, offset), rows
    auto push_back = [&](int slot) {
        if (look_done) { f_n[slot] = 0; return; }
        const int tok = look.t0 + (warp + NW * look_i) * TT;
        f_pb[slot] = __ldg(look.trow + block_index(tok));
        f_row[slot] = look.kvh * bs + block_offset(tok);  // + pb * Hkv * bs once the entry is in
        f_n[slot] = min(TT, look.t1 - tok);
        if (++look_i >= look.nkw) { ++look_j; look_unit(); }
    };
    int n_issued = 0;
    auto issue_front = [&]() {  // copy the FIFO's front position into the next stage, refill the FIFO
        const int s = n_issued % NST;
        const uint32_t bar = bar0 + 8 * s;
        if (f_n[0] > 0) {
            const int pb = f_pb[0];
            if (pb >= 0 && (long long)pb < p.num_blocks) {
                const uint32_t bytes = uint32_t(f_n[0]) * ROW;
                const size_t row = size_t(pb) * Hkv * bs + size_t(f_row[0]);
                const uint32_t dst = stage0 + uint32_t(s) * 2 * TILE;
                my_bad[s] = 0;
                mbar_arrive_expect_tx(bar, 2 * bytes);
                bulk_copy_g2s(dst, p.k_cache + row * D, bytes, bar, policy);
                bulk_copy_g2s(dst + TILE, p.v_cache + row * D, bytes, bar, policy);
            } else {
                my_bad[s] = 1;  // no copy: the unit's partial ends up NaN
                set_error(p.err, ERR_BOUNDS);
                mbar_arrive(bar);
            }
            ++n_issued;
        }
#pragma unroll
        for (int k = 0; k < R - 1; ++k) {
            f_pb[k] = f_pb[k + 1];
            f_row[k] = f_row[k + 1];
            f_n[k] = f_n[k + 1];
        }
        push_back(R - 1);
    };
    if (lane == 0) {
        look_unit();
#pragma unroll
        for (int k = 0; k < R; ++k) push_back(k);
#pragma unroll
        for (int k = 0; k < NST; ++k) issue_front();
    }

    // ---- consumer: the same positions, unit by unit
    WarpAttention<D, G> wa;
    wa.init(lane);
    __shared__ int unit_failed[NW];
    int n = 0;             // positions consumed: stage n % NST, phase (n / NST) & 1
    bool dead = false;     // a wait gave up: consume nothing more, keep the CTA's barriers
    int q_seq = -1, q_kvh = -1;
    for (int j = 0;; ++j) {
        const int u = int(blockIdx.x) + j * int(gridDim.x);
        if (u >= U) break;
        const PartUnit x = decode_unit<NW>(p, keys, u, warp);
        if (x.seq != q_seq || x.kvh != q_kvh) {
            wa.load_q(p.q + (size_t(x.seq) * Hq + x.kvh * G) * D);
            q_seq = x.seq;
            q_kvh = x.kvh;
        }
        wa.reset();
        bool failed = x.bad || dead;
        for (int i = 0; i < x.nkw && !dead; ++i) {
            const int s = n % NST;
            const bool ok = mbar_wait_bounded(bar0 + 8 * s, (n / NST) & 1, p.wait_limit_ns);
            if (__any_sync(FULL_MASK, !ok)) {
                dead = true;
                failed = true;
                if (lane == 0) set_error(p.err, ERR_TIMEOUT);
                break;
            }
            if (my_bad[s]) failed = true;
            const unsigned char* Ks = my_stages + size_t(s) * 2 * TILE;
            const int tok = x.t0 + (warp + NW * i) * TT;
            wa.tile(Ks, Ks + TILE, min(TT, x.t1 - tok), psm, p.scale_log2);
            ++n;
            if (lane == 0) issue_front();
        }
        wa.stash(mml + warp * 2 * G, macc + warp * G * D);
        if (lane == 0) unit_failed[warp] = failed ? 1 : 0;
        __syncthreads();
        bool any_failed = false;
#pragma unroll
        for (int w = 0; w < NW; ++w) any_failed = any_failed || unit_failed[w] != 0;
        if (x.bad && threadIdx.x == 0) set_error(p.err, ERR_BOUNDS);
        const size_t slot0 = (size_t(x.seq) * Hq + x.kvh * G) * p.num_partitions + x.part;
        merge_warps_and_store<D, G, NW>([&](int w) { return mml + w * 2 * G; },
                                        [&](int w) { return (const float*)(macc + w * G * D); }, any_failed,
                                        p.out + slot0 * D, p.part_m + slot0, p.part_l + slot0,
                                        size_t(p.num_partitions));
        __syncthreads();
    }
    if (lane == 0) {
        // no copy may still be landing when the CTA exits (only after a wait gave up)
        for (int k = n; k < n_issued; ++k) mbar_wait_bounded(bar0 + 8 * (k % NST), (k / NST) & 1, p.wait_limit_ns);
    }
    __syncwarp();
}

}  // namespace pf

namespace pf {

template <int D, int G, int NW, int NST>
cudaError_t launch_partition_persistent(const DecodeParams& p, cudaStream_t stream) {
    using Lay = PersistentLayout<D, G, NW, NST>;
    auto kern = paged_partition_persistent_kernel<D, G, NW, NST>;
    static std::atomic<unsigned long long> configured{0};  // one bit per device ordinal
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Lay::max_bytes()));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    const size_t smem = Lay::bytes(p.num_seqs);
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem);
    if (e != cudaSuccess) return e;
    e = sm_count(&sms);
    if (e != cudaSuccess) return e;
    const long long upper = (long long)p.num_partitions * p.num_kv_heads * p.num_seqs;  // units can't exceed it
    long long grid = (long long)sms * (per_sm > 0 ? per_sm : 1);
    if (grid > upper) grid = upper;
    if (grid <= 0) return cudaSuccess;
    kern<<<unsigned(grid), NW * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int D, int G, int NW, int NST>
cudaError_t launch_decode_mode(const DecodeParams& p, int mode, cudaStream_t stream) {
    switch (mode) {
        case MODE_DECODE: return launch_decode_variant<D, G, NW, NST, MODE_DECODE>(p, stream);
        case MODE_PARTITION:
            // the persistent pass needs the flattened (sorted) unit order
            return p.order_mode == ORDER_SORTED ? launch_partition_persistent<D, G, NW, NST>(p, stream)
                                                : launch_decode_variant<D, G, NW, NST, MODE_PARTITION>(p, stream);
        case MODE_DECODE_APPEND: return launch_decode_variant<D, G, NW, NST, MODE_DECODE_APPEND>(p, stream);
        case MODE_CLUSTER: return launch_decode_cluster<D, G, NW, NST>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D, int NW, int NST>
cudaError_t launch_decode_for_dim(const DecodeParams& p, int group, int mode, cudaStream_t stream) {
    switch (group) {
        case 1: return launch_decode_mode<D, 1, NW, NST>(p, mode, stream);
        case 2: return launch_decode_mode<D, 2, NW, NST>(p, mode, stream);
        case 4: return launch_decode_mode<D, 4, NW, NST>(p, mode, stream);
        case 8: return launch_decode_mode<D, 8, NW, NST>(p, mode, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pf

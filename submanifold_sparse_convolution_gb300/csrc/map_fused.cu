// The whole kernel-map build in one launch: a single thread-block cluster
// (up to 16 CTAs x 1024 threads) runs every phase -- key packing, the
// coordinate sort, neighbour search (or the dense presence grid), masks,
// the mask sort and the compaction -- separated by hardware cluster barriers
// instead of kernel boundaries.  For the voxel counts of one or a few LiDAR
// frames (10^3..10^6 rows) the build is latency-bound: the pages measured
// their compaction dominated by launch and synchronisation glue rather than
// data movement (FlyDSL PR #942, "move pair compaction from torch onto three
// fx kernels": a single read of the LUT takes 25 us of 120 us).  Here the
// phases exchange data through global memory (L2-resident at these sizes)
// with cluster-scope release/acquire barriers, and the per-CTA radix
// histograms of the next pass are accumulated during the scatter of the
// current one, so each sort pass costs one barrier.
//
// Results are bit-identical to the multi-kernel pipeline in map.cu: the
// same packed keys, the same stable order (ties by row), the same outputs.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "map_internal.cuh"

namespace spconv {
namespace {

constexpr int FT = 1024;          // threads per CTA
constexpr int FW = FT / 32;       // warps per CTA
constexpr int IPT = 4;            // items per thread per ranking round
constexpr int RS = FT * IPT;      // elements per ranking round
constexpr int kDigitMax = 10;                 // widest radix digit (bits)
constexpr int BINS = 1 << kDigitMax;          // histogram capacity per CTA and pass
static_assert(BINS == kFusedBins, "host and kernel agree on the histogram width");
constexpr int kMaxCluster = 16;
constexpr int kTilesPerRound = FW / 4;   // 4 warps (128 rows) per tile
// Launch parts: the coordinate sort, then (after the whole-GPU neighbour
// search) masks, mask sort and compaction.  The dense-grid mapper runs
// everything in the second part.
constexpr int kPartSort = 0;
constexpr int kPartRest = 1;
static_assert(FT == BINS && FW == 32, "one thread per digit value, 32 warps per CTA");

struct FusedSmem {
    uint16_t cnt[FW][BINS];        // ranking: per (warp, digit) counts of a round, then offsets
    int32_t base[BINS];
    int32_t run[BINS];
    int32_t scan[BINS];
    int32_t pre[BINS];
    int32_t rtot[BINS];
    int32_t tmp[FW];
    int32_t tap_pos[kTaps];
    int32_t tap_base[kTaps];
    int32_t bkt_base[kTaps + 1];
    int32_t qcnt[kTilesPerRound][4][kTaps];
    int32_t ctot[kMaxCluster * kTaps];             // every CTA's tap totals
    int32_t ctab[kMaxCluster * (kTaps + 1)];       // every CTA's bucket counts
    int32_t taps[kTaps];                           // this CTA's tap counts (then the global ones)
    int32_t err;
};

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scan of a[0..count) in place, count <= FT (all threads call).
__device__ void block_scan(int32_t* a, int count, int32_t* tmp) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int32_t v = t < count ? a[t] : 0;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) tmp[w] = incl;
    __syncthreads();
    if (w == 0) {
        const int32_t x = tmp[lane];
        int32_t y = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t z = __shfl_up_sync(0xFFFFFFFFu, y, o);
            if (lane >= o) y += z;
        }
        tmp[lane] = y - x;     // exclusive prefix of the warp totals
    }
    __syncthreads();
    if (t < count) a[t] = tmp[w] + incl - v;
    __syncthreads();
}

// One stable LSD pass over this CTA's part [c*chunk, min(n, (c+1)*chunk)) of
// `in`, by the digit of `width` bits at `shift`.  hc: every CTA's digit counts
// of its part ([C][BINS]).  When hn != nullptr the counts of the next digit
// (next_width bits at next_shift) of every element are accumulated into hn by
// the CTA whose part the element lands in.
__device__ void radix_pass(const uint64_t* __restrict__ in, uint64_t* __restrict__ out, int64_t n,
                           int64_t chunk, int C, int c, int shift, int width, const int32_t* hc,
                           int32_t* hn, int next_shift, int next_width, FusedSmem& sm) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int bins = 1 << width;
    const uint64_t dmask = static_cast<uint64_t>(bins - 1);
    const uint64_t nmask = (uint64_t(1) << next_width) - 1;
    const int64_t lo = static_cast<int64_t>(c) * chunk;
    const int64_t hi = lo + chunk < n ? lo + chunk : n;
    // A round is RS consecutive elements; warp w owns the 32*IPT of them
    // starting at w*32*IPT (item j of lane l at w*32*IPT + 32*j + l), so the
    // stable order inside a round is (warp, item, lane).
    uint64_t v[IPT];
    auto load_round = [&](int64_t r0) {
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const int64_t idx = r0 + static_cast<int64_t>(w) * 32 * IPT + 32 * j + lane;
            v[j] = idx < hi ? __ldcg(in + idx) : 0ull;
        }
    };
    // the first round's keys are requested before the counts are read, so the two waits overlap
    load_round(lo);
    if (t < bins) {
        int32_t h[kMaxCluster];
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q) h[q] = q < C ? __ldcg(hc + q * BINS + t) : 0;   // loads in flight together
        int32_t tot = 0, pre = 0;
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q) {
            tot += h[q];
            pre += q < c ? h[q] : 0;
        }
        sm.scan[t] = tot;
        sm.pre[t] = pre;
        sm.run[t] = 0;
    }
    __syncthreads();
    block_scan(sm.scan, bins, sm.tmp);
    if (t < bins) sm.base[t] = sm.scan[t] + sm.pre[t];
    const uint32_t lt = lanemask_lt();
    for (int64_t r0 = lo; r0 < hi; r0 += RS) {
        if (r0 != lo) load_round(r0);
        uint32_t* cz = reinterpret_cast<uint32_t*>(&sm.cnt[0][0]);
        for (int i = t; i < FW * BINS / 2; i += FT) cz[i] = 0;
        __syncthreads();
        int d[IPT], rk[IPT];
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const int64_t idx = r0 + static_cast<int64_t>(w) * 32 * IPT + 32 * j + lane;
            const bool valid = idx < hi;
            d[j] = valid ? static_cast<int>((v[j] >> shift) & dmask) : BINS;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d[j]);
            const int prior = valid ? sm.cnt[w][d[j]] : 0;
            rk[j] = prior + __popc(peers & lt);
            __syncwarp();
            if (valid && lane == __ffs(peers) - 1) sm.cnt[w][d[j]] = static_cast<uint16_t>(prior + __popc(peers));
            __syncwarp();
        }
        __syncthreads();
        if (t < bins) {   // exclusive prefix over the warps, per digit (loads batched ahead of the stores)
            int32_t pre = 0;
#pragma unroll
            for (int q0 = 0; q0 < FW; q0 += 16) {
                int32_t x[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) x[q] = sm.cnt[q0 + q][t];
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    sm.cnt[q0 + q][t] = static_cast<uint16_t>(pre);
                    pre += x[q];
                }
            }
            sm.rtot[t] = pre;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const bool valid = d[j] < BINS;
            int64_t dst = 0;
            bool ok = false;
            if (valid) {
                dst = static_cast<int64_t>(sm.base[d[j]]) + sm.run[d[j]] + sm.cnt[w][d[j]] + rk[j];
                ok = dst >= 0 && dst < n;
                if (ok)
                    out[dst] = v[j];
                else
                    atomicOr(&sm.err, kStatusInternal);
            }
            if (hn != nullptr) {
                const int dc = ok ? static_cast<int>(dst / chunk) : 0;
                const int key2 = ok ? dc * BINS + static_cast<int>((v[j] >> next_shift) & nmask) : -1;
                const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key2);
                if (ok && lane == __ffs(peers) - 1) atomicAdd(hn + key2, __popc(peers));
            }
        }
        __syncthreads();
        if (t < bins) sm.run[t] += sm.rtot[t];
    }
    __syncthreads();
}

// Adds this warp's tap counts to the CTA's shared counters.
__device__ __forceinline__ void add_tap_counts(uint32_t m, int32_t* cta_taps) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
        if (lane == 0 && b) atomicAdd(cta_taps + k, __popc(b));
    }
}

__device__ __forceinline__ void store_row(int32_t* __restrict__ nbr, int64_t r, const int32_t (&v)[kNbrStride]) {
    int4* dst = reinterpret_cast<int4*>(nbr + r * kNbrStride);
#pragma unroll
    for (int q = 0; q < kNbrStride / 4; ++q) dst[q] = make_int4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

__global__ void __launch_bounds__(FT, 1) k_map_fused(const FusedArgs a, int part) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    FusedSmem& sm = *reinterpret_cast<FusedSmem*>(smem_raw);
    const int C = static_cast<int>(gridDim.x);
    const int c = static_cast<int>(blockIdx.x);
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int64_t n = a.n;
    const int64_t chunk = (n + C - 1) / C;
    const int64_t lo = static_cast<int64_t>(c) * chunk;
    const int64_t hi = lo + chunk < n ? lo + chunk : n;
    const int rb = a.row_bits;
    const uint64_t rmask = (uint64_t(1) << rb) - 1;
    int32_t* H[3] = {a.hist, a.hist + C * BINS, a.hist + 2 * C * BINS};
    // digit widths: the fewest passes of at most kDigitMax bits
    const int key_passes = (a.key_bits + kDigitMax - 1) / kDigitMax;
    const int key_w = (a.key_bits + key_passes - 1) / key_passes;
    constexpr int kMaskPasses = (kTaps + kDigitMax - 1) / kDigitMax;
    constexpr int kMaskW = (kTaps + kMaskPasses - 1) / kMaskPasses;
    if (t == 0) sm.err = 0;
    if (t < kTaps) sm.taps[t] = 0;
    if (part == kPartRest) pdl_wait();   // launched early: the neighbour search must have finished

    // ---------------- phase 0: reset counters, pack keys / clear the grid
    const bool starts = part == kPartSort || a.mapper == SPCONV_MAPPER_DENSE;
    if (starts && c == 0 && t < kTaps) a.tap_count[t] = 0;
    if (starts && c == 0 && t == 0) {
        *a.status = 0;
        a.totals[0] = 0;
        a.totals[1] = 0;
    }
    H[1][c * BINS + t] = 0;
    H[2][c * BINS + t] = 0;
    __syncthreads();
    if (part == kPartSort) {
        // packed keys, and the first digit's counts of this CTA's part
        const uint64_t invalid = ((uint64_t(1) << a.key_bits) - 1) << rb;
        const uint64_t dmask0 = (uint64_t(1) << key_w) - 1;
        sm.scan[t] = 0;
        __syncthreads();
        for (int64_t i0 = lo; i0 < hi; i0 += FT) {
            const int64_t i = i0 + t;
            int dg = BINS;
            if (i < hi) {
                const int4 q = a.coords[i];
                uint64_t key = invalid;
                if (q.x >= 0 && q.x < a.batch && q.y >= 0 && q.y < a.shape.x && q.z >= 0 && q.z < a.shape.y &&
                    q.w >= 0 && q.w < a.shape.z) {
                    key = (((((static_cast<uint64_t>(q.x) << a.wx) | static_cast<uint64_t>(q.y + 1)) << a.wy) |
                            static_cast<uint64_t>(q.z + 1))
                           << a.wz |
                           static_cast<uint64_t>(q.w + 1))
                          << rb;
                } else {
                    atomicOr(&sm.err, kStatusRange);
                }
                a.va[i] = key | static_cast<uint64_t>(i);
                dg = static_cast<int>((key >> rb) & dmask0);
            }
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, dg);
            if (dg < BINS && lane == __ffs(peers) - 1) atomicAdd(&sm.scan[dg], __popc(peers));
        }
        __syncthreads();
        H[0][c * BINS + t] = sm.scan[t];
    } else if (a.mapper == SPCONV_MAPPER_DENSE) {
        const int64_t per = (a.cells + C - 1) / C;
        const int64_t g0 = static_cast<int64_t>(c) * per;
        const int64_t g1 = g0 + per < a.cells ? g0 + per : a.cells;
        for (int64_t i = g0 + t; i < g1; i += FT) a.grid[i] = -1;
    }
    cluster_sync_all();

    if (part == kPartSort) {
        // ---------------- coordinate sort: one barrier per pass
        for (int p = 0; p < key_passes; ++p) {
            const uint64_t* in = (p & 1) ? a.vb : a.va;
            uint64_t* out = (p & 1) ? a.va : a.vb;
            H[(p + 2) % 3][c * BINS + t] = 0;
            radix_pass(in, out, n, chunk, C, c, rb + key_w * p, key_w, H[p % 3],
                       p + 1 < key_passes ? H[(p + 1) % 3] : nullptr, rb + key_w * (p + 1), key_w, sm);
            cluster_sync_all();
        }
        if (t == 0 && sm.err) atomicOr(a.status, sm.err);
        pdl_trigger();
        return;   // the neighbour search runs next on the whole GPU (k_search_window)
    } else if (a.mapper == SPCONV_MAPPER_DENSE) {
        // ---------------- dense grid: scatter row ids, then 27 lookups per row
        for (int64_t i = lo + t; i < hi; i += FT) {
            const int4 q = a.coords[i];
            if (q.x >= 0 && q.x < a.batch && q.y >= 0 && q.y < a.shape.x && q.z >= 0 && q.z < a.shape.y &&
                q.w >= 0 && q.w < a.shape.z) {
                const int64_t cell = q.x * a.gsb + static_cast<int64_t>(q.y + 1) * a.gsx +
                                     static_cast<int64_t>(q.z + 1) * a.gsy + (q.w + 1);
                if (atomicCAS(a.grid + cell, -1, static_cast<int32_t>(i)) != -1) atomicOr(&sm.err, kStatusDuplicate);
            } else {
                atomicOr(&sm.err, kStatusRange);
            }
        }
        cluster_sync_all();
        for (int64_t i0 = lo; i0 < hi; i0 += FT) {
            const int64_t i = i0 + t;
            uint32_t m = 0;
            if (i < hi) {
                const int4 q = a.coords[i];
                int32_t v[kNbrStride];
#pragma unroll
                for (int k = 0; k < kNbrStride; ++k) v[k] = -1;
                if (q.x >= 0 && q.x < a.batch && q.y >= 0 && q.y < a.shape.x && q.z >= 0 && q.z < a.shape.y &&
                    q.w >= 0 && q.w < a.shape.z) {
                    const int64_t cell = q.x * a.gsb + static_cast<int64_t>(q.y + 1) * a.gsx +
                                         static_cast<int64_t>(q.z + 1) * a.gsy + (q.w + 1);
#pragma unroll
                    for (int k = 0; k < kTaps; ++k) {
                        v[k] = __ldcg(a.grid + cell + a.goff[k]);
                        m |= (v[k] >= 0 ? 1u : 0u) << k;
                    }
                }
                store_row(a.nbr, i, v);
                a.mask[i] = m;
            }
            add_tap_counts(m, sm.taps);
        }
    }
    __syncthreads();
    if (t < kTaps && sm.taps[t]) atomicAdd(a.tap_count + t, sm.taps[t]);
    if (a.mapper == SPCONV_MAPPER_DENSE) cluster_sync_all();

    // ---------------- mask sort keys (tap order from the counts) + first histogram
    if (t < kTaps) sm.taps[t] = __ldcg(a.tap_count + t);
    __syncthreads();
    if (t < kTaps) {
        int32_t rank = t;
        if (a.calibrated) {
            const int32_t ck = sm.taps[t];
            rank = 0;
            for (int j = 0; j < kTaps; ++j) {
                const int32_t cj = sm.taps[j];
                rank += (cj > ck || (cj == ck && j < t)) ? 1 : 0;
            }
        }
        sm.tap_pos[t] = rank;
    }
    H[1][c * BINS + t] = 0;
    H[2][c * BINS + t] = 0;
    __syncthreads();
    sm.scan[t] = 0;
    __syncthreads();
    for (int64_t i0 = lo; i0 < hi; i0 += FT) {   // keys and their first-digit histogram in one pass
        const int64_t i = i0 + t;
        int dg = BINS;
        if (i < hi) {
            const uint32_t m = __ldcg(a.mask + i);
            uint32_t key = 0;
#pragma unroll
            for (int k = 0; k < kTaps; ++k) key |= ((m >> k) & 1u) << sm.tap_pos[k];
            a.va[i] = (static_cast<uint64_t>(key) << rb) | static_cast<uint64_t>(i);
            dg = static_cast<int>(key & ((1u << kMaskW) - 1));
        }
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, dg);
        if (dg < BINS && lane == __ffs(peers) - 1) atomicAdd(&sm.scan[dg], __popc(peers));
    }
    __syncthreads();
    H[0][c * BINS + t] = sm.scan[t];
    cluster_sync_all();
    for (int p = 0; p < kMaskPasses; ++p) {
        const uint64_t* in = (p & 1) ? a.vb : a.va;
        uint64_t* out = (p & 1) ? a.va : a.vb;
        H[(p + 2) % 3][c * BINS + t] = 0;
        radix_pass(in, out, n, chunk, C, c, rb + kMaskW * p, kMaskW, H[p % 3],
                   p + 1 < kMaskPasses ? H[(p + 1) % 3] : nullptr, rb + kMaskW * (p + 1), kMaskW, sm);
        cluster_sync_all();
    }
    const uint64_t* ms = (kMaskPasses & 1) ? a.vb : a.va;   // where the last pass left the pairs

    // ---------------- compaction, count: per tile and tap, CTA totals, bucket counts
    const int64_t T = a.n_tiles;
    const int64_t tpc = (T + C - 1) / C;
    const int64_t ta = static_cast<int64_t>(c) * tpc;
    const int64_t tb = ta + tpc < T ? ta + tpc : T;
    const int nt = static_cast<int>(tb > ta ? tb - ta : 0);
    int32_t* tcnt = reinterpret_cast<int32_t*>(smem_raw + sizeof(FusedSmem));   // [nt][27]
    int32_t* tbkt = tcnt + static_cast<int64_t>(nt) * kTaps;                    // [nt]
    uint32_t* tuni = reinterpret_cast<uint32_t*>(tbkt + nt);                     // [nt]
    for (int i = t; i < nt * kTaps; i += FT) tcnt[i] = 0;
    if (t <= kTaps) sm.scan[t] = 0;   // bucket counts of this CTA's tiles
    __syncthreads();
    for (int tr = 0; tr < nt; tr += kTilesPerRound) {
        const int tl = tr + (w >> 2);
        const int64_t s = (ta + tl) * kTileRows + (w & 3) * 32 + lane;
        uint32_t m = 0;
        if (tl < nt && s < n) {
            const int64_t r = static_cast<int64_t>(__ldcg(ms + s) & rmask);
            if (r < n)
                m = __ldcg(a.mask + r);
            else
                atomicOr(&sm.err, kStatusInternal);
        }
        if (tl < nt) {
#pragma unroll
            for (int k = 0; k < kTaps; ++k) {
                const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
                if (lane == 0 && b) atomicAdd(&tcnt[tl * kTaps + k], __popc(b));
            }
        }
    }
    __syncthreads();
    for (int i = t; i < nt; i += FT) {
        uint32_t uni = 0;
        for (int k = 0; k < kTaps; ++k) uni |= (tcnt[i * kTaps + k] > 0 ? 1u : 0u) << k;
        const int u = __popc(uni);
        tuni[i] = uni;
        tbkt[i] = kTaps - u;
        atomicAdd(&sm.scan[kTaps - u], 1);
    }
    __syncthreads();
    if (t <= kTaps) a.cta_bkt[c * (kTaps + 1) + t] = sm.scan[t];
    // per tap (one warp each): CTA total, then exclusive prefix over this CTA's tiles in place
    if (w < kTaps) {
        int32_t run = 0;
        for (int i0 = 0; i0 < nt; i0 += 32) {
            const int i = i0 + lane;
            const int32_t x = i < nt ? tcnt[i * kTaps + w] : 0;
            int32_t incl = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            if (i < nt) tcnt[i * kTaps + w] = run + incl - x;
            run += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) a.cta_tot[c * kTaps + w] = run;
    }
    cluster_sync_all();

    // ---------------- compaction, write
    for (int i = t; i < C * kTaps; i += FT) sm.ctot[i] = __ldcg(a.cta_tot + i);
    for (int i = t; i < C * (kTaps + 1); i += FT) sm.ctab[i] = __ldcg(a.cta_bkt + i);
    __syncthreads();
    // per tap: total over all CTAs and this CTA's offset among them; per
    // bucket likewise (one thread each, C steps), then short scans
    if (t < kTaps) {
        int32_t all_k = 0, mine = 0;
        for (int q = 0; q < C; ++q) {
            const int32_t x = sm.ctot[q * kTaps + t];
            all_k += x;
            if (q < c) mine += x;
        }
        sm.scan[t] = all_k;
        sm.pre[t] = mine;
    }
    if (t >= 32 && t < 32 + kTaps + 1) {
        const int b = t - 32;
        int32_t all_b = 0, mine = 0;
        for (int q = 0; q < C; ++q) {
            const int32_t x = sm.ctab[q * (kTaps + 1) + b];
            all_b += x;
            if (q < c) mine += x;
        }
        sm.scan[64 + b] = all_b;
        sm.pre[64 + b] = mine;
    }
    __syncthreads();
    if (w == 0) {   // exclusive scans over the 27 taps and over the 28 buckets
        const int32_t xt = lane < kTaps ? sm.scan[lane] : 0;
        const int32_t xb = lane <= kTaps ? sm.scan[64 + lane] : 0;
        int32_t it = xt, ib = xb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t yt = __shfl_up_sync(0xFFFFFFFFu, it, o);
            const int32_t yb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
            if (lane >= o) {
                it += yt;
                ib += yb;
            }
        }
        if (lane < kTaps) {
            sm.tap_base[lane] = it - xt + sm.pre[lane];
            if (c == 0) a.tap_off[lane] = it - xt;
        }
        if (lane == kTaps - 1 && c == 0) {
            a.tap_off[kTaps] = it;
            a.totals[0] = it;
        }
        if (lane <= kTaps) sm.bkt_base[lane] = ib - xb + sm.pre[64 + lane];
        // sum of union sizes over all tiles: bucket b holds tiles with 27 - b taps
        int32_t taps = lane <= kTaps ? (kTaps - lane) * xb : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) taps += __shfl_xor_sync(0xFFFFFFFFu, taps, o);
        if (lane == 0 && c == 0) a.totals[1] = taps;
    }
    __syncthreads();
    // tiles by descending union size, stable in the tile index
    for (int i = t; i < nt; i += FT) {
        const int b = tbkt[i];
        int32_t at = sm.bkt_base[b];
        for (int j = 0; j < i; ++j) at += tbkt[j] == b ? 1 : 0;
        if (at >= 0 && at < T)
            a.tile_order[at] = static_cast<int32_t>(ta + i);
        else
            atomicOr(&sm.err, kStatusInternal);
    }
    // offsets of every (tap, tile) pair run and the tile unions, for the
    // whole-GPU write kernel that follows (k_tile_write_packed)
    for (int i = t; i < nt * kTaps; i += FT) {
        const int tl = i / kTaps, k = i % kTaps;
        a.seg_off[static_cast<int64_t>(k) * T + ta + tl] = sm.tap_base[k] + tcnt[i];
    }
    for (int i = t; i < nt; i += FT) a.tile_union[ta + i] = tuni[i];
    if (t == 0 && sm.err) atomicOr(a.status, sm.err);
    pdl_trigger();
}

// One block of 128 threads per tile of the mask-sorted order: perm, the
// per-tap pair lists and the GEMM gather table.  Reads the sorted packed
// (mask key << rb | row) array, the masks, the kernel map and the (tap, tile)
// offsets published by the cluster part; only the taps of the tile's union
// get gather-table entries (the GEMM reads no others).
__global__ void __launch_bounds__(kTileRows) k_tile_write_packed(const FusedArgs a, const uint64_t* __restrict__ ms) {
    __shared__ int32_t wc[kTileRows / 32][kTaps];
    __shared__ int32_t seg[kTaps];   // the tile's first pair in every tap's list
    __shared__ int32_t err;
    const int64_t t = blockIdx.x;
    const int64_t T = a.n_tiles;
    const int64_t n = a.n;
    const int rb = a.row_bits;
    const uint64_t rmask = (uint64_t(1) << rb) - 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) err = 0;
    pdl_wait();   // the mask sort and the (tap, tile) offsets must be complete
    // read once here, not in the per-tap loop behind the pair stores
    if (threadIdx.x < kTaps) seg[threadIdx.x] = a.seg_off[static_cast<int64_t>(threadIdx.x) * T + t];
    const int64_t s = t * kTileRows + threadIdx.x;
    int32_t r = s < n ? static_cast<int32_t>(ms[s] & rmask) : -1;
    if (r >= n) {
        r = -1;
        atomicOr(&err, kStatusInternal);
    }
    const uint32_t m = r >= 0 ? a.mask[r] : 0u;
    const uint32_t uni = a.tile_union[t];
    int32_t v[kNbrStride];
    if (r >= 0) {
        const int4* src = reinterpret_cast<const int4*>(a.nbr + static_cast<int64_t>(r) * kNbrStride);
#pragma unroll
        for (int q = 0; q < kNbrStride / 4; ++q) {
            const int4 x = src[q];
            v[4 * q] = x.x;
            v[4 * q + 1] = x.y;
            v[4 * q + 2] = x.z;
            v[4 * q + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < kNbrStride; ++k) v[k] = -1;
    }
    uint32_t ball[kTaps];
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
        ball[k] = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
        if (lane == 0) wc[warp][k] = __popc(ball[k]);
    }
    __syncthreads();
    a.perm[s] = r;
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
        if (!((uni >> k) & 1u)) continue;
        const bool present = (m >> k) & 1u;
        if (present) {
            int64_t off = seg[k] + __popc(ball[k] & lt);
            for (int q = 0; q < warp; ++q) off += wc[q][k];
            if (off >= 0 && off < kTaps * n) {
                a.in_rows[off] = v[k];
                a.out_rows[off] = r;
            } else {
                atomicOr(&err, kStatusInternal);
            }
        }
        a.gtab[static_cast<int64_t>(k) * a.n_pad + s] = present ? v[k] : -1;
    }
    __syncthreads();
    if (threadIdx.x == 0 && err) atomicOr(a.status, err);
    pdl_trigger();
}

}  // namespace

// Tiles per CTA are bounded by kFusedMaxRows / kTileRows / (smallest cluster).
constexpr int kMinCluster = 16;
constexpr size_t kFusedSmem = sizeof(FusedSmem) +
    static_cast<size_t>(kFusedMaxRows / kTileRows / kMinCluster) * (kTaps + 2) * sizeof(int32_t);

int fused_cluster_size(cudaStream_t s) {
    static int cached = -1;
    if (cached >= 0) return cached;
    int result = 0;
    if (cudaFuncSetAttribute(k_map_fused, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kFusedSmem)) != cudaSuccess ||
        cudaFuncSetAttribute(k_map_fused, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        cached = 0;
        return 0;
    }
    for (int cs = kMaxCluster; cs >= kMinCluster; cs >>= 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs);
        cfg.blockDim = dim3(FT);
        cfg.dynamicSmemBytes = kFusedSmem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, k_map_fused, &cfg) == cudaSuccess && clusters > 0) {
            result = cs;
            break;
        }
        cudaGetLastError();
    }
    cached = result;
    return result;
}

int launch_map_fused(const FusedArgs& a, int cluster, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster);
    cfg.blockDim = dim3(FT);
    cfg.dynamicSmemBytes = kFusedSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.mapper == SPCONV_MAPPER_SORTED) {
        SPCONV_CHECK_CUDA(cudaLaunchKernelEx(&cfg, k_map_fused, a, static_cast<int>(kPartSort)));
        const int key_passes = (a.key_bits + kDigitMax - 1) / kDigitMax;
        SPCONV_CHECK(launch_search_window((key_passes & 1) ? a.vb : a.va, a.n, a.row_bits, a.key_bits, a.koff, a.nbr,
                                          a.mask, a.tap_count, a.status, s));
        count_launch(2);
    }
    {   // after the search: may start while it finishes (the dense mapper has no search before it)
        cudaLaunchAttribute rattr[2] = {attr[0], pdl_attr()};
        cudaLaunchConfig_t rcfg = cfg;
        rcfg.attrs = rattr;
        rcfg.numAttrs = a.mapper == SPCONV_MAPPER_SORTED ? 2 : 1;
        SPCONV_CHECK_CUDA(cudaLaunchKernelEx(&rcfg, k_map_fused, a, static_cast<int>(kPartRest)));
    }
    // the mask sort has an odd or even number of passes: the packed pairs end in vb or va
    constexpr int kMaskPasses = (kTaps + kDigitMax - 1) / kDigitMax;
    cudaLaunchConfig_t wcfg = {};
    wcfg.gridDim = dim3(static_cast<unsigned>(a.n_tiles));
    wcfg.blockDim = dim3(kTileRows);
    wcfg.stream = s;
    cudaLaunchAttribute wattr[1] = {pdl_attr()};
    wcfg.attrs = wattr;
    wcfg.numAttrs = 1;
    const uint64_t* ms = (kMaskPasses & 1) ? a.vb : a.va;
    SPCONV_CHECK_CUDA(cudaLaunchKernelEx(&wcfg, k_tile_write_packed, a, ms));
    count_launch(2);
    return SPCONV_OK;
}

}  // namespace spconv

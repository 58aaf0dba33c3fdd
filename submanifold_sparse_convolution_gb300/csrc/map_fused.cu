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
constexpr int BINS = 256;
constexpr int kMaxCluster = 16;
constexpr int kTilesPerRound = FW / 4;   // 4 warps (128 rows) per tile

struct FusedSmem {
    uint16_t cnt[IPT][FW][BINS];   // ranking: per (item slot, warp, digit) counts, then offsets
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

// Exclusive scan of a[0..255] in place (all threads call; uses the first 8 warps).
__device__ int32_t block_scan256(int32_t* a, int32_t* tmp) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    int32_t v = 0, incl = 0;
    if (t < BINS) {
        v = a[t];
        incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += x;
        }
        if (lane == 31) tmp[w] = incl;
    }
    __syncthreads();
    int32_t total = 0;
    for (int i = 0; i < BINS / 32; ++i) total += tmp[i];
    if (t < BINS) {
        int32_t wpre = 0;
        for (int i = 0; i < w; ++i) wpre += tmp[i];
        a[t] = wpre + incl - v;
    }
    __syncthreads();
    return total;
}

// One stable LSD pass over this CTA's part [c*chunk, min(n, (c+1)*chunk)) of
// `in`, by digit (v >> shift) & 255.  hc: every CTA's digit counts of its
// part ([C][256]).  When hn != nullptr the counts of the next digit
// (v >> next_shift) of every element are accumulated into hn by the CTA
// whose part the element lands in.
__device__ void radix_pass(const uint64_t* __restrict__ in, uint64_t* __restrict__ out, int64_t n,
                           int64_t chunk, int C, int c, int shift, const int32_t* hc, int32_t* hn,
                           int next_shift, FusedSmem& sm) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    if (t < BINS) {
        int32_t tot = 0, pre = 0;
        for (int q = 0; q < C; ++q) {
            const int32_t h = __ldcg(hc + q * BINS + t);
            tot += h;
            if (q < c) pre += h;
        }
        sm.scan[t] = tot;
        sm.pre[t] = pre;
        sm.run[t] = 0;
    }
    __syncthreads();
    block_scan256(sm.scan, sm.tmp);
    if (t < BINS) sm.base[t] = sm.scan[t] + sm.pre[t];
    const int64_t lo = static_cast<int64_t>(c) * chunk;
    const int64_t hi = lo + chunk < n ? lo + chunk : n;
    const uint32_t lt = lanemask_lt();
    for (int64_t r0 = lo; r0 < hi; r0 += RS) {
        uint32_t* cz = reinterpret_cast<uint32_t*>(&sm.cnt[0][0][0]);
        for (int i = t; i < IPT * FW * BINS / 2; i += FT) cz[i] = 0;
        __syncthreads();
        uint64_t v[IPT];
        int d[IPT], rk[IPT];
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const int64_t idx = r0 + j * FT + t;
            const bool valid = idx < hi;
            v[j] = valid ? __ldcg(in + idx) : 0ull;
            d[j] = valid ? static_cast<int>((v[j] >> shift) & 0xFF) : BINS;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d[j]);
            rk[j] = __popc(peers & lt);
            if (valid && lane == __ffs(peers) - 1) sm.cnt[j][w][d[j]] = static_cast<uint16_t>(__popc(peers));
        }
        __syncthreads();
        if (t < BINS) {
            uint32_t running = 0;
            for (int j = 0; j < IPT; ++j)
                for (int q = 0; q < FW; ++q) {
                    const uint32_t x = sm.cnt[j][q][t];
                    sm.cnt[j][q][t] = static_cast<uint16_t>(running);
                    running += x;
                }
            sm.rtot[t] = static_cast<int32_t>(running);
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < IPT; ++j) {
            const bool valid = d[j] < BINS;
            int64_t dst = 0;
            bool ok = false;
            if (valid) {
                dst = static_cast<int64_t>(sm.base[d[j]]) + sm.run[d[j]] + sm.cnt[j][w][d[j]] + rk[j];
                ok = dst >= 0 && dst < n;
                if (ok)
                    out[dst] = v[j];
                else
                    atomicOr(&sm.err, kStatusInternal);
            }
            if (hn != nullptr) {
                const int dc = ok ? static_cast<int>(dst / chunk) : 0;
                const int key2 = ok ? dc * BINS + static_cast<int>((v[j] >> next_shift) & 0xFF) : -1;
                const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key2);
                if (ok && lane == __ffs(peers) - 1) atomicAdd(hn + key2, __popc(peers));
            }
        }
        __syncthreads();
        if (t < BINS) sm.run[t] += sm.rtot[t];
    }
    __syncthreads();
}

// Local (this CTA only) digit histogram of in[lo, hi) written to h[c][*].
__device__ void local_hist(const uint64_t* __restrict__ in, int64_t lo, int64_t hi, int shift,
                           int32_t* h, FusedSmem& sm) {
    const int t = threadIdx.x, lane = t & 31;
    if (t < BINS) sm.scan[t] = 0;
    __syncthreads();
    for (int64_t i0 = lo; i0 < hi; i0 += FT) {
        const int64_t i = i0 + t;
        const int dg = i < hi ? static_cast<int>((__ldcg(in + i) >> shift) & 0xFF) : BINS;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, dg);
        if (dg < BINS && lane == __ffs(peers) - 1) atomicAdd(&sm.scan[dg], __popc(peers));
    }
    __syncthreads();
    if (t < BINS) h[t] = sm.scan[t];
    __syncthreads();
}

__device__ __forceinline__ void add_tap_counts(uint32_t m, int32_t* tap_count) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
        if (lane == 0 && b) atomicAdd(tap_count + k, __popc(b));
    }
}

__device__ __forceinline__ void store_row(int32_t* __restrict__ nbr, int64_t r, const int32_t (&v)[kNbrStride]) {
    int4* dst = reinterpret_cast<int4*>(nbr + r * kNbrStride);
#pragma unroll
    for (int q = 0; q < kNbrStride / 4; ++q) dst[q] = make_int4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

__global__ void __launch_bounds__(FT, 1) k_map_fused(const FusedArgs a) {
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
    if (t == 0) sm.err = 0;

    // ---------------- phase 0: reset counters, pack keys / clear the grid
    if (c == 0 && t < kTaps) a.tap_count[t] = 0;
    if (c == 0 && t == 0) {
        *a.status = 0;
        a.totals[0] = 0;
        a.totals[1] = 0;
    }
    if (t < BINS) {
        H[1][c * BINS + t] = 0;
        H[2][c * BINS + t] = 0;
    }
    __syncthreads();
    if (a.mapper == SPCONV_MAPPER_SORTED) {
        const uint64_t invalid = ((uint64_t(1) << a.key_bits) - 1) << rb;
        for (int64_t i = lo + t; i < hi; i += FT) {
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
        }
        __syncthreads();
        local_hist(a.va, lo, hi, rb, H[0] + c * BINS, sm);
    } else {
        const int64_t per = (a.cells + C - 1) / C;
        const int64_t g0 = static_cast<int64_t>(c) * per;
        const int64_t g1 = g0 + per < a.cells ? g0 + per : a.cells;
        for (int64_t i = g0 + t; i < g1; i += FT) a.grid[i] = -1;
    }
    cluster_sync_all();

    if (a.mapper == SPCONV_MAPPER_SORTED) {
        // ---------------- coordinate sort: one barrier per 8-bit pass
        const int passes = (a.key_bits + 7) / 8;
        for (int p = 0; p < passes; ++p) {
            const uint64_t* in = (p & 1) ? a.vb : a.va;
            uint64_t* out = (p & 1) ? a.va : a.vb;
            if (t < BINS) H[(p + 2) % 3][c * BINS + t] = 0;
            radix_pass(in, out, n, chunk, C, c, rb + 8 * p, H[p % 3], p + 1 < passes ? H[(p + 1) % 3] : nullptr,
                       rb + 8 * (p + 1), sm);
            cluster_sync_all();
        }
        const uint64_t* sv = (passes & 1) ? a.vb : a.va;
        const uint64_t invalid_key = (uint64_t(1) << a.key_bits) - 1;
        // ---------------- neighbour search: one lower_bound per (dx, dy) column
        // Each thread takes a contiguous run of sorted positions.  The first
        // is searched in lockstep over the whole array; later ones gallop
        // forward from the previous bounds, since every column's target grows
        // with the key.  The sorted array is read through L1: no thread has
        // read it through L1 before, so no stale line can be there.
        const int64_t per = (hi - lo + FT - 1) / FT;
        const int64_t sa = lo + static_cast<int64_t>(t) * per;
        const int64_t sb = sa + per < hi ? sa + per : hi;
        int64_t pos[9];
        bool have = false;
        for (int64_t e = 0; e < per; ++e) {
            const int64_t s = sa + e;
            uint32_t m = 0;
            if (s < sb) {
                const uint64_t vs = __ldg(sv + s);
                const uint64_t q = vs >> rb;
                int64_t r = static_cast<int64_t>(vs & rmask);
                if (r >= n) {
                    atomicOr(&sm.err, kStatusInternal);
                    r = -1;
                }
                int32_t v[kNbrStride];
#pragma unroll
                for (int k = 0; k < kNbrStride; ++k) v[k] = -1;
                if (q != invalid_key) {
                    if (s > 0 && (__ldg(sv + s - 1) >> rb) == q) atomicOr(&sm.err, kStatusDuplicate);
                    uint64_t tl[9];
#pragma unroll
                    for (int cc = 0; cc < 9; ++cc) tl[cc] = (q + a.koff[3 * cc]) << rb;
                    if (!have) {
                        lower_bound9(sv, n, tl, pos);
                        have = true;
                    } else {
#pragma unroll
                        for (int cc = 0; cc < 9; ++cc) pos[cc] = lower_bound_from(sv, n, pos[cc], tl[cc]);
                    }
#pragma unroll
                    for (int cc = 0; cc < 9; ++cc) {
                        const uint64_t hi_k = q + a.koff[3 * cc + 2];
#pragma unroll
                        for (int j = 0; j < 3; ++j) {
                            const int64_t pp = pos[cc] + j;
                            if (pp < n) {
                                const uint64_t vv = __ldg(sv + pp);
                                const uint64_t kk = vv >> rb;
                                if (kk <= hi_k) {
                                    const uint64_t dz = kk - (tl[cc] >> rb);
                                    const int32_t row = static_cast<int32_t>(vv & rmask) < n
                                                            ? static_cast<int32_t>(vv & rmask) : -1;
                                    if (dz == 0) v[3 * cc] = row;
                                    if (dz == 1) v[3 * cc + 1] = row;
                                    if (dz == 2) v[3 * cc + 2] = row;
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int k = 0; k < kTaps; ++k) m |= (v[k] >= 0 ? 1u : 0u) << k;
                }
                if (r >= 0) {
                    store_row(a.nbr, r, v);
                    a.mask[r] = m;
                }
            }
            add_tap_counts(m, a.tap_count);
        }
    } else {
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
                        v[k] = __ldg(a.grid + cell + a.goff[k]);
                        m |= (v[k] >= 0 ? 1u : 0u) << k;
                    }
                }
                store_row(a.nbr, i, v);
                a.mask[i] = m;
            }
            add_tap_counts(m, a.tap_count);
        }
    }
    cluster_sync_all();

    // ---------------- mask sort keys (tap order from the counts) + first histogram
    if (t < kTaps) {
        int32_t rank = t;
        if (a.calibrated) {
            const int32_t ck = __ldcg(a.tap_count + t);
            rank = 0;
            for (int j = 0; j < kTaps; ++j) {
                const int32_t cj = __ldcg(a.tap_count + j);
                rank += (cj > ck || (cj == ck && j < t)) ? 1 : 0;
            }
        }
        sm.tap_pos[t] = rank;
    }
    if (t < BINS) {
        H[1][c * BINS + t] = 0;
        H[2][c * BINS + t] = 0;
    }
    __syncthreads();
    for (int64_t i = lo + t; i < hi; i += FT) {
        const uint32_t m = __ldcg(a.mask + i);
        uint32_t key = 0;
#pragma unroll
        for (int k = 0; k < kTaps; ++k) key |= ((m >> k) & 1u) << sm.tap_pos[k];
        a.va[i] = (static_cast<uint64_t>(key) << rb) | static_cast<uint64_t>(i);
    }
    __syncthreads();
    local_hist(a.va, lo, hi, rb, H[0] + c * BINS, sm);
    cluster_sync_all();
    for (int p = 0; p < 4; ++p) {
        const uint64_t* in = (p & 1) ? a.vb : a.va;
        uint64_t* out = (p & 1) ? a.va : a.vb;
        if (t < BINS) H[(p + 2) % 3][c * BINS + t] = 0;
        radix_pass(in, out, n, chunk, C, c, rb + 8 * p, H[p % 3], p + 1 < 4 ? H[(p + 1) % 3] : nullptr,
                   rb + 8 * (p + 1), sm);
        cluster_sync_all();
    }
    const uint64_t* ms = a.va;   // 4 passes: the sorted (key, row) pairs are back in va

    // ---------------- compaction, count: per tile and tap, CTA totals, bucket counts
    const int64_t T = a.n_tiles;
    const int64_t tpc = (T + C - 1) / C;
    const int64_t ta = static_cast<int64_t>(c) * tpc;
    const int64_t tb = ta + tpc < T ? ta + tpc : T;
    const int nt = static_cast<int>(tb > ta ? tb - ta : 0);
    int32_t* tcnt = reinterpret_cast<int32_t*>(smem_raw + sizeof(FusedSmem));   // [nt][27]
    int32_t* tbkt = tcnt + static_cast<int64_t>(nt) * kTaps;                    // [nt]
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
        int u = 0;
        for (int k = 0; k < kTaps; ++k) u += tcnt[i * kTaps + k] > 0 ? 1 : 0;
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
    if (t < kTaps) {
        int32_t before = 0, mine = 0;
        for (int k = 0; k < t; ++k)
            for (int q = 0; q < C; ++q) before += __ldcg(a.cta_tot + q * kTaps + k);
        for (int q = 0; q < c; ++q) mine += __ldcg(a.cta_tot + q * kTaps + t);
        sm.tap_base[t] = before + mine;
        if (c == 0) a.tap_off[t] = before;
        if (c == 0 && t == kTaps - 1) {
            int32_t all = before;
            for (int q = 0; q < C; ++q) all += __ldcg(a.cta_tot + q * kTaps + t);
            a.tap_off[kTaps] = all;
            a.totals[0] = all;
        }
    }
    if (t >= 32 && t < 32 + kTaps + 1) {
        const int b = t - 32;
        int32_t before = 0, mine = 0;
        for (int bb = 0; bb < b; ++bb)
            for (int q = 0; q < C; ++q) before += __ldcg(a.cta_bkt + q * (kTaps + 1) + bb);
        for (int q = 0; q < c; ++q) mine += __ldcg(a.cta_bkt + q * (kTaps + 1) + b);
        sm.bkt_base[b] = before + mine;
        if (c == 0 && b == 0) {
            int32_t taps = 0;
            for (int bb = 0; bb <= kTaps; ++bb)
                for (int q = 0; q < C; ++q) taps += (kTaps - bb) * __ldcg(a.cta_bkt + q * (kTaps + 1) + bb);
            a.totals[1] = taps;
        }
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
    const uint32_t lt = lanemask_lt();
    for (int tr = 0; tr < nt; tr += kTilesPerRound) {
        const int tl = tr + (w >> 2);
        const int quarter = w & 3;
        const int64_t s = (ta + tl) * kTileRows + quarter * 32 + lane;
        const bool in_tile = tl < nt;
        const bool valid = in_tile && s < n;
        int32_t r = valid ? static_cast<int32_t>(__ldcg(ms + s) & rmask) : -1;
        if (r >= n) r = -1;
        const uint32_t m = r >= 0 ? __ldcg(a.mask + r) : 0u;
        uint32_t ball[kTaps];
#pragma unroll
        for (int k = 0; k < kTaps; ++k) {
            ball[k] = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
            if (lane == 0) sm.qcnt[w >> 2][quarter][k] = __popc(ball[k]);
        }
        __syncthreads();
        if (in_tile) {
            int32_t v[kNbrStride];
            if (r >= 0) {
                const int4* src = reinterpret_cast<const int4*>(a.nbr + static_cast<int64_t>(r) * kNbrStride);
#pragma unroll
                for (int q = 0; q < kNbrStride / 4; ++q) {
                    const int4 x = __ldcg(src + q);
                    v[4 * q] = x.x;
                    v[4 * q + 1] = x.y;
                    v[4 * q + 2] = x.z;
                    v[4 * q + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int k = 0; k < kNbrStride; ++k) v[k] = -1;
            }
            uint32_t uni = 0;
#pragma unroll
            for (int k = 0; k < kTaps; ++k) {
                const bool present = (m >> k) & 1u;
                int32_t tile_k = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) tile_k += sm.qcnt[w >> 2][q][k];
                uni |= (tile_k > 0 ? 1u : 0u) << k;
                if (present) {
                    int64_t off = sm.tap_base[k] + tcnt[tl * kTaps + k] + __popc(ball[k] & lt);
                    for (int q = 0; q < quarter; ++q) off += sm.qcnt[w >> 2][q][k];
                    if (off >= 0 && off < kTaps * n) {
                        a.in_rows[off] = v[k];
                        a.out_rows[off] = r;
                    } else {
                        atomicOr(&sm.err, kStatusInternal);
                    }
                }
                a.gtab[k * a.n_pad + s] = present ? v[k] : -1;
            }
            a.perm[s] = r;
            if (quarter == 0 && lane == 0) a.tile_union[ta + tl] = uni;
        }
        __syncthreads();
    }
    if (t == 0 && sm.err) atomicOr(a.status, sm.err);
}

}  // namespace

// Tiles per CTA are bounded by kFusedMaxRows / kTileRows / (smallest cluster).
constexpr int kMinCluster = 8;
constexpr size_t kFusedSmem = sizeof(FusedSmem) +
    static_cast<size_t>(kFusedMaxRows / kTileRows / kMinCluster) * (kTaps + 1) * sizeof(int32_t);

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
    SPCONV_CHECK_CUDA(cudaLaunchKernelEx(&cfg, k_map_fused, a));
    count_launch();
    return SPCONV_OK;
}

}  // namespace spconv

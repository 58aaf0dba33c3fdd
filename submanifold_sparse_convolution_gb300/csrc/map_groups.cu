// Kernel maps for any odd kernel size K (3 or 5: 27 or 125 taps) with the
// taps split into G offset groups of V / G consecutive taps, each group with
// its own neighbour masks, calibrated bit order, row order, 128-row tiles and
// tile unions.
//
// "Sparse convolution in FP32", "Offset-group partitioning": one row order for
// all 27 offsets leaves every tile executing the union of its rows' masks;
// one pass per offset has no waste but writes the output 27 times; a few
// groups, each with its own row order, sit in between.  Building every
// group's order with one radix sort (the group index as the most significant
// key digit) rather than one sort per group kept the preparation cost near
// that of a single order.  A 5x5x5 kernel (FlyDSL PR #942 tests K = 3 and
// K = 5) has 125 taps, more than one 32-bit mask holds, so it always runs in
// K groups of 25 (the taps with the same dx).
//
// Steps (one kernel each, stream-ordered, no host synchronisation):
//   sorted mapper: pack (b, x + r, y + r, z + r) into a 64-bit key
//     (r = (K - 1) / 2: the padding makes packed(q + d) = packed(q) +
//     packed(d) for every offset), radix-sort (key, row), then per row one
//     lower bound per (dx, dy) column and a check of the K keys that follow
//     (FlyDSL PR #942, "Two mappers, both required": K^2 searches, not K^3);
//   dense mapper: scatter row ids into the padded grid, K^3 lookups per row;
//   per group, the masks and calibrated sort keys, all groups in one sort;
//   per (group, tile) tap counts and unions, one scan of the counts into the
//   per-tap pair offsets, and the write of the pair lists and gather table.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "radix_sort.cuh"

namespace spconv {
namespace {

constexpr int kGBlock = 256;
constexpr int kMaxCols = kMaxKernel * kMaxKernel;
constexpr int kMaxGroups = kMaxKernel;
static_assert(kMaxGroups <= 32, "the tile scan places one group per warp");
constexpr uint64_t kNoKey = ~0ull;

struct GLayout {
    int K, r, V, stride;          // kernel size, radius, taps, nbr row width
    int wz, wy, wx;               // key field widths (bits)
    uint64_t col_off[kMaxCols];   // packed(dx, dy, -r) of column c = K (dx + r) + (dy + r), two's complement
    int64_t gsy, gsx, gsb;        // dense grid strides of y, x, b (z stride 1)
    int64_t goff[kMaxTaps];       // dense grid offset of each tap
};

int bit_len(uint64_t v) {
    int b = 0;
    while (v) {
        ++b;
        v >>= 1;
    }
    return b;
}

inline unsigned blocks(int64_t n, int per) { return static_cast<unsigned>((n + per - 1) / per); }

template <typename T>
T* take(char*& p, size_t count) {
    T* r = reinterpret_cast<T*>(p);
    p += (count * sizeof(T) + 255) / 256 * 256;
    return r;
}

__device__ __forceinline__ bool in_range(int4 c, int3 shape, int batch) {
    return c.x >= 0 && c.x < batch && c.y >= 0 && c.y < shape.x && c.z >= 0 && c.z < shape.y &&
           c.w >= 0 && c.w < shape.z;
}

// ---------------------------------------------------------------------------
// sorted-key mapper
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kGBlock) kg_pack_keys(const int4* __restrict__ coords, int64_t n, int3 shape,
                                                        int batch, const GLayout L, uint64_t* __restrict__ keys,
                                                        uint32_t* __restrict__ vals, int32_t* __restrict__ status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    uint64_t key = kNoKey;
    if (in_range(c, shape, batch)) {
        key = ((((static_cast<uint64_t>(c.x) << L.wx) | static_cast<uint64_t>(c.y + L.r)) << L.wy |
                static_cast<uint64_t>(c.z + L.r))
               << L.wz) |
              static_cast<uint64_t>(c.w + L.r);
    } else {
        atomicOr(status, kStatusRange);
    }
    keys[i] = key;
    vals[i] = static_cast<uint32_t>(i);
}

// First index in [lo, hi) with keys[idx] >= t (hi if none).
__device__ __forceinline__ int64_t first_not_less(const uint64_t* __restrict__ keys, int64_t lo, int64_t hi,
                                                  uint64_t t) {
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (__ldg(keys + mid) < t)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// One thread per sorted position s: for each (dx, dy) column, the lower bound
// of (dx, dy, -r) and the K keys from there.  Columns before the centre column
// hold smaller keys than the row's own, columns after it larger ones, so each
// search runs on one side of s.  nbr is cleared to -1 beforehand; only the
// present neighbours are written.
__global__ void __launch_bounds__(kGBlock) kg_search(const uint64_t* __restrict__ skeys,
                                                     const uint32_t* __restrict__ svals, int64_t n,
                                                     const GLayout L, int32_t* __restrict__ nbr,
                                                     int32_t* __restrict__ tap_count,
                                                     int32_t* __restrict__ status) {
    __shared__ int32_t cnt[kMaxTaps];
    for (int k = threadIdx.x; k < L.V; k += kGBlock) cnt[k] = 0;
    __syncthreads();
    const int64_t s = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (s < n) {
        const uint64_t q = skeys[s];
        const int64_t row = svals[s];
        if (q != kNoKey) {
            if (s > 0 && skeys[s - 1] == q) atomicOr(status, kStatusDuplicate);
            const int cols = L.K * L.K, centre = (cols - 1) / 2;
            for (int c = 0; c < cols; ++c) {
                const uint64_t lo_t = q + L.col_off[c];
                const uint64_t hi_t = lo_t + static_cast<uint64_t>(2 * L.r);
                int64_t lo = 0, hi = n;
                if (c < centre) hi = s;
                if (c > centre) lo = s + 1;
                if (c == centre) {
                    lo = s > L.r ? s - L.r : 0;
                    hi = s + L.r + 1 < n ? s + L.r + 1 : n;
                }
                const int64_t pos = first_not_less(skeys, lo, hi, lo_t);
                for (int j = 0; j < L.K; ++j) {
                    const int64_t p = pos + j;
                    if (p >= n) break;
                    const uint64_t kk = __ldg(skeys + p);
                    if (kk > hi_t) break;
                    const int k = c * L.K + static_cast<int>(kk - lo_t);
                    nbr[row * L.stride + k] = static_cast<int32_t>(__ldg(svals + p));
                    atomicAdd(&cnt[k], 1);
                }
            }
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < L.V; k += kGBlock)
        if (cnt[k]) atomicAdd(&tap_count[k], cnt[k]);
}

// ---------------------------------------------------------------------------
// hash mapper: the packed keys in a table of 4-slot buckets (bucketed linear
// probing, 16 slots per row), hashed by key >> 1 so that a z pair shares a
// bucket; a (dx, dy) column's K keys (dz = -r .. r) lie in at most r + 1
// pairs.  Within a bucket the slots fill in order and never empty again, and
// a pair's entries go to its bucket or the ones after it, so a bucket with an
// empty slot holds every entry of its pairs.
// ---------------------------------------------------------------------------
constexpr int kGHashBucket = 4;
constexpr int kGHashSlotsPerRow = 16;

__device__ __forceinline__ uint64_t g_bucket(uint64_t pair, int lb) {
    return (pair * 0x9E3779B97F4A7C15ull) >> (64 - lb);   // multiplicative (Fibonacci) hashing
}

// One bucket (4 slots, 32 bytes, 32-byte aligned) in a single 256-bit load
// through L2 (the table was written by the kernel before this one).
__device__ __forceinline__ void g_load_bucket(const uint64_t* b, ulonglong2& lo, ulonglong2& hi) {
    asm volatile("ld.global.cg.v4.u64 {%0, %1, %2, %3}, [%4];"
                 : "=l"(lo.x), "=l"(lo.y), "=l"(hi.x), "=l"(hi.y)
                 : "l"(b));
}

__device__ __forceinline__ uint64_t g_key(int4 c, const GLayout& L) {
    return ((((static_cast<uint64_t>(c.x) << L.wx) | static_cast<uint64_t>(c.y + L.r)) << L.wy |
             static_cast<uint64_t>(c.z + L.r))
            << L.wz) |
           static_cast<uint64_t>(c.w + L.r);
}

__global__ void __launch_bounds__(kGBlock) kg_hash_insert(const int4* __restrict__ coords, int64_t n, int3 shape,
                                                          int batch, const GLayout L, uint64_t* __restrict__ table,
                                                          int log2, int row_bits, int32_t* __restrict__ status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    if (!in_range(c, shape, batch)) {
        atomicOr(status, kStatusRange);
        return;
    }
    const uint64_t key = g_key(c, L);   // >= 1: every field is offset by r >= 1
    const uint64_t entry = (key << row_bits) | static_cast<uint64_t>(i);
    const int lb = log2 - 2;
    const uint64_t bmask = (uint64_t(1) << lb) - 1;
    uint64_t b = g_bucket(key >> 1, lb);
    for (uint64_t probe = 0; probe <= bmask; ++probe, b = (b + 1) & bmask) {
        for (int j = 0; j < kGHashBucket; ++j) {
            const unsigned long long prev = atomicCAS(
                reinterpret_cast<unsigned long long*>(table + b * kGHashBucket + j), 0ull,
                static_cast<unsigned long long>(entry));
            if (prev == 0ull) return;
            if ((prev >> row_bits) == key) {   // the same voxel twice
                atomicOr(status, kStatusDuplicate);
                return;
            }
        }
    }
    atomicOr(status, kStatusInternal);   // a full table: cannot happen at load <= 1/16
}

// One thread per row, one dx plane at a time: the plane's K columns' bucket
// reads (r + 1 pairs each) in flight together; the rare reads that meet a
// full bucket go on, all of the warp's in the same extra round.  nbr is
// cleared to -1 beforehand; only present neighbours are written.
template <int K>
__global__ void __launch_bounds__(kGBlock) kg_hash_lookup(const int4* __restrict__ coords, int64_t n, int3 shape,
                                                          int batch, const GLayout L,
                                                          const uint64_t* __restrict__ table, int log2,
                                                          int row_bits, int32_t* __restrict__ nbr,
                                                          int32_t* __restrict__ tap_count) {
    constexpr int r = (K - 1) / 2, V = K * K * K, NP = r + 1;   // pairs per column
    __shared__ int32_t cnt[V];
    for (int k = threadIdx.x; k < V; k += kGBlock) cnt[k] = 0;
    __syncthreads();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    const bool ok = i < n && in_range(coords[i], shape, batch);
    const uint64_t key = ok ? g_key(coords[i], L) : 0ull;
    const int lb = log2 - 2;
    const uint64_t bmask = (uint64_t(1) << lb) - 1;
    const uint64_t rmask = (uint64_t(1) << row_bits) - 1;
    for (int p = 0; p < K; ++p) {   // dx plane
        ulonglong2 lo[K * NP], hi[K * NP];
        uint64_t first_pair[K];
        uint32_t pending = 0, found = 0;   // found: bit K c + dz of this plane (a bucket may be read twice)
#pragma unroll
        for (int c = 0; c < K; ++c) first_pair[c] = (key + L.col_off[K * p + c]) >> 1;
#pragma unroll
        for (int q = 0; q < K * NP; ++q) {
            if (ok) {
                const uint64_t b = g_bucket(first_pair[q / NP] + q % NP, lb);
                g_load_bucket(table + b * kGHashBucket, lo[q], hi[q]);
            }
        }
        for (uint64_t step = 0;; ++step) {
#pragma unroll
            for (int q = 0; q < K * NP; ++q) {
                if (!ok || (step > 0 && !((pending >> q) & 1u))) continue;
                const int c = q / NP;
                const uint64_t lo_t = key + L.col_off[K * p + c];   // the column's dz = -r key
                const uint64_t sl[4] = {lo[q].x, lo[q].y, hi[q].x, hi[q].y};
                bool open = false;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    open |= sl[j] == 0ull;
                    const uint64_t d = (sl[j] >> row_bits) - lo_t;
                    if (sl[j] != 0ull && d < static_cast<uint64_t>(K)) {
                        nbr[i * L.stride + K * K * p + K * c + static_cast<int>(d)] = static_cast<int32_t>(sl[j] & rmask);
                        found |= 1u << (K * c + static_cast<int>(d));
                    }
                }
                if (open) pending &= ~(1u << q);
                else pending |= 1u << q;
            }
            if (!__any_sync(0xFFFFFFFFu, pending != 0u) || step >= bmask) {
                for (uint32_t f = found; f; f &= f - 1) atomicAdd(&cnt[K * K * p + __ffs(f) - 1], 1);
                break;
            }
#pragma unroll
            for (int q = 0; q < K * NP; ++q) {
                if ((pending >> q) & 1u) {
                    const uint64_t b = (g_bucket(first_pair[q / NP] + q % NP, lb) + step + 1) & bmask;
                    g_load_bucket(table + b * kGHashBucket, lo[q], hi[q]);
                }
            }
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < V; k += kGBlock)
        if (cnt[k]) atomicAdd(&tap_count[k], cnt[k]);
}

// ---------------------------------------------------------------------------
// dense presence-grid mapper (grid over the extents padded by r per side)
// ---------------------------------------------------------------------------
__device__ __forceinline__ int64_t cell_of(int4 c, const GLayout& L) {
    return c.x * L.gsb + static_cast<int64_t>(c.y + L.r) * L.gsx + static_cast<int64_t>(c.z + L.r) * L.gsy +
           (c.w + L.r);
}

__global__ void __launch_bounds__(kGBlock) kg_grid_scatter(const int4* __restrict__ coords, int64_t n, int3 shape,
                                                           int batch, const GLayout L, int32_t* __restrict__ grid,
                                                           int32_t* __restrict__ status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    if (!in_range(c, shape, batch)) {
        atomicOr(status, kStatusRange);
        return;
    }
    if (atomicCAS(grid + cell_of(c, L), -1, static_cast<int32_t>(i)) != -1) atomicOr(status, kStatusDuplicate);
}

__global__ void __launch_bounds__(kGBlock) kg_grid_lookup(const int4* __restrict__ coords, int64_t n, int3 shape,
                                                          int batch, const GLayout L,
                                                          const int32_t* __restrict__ grid,
                                                          int32_t* __restrict__ nbr,
                                                          int32_t* __restrict__ tap_count) {
    __shared__ int32_t cnt[kMaxTaps];
    for (int k = threadIdx.x; k < L.V; k += kGBlock) cnt[k] = 0;
    __syncthreads();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (i < n) {
        const int4 c = coords[i];
        if (in_range(c, shape, batch)) {
            const int64_t cell = cell_of(c, L);
            for (int k = 0; k < L.V; ++k) {
                const int32_t v = __ldg(grid + cell + L.goff[k]);
                if (v >= 0) {
                    nbr[i * L.stride + k] = v;
                    atomicAdd(&cnt[k], 1);
                }
            }
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < L.V; k += kGBlock)
        if (cnt[k]) atomicAdd(&tap_count[k], cnt[k]);
}

// ---------------------------------------------------------------------------
// per-group masks and row orders
// ---------------------------------------------------------------------------
// tap_pos[k] = key bit of tap k within its group.  Calibrated: the group's
// taps ranked by descending count (ties by ascending tap), the commonest at
// bit 0, so the rarest is the most significant ("Calibrated bit order").
__global__ void kg_tap_order(const int32_t* __restrict__ tap_count, int V, int kg, int calibrated,
                             int32_t* __restrict__ tap_pos) {
    for (int k = threadIdx.x; k < V; k += blockDim.x) {
        const int g0 = k / kg * kg;
        if (!calibrated) {
            tap_pos[k] = k - g0;
            continue;
        }
        const int32_t ck = tap_count[k];
        int rank = 0;
        for (int j = g0; j < g0 + kg; ++j) {
            const int32_t cj = tap_count[j];
            rank += (cj > ck || (cj == ck && j < k)) ? 1 : 0;
        }
        tap_pos[k] = rank;
    }
}

// One thread per (group g, row i), i fastest: the group's mask of row i and
// its sort key (g << kg) | calibrated key, so that one stable sort of all G n
// entries leaves group g's row order in positions [g n, (g + 1) n).
__global__ void __launch_bounds__(kGBlock) kg_mask_keys(const int32_t* __restrict__ nbr, int64_t n, int stride,
                                                        int G, int kg, const int32_t* __restrict__ tap_pos,
                                                        uint32_t* __restrict__ mask, uint32_t* __restrict__ keys,
                                                        uint32_t* __restrict__ vals) {
    __shared__ int32_t pos[kMaxTaps];
    for (int k = threadIdx.x; k < G * kg; k += kGBlock) pos[k] = tap_pos[k];
    __syncthreads();
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (idx >= G * n) return;
    const int g = static_cast<int>(idx / n);
    const int64_t i = idx - g * n;
    const int32_t* row = nbr + i * stride + g * kg;
    uint32_t m = 0, key = 0;
    for (int j = 0; j < kg; ++j) {
        if (row[j] >= 0) {
            m |= 1u << j;
            key |= 1u << pos[g * kg + j];
        }
    }
    mask[idx] = m;
    keys[idx] = (static_cast<uint32_t>(g) << kg) | key;
    vals[idx] = static_cast<uint32_t>(i);
}

// ---------------------------------------------------------------------------
// compaction: per-(tap, tile) counts -> scan -> pair lists, gather table
// ---------------------------------------------------------------------------
// Block (g, t): tile t of group g's order.  counts[k][t] for the group's taps
// k; the tile's union (bit j: tap g kg + j) in tile_union[g][t].
__global__ void __launch_bounds__(kTileRows) kg_tile_count(const int32_t* __restrict__ perm,
                                                           const uint32_t* __restrict__ mask, int64_t n,
                                                           int64_t n_tiles, int kg, int32_t* __restrict__ counts,
                                                           uint32_t* __restrict__ tile_union) {
    __shared__ int32_t wc[kTileRows / 32][kMaxGroupTaps];
    const int64_t g = blockIdx.x / n_tiles, t = blockIdx.x % n_tiles;
    const int64_t s = t * kTileRows + threadIdx.x;
    const uint32_t m = s < n ? mask[g * n + perm[g * n + s]] : 0u;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int j = 0; j < kg; ++j) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> j) & 1u);
        if (lane == 0) wc[warp][j] = __popc(b);
    }
    __syncthreads();
    if (warp == 0) {
        int32_t c = 0;
        if (lane < kg) {
            for (int w = 0; w < kTileRows / 32; ++w) c += wc[w][lane];
            counts[(g * kg + lane) * n_tiles + t] = c;
        }
        const uint32_t u = __ballot_sync(0xFFFFFFFFu, lane < kg && c > 0);
        if (lane == 0) tile_union[g * n_tiles + t] = u;
    }
}

// One block: exclusive scan of counts[V][T] into seg_off, the tap offsets and
// the pair total; each group's tiles ordered by descending union size
// (stable), with the number of tiles whose union is not empty (they come
// first); the sum of union sizes over all tiles.
__global__ void __launch_bounds__(1024) kg_scan_tiles(const int32_t* __restrict__ counts, int V, int G, int kg,
                                                      int64_t n_tiles, const uint32_t* __restrict__ tile_union,
                                                      int32_t* __restrict__ seg_off, int32_t* __restrict__ tap_off,
                                                      int32_t* __restrict__ totals,
                                                      int32_t* __restrict__ tile_order,
                                                      int32_t* __restrict__ nonempty) {
    __shared__ int32_t hist[kMaxGroups][kMaxGroupTaps + 1];
    for (int i = threadIdx.x; i < kMaxGroups * (kMaxGroupTaps + 1); i += 1024) (&hist[0][0])[i] = 0;
    const int64_t m = V * n_tiles;
    // seg_off is the exclusive scan of counts; a tap's list starts at the
    // offset of its first tile (one division per run of entries)
    const int32_t total = rsort::block_scan_exclusive(
        counts, seg_off, m, [&](int64_t i0, const int32_t (&v)[rsort::kScanPer]) {
            int64_t k = i0 / n_tiles, t = i0 - k * n_tiles;
#pragma unroll
            for (int j = 0; j < rsort::kScanPer; ++j) {
                if (t == 0 && i0 + j < m) tap_off[k] = v[j];
                if (++t == n_tiles) {
                    t = 0;
                    ++k;
                }
            }
        });
    if (threadIdx.x == 0) {
        tap_off[V] = total;
        totals[0] = total;
    }
    if (n_tiles == 0)
        for (int k = threadIdx.x; k < V; k += 1024) tap_off[k] = 0;
    __syncthreads();
    // per group, a counting sort of its tiles by descending union size, stable in t
    int32_t tap_sum = 0;
    for (int64_t i = threadIdx.x; i < G * n_tiles; i += 1024) {
        const int c = __popc(tile_union[i]);
        atomicAdd(&hist[i / n_tiles][kg - c], 1);
        tap_sum += c;
    }
    // one atomic per warp
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tap_sum += __shfl_down_sync(0xFFFFFFFFu, tap_sum, o);
    if ((threadIdx.x & 31) == 0 && tap_sum != 0) atomicAdd(&totals[1], tap_sum);
    __syncthreads();
    if (threadIdx.x < G) {
        nonempty[threadIdx.x] = static_cast<int32_t>(n_tiles) - hist[threadIdx.x][kg];
        int32_t r = 0;
        for (int b = 0; b <= kg; ++b) {
            const int32_t c = hist[threadIdx.x][b];
            hist[threadIdx.x][b] = r;
            r += c;
        }
    }
    __syncthreads();
    // warp g places group g's tiles, 32 at a time: each at its bucket's next
    // free position, tiles of one bucket in t order (ranked among the lanes
    // that share the bucket)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp < G) {
        const uint32_t* un = tile_union + warp * n_tiles;
        int32_t* ord = tile_order + warp * n_tiles;
        const uint32_t lt = rsort::lanemask_lt();
        for (int64_t t0 = 0; t0 < n_tiles; t0 += 32) {
            const int64_t t = t0 + lane;
            const int b = t < n_tiles ? kg - __popc(un[t]) : kg + 1;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, b);
            if (b <= kg) ord[hist[warp][b] + __popc(peers & lt)] = static_cast<int32_t>(t);
            __syncwarp();
            if (b <= kg && lane == __ffs(peers) - 1) hist[warp][b] += __popc(peers);
            __syncwarp();
        }
    }
}

// Block (g, t): the pairs of the group's taps for the rows of tile t, at the
// tile's offsets in each tap's list, ranked by position in the tile; and
// gtab[k][s] = neighbour of the row at position s of the group's order (-1
// when absent or past n).
__global__ void __launch_bounds__(kTileRows) kg_tile_write(const int32_t* __restrict__ perm,
                                                           const uint32_t* __restrict__ mask,
                                                           const int32_t* __restrict__ nbr, int stride, int64_t n,
                                                           int64_t n_tiles, int64_t n_pad, int kg,
                                                           const int32_t* __restrict__ seg_off,
                                                           int32_t* __restrict__ in_rows,
                                                           int32_t* __restrict__ out_rows,
                                                           int32_t* __restrict__ gtab) {
    __shared__ int32_t wc[kTileRows / 32][kMaxGroupTaps];
    __shared__ int32_t seg[kMaxGroupTaps];
    const int64_t g = blockIdx.x / n_tiles, t = blockIdx.x % n_tiles;
    const int64_t s = t * kTileRows + threadIdx.x;
    const bool valid = s < n;
    const int32_t r = valid ? perm[g * n + s] : -1;
    const uint32_t m = valid ? mask[g * n + r] : 0u;
    if (threadIdx.x < kg) seg[threadIdx.x] = seg_off[(g * kg + threadIdx.x) * n_tiles + t];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int j = 0; j < kg; ++j) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> j) & 1u);
        if (lane == 0) wc[warp][j] = __popc(b);
    }
    __syncthreads();
    const uint32_t lt = rsort::lanemask_lt();
    for (int j = 0; j < kg; ++j) {
        const int64_t k = g * kg + j;
        const bool present = (m >> j) & 1u;
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, present);
        int32_t v = -1;
        if (present) {
            v = nbr[static_cast<int64_t>(r) * stride + k];
            int32_t off = seg[j] + __popc(b & lt);
            for (int w = 0; w < warp; ++w) off += wc[w][j];
            in_rows[off] = v;
            out_rows[off] = r;
        }
        gtab[k * n_pad + s] = v;
    }
}

// ---------------------------------------------------------------------------
// strided maps: the output sites and the query sites 2o
// ---------------------------------------------------------------------------
// Output key of site (b, x, y, z) of the strided grid: fields of widths
// ow[0..2] (x, y, z), the batch above them; ~0 for no site.
struct OutLayout {
    int wx, wy, wz;
    int3 shape;   // output shape
};

__device__ __forceinline__ uint64_t out_key(int b, int x, int y, int z, const OutLayout& O) {
    return ((((static_cast<uint64_t>(b) << O.wx) | static_cast<uint64_t>(x)) << O.wy | static_cast<uint64_t>(y))
            << O.wz) |
           static_cast<uint64_t>(z);
}

// Per input site, the up to 8 output sites whose window {2o + d} holds it:
// o = (c - d) / 2 for the d of matching parity on each axis, inside the
// output shape.  cand[8 i + j] (~0 where there is none).
__global__ void __launch_bounds__(kGBlock) kst_candidates(const int4* __restrict__ coords, int64_t n, int3 shape,
                                                          int batch, const OutLayout O, uint64_t* __restrict__ cand,
                                                          uint32_t* __restrict__ vals) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    const bool ok = in_range(c, shape, batch);
    int j = 0;
    for (int dx = -1; dx <= 1; ++dx)
        for (int dy = -1; dy <= 1; ++dy)
            for (int dz = -1; dz <= 1; ++dz) {
                const int px = c.y - dx, py = c.z - dy, pz = c.w - dz;
                if (!ok || px < 0 || py < 0 || pz < 0 || (px & 1) || (py & 1) || (pz & 1)) continue;
                const int ox = px >> 1, oy = py >> 1, oz = pz >> 1;
                if (ox >= O.shape.x || oy >= O.shape.y || oz >= O.shape.z) continue;
                cand[8 * i + j] = out_key(c.x, ox, oy, oz, O);
                vals[8 * i + j] = 0;
                ++j;
            }
    for (; j < 8; ++j) {
        cand[8 * i + j] = kNoKey;
        vals[8 * i + j] = 0;
    }
}

// flags[j] = 1 for the first of each run of equal sorted keys (not ~0).
__global__ void __launch_bounds__(kGBlock) kst_first(const uint64_t* __restrict__ keys, int64_t m,
                                                     int32_t* __restrict__ flags) {
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (j >= m) return;
    const uint64_t k = keys[j];
    flags[j] = (k != kNoKey && (j == 0 || keys[j - 1] != k)) ? 1 : 0;
}

// Exclusive scan of the first-of-run flags over the whole grid, in three
// steps: per 1024-entry block the number of flags, one CTA's scan of the
// block counts, then each block's ranks (a single-CTA scan over 8 n entries
// was a serial walk of thousands of values per thread).
constexpr int kRankBlock = 1024;

__global__ void __launch_bounds__(kRankBlock) kst_block_count(const int32_t* __restrict__ flags, int64_t m,
                                                              int32_t* __restrict__ bcount) {
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kRankBlock + threadIdx.x;
    const int f = j < m ? flags[j] : 0;
    const int c = __syncthreads_count(f);
    if (threadIdx.x == 0) bcount[blockIdx.x] = c;
}

__global__ void __launch_bounds__(kRankBlock) kst_block_scan(int32_t* __restrict__ bcount, int64_t nb) {
    __shared__ int32_t carry;
    __shared__ int32_t wsum[kRankBlock / 32];
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    if (t == 0) carry = 0;
    __syncthreads();
    for (int64_t b0 = 0; b0 < nb; b0 += kRankBlock) {
        const int64_t i = b0 + t;
        const int32_t v = i < nb ? bcount[i] : 0;
        int32_t inc = v;
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) wsum[w] = inc;
        __syncthreads();
        int32_t before = 0, total = 0;
        for (int q = 0; q < kRankBlock / 32; ++q) {
            before += q < w ? wsum[q] : 0;
            total += wsum[q];
        }
        if (i < nb) bcount[i] = carry + before + inc - v;
        __syncthreads();
        if (t == 0) carry += total;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kRankBlock) kst_block_rank(const int32_t* __restrict__ flags, int64_t m,
                                                             const int32_t* __restrict__ bbase,
                                                             int32_t* __restrict__ rank) {
    __shared__ int32_t wsum[kRankBlock / 32];
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kRankBlock + t;
    const int32_t f = j < m ? flags[j] : 0;
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, f != 0);
    if (lane == 0) wsum[w] = __popc(b);
    __syncthreads();
    int32_t before = 0;
    for (int q = 0; q < w; ++q) before += wsum[q];
    if (j < m) rank[j] = bbase[blockIdx.x] + before + __popc(b & ((1u << lane) - 1u));
}

// After the exclusive scan of the flags: output row rank[j] is site keys[j];
// writes its coordinates, its query site 2o in input coordinates, and the
// count of sites (into *count, by the last entry).
__global__ void __launch_bounds__(kGBlock) kst_outputs(const uint64_t* __restrict__ keys,
                                                       const int32_t* __restrict__ flags_first,
                                                       const int32_t* __restrict__ rank, int64_t m, const OutLayout O,
                                                       int4* __restrict__ out_coords, int4* __restrict__ query,
                                                       int64_t cap, int64_t* __restrict__ count) {
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (j >= m) return;
    if (j == m - 1) *count = static_cast<int64_t>(rank[j]) + flags_first[j];
    if (!flags_first[j]) return;
    const uint64_t k = keys[j];
    const int z = static_cast<int>(k & ((uint64_t(1) << O.wz) - 1));
    const int y = static_cast<int>((k >> O.wz) & ((uint64_t(1) << O.wy) - 1));
    const int x = static_cast<int>((k >> (O.wz + O.wy)) & ((uint64_t(1) << O.wx) - 1));
    const int b = static_cast<int>(k >> (O.wz + O.wy + O.wx));
    const int64_t r = rank[j];
    if (r < cap) {
        out_coords[r] = make_int4(b, x, y, z);
        query[r] = make_int4(b, 2 * x, 2 * y, 2 * z);
    }
}

// Inverse map: for every (o, k) of the strided map with input row i,
// inv[i][k] = o (one writer per entry: o is fixed by i and k).
__global__ void __launch_bounds__(kGBlock) kg_inverse_scatter(const int32_t* __restrict__ nbr, int stride, int64_t n,
                                                              int32_t* __restrict__ inv, int inv_stride) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (idx >= n * kTaps) return;
    const int64_t o = idx / kTaps;
    const int k = static_cast<int>(idx % kTaps);
    const int32_t i = nbr[o * stride + k];
    if (i >= 0) inv[static_cast<int64_t>(i) * inv_stride + k] = static_cast<int32_t>(o);
}

// The whole grouped build for one of three sources of the neighbours: the
// sites themselves (coords, n_table = h->n rows), the input sites of a
// strided map (table coords [n_table], query sites [h->n], hash mapper), or
// the inverse of strided map src.
int grouped_core(MapHandle* h, const spconv_options_t* opt, const int32_t* coords, int64_t n_table,
                 const int32_t* query, const MapHandle* src);

}  // namespace

int build_map_grouped(MapHandle* h, const int32_t* coords, const spconv_options_t* opt) {
    return grouped_core(h, opt, coords, h->n, nullptr, nullptr);
}

namespace {
int grouped_core(MapHandle* h, const spconv_options_t* opt, const int32_t* coords, int64_t n_table,
                 const int32_t* query, const MapHandle* src) {
    cudaStream_t s = h->stream;
    const int64_t n = h->n;
    const int64_t T = (n + kTileRows - 1) / kTileRows;
    h->n_tiles = T;
    h->n_pad = T * kTileRows;
    const int K = h->kernel_size, r = (K - 1) / 2, V = K * K * K, G = h->groups, kg = V / G;
    if (K < 1 || K > kMaxKernel || K % 2 == 0 || G < 1 || G > kMaxGroups || V % G != 0 || kg > kMaxGroupTaps)
        return SPCONV_ERR_UNSUPPORTED;
    h->taps = V;
    h->group_taps = kg;
    h->nbr_stride = (V + 3) / 4 * 4;
    const int X = h->shape[0], Y = h->shape[1], Z = h->shape[2], B = h->batch;

    GLayout L = {};
    L.K = K;
    L.r = r;
    L.V = V;
    L.stride = h->nbr_stride;
    // coordinates + r lie in [r, extent - 1 + r], neighbours in [0, extent - 1 + 2r]
    L.wz = bit_len(static_cast<uint64_t>(Z) - 1 + 2 * r);
    L.wy = bit_len(static_cast<uint64_t>(Y) - 1 + 2 * r);
    L.wx = bit_len(static_cast<uint64_t>(X) - 1 + 2 * r);
    const int wb = bit_len(static_cast<uint64_t>(B) - 1);
    const int key_bits = L.wz + L.wy + L.wx + wb;
    h->key_bits = key_bits;
    for (int dx = -r; dx <= r; ++dx)
        for (int dy = -r; dy <= r; ++dy) {
            const int64_t o = static_cast<int64_t>(dx) * (int64_t(1) << (L.wy + L.wz)) +
                              static_cast<int64_t>(dy) * (int64_t(1) << L.wz) - r;
            L.col_off[K * (dx + r) + (dy + r)] = static_cast<uint64_t>(o);
        }
    L.gsy = Z + 2 * r;
    L.gsx = static_cast<int64_t>(Y + 2 * r) * L.gsy;
    L.gsb = static_cast<int64_t>(X + 2 * r) * L.gsx;
    for (int dx = -r; dx <= r; ++dx)
        for (int dy = -r; dy <= r; ++dy)
            for (int dz = -r; dz <= r; ++dz)
                L.goff[K * K * (dx + r) + K * (dy + r) + (dz + r)] = dx * L.gsx + dy * L.gsy + dz;

    const double cells_d = static_cast<double>(B) * (X + 2 * r) * (Y + 2 * r) * (Z + 2 * r);
    const int64_t cells = cells_d > 9.0e18 ? 0 : static_cast<int64_t>(B) * L.gsb;
    int mapper = opt ? opt->mapper : SPCONV_MAPPER_AUTO;
    const int64_t dense_max = (opt && opt->dense_max_cells > 0) ? opt->dense_max_cells : (int64_t(1) << 24);
    const int row_bits = std::max(1, bit_len(static_cast<uint64_t>(n_table > 0 ? n_table - 1 : 0)));
    // AUTO: the dense grid on small boxes; else, for K = 3, hashed keys when they
    // pack with the row (outdoor in 3 groups: map 197 -> 130 us), and sorted keys
    // for K = 5, where the per-row hash lookup of 125 taps measured slower (outdoor
    // 339 vs 354 us, 240k rows 1364 vs 1747 us)
    if (query) {   // strided: the input sites go in a hash table
        if (mapper != SPCONV_MAPPER_AUTO && mapper != SPCONV_MAPPER_HASH) return SPCONV_ERR_UNSUPPORTED;
        mapper = SPCONV_MAPPER_HASH;
    }
    if (src) mapper = src->mapper;   // inverse: read off the strided map (reported as its mapper)
    if (mapper == SPCONV_MAPPER_AUTO)
        mapper = (cells_d <= 9.0e18 && cells <= dense_max) ? SPCONV_MAPPER_DENSE
                 : (K == 3 && key_bits + row_bits <= 64) ? SPCONV_MAPPER_HASH : SPCONV_MAPPER_SORTED;
    if (mapper == SPCONV_MAPPER_SORTED && key_bits > 63) return SPCONV_ERR_UNSUPPORTED;
    if (mapper == SPCONV_MAPPER_HASH && key_bits + row_bits > 64) return SPCONV_ERR_UNSUPPORTED;
    if (mapper == SPCONV_MAPPER_DENSE && (cells_d > 9.0e18 || cells > (int64_t(1) << 34))) return SPCONV_ERR_UNSUPPORTED;
    h->mapper = mapper;
    h->bit_order = opt ? opt->bit_order : SPCONV_ORDER_CALIBRATED;
    h->gemm = SPCONV_GEMM_TILE_UNION;
    h->pipeline = SPCONV_PIPELINE_MULTI;

    // ---- one arena
    const int64_t n1 = std::max<int64_t>(1, n);
    const int64_t gn = std::max<int64_t>(1, G * n);
    const int64_t np = std::max<int64_t>(1, h->n_pad);
    const int64_t t1 = std::max<int64_t>(1, T);
    const int64_t nb = std::max<int64_t>(1, rsort::num_tiles(std::max(G * n, mapper == SPCONV_MAPPER_SORTED ? n : 0)));
    const int64_t nt1 = std::max<int64_t>(1, n_table);
    size_t bytes = 0;
    auto add = [&](size_t count, size_t elem) { bytes += (count * elem + 255) / 256 * 256; };
    add(4, 4);                                        // status
    add(n1 * h->nbr_stride, 4);                       // nbr
    add(gn, 4);                                       // masks [G][n]
    add(V, 4); add(V, 4); add(V + 1, 4); add(2, 4);   // tap_count, tap_pos, tap_off, totals
    add(V * n1, 4); add(V * n1, 4);                   // in_rows, out_rows
    add(V * np, 4);                                   // gtab
    add(G * t1, 4); add(G * t1, 4);                   // unions, tile orders
    add(V * t1, 4); add(V * t1, 4);                   // counts, seg_off
    add(G, 4);                                        // nonempty tiles per group
    add(gn, 4); add(gn, 4); add(gn, 4); add(gn, 4);   // mask keys and row ids, ping-pong
    add(rsort::kBins * nb, 4);                        // radix histograms
    int table_log2 = 11;
    while ((int64_t(1) << table_log2) < kGHashSlotsPerRow * nt1) ++table_log2;
    if (src) {
        // the neighbours come from the strided map
    } else if (mapper == SPCONV_MAPPER_SORTED) {
        add(n1, 8); add(n1, 8); add(n1, 4); add(n1, 4);   // coordinate keys and rows, ping-pong
    } else if (mapper == SPCONV_MAPPER_HASH) {
        add(size_t(1) << table_log2, 8);                 // hash table
    } else {
        add(static_cast<size_t>(cells), 4);              // presence grid
    }
    void* arena = nullptr;
    if (pool_alloc(&arena, bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_OOM;
    }
    h->arena = arena;
    h->arena_bytes = bytes;
    char* p = static_cast<char*>(arena);
    h->status = take<int32_t>(p, 4);
    h->nbr = take<int32_t>(p, n1 * h->nbr_stride);
    h->mask = take<uint32_t>(p, gn);
    h->tap_count = take<int32_t>(p, V);
    h->tap_pos = take<int32_t>(p, V);
    h->tap_off = take<int32_t>(p, V + 1);
    h->totals = take<int32_t>(p, 2);
    h->in_rows = take<int32_t>(p, V * n1);
    h->out_rows = take<int32_t>(p, V * n1);
    h->gtab = take<int32_t>(p, V * np);
    h->tile_union = take<uint32_t>(p, G * t1);
    h->tile_order = take<int32_t>(p, G * t1);
    int32_t* counts = take<int32_t>(p, V * t1);
    h->seg_off = take<int32_t>(p, V * t1);
    h->tile_nonempty = take<int32_t>(p, G);
    uint32_t* mkey_a = take<uint32_t>(p, gn);
    uint32_t* mkey_b = take<uint32_t>(p, gn);
    uint32_t* perm_a = take<uint32_t>(p, gn);
    uint32_t* perm_b = take<uint32_t>(p, gn);
    int32_t* hist = take<int32_t>(p, rsort::kBins * nb);

    SPCONV_CHECK_CUDA(cudaMemsetAsync(h->status, 0, 4 * sizeof(int32_t), s));
    SPCONV_CHECK_CUDA(cudaMemsetAsync(h->tap_count, 0, V * sizeof(int32_t), s));
    SPCONV_CHECK_CUDA(cudaMemsetAsync(h->totals, 0, 2 * sizeof(int32_t), s));
    h->perm = reinterpret_cast<int32_t*>(perm_a);
    if (n == 0) {
        SPCONV_CHECK_CUDA(cudaMemsetAsync(h->tap_off, 0, (V + 1) * sizeof(int32_t), s));
        return cuda_status(cudaGetLastError());
    }
    SPCONV_CHECK_CUDA(cudaMemsetAsync(h->nbr, 0xFF, static_cast<size_t>(n) * h->nbr_stride * sizeof(int32_t), s));

    const int4* c4 = reinterpret_cast<const int4*>(coords);
    const int3 shape3 = make_int3(X, Y, Z);
    int launches = 0;
    if (src) {
        // the strided map read backwards; the tap counts are the same incidences
        kg_inverse_scatter<<<blocks(src->n * kTaps, kGBlock), kGBlock, 0, s>>>(src->nbr, src->nbr_stride, src->n,
                                                                              h->nbr, h->nbr_stride);
        SPCONV_CHECK_CUDA(cudaMemcpyAsync(h->tap_count, src->tap_count, V * sizeof(int32_t),
                                          cudaMemcpyDeviceToDevice, s));
        SPCONV_CHECK_CUDA(cudaMemcpyAsync(h->status, src->status, sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
        ++launches;
    } else if (mapper == SPCONV_MAPPER_SORTED) {
        uint64_t* ck_a = take<uint64_t>(p, n1);
        uint64_t* ck_b = take<uint64_t>(p, n1);
        uint32_t* cv_a = take<uint32_t>(p, n1);
        uint32_t* cv_b = take<uint32_t>(p, n1);
        kg_pack_keys<<<blocks(n, kGBlock), kGBlock, 0, s>>>(c4, n, shape3, B, L, ck_a, cv_a, h->status);
        ++launches;
        // out-of-range rows carry the all-ones key: one bit above the live ones orders them last
        const bool in_b = rsort::sort_pairs<uint64_t>(ck_a, cv_a, ck_b, cv_b, n, std::min(64, key_bits + 1), hist, s,
                                                      &launches);
        kg_search<<<blocks(n, kGBlock), kGBlock, 0, s>>>(in_b ? ck_b : ck_a, in_b ? cv_b : cv_a, n, L, h->nbr,
                                                         h->tap_count, h->status);
        ++launches;
    } else if (mapper == SPCONV_MAPPER_HASH) {
        uint64_t* table = take<uint64_t>(p, size_t(1) << table_log2);
        SPCONV_CHECK_CUDA(cudaMemsetAsync(table, 0, (size_t(1) << table_log2) * 8, s));
        kg_hash_insert<<<blocks(n_table, kGBlock), kGBlock, 0, s>>>(c4, n_table, shape3, B, L, table, table_log2,
                                                                    row_bits, h->status);
        const int4* q4 = query ? reinterpret_cast<const int4*>(query) : c4;
        if (K == 3)
            kg_hash_lookup<3><<<blocks(n, kGBlock), kGBlock, 0, s>>>(q4, n, shape3, B, L, table, table_log2, row_bits,
                                                                     h->nbr, h->tap_count);
        else
            kg_hash_lookup<5><<<blocks(n, kGBlock), kGBlock, 0, s>>>(q4, n, shape3, B, L, table, table_log2, row_bits,
                                                                     h->nbr, h->tap_count);
        launches += 2;
    } else {
        int32_t* grid = take<int32_t>(p, static_cast<size_t>(cells));
        SPCONV_CHECK_CUDA(cudaMemsetAsync(grid, 0xFF, static_cast<size_t>(cells) * 4, s));
        kg_grid_scatter<<<blocks(n, kGBlock), kGBlock, 0, s>>>(c4, n, shape3, B, L, grid, h->status);
        kg_grid_lookup<<<blocks(n, kGBlock), kGBlock, 0, s>>>(c4, n, shape3, B, L, grid, h->nbr, h->tap_count);
        launches += 2;
    }
    kg_tap_order<<<1, 128, 0, s>>>(h->tap_count, V, kg, h->bit_order == SPCONV_ORDER_CALIBRATED, h->tap_pos);
    kg_mask_keys<<<blocks(G * n, kGBlock), kGBlock, 0, s>>>(h->nbr, n, h->nbr_stride, G, kg, h->tap_pos, h->mask,
                                                            mkey_a, perm_a);
    launches += 2;
    const bool perm_in_b = rsort::sort_pairs<uint32_t>(mkey_a, perm_a, mkey_b, perm_b, G * n,
                                                       kg + bit_len(static_cast<uint64_t>(G) - 1), hist, s, &launches);
    h->perm = reinterpret_cast<int32_t*>(perm_in_b ? perm_b : perm_a);
    const unsigned tiles = static_cast<unsigned>(G * T);
    kg_tile_count<<<tiles, kTileRows, 0, s>>>(h->perm, h->mask, n, T, kg, counts, h->tile_union);
    kg_scan_tiles<<<1, 1024, 0, s>>>(counts, V, G, kg, T, h->tile_union, h->seg_off, h->tap_off, h->totals,
                                     h->tile_order, h->tile_nonempty);
    kg_tile_write<<<tiles, kTileRows, 0, s>>>(h->perm, h->mask, h->nbr, h->nbr_stride, n, T, h->n_pad, kg,
                                              h->seg_off, h->in_rows, h->out_rows, h->gtab);
    launches += 3;
    count_launch(launches);
    return cuda_status(cudaGetLastError());
}
}  // namespace

int build_map_strided(MapHandle* h, const int32_t* coords, int64_t n_in, const spconv_options_t* opt) {
    cudaStream_t s = h->stream;
    OutLayout O;
    O.shape = make_int3((h->shape[0] - 1) / 2 + 1, (h->shape[1] - 1) / 2 + 1, (h->shape[2] - 1) / 2 + 1);
    O.wx = std::max(1, bit_len(static_cast<uint64_t>(O.shape.x - 1)));
    O.wy = std::max(1, bit_len(static_cast<uint64_t>(O.shape.y - 1)));
    O.wz = std::max(1, bit_len(static_cast<uint64_t>(O.shape.z - 1)));
    const int okey_bits = O.wx + O.wy + O.wz + bit_len(static_cast<uint64_t>(h->batch) - 1);
    if (okey_bits > 62) return SPCONV_ERR_UNSUPPORTED;
    h->conv = kConvStrided;
    h->n_in = n_in;
    h->out_shape[0] = O.shape.x;
    h->out_shape[1] = O.shape.y;
    h->out_shape[2] = O.shape.z;
    // ---- the output sites: 8 candidates per input site, sorted, the first of each run kept
    const int64_t m = 8 * std::max<int64_t>(1, n_in);
    size_t bytes = 0;
    auto add = [&](size_t count, size_t elem) { bytes += (count * elem + 255) / 256 * 256; };
    const int64_t nb = rsort::num_tiles(m);
    add(m, 8); add(m, 8); add(m, 4); add(m, 4);   // candidate keys and (unused) values, ping-pong
    add(m, 4); add(m, 4);                         // first-of-run flags, their exclusive scan
    add((m + kRankBlock - 1) / kRankBlock, 4);    // per-block flag counts
    add(rsort::kBins * std::max<int64_t>(1, nb), 4);
    add(m, 16); add(1, 8);                        // query sites, the output count
    void* scratch = nullptr;
    if (pool_alloc(&scratch, bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_OOM;
    }
    char* p = static_cast<char*>(scratch);
    uint64_t* ka = take<uint64_t>(p, m);
    uint64_t* kb = take<uint64_t>(p, m);
    uint32_t* va = take<uint32_t>(p, m);
    uint32_t* vb = take<uint32_t>(p, m);
    int32_t* flags = take<int32_t>(p, m);
    int32_t* rank = take<int32_t>(p, m);
    const int64_t rb = (m + kRankBlock - 1) / kRankBlock;
    int32_t* bcount = take<int32_t>(p, rb);
    int32_t* hist = take<int32_t>(p, rsort::kBins * std::max<int64_t>(1, nb));
    int4* query = take<int4>(p, m);
    int64_t* count = take<int64_t>(p, 1);
    void* outs = nullptr;
    if (pool_alloc(&outs, static_cast<size_t>(m) * 16, s) != cudaSuccess) {
        cudaGetLastError();
        cudaFreeAsync(scratch, s);
        return SPCONV_ERR_OOM;
    }
    h->out_alloc = outs;
    h->out_coords = static_cast<int32_t*>(outs);
    int launches = 0;
    int64_t n_out = 0;
    SPCONV_CHECK_CUDA(cudaMemsetAsync(count, 0, 8, s));
    if (n_in > 0) {
        kst_candidates<<<blocks(n_in, kGBlock), kGBlock, 0, s>>>(reinterpret_cast<const int4*>(coords), n_in,
                                                                  make_int3(h->shape[0], h->shape[1], h->shape[2]),
                                                                  h->batch, O, ka, va);
        ++launches;
        const bool in_b = rsort::sort_pairs<uint64_t>(ka, va, kb, vb, m, okey_bits + 1, hist, s, &launches);
        const uint64_t* sk = in_b ? kb : ka;
        kst_first<<<blocks(m, kGBlock), kGBlock, 0, s>>>(sk, m, flags);
        kst_block_count<<<static_cast<unsigned>(rb), kRankBlock, 0, s>>>(flags, m, bcount);
        kst_block_scan<<<1, kRankBlock, 0, s>>>(bcount, rb);
        kst_block_rank<<<static_cast<unsigned>(rb), kRankBlock, 0, s>>>(flags, m, bcount, rank);
        launches += 2;
        kst_outputs<<<blocks(m, kGBlock), kGBlock, 0, s>>>(sk, flags, rank, m, O,
                                                           reinterpret_cast<int4*>(h->out_coords), query, m, count);
        launches += 3;
        // the one synchronisation: the output count sizes the map
        SPCONV_CHECK_CUDA(cudaMemcpyAsync(&n_out, count, 8, cudaMemcpyDeviceToHost, s));
        SPCONV_CHECK_CUDA(cudaStreamSynchronize(s));
    }
    count_launch(launches);
    h->n = n_out;
    const int rc = grouped_core(h, opt, coords, n_in, reinterpret_cast<const int32_t*>(query), nullptr);
    cudaFreeAsync(scratch, s);   // stream-ordered: after the kernels that read it
    return rc;
}

int build_map_inverse(MapHandle* h, const MapHandle* src, const spconv_options_t* opt) {
    h->conv = kConvInverse;
    h->n = src->n_in;
    h->n_in = src->n;
    std::memcpy(h->out_shape, src->shape, sizeof(h->out_shape));
    std::memcpy(h->shape, src->shape, sizeof(h->shape));
    h->batch = src->batch;
    return grouped_core(h, opt, nullptr, src->n, nullptr, src);
}

}  // namespace spconv

// Kernel-map construction: coordinate mapper (sorted 64-bit keys or dense
// presence grid), 27-bit neighbour masks, mask-sorted row order, per-tap pair
// lists and the 128-row tile work list.
//
// FlyDSL PR #942 ("Two mappers, both required"): a dense grid is fastest on
// compact boxes but is O(volume) and overflows 32-bit indexing past 2^31
// cells; the sorted-key mapper packs coordinates so that
// packed(q + d) == packed(q) + packed(d), sorts once, and needs one binary
// search per (dx, dy) column (K^2 searches instead of K^3) since the three z
// neighbours of a column are adjacent in key order.
// "Sparse convolution in FP32" ("Neighbour masks and sorted rows"): the map
// builder emits a 27-bit mask per row and the rows are radix-sorted by it so
// that a tile of rows only visits the union of its rows' taps.
// FlyDSL PR #942 ("scan the pair counts on the device"): pair lists are written
// from a scan over small per-(tap, tile) counts, not through atomic counters,
// with no host synchronisation.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "map_internal.cuh"
#include "radix_sort.cuh"

namespace spconv {
namespace {

constexpr uint64_t kInvalidKey = ~0ull;
constexpr int kBlock = 256;

struct KeyLayout {
    int wz, wy, wx, wb;          // field widths (bits)
    uint64_t off[kTaps];         // packed(d_k) as a two's-complement 64-bit addend
};

int bit_length(uint64_t v) {
    int b = 0;
    while (v) {
        ++b;
        v >>= 1;
    }
    return b;
}

__device__ __forceinline__ bool coord_valid(int4 c, int3 shape, int batch) {
    return c.x >= 0 && c.x < batch && c.y >= 0 && c.y < shape.x && c.z >= 0 && c.z < shape.y &&
           c.w >= 0 && c.w < shape.z;
}

// ---------------------------------------------------------------------------
// sorted-key mapper
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBlock) k_pack_keys(const int4* __restrict__ coords, int64_t n,
                                                      int3 shape, int batch, int wz, int wy, int wx,
                                                      uint64_t* __restrict__ keys,
                                                      uint32_t* __restrict__ vals,
                                                      int32_t* __restrict__ status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    uint64_t key = kInvalidKey;
    if (coord_valid(c, shape, batch)) {
        key = ((((static_cast<uint64_t>(c.x) << wx) | static_cast<uint64_t>(c.y + 1)) << wy |
                static_cast<uint64_t>(c.z + 1))
               << wz) |
              static_cast<uint64_t>(c.w + 1);
    } else {
        atomicOr(status, kStatusRange);
    }
    keys[i] = key;
    vals[i] = static_cast<uint32_t>(i);
}

// First index in [lo, hi) with keys[idx] >= t (hi if none).
__device__ __forceinline__ int64_t lower_bound(const uint64_t* __restrict__ keys, int64_t lo,
                                               int64_t hi, uint64_t t) {
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (__ldg(keys + mid) < t)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// Adds the per-block tap counts of this thread's mask to smem counters with
// one atomic per distinct (warp, tap).
__device__ __forceinline__ void count_taps(uint32_t m, int32_t* cnt) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
        if (lane == 0 && b) atomicAdd(&cnt[k], __popc(b));
    }
}

__device__ __forceinline__ void store_nbr_row(int32_t* __restrict__ nbr, int64_t r,
                                              const int32_t (&v)[kNbrStride]) {
    int4* dst = reinterpret_cast<int4*>(nbr + r * kNbrStride);
#pragma unroll
    for (int q = 0; q < kNbrStride / 4; ++q) dst[q] = make_int4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// One thread per sorted position s.  Finds the 27 neighbours of the voxel at
// s: for each of the 9 (dx, dy) columns one lower_bound on the key of
// (dx, dy, dz = -1), then at most 3 consecutive keys for dz = -1, 0, +1.
__global__ void __launch_bounds__(kBlock) k_search(const uint64_t* __restrict__ skeys,
                                                   const uint32_t* __restrict__ svals, int64_t n,
                                                   KeyLayout lay, int32_t* __restrict__ nbr,
                                                   uint32_t* __restrict__ mask,
                                                   int32_t* __restrict__ tap_count,
                                                   int32_t* __restrict__ status) {
    __shared__ int32_t cnt[kTaps];
    if (threadIdx.x < kTaps) cnt[threadIdx.x] = 0;
    __syncthreads();
    const int64_t s = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    uint32_t m = 0;
    if (s < n) {
        const uint64_t q = skeys[s];
        const int64_t r = svals[s];
        int32_t v[kNbrStride];
#pragma unroll
        for (int k = 0; k < kNbrStride; ++k) v[k] = -1;
        if (q != kInvalidKey) {
            if (s > 0 && skeys[s - 1] == q) atomicOr(status, kStatusDuplicate);
#pragma unroll
            for (int c = 0; c < 9; ++c) {
                const uint64_t lo_t = q + lay.off[3 * c];
                const uint64_t hi_t = q + lay.off[3 * c + 2];
                // columns before (dx,dy)=(0,0) hold smaller keys, after it larger ones
                int64_t lo = 0, hi = n;
                if (c < 4) hi = s;
                if (c > 4) lo = s + 1;
                if (c == 4) {
                    lo = s > 0 ? s - 1 : 0;
                    hi = s + 2 < n ? s + 2 : n;
                }
                const int64_t pos = lower_bound(skeys, lo, hi, lo_t);
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const int64_t p = pos + j;
                    if (p < n) {
                        const uint64_t kk = __ldg(skeys + p);
                        if (kk <= hi_t) {
                            const uint64_t dz = kk - lo_t;
                            const int32_t row = static_cast<int32_t>(__ldg(svals + p));
                            if (dz == 0) v[3 * c] = row;
                            if (dz == 1) v[3 * c + 1] = row;
                            if (dz == 2) v[3 * c + 2] = row;
                        }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kTaps; ++k) m |= (v[k] >= 0 ? 1u : 0u) << k;
        }
        store_nbr_row(nbr, r, v);
        mask[r] = m;
    }
    count_taps(m, cnt);
    __syncthreads();
    if (threadIdx.x < kTaps && cnt[threadIdx.x]) atomicAdd(&tap_count[threadIdx.x], cnt[threadIdx.x]);
}

// ---------------------------------------------------------------------------
// dense presence-grid mapper
// ---------------------------------------------------------------------------
struct GridLayout {
    int64_t sy, sx, sb;   // strides of y, x, b in cells (z stride 1)
    int64_t off[kTaps];   // cell offset of each tap
};

__device__ __forceinline__ int64_t grid_cell(int4 c, const GridLayout& g) {
    return c.x * g.sb + static_cast<int64_t>(c.y + 1) * g.sx + static_cast<int64_t>(c.z + 1) * g.sy +
           (c.w + 1);
}

__global__ void __launch_bounds__(kBlock) k_grid_scatter(const int4* __restrict__ coords, int64_t n,
                                                         int3 shape, int batch, GridLayout g,
                                                         int32_t* __restrict__ grid,
                                                         int32_t* __restrict__ status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    if (!coord_valid(c, shape, batch)) {
        atomicOr(status, kStatusRange);
        return;
    }
    const int32_t prev = atomicCAS(grid + grid_cell(c, g), -1, static_cast<int32_t>(i));
    if (prev != -1) atomicOr(status, kStatusDuplicate);
}

__global__ void __launch_bounds__(kBlock) k_grid_lookup(const int4* __restrict__ coords, int64_t n,
                                                        int3 shape, int batch, GridLayout g,
                                                        const int32_t* __restrict__ grid,
                                                        int32_t* __restrict__ nbr,
                                                        uint32_t* __restrict__ mask,
                                                        int32_t* __restrict__ tap_count) {
    __shared__ int32_t cnt[kTaps];
    if (threadIdx.x < kTaps) cnt[threadIdx.x] = 0;
    __syncthreads();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    uint32_t m = 0;
    if (i < n) {
        const int4 c = coords[i];
        int32_t v[kNbrStride];
#pragma unroll
        for (int k = 0; k < kNbrStride; ++k) v[k] = -1;
        if (coord_valid(c, shape, batch)) {
            const int64_t cell = grid_cell(c, g);
#pragma unroll
            for (int k = 0; k < kTaps; ++k) {
                v[k] = __ldg(grid + cell + g.off[k]);
                m |= (v[k] >= 0 ? 1u : 0u) << k;
            }
        }
        store_nbr_row(nbr, i, v);
        mask[i] = m;
    }
    count_taps(m, cnt);
    __syncthreads();
    if (threadIdx.x < kTaps && cnt[threadIdx.x]) atomicAdd(&tap_count[threadIdx.x], cnt[threadIdx.x]);
}

// ---------------------------------------------------------------------------
// mask order
// ---------------------------------------------------------------------------
// tap_pos[k] = key bit of tap k.  Calibrated: taps ranked by descending count
// (ties by ascending tap), the most frequent tap at bit 0.
__global__ void k_tap_order(const int32_t* __restrict__ tap_count, int calibrated,
                            int32_t* __restrict__ tap_pos) {
    const int k = threadIdx.x;
    if (k >= kTaps) return;
    if (!calibrated) {
        tap_pos[k] = k;
        return;
    }
    const int32_t ck = tap_count[k];
    int rank = 0;
    for (int j = 0; j < kTaps; ++j) {
        const int32_t cj = tap_count[j];
        rank += (cj > ck || (cj == ck && j < k)) ? 1 : 0;
    }
    tap_pos[k] = rank;
}

__global__ void __launch_bounds__(kBlock) k_mask_keys(const uint32_t* __restrict__ mask, int64_t n,
                                                      const int32_t* __restrict__ tap_pos,
                                                      uint32_t* __restrict__ keys,
                                                      uint32_t* __restrict__ vals) {
    __shared__ int32_t pos[kTaps];
    if (threadIdx.x < kTaps) pos[threadIdx.x] = tap_pos[threadIdx.x];
    __syncthreads();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (i >= n) return;
    const uint32_t m = mask[i];
    uint32_t key = 0;
#pragma unroll
    for (int k = 0; k < kTaps; ++k) key |= ((m >> k) & 1u) << pos[k];
    keys[i] = key;
    vals[i] = static_cast<uint32_t>(i);
}

// ---------------------------------------------------------------------------
// compaction: per-(tap, tile) counts -> scan -> pair lists, gather table
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTileRows) k_tile_count(const int32_t* __restrict__ perm,
                                                          const uint32_t* __restrict__ mask, int64_t n,
                                                          int64_t n_tiles, int32_t* __restrict__ counts,
                                                          uint32_t* __restrict__ tile_union) {
    __shared__ int32_t wc[kTileRows / 32][kTaps];
    const int64_t t = blockIdx.x;
    const int64_t s = t * kTileRows + threadIdx.x;
    const uint32_t m = s < n ? mask[perm[s]] : 0u;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
        if (lane == 0) wc[warp][k] = __popc(b);
    }
    __syncthreads();
    if (threadIdx.x < kTaps) {
        int32_t c = 0;
        for (int w = 0; w < kTileRows / 32; ++w) c += wc[w][threadIdx.x];
        counts[threadIdx.x * n_tiles + t] = c;
        const uint32_t u = __ballot_sync(0x07FFFFFFu, c > 0);
        if (threadIdx.x == 0) tile_union[t] = u;
    }
}

// One block: exclusive scan of counts[27][T] into seg_off, tap offsets, totals,
// and the tiles ordered by descending union size (stable).
__global__ void __launch_bounds__(1024) k_scan_tiles(const int32_t* __restrict__ counts,
                                                     int64_t n_tiles, const uint32_t* __restrict__ tile_union,
                                                     int32_t* __restrict__ seg_off,
                                                     int32_t* __restrict__ tap_off,
                                                     int32_t* __restrict__ totals,
                                                     int32_t* __restrict__ tile_order) {
    __shared__ int32_t hist[kTaps + 1];
    if (threadIdx.x <= kTaps) hist[threadIdx.x] = 0;
    const int64_t m = kTaps * n_tiles;
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
        tap_off[kTaps] = total;
        totals[0] = total;
    }
    if (n_tiles == 0 && threadIdx.x < kTaps) tap_off[threadIdx.x] = 0;
    __syncthreads();
    // counting sort of tiles by descending union size (27..0), stable in t
    int32_t tap_sum = 0;
    for (int64_t t = threadIdx.x; t < n_tiles; t += 1024) {
        const int c = __popc(tile_union[t]);
        atomicAdd(&hist[kTaps - c], 1);
        tap_sum += c;
    }
    // one atomic per warp
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tap_sum += __shfl_down_sync(0xFFFFFFFFu, tap_sum, o);
    if ((threadIdx.x & 31) == 0 && tap_sum != 0) atomicAdd(&totals[1], tap_sum);
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t r = 0;
        for (int b = 0; b <= kTaps; ++b) {
            const int32_t c = hist[b];
            hist[b] = r;
            r += c;
        }
    }
    __syncthreads();
    // stable scatter by warp 0, 32 tiles at a time: each at its bucket's next
    // free position, tiles of one bucket in t order
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const uint32_t lt = rsort::lanemask_lt();
        for (int64_t t0 = 0; t0 < n_tiles; t0 += 32) {
            const int64_t t = t0 + lane;
            const int b = t < n_tiles ? kTaps - __popc(tile_union[t]) : kTaps + 1;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, b);
            if (b <= kTaps) tile_order[hist[b] + __popc(peers & lt)] = static_cast<int32_t>(t);
            __syncwarp();
            if (b <= kTaps && lane == __ffs(peers) - 1) hist[b] += __popc(peers);
            __syncwarp();
        }
    }
}

__global__ void __launch_bounds__(kTileRows) k_tile_write(int32_t* __restrict__ perm,
                                                          const uint32_t* __restrict__ mask,
                                                          const int32_t* __restrict__ nbr, int64_t n,
                                                          int64_t n_tiles, int64_t n_pad,
                                                          const int32_t* __restrict__ seg_off,
                                                          int32_t* __restrict__ in_rows,
                                                          int32_t* __restrict__ out_rows,
                                                          int32_t* __restrict__ gtab) {
    __shared__ int32_t wc[kTileRows / 32][kTaps];
    const int64_t t = blockIdx.x;
    const int64_t s = t * kTileRows + threadIdx.x;
    const bool valid = s < n;
    const int32_t r = valid ? perm[s] : -1;
    if (!valid) perm[s] = -1;
    const uint32_t m = valid ? mask[r] : 0u;
    int32_t v[kNbrStride];
    if (valid) {
        const int4* src = reinterpret_cast<const int4*>(nbr + static_cast<int64_t>(r) * kNbrStride);
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
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t ball[kTaps];
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
        ball[k] = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
        if (lane == 0) wc[warp][k] = __popc(ball[k]);
    }
    __syncthreads();
    const uint32_t lt = rsort::lanemask_lt();
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
        const bool present = (m >> k) & 1u;
        if (present) {
            int32_t off = seg_off[k * n_tiles + t] + __popc(ball[k] & lt);
            for (int w = 0; w < warp; ++w) off += wc[w][k];
            in_rows[off] = v[k];
            out_rows[off] = r;
        }
        gtab[k * n_pad + s] = present ? v[k] : -1;
    }
}

// ---------------------------------------------------------------------------
// derived shape / batch
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBlock) k_coord_extent(const int4* __restrict__ coords, int64_t n,
                                                         int32_t* __restrict__ ext) {
    int4 mx = make_int4(-1, -1, -1, -1);
    int mn = 0;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * kBlock) {
        const int4 c = coords[i];
        mx.x = max(mx.x, c.x);
        mx.y = max(mx.y, c.y);
        mx.z = max(mx.z, c.z);
        mx.w = max(mx.w, c.w);
        mn = min(mn, min(min(c.x, c.y), min(c.z, c.w)));
    }
    atomicMax(ext + 0, mx.x);
    atomicMax(ext + 1, mx.y);
    atomicMax(ext + 2, mx.z);
    atomicMax(ext + 3, mx.w);
    atomicMin(ext + 4, mn);
}

template <typename T>
T* carve(char*& p, size_t count) {
    T* r = reinterpret_cast<T*>(p);
    p += (count * sizeof(T) + 255) / 256 * 256;
    return r;
}

inline unsigned blocks_for(int64_t n, int per) { return static_cast<unsigned>((n + per - 1) / per); }

}  // namespace

int derive_shape(const int32_t* coords, int64_t n, cudaStream_t stream, int32_t shape[3],
                 int32_t* batch) {
    int32_t* ext = nullptr;
    SPCONV_CHECK_CUDA(cudaMallocAsync(&ext, 8 * sizeof(int32_t), stream));
    int32_t init[8] = {-1, -1, -1, -1, 0, 0, 0, 0};
    cudaError_t e = cudaMemcpyAsync(ext, init, sizeof(init), cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && n > 0) {
        const unsigned grid = std::min<int64_t>(blocks_for(n, kBlock), 1024);
        k_coord_extent<<<grid, kBlock, 0, stream>>>(reinterpret_cast<const int4*>(coords), n, ext);
        count_launch();
        e = cudaGetLastError();
    }
    int32_t host[8];
    if (e == cudaSuccess) e = cudaMemcpyAsync(host, ext, sizeof(host), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    cudaFreeAsync(ext, stream);
    if (e != cudaSuccess) return SPCONV_ERR_CUDA;
    if (host[4] < 0) return SPCONV_ERR_COORD_RANGE;
    if (shape) {
        shape[0] = std::max(1, host[1] + 1);
        shape[1] = std::max(1, host[2] + 1);
        shape[2] = std::max(1, host[3] + 1);
    }
    if (batch) *batch = std::max(1, host[0] + 1);
    return SPCONV_OK;
}

int build_map_impl(MapHandle* h, const int32_t* coords, const spconv_options_t* opt) {
    if (h->kernel_size != 3 || h->groups != 1) return build_map_grouped(h, coords, opt);
    cudaStream_t s = h->stream;
    const int64_t n = h->n;
    const int64_t T = (n + kTileRows - 1) / kTileRows;
    h->n_tiles = T;
    h->n_pad = T * kTileRows;
    const int X = h->shape[0], Y = h->shape[1], Z = h->shape[2], B = h->batch;

    // key layout over padded extents (coordinate + 1 in [1, extent], neighbours in [0, extent + 1])
    KeyLayout lay;
    lay.wz = bit_length(static_cast<uint64_t>(Z) + 1);
    lay.wy = bit_length(static_cast<uint64_t>(Y) + 1);
    lay.wx = bit_length(static_cast<uint64_t>(X) + 1);
    lay.wb = bit_length(static_cast<uint64_t>(B) - 1);
    const int key_bits = lay.wz + lay.wy + lay.wx + lay.wb;
    h->key_bits = key_bits;
    for (int dx = -1; dx <= 1; ++dx)
        for (int dy = -1; dy <= 1; ++dy)
            for (int dz = -1; dz <= 1; ++dz) {
                const int64_t o = static_cast<int64_t>(dx) * (int64_t(1) << (lay.wy + lay.wz)) +
                                  static_cast<int64_t>(dy) * (int64_t(1) << lay.wz) + dz;
                lay.off[9 * (dx + 1) + 3 * (dy + 1) + (dz + 1)] = static_cast<uint64_t>(o);
            }

    const int64_t cells = static_cast<int64_t>(B) * (X + 2) * (Y + 2) * (Z + 2);
    const bool cells_overflow = static_cast<double>(B) * (X + 2) * (Y + 2) * (Z + 2) > 9.0e18;
    int mapper = opt ? opt->mapper : SPCONV_MAPPER_AUTO;
    const int64_t dense_max = (opt && opt->dense_max_cells > 0) ? opt->dense_max_cells : (int64_t(1) << 24);
    // AUTO: the dense grid on small boxes, else packed keys -- in a hash table
    // when the whole-GPU pipeline builds the map, else sorted (decided below)
    const bool auto_keys = mapper == SPCONV_MAPPER_AUTO && !(!cells_overflow && cells <= dense_max);
    if (mapper == SPCONV_MAPPER_AUTO) mapper = auto_keys ? SPCONV_MAPPER_SORTED : SPCONV_MAPPER_DENSE;
    if ((mapper == SPCONV_MAPPER_SORTED || mapper == SPCONV_MAPPER_HASH) && key_bits > 63) return SPCONV_ERR_UNSUPPORTED;
    if (mapper == SPCONV_MAPPER_DENSE && (cells_overflow || cells > (int64_t(1) << 34))) return SPCONV_ERR_UNSUPPORTED;
    h->bit_order = opt ? opt->bit_order : SPCONV_ORDER_CALIBRATED;
    h->gemm = (opt && opt->gemm == SPCONV_GEMM_TAP_MAJOR) ? SPCONV_GEMM_TAP_MAJOR : SPCONV_GEMM_TILE_UNION;

    // ---- pipeline: the whole-GPU one when the keys fit it, else one cluster
    // launch when the rows fit, else the plain one kernel per step
    const int row_bits = std::max(1, bit_length(static_cast<uint64_t>(n > 0 ? n - 1 : 0)));
    const int want = opt ? opt->pipeline : SPCONV_PIPELINE_AUTO;
    const bool packs = mapper == SPCONV_MAPPER_DENSE || key_bits + row_bits <= 64;
    const bool hash_ok = n <= kWideMaxRows && key_bits + row_bits <= 64 &&
                         (want == SPCONV_PIPELINE_AUTO || want == SPCONV_PIPELINE_WIDE);
    if (auto_keys && hash_ok) mapper = SPCONV_MAPPER_HASH;
    if (mapper == SPCONV_MAPPER_HASH && !hash_ok) return SPCONV_ERR_UNSUPPORTED;
    h->mapper = mapper;
    const bool wide_ok = n <= kWideMaxRows && packs &&
                         (mapper != SPCONV_MAPPER_SORTED || wide_key_passes(key_bits) <= kWideKeyPassesMax);
    bool fused_ok = n <= kFusedMaxRows && packs;
    int cluster = 0;
    if (fused_ok && (want == SPCONV_PIPELINE_FUSED || (want == SPCONV_PIPELINE_AUTO && !wide_ok)) && n > 0) {
        cluster = fused_cluster_size(s);
        fused_ok = cluster > 0;
    }
    if (want == SPCONV_PIPELINE_FUSED && !fused_ok) return SPCONV_ERR_UNSUPPORTED;
    if (want == SPCONV_PIPELINE_WIDE && !wide_ok) return SPCONV_ERR_UNSUPPORTED;
    const bool wide = want == SPCONV_PIPELINE_WIDE || (want == SPCONV_PIPELINE_AUTO && wide_ok);
    const bool fused = !wide && want != SPCONV_PIPELINE_MULTI && fused_ok;
    h->pipeline = wide ? SPCONV_PIPELINE_WIDE : fused ? SPCONV_PIPELINE_FUSED : SPCONV_PIPELINE_MULTI;

    // ---- one arena for everything the map keeps or needs while building
    const int64_t nb = std::max<int64_t>(1, rsort::num_tiles(n));
    const int64_t np = std::max<int64_t>(1, h->n_pad);
    const int64_t n1 = std::max<int64_t>(1, n);
    const int64_t t1 = std::max<int64_t>(1, T);
    const int64_t cl = std::max(1, cluster);
    size_t bytes = 0;
    auto add = [&](size_t count, size_t elem) { bytes += (count * elem + 255) / 256 * 256; };
    add(4, 4);                          // status (+ pad)
    add(n1 * kNbrStride, 4);            // nbr
    add(n1, 4);                         // mask
    add(kTaps, 4); add(kTaps, 4); add(kTaps + 1, 4); add(2, 4);  // tap_count, tap_pos, tap_off, totals
    add(kTaps * n1, 4); add(kTaps * n1, 4);                      // in_rows, out_rows
    add(kTaps * np, 4);                 // gtab
    add(t1, 4); add(t1, 4); add(kTaps * t1, 4); add(kTaps * t1, 4);  // union, order, counts, seg_off
    add(np, 4); add(np, 4);             // perm ping-pong
    const int64_t parts = std::max<int64_t>(1, (n + kWideKeysPerCta - 1) / kWideKeysPerCta);
    if (wide) {
        add(n1, 8); add(n1, 8);         // packed (key, row) ping-pong
        add((kWideKeyPassesMax + kWideMaskPasses) * kWideBins, 4); add(kWideCounters, 4);
        add(parts * kWideBins, 8);      // look-back states
    } else if (fused) {
        add(n1, 8); add(n1, 8);         // packed (key, row) ping-pong
        add(3 * cl * kFusedBins, 4); add(cl * kTaps, 4); add(cl * (kTaps + 1), 4);
    } else {
        add(n1, 4); add(n1, 4);         // mask-sort keys ping-pong
        add(rsort::kBins * nb, 4);      // radix histograms
        if (mapper == SPCONV_MAPPER_SORTED) {
            add(n1, 8); add(n1, 8); add(n1, 4); add(n1, 4);  // coordinate keys, row ids (ping-pong)
        }
    }
    if (mapper == SPCONV_MAPPER_DENSE) add(static_cast<size_t>(cells), 4);   // presence grid
    const int table_log2 = mapper == SPCONV_MAPPER_HASH ? hash_table_log2(n) : 0;
    if (mapper == SPCONV_MAPPER_HASH) add(size_t(1) << table_log2, 8);       // hash table
    void* arena = nullptr;
    if (pool_alloc(&arena, bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return SPCONV_ERR_OOM;
    }
    h->arena = arena;
    h->arena_bytes = bytes;
    char* p = static_cast<char*>(arena);
    h->status = carve<int32_t>(p, 4);
    h->nbr = carve<int32_t>(p, n1 * kNbrStride);
    h->mask = carve<uint32_t>(p, n1);
    h->tap_count = carve<int32_t>(p, kTaps);
    h->tap_pos = carve<int32_t>(p, kTaps);
    h->tap_off = carve<int32_t>(p, kTaps + 1);
    h->totals = carve<int32_t>(p, 2);
    h->in_rows = carve<int32_t>(p, kTaps * n1);
    h->out_rows = carve<int32_t>(p, kTaps * n1);
    h->gtab = carve<int32_t>(p, kTaps * np);
    h->tile_union = carve<uint32_t>(p, t1);
    h->tile_order = carve<int32_t>(p, t1);
    int32_t* counts = carve<int32_t>(p, kTaps * t1);
    h->seg_off = carve<int32_t>(p, kTaps * t1);
    int32_t* perm_a = carve<int32_t>(p, np);
    int32_t* perm_b = carve<int32_t>(p, np);

    if (wide) {
        WideArgs wa;
        wa.va = carve<uint64_t>(p, n1);
        wa.vb = carve<uint64_t>(p, n1);
        wa.gh = carve<int32_t>(p, (kWideKeyPassesMax + kWideMaskPasses) * kWideBins);
        wa.tickets = carve<int32_t>(p, kWideCounters);
        wa.look = carve<uint64_t>(p, parts * kWideBins);
        wa.grid = mapper == SPCONV_MAPPER_DENSE ? carve<int32_t>(p, static_cast<size_t>(cells)) : nullptr;
        wa.table = mapper == SPCONV_MAPPER_HASH ? carve<uint64_t>(p, size_t(1) << table_log2) : nullptr;
        wa.table_log2 = table_log2;
        h->perm = perm_a;
        if (n == 0) {
            SPCONV_CHECK_CUDA(cudaMemsetAsync(h->status, 0, 256, s));
            SPCONV_CHECK_CUDA(cudaMemsetAsync(h->tap_off, 0, 256, s));
            SPCONV_CHECK_CUDA(cudaMemsetAsync(h->totals, 0, 256, s));
            return cuda_status(cudaGetLastError());
        }
        wa.coords = reinterpret_cast<const int4*>(coords);
        wa.n = n;
        wa.shape = make_int3(X, Y, Z);
        wa.batch = B;
        wa.mapper = mapper;
        wa.calibrated = h->bit_order == SPCONV_ORDER_CALIBRATED;
        wa.wz = lay.wz;
        wa.wy = lay.wy;
        wa.wx = lay.wx;
        wa.key_bits = key_bits;
        wa.row_bits = row_bits;
        for (int k = 0; k < kTaps; ++k) wa.koff[k] = lay.off[k];
        wa.gsy = Z + 2;
        wa.gsx = static_cast<int64_t>(Y + 2) * (Z + 2);
        wa.gsb = static_cast<int64_t>(X + 2) * wa.gsx;
        wa.cells = cells;
        for (int dx = -1; dx <= 1; ++dx)
            for (int dy = -1; dy <= 1; ++dy)
                for (int dz = -1; dz <= 1; ++dz)
                    wa.goff[9 * (dx + 1) + 3 * (dy + 1) + (dz + 1)] = dx * wa.gsx + dy * wa.gsy + dz;
        wa.nbr = h->nbr;
        wa.mask = h->mask;
        wa.tap_count = h->tap_count;
        wa.perm = h->perm;
        wa.tap_off = h->tap_off;
        wa.totals = h->totals;
        wa.in_rows = h->in_rows;
        wa.out_rows = h->out_rows;
        wa.gtab = h->gtab;
        wa.tile_union = h->tile_union;
        wa.tile_order = h->tile_order;
        wa.seg_off = h->seg_off;
        wa.status = h->status;
        wa.n_tiles = T;
        wa.n_pad = h->n_pad;
        int sms = 0;
        SPCONV_CHECK_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device));
        return launch_map_wide(wa, sms, s);
    }

    if (fused) {
        FusedArgs fa;
        fa.va = carve<uint64_t>(p, n1);
        fa.vb = carve<uint64_t>(p, n1);
        fa.hist = carve<int32_t>(p, 3 * cl * kFusedBins);
        fa.cta_tot = carve<int32_t>(p, cl * kTaps);
        fa.cta_bkt = carve<int32_t>(p, cl * (kTaps + 1));
        fa.grid = mapper == SPCONV_MAPPER_DENSE ? carve<int32_t>(p, static_cast<size_t>(cells)) : nullptr;
        h->perm = perm_a;
        if (n == 0) {
            SPCONV_CHECK_CUDA(cudaMemsetAsync(h->status, 0, 256, s));
            SPCONV_CHECK_CUDA(cudaMemsetAsync(h->tap_off, 0, 256, s));
            SPCONV_CHECK_CUDA(cudaMemsetAsync(h->totals, 0, 256, s));
            return cuda_status(cudaGetLastError());
        }
        fa.coords = reinterpret_cast<const int4*>(coords);
        fa.n = n;
        fa.shape = make_int3(X, Y, Z);
        fa.batch = B;
        fa.mapper = mapper;
        fa.calibrated = h->bit_order == SPCONV_ORDER_CALIBRATED;
        fa.wz = lay.wz;
        fa.wy = lay.wy;
        fa.wx = lay.wx;
        fa.key_bits = key_bits;
        fa.row_bits = row_bits;
        for (int k = 0; k < kTaps; ++k) fa.koff[k] = lay.off[k];
        fa.gsy = Z + 2;
        fa.gsx = static_cast<int64_t>(Y + 2) * (Z + 2);
        fa.gsb = static_cast<int64_t>(X + 2) * fa.gsx;
        fa.cells = cells;
        for (int dx = -1; dx <= 1; ++dx)
            for (int dy = -1; dy <= 1; ++dy)
                for (int dz = -1; dz <= 1; ++dz)
                    fa.goff[9 * (dx + 1) + 3 * (dy + 1) + (dz + 1)] = dx * fa.gsx + dy * fa.gsy + dz;
        fa.nbr = h->nbr;
        fa.mask = h->mask;
        fa.tap_count = h->tap_count;
        fa.perm = h->perm;
        fa.tap_off = h->tap_off;
        fa.totals = h->totals;
        fa.in_rows = h->in_rows;
        fa.out_rows = h->out_rows;
        fa.gtab = h->gtab;
        fa.tile_union = h->tile_union;
        fa.tile_order = h->tile_order;
        fa.seg_off = h->seg_off;
        fa.status = h->status;
        fa.n_tiles = T;
        fa.n_pad = h->n_pad;
        return launch_map_fused(fa, cluster, s);
    }

    uint32_t* mkey_a = carve<uint32_t>(p, n1);
    uint32_t* mkey_b = carve<uint32_t>(p, n1);
    int32_t* hist = carve<int32_t>(p, rsort::kBins * nb);
    uint64_t *ckey_a = nullptr, *ckey_b = nullptr;
    uint32_t *cval_a = nullptr, *cval_b = nullptr;
    int32_t* grid = nullptr;
    if (mapper == SPCONV_MAPPER_SORTED) {
        ckey_a = carve<uint64_t>(p, n1);
        ckey_b = carve<uint64_t>(p, n1);
        cval_a = carve<uint32_t>(p, n1);
        cval_b = carve<uint32_t>(p, n1);
    } else {
        grid = carve<int32_t>(p, static_cast<size_t>(cells));
    }

    // status, tap counters, totals: zero (they are contiguous in the arena's head)
    SPCONV_CHECK_CUDA(cudaMemsetAsync(h->status, 0, 256, s));
    SPCONV_CHECK_CUDA(cudaMemsetAsync(h->tap_count, 0, 256, s));
    SPCONV_CHECK_CUDA(cudaMemsetAsync(h->totals, 0, 256, s));
    if (n == 0) {
        SPCONV_CHECK_CUDA(cudaMemsetAsync(h->tap_off, 0, 256, s));
        h->perm = perm_a;
        return cuda_status(cudaGetLastError());
    }

    const int4* c4 = reinterpret_cast<const int4*>(coords);
    const int3 shape3 = make_int3(X, Y, Z);
    int launches = 0;
    if (mapper == SPCONV_MAPPER_SORTED) {
        k_pack_keys<<<blocks_for(n, kBlock), kBlock, 0, s>>>(c4, n, shape3, B, lay.wz, lay.wy, lay.wx,
                                                            ckey_a, cval_a, h->status);
        ++launches;
        // out-of-range rows carry the all-ones key: sort all 64 bits if any could be present
        const bool in_b = rsort::sort_pairs<uint64_t>(ckey_a, cval_a, ckey_b, cval_b, n,
                                                      std::min(64, key_bits + 1), hist, s, &launches);
        const uint64_t* sk = in_b ? ckey_b : ckey_a;
        const uint32_t* sv = in_b ? cval_b : cval_a;
        k_search<<<blocks_for(n, kBlock), kBlock, 0, s>>>(sk, sv, n, lay, h->nbr, h->mask, h->tap_count,
                                                          h->status);
        ++launches;
    } else {
        GridLayout g;
        g.sy = Z + 2;
        g.sx = static_cast<int64_t>(Y + 2) * (Z + 2);
        g.sb = static_cast<int64_t>(X + 2) * g.sx;
        for (int dx = -1; dx <= 1; ++dx)
            for (int dy = -1; dy <= 1; ++dy)
                for (int dz = -1; dz <= 1; ++dz)
                    g.off[9 * (dx + 1) + 3 * (dy + 1) + (dz + 1)] = dx * g.sx + dy * g.sy + dz;
        SPCONV_CHECK_CUDA(cudaMemsetAsync(grid, 0xFF, static_cast<size_t>(cells) * 4, s));
        k_grid_scatter<<<blocks_for(n, kBlock), kBlock, 0, s>>>(c4, n, shape3, B, g, grid, h->status);
        k_grid_lookup<<<blocks_for(n, kBlock), kBlock, 0, s>>>(c4, n, shape3, B, g, grid, h->nbr, h->mask,
                                                               h->tap_count);
        launches += 2;
    }
    k_tap_order<<<1, 32, 0, s>>>(h->tap_count, h->bit_order == SPCONV_ORDER_CALIBRATED, h->tap_pos);
    k_mask_keys<<<blocks_for(n, kBlock), kBlock, 0, s>>>(h->mask, n, h->tap_pos, mkey_a,
                                                         reinterpret_cast<uint32_t*>(perm_a));
    launches += 2;
    const bool perm_in_b = rsort::sort_pairs<uint32_t>(mkey_a, reinterpret_cast<uint32_t*>(perm_a), mkey_b,
                                                       reinterpret_cast<uint32_t*>(perm_b), n, kTaps, hist, s,
                                                       &launches);
    h->perm = perm_in_b ? perm_b : perm_a;
    k_tile_count<<<static_cast<unsigned>(T), kTileRows, 0, s>>>(h->perm, h->mask, n, T, counts, h->tile_union);
    k_scan_tiles<<<1, 1024, 0, s>>>(counts, T, h->tile_union, h->seg_off, h->tap_off, h->totals,
                                    h->tile_order);
    k_tile_write<<<static_cast<unsigned>(T), kTileRows, 0, s>>>(h->perm, h->mask, h->nbr, n, T, h->n_pad,
                                                                h->seg_off, h->in_rows, h->out_rows, h->gtab);
    launches += 3;
    count_launch(launches);
    return cuda_status(cudaGetLastError());
}

}  // namespace spconv

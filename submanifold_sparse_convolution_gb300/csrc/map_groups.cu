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
#include "map_internal.cuh"
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
// Launch with programmatic dependent launch: the kernel may be scheduled
// while the kernel before it finishes (that kernel's CTAs have all started);
// every kernel launched this way begins with pdl_trigger(); pdl_wait(), so it
// touches global memory only once the kernels before it have completed.
template <typename Kernel, typename... Args>
int launch_chained(Kernel kernel, unsigned grid, unsigned block, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kernel, args...));
}

// grid of a grid-stride kernel over n entries (kGBlock threads per CTA)
inline unsigned capped_blocks(int64_t n) {
    const unsigned b = blocks(n, kGBlock);
    return b < 2048 ? (b < 1 ? 1 : b) : 2048;
}

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
    pdl_trigger();
    pdl_wait();
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

// The same keys packed with the row for the whole-GPU sort: (key << rbits) |
// row, the key kb = key_bits + 1 bits wide (all ones for an out-of-range
// row, which orders it last); counts the digits of the passes in d (the
// caller passes none where no pass reads the totals).  Grid-stride, so that
// whole warps take part in the digit counts.
__global__ void __launch_bounds__(kGBlock) kg_pack_keys_packed(const int4* __restrict__ coords, int64_t n, int3 shape,
                                                               int batch, const GLayout L, int kb, int rbits,
                                                               const WideDigits d, uint64_t* __restrict__ packed,
                                                               int32_t* __restrict__ gh,
                                                               int32_t* __restrict__ status) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t h[kWideKeyPassesMax][kWideBins];
    for (int i = threadIdx.x; i < kWideKeyPassesMax * kWideBins; i += kGBlock) (&h[0][0])[i] = 0;
    __syncthreads();
    const uint64_t none = (uint64_t(1) << kb) - 1;
    int32_t err = 0;
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * kGBlock; i0 < n; i0 += static_cast<int64_t>(gridDim.x) * kGBlock) {
        const int64_t i = i0 + threadIdx.x;
        const bool valid = i < n;
        uint64_t v = 0;
        if (valid) {
            const int4 c = coords[i];
            uint64_t key = none;
            if (in_range(c, shape, batch)) {
                key = ((((static_cast<uint64_t>(c.x) << L.wx) | static_cast<uint64_t>(c.y + L.r)) << L.wy |
                        static_cast<uint64_t>(c.z + L.r))
                       << L.wz) |
                      static_cast<uint64_t>(c.w + L.r);
            } else {
                err |= kStatusRange;
            }
            v = (key << rbits) | static_cast<uint64_t>(i);
            packed[i] = v;
        }
        wide_count_digits(v, valid, d, h);
    }
    if (err) atomicOr(status, err);
    __syncthreads();
    wide_flush_digits(d, h, gh);
}

// One thread per sorted position s: for each (dx, dy) column, the lower bound
// of (dx, dy, -r) and the K keys from there.  Columns before the centre column
// hold smaller keys than the row's own, columns after it larger ones, so each
// search runs on one side of s.  nbr is cleared to -1 beforehand; only the
// present neighbours are written.
// kPacked: skeys holds (key << rbits) | row (the whole-GPU sort's values),
// no_key the key of an out-of-range row; else keys and rows are separate.
template <bool kPacked>
__global__ void __launch_bounds__(kGBlock) kg_search(const uint64_t* __restrict__ skeys,
                                                     const uint32_t* __restrict__ svals, int64_t n, int rbits,
                                                     uint64_t no_key, const GLayout L, int32_t* __restrict__ nbr,
                                                     int32_t* __restrict__ tap_count,
                                                     int32_t* __restrict__ status) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t cnt[kMaxTaps];
    for (int k = threadIdx.x; k < L.V; k += kGBlock) cnt[k] = 0;
    __syncthreads();
    const uint64_t rmask = (uint64_t(1) << rbits) - 1;
    auto key_at = [&](int64_t p) -> uint64_t { return kPacked ? (__ldcg(skeys + p) >> rbits) : __ldcg(skeys + p); };
    auto row_at = [&](int64_t p) -> int64_t {
        return kPacked ? static_cast<int64_t>(__ldcg(skeys + p) & rmask) : static_cast<int64_t>(__ldcg(svals + p));
    };
    const int64_t s = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (s < n) {
        const uint64_t q = key_at(s);
        const int64_t row = row_at(s);
        if (q != no_key) {
            if (s > 0 && key_at(s - 1) == q) atomicOr(status, kStatusDuplicate);
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
                int64_t pos = lo, top = hi;   // first position in [lo, hi) with key >= lo_t
                while (pos < top) {
                    const int64_t mid = (pos + top) >> 1;
                    if (key_at(mid) < lo_t)
                        pos = mid + 1;
                    else
                        top = mid;
                }
                for (int j = 0; j < L.K; ++j) {
                    const int64_t p = pos + j;
                    if (p >= n) break;
                    const uint64_t kk = key_at(p);
                    if (kk > hi_t) break;
                    const int k = c * L.K + static_cast<int>(kk - lo_t);
                    nbr[row * L.stride + k] = static_cast<int32_t>(row_at(p));
                    atomicAdd(&cnt[k], 1);
                }
            }
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < L.V; k += kGBlock)
        if (cnt[k]) atomicAdd(&tap_count[k], cnt[k]);
}

// The kernel-map row width of kernel size K (V taps rounded up to whole
// 16-byte words), which the staged search and lookup below write whole.
template <int K>
struct NbrStride {
    static constexpr int value = (K * K * K + 3) / 4 * 4;
};

// A block's kernel-map rows, assembled in shared memory (initialised to -1)
// and written whole, 16 bytes a thread: rows_s[j] goes to row rid(j) of nbr
// (skipped when rid(j) < 0).  Every thread of the block calls it.
template <int RB, int ST, typename RowOf>
__device__ __forceinline__ void write_rows(const int32_t (&rows_s)[RB][ST], RowOf rid, int32_t* __restrict__ nbr) {
    static_assert(ST % 4 == 0, "rows of whole 16-byte words");
    constexpr int Q = ST / 4;
    for (int t = threadIdx.x; t < RB * Q; t += blockDim.x) {
        const int j = t / Q, c = t % Q;
        const int64_t r = rid(j);
        if (r >= 0)
            reinterpret_cast<int4*>(nbr + r * ST)[c] = reinterpret_cast<const int4*>(&rows_s[j][0])[c];
    }
}

// The same search over the packed values (key << rbits | row) for kernel size
// K, with the K^2 column searches of a row in lockstep: every step of the
// binary searches issues the probes of all columns still open at once, and
// the K keys after every lower bound are read together, so a row waits
// ~log2(n) memory round trips rather than K^2 log2(n).
// The block's rows (at their original row index, scattered) are assembled in
// shared memory and written whole, so the map needs no -1 fill first (kernel
// size 5: its 16.6 MB memset and ~50 scattered 4-byte stores per row gone).
template <int K>
struct LockRows {   // rows per block; K threads per row, one per dx plane
    static constexpr int value = K == 3 ? 128 : 64;
};

template <int K>
__global__ void __launch_bounds__(LockRows<K>::value * K) kg_search_lockstep(const uint64_t* __restrict__ sv, int64_t n,
                                                                             int rbits, uint64_t no_key, const GLayout L,
                                                                             int32_t* __restrict__ nbr,
                                                                             int32_t* __restrict__ tap_count,
                                                                             int32_t* __restrict__ status) {
    pdl_trigger();
    pdl_wait();
    constexpr int R = (K - 1) / 2, V = K * K * K, LR = LockRows<K>::value, ST = NbrStride<K>::value;
    __shared__ int32_t cnt[V];
    __shared__ __align__(16) int32_t rows_s[LR][ST];
    __shared__ int64_t rid[LR];
    for (int k = threadIdx.x; k < V; k += LR * K) cnt[k] = 0;
    for (int k = threadIdx.x; k < LR * ST; k += LR * K) (&rows_s[0][0])[k] = -1;
    const int plane = threadIdx.x / LR;   // dx = plane - R (warp-uniform)
    const int rl = threadIdx.x % LR;
    const uint64_t rmask = (uint64_t(1) << rbits) - 1;
    const int64_t s = static_cast<int64_t>(blockIdx.x) * LR + rl;
    bool ok = s < n;
    uint64_t q = 0;
    int64_t row = 0;
    if (ok) {
        const uint64_t v = __ldcg(sv + s);
        q = v >> rbits;
        row = static_cast<int64_t>(v & rmask);
        ok = q != no_key;
        if (ok && plane == R && s > 0 && (__ldcg(sv + s - 1) >> rbits) == q) atomicOr(status, kStatusDuplicate);
    }
    if (plane == 0) rid[rl] = s < n ? row : -1;   // (a row out of range is written as all -1)
    __syncthreads();
    if (ok) {
        // the plane's K columns c = K plane + e; those before the row's own
        // column hold smaller keys than its own, those after it larger ones
        int32_t lo[K], hi[K];
#pragma unroll
        for (int e = 0; e < K; ++e) {
            const int rel = (plane - R) * K + (e - R);   // sign of the column's offset from the row's own
            lo[e] = rel < 0 ? 0 : (rel > 0 ? static_cast<int32_t>(s + 1) : static_cast<int32_t>(s > R ? s - R : 0));
            hi[e] = rel < 0 ? static_cast<int32_t>(s)
                            : (rel > 0 ? static_cast<int32_t>(n) : static_cast<int32_t>(s + R + 1 < n ? s + R + 1 : n));
        }
        for (int it = 0; it < 40; ++it) {
            uint64_t kk[K];
#pragma unroll
            for (int e = 0; e < K; ++e) kk[e] = lo[e] < hi[e] ? (__ldcg(sv + ((lo[e] + hi[e]) >> 1)) >> rbits) : 0ull;
            bool open = false;
#pragma unroll
            for (int e = 0; e < K; ++e) {
                if (lo[e] < hi[e]) {
                    const int32_t mid = (lo[e] + hi[e]) >> 1;
                    if (kk[e] < q + L.col_off[plane * K + e])
                        lo[e] = mid + 1;
                    else
                        hi[e] = mid;
                    open |= lo[e] < hi[e];
                }
            }
            if (!open) break;
        }
        // at most K keys from each lower bound lie in the column (keys are unique)
#pragma unroll
        for (int e = 0; e < K; ++e) {
            const int c = plane * K + e;
            const uint64_t lo_t = q + L.col_off[c];
            uint64_t vv[K];
#pragma unroll
            for (int j = 0; j < K; ++j) vv[j] = lo[e] + j < n ? __ldcg(sv + lo[e] + j) : ~0ull;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const uint64_t d = (vv[j] >> rbits) - lo_t;
                if (vv[j] != ~0ull && d <= static_cast<uint64_t>(2 * R)) {
                    const int k = c * K + static_cast<int>(d);
                    rows_s[rl][k] = static_cast<int32_t>(vv[j] & rmask);
                    atomicAdd(&cnt[k], 1);
                }
            }
        }
    }
    __syncthreads();
    write_rows(rows_s, [&](int j) { return rid[j]; }, nbr);
    for (int k = threadIdx.x; k < V; k += LR * K)
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

// ---------------------------------------------------------------------------
// column index over the sorted keys: z is the key's lowest field, so the
// voxels of one (b, x, y) column are one run of the sorted array.  A table of
// (column key + 1, run start | run length << 32) entries, two per 32-byte
// bucket, lets a row find each of its K^2 neighbour columns with one bucket
// read and the run's few keys, instead of a binary search of ~log2(n) round
// trips per column.
// ---------------------------------------------------------------------------
constexpr int kColBucket = 2;   // entries (16 bytes each) per 32-byte bucket
constexpr int64_t kColIndexRows = 65536;

// Entries of the column table for n rows: at least 4 n (columns number at
// most n, so a bucket is rarely full), a power of two.
inline int col_table_log2(int64_t n) {
    int l = 11;
    while ((int64_t(1) << l) < 4 * std::max<int64_t>(1, n)) ++l;
    return l;
}

// The thread of each column's first sorted position measures the run and
// enters it; the table is zero before.  Out-of-range rows (the all-ones key)
// sort last and are skipped.
__global__ void __launch_bounds__(kGBlock) kg_col_insert(const uint64_t* __restrict__ sv, int64_t n, int rbits,
                                                         uint64_t no_key, int wz, int log2,
                                                         uint64_t* __restrict__ table,
                                                         int32_t* __restrict__ status) {
    pdl_trigger();
    pdl_wait();
    const int64_t s = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (s >= n) return;
    const uint64_t q = __ldcg(sv + s) >> rbits;
    if (q == no_key) return;
    const uint64_t ck = q >> wz;
    if (s > 0 && ((__ldcg(sv + s - 1) >> rbits) >> wz) == ck) return;   // not the run's first voxel
    int64_t e = s + 1;
    while (e < n) {
        const uint64_t qe = __ldcg(sv + e) >> rbits;
        if (qe == no_key || (qe >> wz) != ck) break;
        ++e;
    }
    const uint64_t val = static_cast<uint64_t>(s) | (static_cast<uint64_t>(e - s) << 32);
    const int lb = log2 - 1;   // buckets of kColBucket entries
    const uint64_t bmask = (uint64_t(1) << lb) - 1;
    uint64_t b = g_bucket(ck, lb);
    for (uint64_t probe = 0; probe <= bmask; ++probe, b = (b + 1) & bmask) {
        for (int j = 0; j < kColBucket; ++j) {
            uint64_t* ent = table + 2 * (b * kColBucket + j);
            if (atomicCAS(reinterpret_cast<unsigned long long*>(ent), 0ull,
                          static_cast<unsigned long long>(ck + 1)) == 0ull) {
                ent[1] = val;
                return;
            }
        }
    }
    atomicOr(status, kStatusInternal);   // a full table: cannot happen at load <= 1/4
}

// The sorted mapper's search through the column index (kernel size K, K
// threads per row, one per dx plane, LockRows<K> rows per block): a plane's K
// (dx, dy) columns are found with their bucket reads in flight together, then
// each column's dz window -- at most K consecutive keys of its run, from the
// first key at or past dz = -r -- is read; a run longer than K is first
// searched for that key (in lockstep over the plane's columns).  Rows are
// staged in shared memory and written whole, as in kg_search_lockstep.
template <int K>
__global__ void __launch_bounds__(LockRows<K>::value * K) kg_col_search(const uint64_t* __restrict__ sv, int64_t n,
                                                                        int rbits, uint64_t no_key, const GLayout L,
                                                                        int log2, const uint64_t* __restrict__ table,
                                                                        int32_t* __restrict__ nbr,
                                                                        int32_t* __restrict__ tap_count,
                                                                        int32_t* __restrict__ status) {
    pdl_trigger();
    pdl_wait();
    constexpr int R = (K - 1) / 2, V = K * K * K, LR = LockRows<K>::value, ST = NbrStride<K>::value;
    __shared__ int32_t cnt[V];
    __shared__ __align__(16) int32_t rows_s[LR][ST];
    __shared__ int64_t rid[LR];
    for (int k = threadIdx.x; k < V; k += LR * K) cnt[k] = 0;
    for (int k = threadIdx.x; k < LR * ST; k += LR * K) (&rows_s[0][0])[k] = -1;
    const int plane = threadIdx.x / LR;   // dx = plane - R (warp-uniform)
    const int rl = threadIdx.x % LR;
    const uint64_t rmask = (uint64_t(1) << rbits) - 1;
    const int64_t s = static_cast<int64_t>(blockIdx.x) * LR + rl;
    bool ok = s < n;
    uint64_t q = 0;
    int64_t row = 0;
    if (ok) {
        const uint64_t v = __ldcg(sv + s);
        q = v >> rbits;
        row = static_cast<int64_t>(v & rmask);
        ok = q != no_key;
        if (ok && plane == R && s > 0 && (__ldcg(sv + s - 1) >> rbits) == q) atomicOr(status, kStatusDuplicate);
    }
    if (plane == 0) rid[rl] = s < n ? row : -1;   // (a row out of range is written as all -1)
    __syncthreads();
    if (ok) {
        const int lb = log2 - 1;
        const uint64_t bmask = (uint64_t(1) << lb) - 1;
        const uint64_t zq = q & ((uint64_t(1) << L.wz) - 1);   // z + r >= r: zq - R >= 0
        // the plane's columns (the +r padding keeps every field in range: no borrow)
        uint64_t cke[K];
        ulonglong2 blo[K], bhi[K];
#pragma unroll
        for (int e = 0; e < K; ++e) {
            cke[e] = (q >> L.wz) + (static_cast<uint64_t>(static_cast<int64_t>(plane - R)) << L.wy) +
                     static_cast<uint64_t>(static_cast<int64_t>(e - R));
            g_load_bucket(table + 2 * kColBucket * g_bucket(cke[e], lb), blo[e], bhi[e]);
        }
        int64_t lo[K], hi[K], re[K];   // search range and run end of each column (empty when absent)
#pragma unroll
        for (int e = 0; e < K; ++e) {
            uint64_t val = 0;
            bool found = false;
            if (blo[e].x == cke[e] + 1) {
                val = blo[e].y;
                found = true;
            } else if (bhi[e].x == cke[e] + 1) {
                val = bhi[e].y;
                found = true;
            } else if (blo[e].x != 0ull && bhi[e].x != 0ull) {
                // a full bucket: the column may sit in the buckets after it (rare)
                uint64_t b = g_bucket(cke[e], lb);
                for (uint64_t probe = 1; probe <= bmask && !found; ++probe) {
                    b = (b + 1) & bmask;
                    ulonglong2 x, y;
                    g_load_bucket(table + 2 * kColBucket * b, x, y);
                    if (x.x == cke[e] + 1) {
                        val = x.y;
                        found = true;
                    } else if (y.x == cke[e] + 1) {
                        val = y.y;
                        found = true;
                    } else if (x.x == 0ull || y.x == 0ull) {
                        break;   // an empty slot: the column has no voxel
                    }
                }
            }
            lo[e] = found ? static_cast<int64_t>(val & 0xFFFFFFFFull) : 0;
            re[e] = found ? lo[e] + static_cast<int64_t>(val >> 32) : 0;
            if (re[e] > n || lo[e] > re[e]) {   // a corrupt entry: never read past the array
                atomicOr(status, kStatusInternal);
                lo[e] = re[e] = 0;
            }
            hi[e] = re[e] - lo[e] > K ? re[e] : lo[e];   // only a run longer than K is searched
        }
        // the first key at or past the column's dz = -r key (lower bound, in
        // lockstep over the plane's columns; a run is at most Z + 2r long)
        for (int it = 0; it < 40; ++it) {
            uint64_t kk[K];
#pragma unroll
            for (int e = 0; e < K; ++e) kk[e] = lo[e] < hi[e] ? (__ldcg(sv + ((lo[e] + hi[e]) >> 1)) >> rbits) : 0ull;
            bool open = false;
#pragma unroll
            for (int e = 0; e < K; ++e) {
                if (lo[e] < hi[e]) {
                    const int64_t mid = (lo[e] + hi[e]) >> 1;
                    if (kk[e] < (cke[e] << L.wz) + zq - R)
                        lo[e] = mid + 1;
                    else
                        hi[e] = mid;
                    open |= lo[e] < hi[e];
                }
            }
            if (!open) break;
        }
        // at most K keys from there lie in the column's dz window (keys are unique)
#pragma unroll
        for (int e = 0; e < K; ++e) {
            const int c = plane * K + e;
            const uint64_t lo_t = (cke[e] << L.wz) + zq - R;   // the column's dz = -r key
            uint64_t vv[K];
#pragma unroll
            for (int j = 0; j < K; ++j) vv[j] = lo[e] + j < re[e] ? __ldcg(sv + lo[e] + j) : ~0ull;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const uint64_t d = (vv[j] >> rbits) - lo_t;
                if (vv[j] != ~0ull && d <= static_cast<uint64_t>(2 * R)) {
                    const int k = c * K + static_cast<int>(d);
                    rows_s[rl][k] = static_cast<int32_t>(vv[j] & rmask);
                    atomicAdd(&cnt[k], 1);
                }
            }
        }
    }
    __syncthreads();
    write_rows(rows_s, [&](int j) { return rid[j]; }, nbr);
    for (int k = threadIdx.x; k < V; k += LR * K)
        if (cnt[k]) atomicAdd(&tap_count[k], cnt[k]);
}

__global__ void __launch_bounds__(kGBlock) kg_hash_insert(const int4* __restrict__ coords, int64_t n, int3 shape,
                                                          int batch, const GLayout L, uint64_t* __restrict__ table,
                                                          int log2, int row_bits, int32_t* __restrict__ status) {
    pdl_trigger();
    pdl_wait();
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

// K threads per row, one per dx plane (kLookRows rows per block, each warp
// in one plane): the plane's K columns' bucket reads (r + 1 pairs each) in
// flight together; the rare reads that meet a full bucket go on, all of the
// warp's in the same extra round.  The block's rows are staged in
// shared memory (absent neighbours -1) and written whole.
template <int K>
struct LookRows {
    static constexpr int value = K == 3 ? 128 : 64;   // 5 x 64 threads keep the 15 bucket reads in registers
};

template <int K>
__global__ void __launch_bounds__(LookRows<K>::value * K) kg_hash_lookup(const int4* __restrict__ coords, int64_t n,
                                                                         int3 shape, int batch, const GLayout L,
                                                                         const uint64_t* __restrict__ table, int log2,
                                                                         int row_bits, int32_t* __restrict__ nbr,
                                                                         int32_t* __restrict__ tap_count) {
    pdl_trigger();
    pdl_wait();
    constexpr int r = (K - 1) / 2, V = K * K * K, NP = r + 1;   // pairs per column
    constexpr int kRows = LookRows<K>::value, ST = NbrStride<K>::value;
    __shared__ int32_t cnt[V];
    // the block's rows (consecutive), written whole at the end: no -1 fill of the map first
    __shared__ __align__(16) int32_t rows_s[kRows][ST];
    for (int k = threadIdx.x; k < V; k += kRows * K) cnt[k] = 0;
    for (int k = threadIdx.x; k < kRows * ST; k += kRows * K) (&rows_s[0][0])[k] = -1;
    __syncthreads();
    const int p = threadIdx.x / kRows;   // this thread's dx plane
    const int il = threadIdx.x % kRows;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRows;
    const int64_t i = row0 + il;
    const bool ok = i < n && in_range(coords[i], shape, batch);
    const uint64_t key = ok ? g_key(coords[i], L) : 0ull;
    const int lb = log2 - 2;
    const uint64_t bmask = (uint64_t(1) << lb) - 1;
    const uint64_t rmask = (uint64_t(1) << row_bits) - 1;
    {
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
                        rows_s[il][K * K * p + K * c + static_cast<int>(d)] = static_cast<int32_t>(sl[j] & rmask);
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
    write_rows(rows_s, [&](int j) { return row0 + j < n ? row0 + j : int64_t(-1); }, nbr);
    for (int k = threadIdx.x; k < V; k += kRows * K)
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
    pdl_trigger();
    pdl_wait();
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
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t cnt[kMaxTaps];
    for (int k = threadIdx.x; k < L.V; k += kGBlock) cnt[k] = 0;
    __syncthreads();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (i < n) {
        const int4 c = coords[i];
        if (in_range(c, shape, batch)) {
            const int64_t cell = cell_of(c, L);
            for (int k = 0; k < L.V; ++k) {
                const int32_t v = __ldcg(grid + cell + L.goff[k]);
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
    pdl_trigger();
    pdl_wait();
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
    pdl_trigger();
    pdl_wait();
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

// The same keys packed with the row for the whole-GPU sort: entry g n + i is
// (((g << kg) | key) << rbits) | i; counts the digits of the passes in d
// (none where no pass reads the totals).
__global__ void __launch_bounds__(kGBlock) kg_mask_keys_packed(const int32_t* __restrict__ nbr, int64_t n, int stride,
                                                               int G, int kg, int rbits,
                                                               const int32_t* __restrict__ tap_pos,
                                                               const WideDigits d, uint32_t* __restrict__ mask,
                                                               uint64_t* __restrict__ packed,
                                                               int32_t* __restrict__ gh) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t pos[kMaxTaps];
    __shared__ int32_t h[kWideKeyPassesMax][kWideBins];
    for (int k = threadIdx.x; k < G * kg; k += kGBlock) pos[k] = tap_pos[k];
    for (int i = threadIdx.x; i < kWideKeyPassesMax * kWideBins; i += kGBlock) (&h[0][0])[i] = 0;
    __syncthreads();
    const int64_t total = G * n;
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * kGBlock; i0 < total;
         i0 += static_cast<int64_t>(gridDim.x) * kGBlock) {
        const int64_t idx = i0 + threadIdx.x;
        const bool valid = idx < total;
        uint64_t v = 0;
        if (valid) {
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
            v = (((static_cast<uint64_t>(g) << kg) | key) << rbits) | static_cast<uint64_t>(i);
            packed[idx] = v;
        }
        wide_count_digits(v, valid, d, h);
    }
    __syncthreads();
    wide_flush_digits(d, h, gh);
}

// The same, four lanes per row for kernel size K: the lanes read the row's
// nbr entries with 16-byte loads (lane q the words q, q + 4, ...), combine
// their presence bits (bit k: tap k) by shuffles, and lane q then writes the
// mask and key of groups q, q + 4, ...; entry g n + i gets group g's.
template <int K>
__global__ void __launch_bounds__(kGBlock) kg_mask_keys_rows(const int32_t* __restrict__ nbr, int64_t n, int G,
                                                             int kg, int rbits, const int32_t* __restrict__ tap_count,
                                                             int calibrated, int32_t* __restrict__ tap_pos,
                                                             const WideDigits d, uint32_t* __restrict__ mask,
                                                             uint64_t* __restrict__ packed,
                                                             int32_t* __restrict__ gh) {
    pdl_trigger();
    pdl_wait();
    constexpr int V = K * K * K, NQ = (V + 3) / 4, NW = (V + 31) / 32;   // taps, 16-byte words of a row, bitmap words
    __shared__ int32_t cnt[V];
    __shared__ int32_t pos[V];
    __shared__ int32_t h[kWideKeyPassesMax][kWideBins];
    for (int k = threadIdx.x; k < V; k += kGBlock) cnt[k] = __ldcg(tap_count + k);
    for (int i = threadIdx.x; i < kWideKeyPassesMax * kWideBins; i += kGBlock) (&h[0][0])[i] = 0;
    __syncthreads();
    // each block ranks the taps itself, as kg_tap_order does (block 0 also stores the ranks)
    for (int k = threadIdx.x; k < V; k += kGBlock) {
        const int g0 = k / kg * kg;
        int rank = k - g0;
        if (calibrated) {
            const int32_t ck = cnt[k];
            rank = 0;
            for (int j = g0; j < g0 + kg; ++j) {
                const int32_t cj = cnt[j];
                rank += (cj > ck || (cj == ck && j < k)) ? 1 : 0;
            }
        }
        pos[k] = rank;
        if (blockIdx.x == 0) tap_pos[k] = rank;
    }
    __syncthreads();
    const int q = threadIdx.x & 3;
    for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * kGBlock; t0 < 4 * n; t0 += static_cast<int64_t>(gridDim.x) * kGBlock) {
        const int64_t i = (t0 + threadIdx.x) >> 2;
        const bool valid = i < n;
        uint32_t pres[NW];
#pragma unroll
        for (int w = 0; w < NW; ++w) pres[w] = 0;
        if (valid) {
            const int4* row = reinterpret_cast<const int4*>(nbr + i * (4 * NQ));
#pragma unroll
            for (int u = 0; u < (NQ + 3) / 4; ++u) {
                const int qd = q + 4 * u;
                if (qd < NQ) {
                    const int4 v = __ldcg(row + qd);
                    const int32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        // tap 4 qd + b: word (4 qd + b) / 32, the same for the four b
                        const uint32_t bit = (4 * qd + b < V && e[b] >= 0) ? 1u << ((4 * qd + b) & 31) : 0u;
#pragma unroll
                        for (int w = 0; w < NW; ++w) pres[w] |= ((4 * qd) >> 5) == w ? bit : 0u;
                    }
                }
            }
        }
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            pres[w] |= __shfl_xor_sync(0xFFFFFFFFu, pres[w], 1);
            pres[w] |= __shfl_xor_sync(0xFFFFFFFFu, pres[w], 2);
        }
        // the presence bits as two 64-bit words (V <= 128)
        uint64_t p0 = pres[0], p1 = 0;
        if (NW > 1) p0 |= static_cast<uint64_t>(pres[NW > 1 ? 1 : 0]) << 32;
        if (NW > 2) p1 = pres[NW > 2 ? 2 : 0];
        if (NW > 3) p1 |= static_cast<uint64_t>(pres[NW > 3 ? 3 : 0]) << 32;
        for (int gi = 0; gi < (G + 3) / 4; ++gi) {
            const int g = q + 4 * gi;
            const bool on = valid && g < G;
            uint64_t v = 0;
            if (on) {
                const int a = g * kg;   // group g's taps are bits [a, a + kg)
                const uint64_t w = a < 64 ? ((p0 >> a) | (a > 0 ? p1 << (64 - a) : 0ull)) : (p1 >> (a - 64));
                const uint32_t m = static_cast<uint32_t>(w) & ((1u << kg) - 1u);
                uint32_t key = 0;
                for (uint32_t b = m; b; b &= b - 1) key |= 1u << pos[a + __ffs(b) - 1];
                v = (((static_cast<uint64_t>(g) << kg) | key) << rbits) | static_cast<uint64_t>(i);
                mask[g * n + i] = m;
                packed[g * n + i] = v;
            }
            wide_count_digits(v, on, d, h);
        }
    }
    __syncthreads();
    wide_flush_digits(d, h, gh);
}

// ---------------------------------------------------------------------------
// compaction: per-(tap, tile) counts -> scan -> pair lists, gather table
// ---------------------------------------------------------------------------
// Block (g, t): tile t of group g's order.  counts[k][t] for the group's taps
// k; the tile's union (bit j: tap g kg + j) in tile_union[g][t].
// kPacked: the row order comes as the sorted packed values (row in the low
// rbits bits) and is written out to perm here.
template <bool kPacked>
__global__ void __launch_bounds__(kTileRows) kg_tile_count(int32_t* __restrict__ perm,
                                                           const uint64_t* __restrict__ sorted, int rbits,
                                                           const uint32_t* __restrict__ mask, int64_t n,
                                                           int64_t n_tiles, int kg, int32_t* __restrict__ counts,
                                                           uint32_t* __restrict__ tile_union) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t wc[kTileRows / 32][kMaxGroupTaps];
    const int64_t g = blockIdx.x / n_tiles, t = blockIdx.x % n_tiles;
    const int64_t s = t * kTileRows + threadIdx.x;
    uint32_t m = 0;
    if (s < n) {
        int32_t r;
        if (kPacked) {
            r = static_cast<int32_t>(sorted[g * n + s] & ((uint64_t(1) << rbits) - 1));
            perm[g * n + s] = r;
        } else {
            r = perm[g * n + s];
        }
        m = mask[g * n + r];
    }
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

// The (tap, tile) counts scanned into the per-tap pair offsets, the tap
// offsets and the pair total; each group's tiles in descending order of
// union size (stable), with the number of tiles whose union is not empty
// (they come first); the sum of union sizes over all tiles.  One launch of
// V + 1 CTAs: CTA k < V scans tap k's T counts from
// the tap's start, the exclusive sum of the per-tap pair totals the search
// counted (a tap whose counts do not add up to its total is reported); CTA V
// does the tile orders.  (One CTA scanning all V T counts took ~29 rounds on
// a kernel-size-5 stage map.)
__global__ void __launch_bounds__(1024) kg_scan_tiles(const int32_t* __restrict__ counts, int V, int G, int kg,
                                                      int64_t n_tiles, const int32_t* __restrict__ tap_count,
                                                      const uint32_t* __restrict__ tile_union,
                                                      int32_t* __restrict__ seg_off, int32_t* __restrict__ tap_off,
                                                      int32_t* __restrict__ totals,
                                                      int32_t* __restrict__ tile_order,
                                                      int32_t* __restrict__ nonempty, int32_t* __restrict__ status) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t hist[kMaxGroups][kMaxGroupTaps + 1];
    __shared__ int32_t pre[kMaxTaps + 1];   // exclusive prefix of the tap totals, and their sum
    __shared__ int32_t wpre[4];
    static_assert(kMaxTaps < 128, "four warps scan the tap totals");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (static_cast<int>(blockIdx.x) < V) {
        const int k = blockIdx.x;
        int32_t tot = 0, inc = 0;
        if (warp < 4) {
            tot = threadIdx.x < V ? __ldcg(tap_count + threadIdx.x) : 0;
            inc = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += y;
            }
            if (lane == 31) wpre[warp] = inc;
        }
        __syncthreads();
        if (warp < 4) {
            int32_t before = 0;
            for (int q = 0; q < warp; ++q) before += wpre[q];
            if (static_cast<int>(threadIdx.x) <= V) pre[threadIdx.x] = before + inc - tot;
        }
        __syncthreads();
        if (k == 0) {   // CTA 0 writes the tap offsets and the pair total
            for (int i = threadIdx.x; i <= V; i += 1024) tap_off[i] = pre[i];
            if (threadIdx.x == 0) totals[0] = pre[V];
        }
        const int32_t end = rsort::block_scan_exclusive(counts + k * n_tiles, seg_off + k * n_tiles, n_tiles,
                                                        rsort::NoVisit(), pre[k]);
        if (threadIdx.x == 0 && end != pre[k + 1]) atomicOr(status, kStatusInternal);
        return;
    }
    for (int i = threadIdx.x; i < kMaxGroups * (kMaxGroupTaps + 1); i += 1024) (&hist[0][0])[i] = 0;
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

// Block (g, i) handles tile t, the i-th of group g's tile order: the pairs of
// the group's taps for the rows of tile t, at the tile's offsets in each
// tap's list, ranked by position in the tile; and
// gtab[k][s] = neighbour of the row at position s of the group's order (-1
// when absent or past n).
__global__ void __launch_bounds__(kTileRows) kg_tile_write(const int32_t* __restrict__ perm,
                                                           const uint32_t* __restrict__ mask,
                                                           const int32_t* __restrict__ nbr, int stride, int64_t n,
                                                           int64_t n_tiles, int64_t n_pad, int kg,
                                                           const int32_t* __restrict__ seg_off,
                                                           const int32_t* __restrict__ tile_order,
                                                           int32_t* __restrict__ in_rows,
                                                           int32_t* __restrict__ out_rows,
                                                           int32_t* __restrict__ gtab) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t wc[kTileRows / 32][kMaxGroupTaps];
    __shared__ int32_t seg[kMaxGroupTaps];
    // block (g, i) takes the i-th tile of group g's tile order (descending
    // union size): the costliest start first, the cheapest fill the last wave
    const int64_t g = blockIdx.x / n_tiles;
    const int64_t t = __ldcg(tile_order + blockIdx.x);
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
    // the row's neighbours of the group's present taps, all requested before
    // the first is stored (a load beside each store would wait for each in turn)
    int32_t vv[kMaxGroupTaps];
    const int32_t* nrow = nbr + (r >= 0 ? static_cast<int64_t>(r) * stride : 0) + g * kg;
#pragma unroll
    for (int j = 0; j < kMaxGroupTaps; ++j) vv[j] = (j < kg && ((m >> j) & 1u)) ? __ldcg(nrow + j) : -1;
#pragma unroll
    for (int j = 0; j < kMaxGroupTaps; ++j) {
        if (j >= kg) break;
        const int64_t k = g * kg + j;
        const bool present = (m >> j) & 1u;
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, present);
        if (present) {
            int32_t off = seg[j] + __popc(b & lt);
            for (int w = 0; w < warp; ++w) off += wc[w][j];
            in_rows[off] = vv[j];
            out_rows[off] = r;
        }
        gtab[k * n_pad + s] = vv[j];
    }
}

// kg_scan_tiles and kg_tile_write in one, for groups of up to
// kPrefixTilesG tiles: block (g, t) finds its own offsets.  Tap k's list
// starts after the pairs of every earlier tap (their totals are the tap
// counts of the lookup), and tile t's part of it after those of tiles
// 0 .. t - 1 (summed here from the raw counts); the tile's place in its
// group's order is the number of the group's tiles with a larger union plus
// those before it with an equal one.  Block (g, 0) writes the group's count
// of tiles with a nonempty union, block (0, 0) the tap offsets and totals.
__global__ void __launch_bounds__(kTileRows) kg_tile_write_prefix(
    const int32_t* __restrict__ perm, const uint32_t* __restrict__ mask, const int32_t* __restrict__ nbr, int stride,
    int64_t n, int64_t n_tiles, int64_t n_pad, int G, int kg, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ tap_count, const uint32_t* __restrict__ tile_union, int32_t* __restrict__ tap_off,
    int32_t* __restrict__ totals, int32_t* __restrict__ tile_order, int32_t* __restrict__ nonempty,
    int32_t* __restrict__ in_rows, int32_t* __restrict__ out_rows, int32_t* __restrict__ gtab) {
    pdl_trigger();
    pdl_wait();
    constexpr int W = kTileRows / 32;
    __shared__ int32_t wc[W][kMaxGroupTaps];
    __shared__ int32_t seg[kMaxGroupTaps];
    __shared__ int32_t tstart[kMaxTaps + 1];
    __shared__ int32_t wsum[W];
    __shared__ int32_t red[4][W];
    const int64_t g = blockIdx.x / n_tiles, t = blockIdx.x % n_tiles;
    const int V = G * kg;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // ---- tap starts: exclusive prefix of the tap counts (V <= kTileRows)
    const int32_t tc = threadIdx.x < V ? tap_count[threadIdx.x] : 0;
    int32_t inc = tc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    int32_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) {
        before += w < warp ? wsum[w] : 0;
        total += wsum[w];
    }
    if (threadIdx.x <= V) tstart[threadIdx.x] = threadIdx.x < V ? before + inc - tc : total;
    // ---- the counts of the group's taps in the tiles before t: warp w sums
    // taps w, w + W, ..., the loads of all its taps in flight together
    constexpr int kTapsPerWarp = (kMaxGroupTaps + W - 1) / W;
    int32_t acc[kTapsPerWarp];
#pragma unroll
    for (int i = 0; i < kTapsPerWarp; ++i) acc[i] = 0;
#pragma unroll 2
    for (int64_t tt = lane; tt < t; tt += 32) {
#pragma unroll
        for (int i = 0; i < kTapsPerWarp; ++i) {
            const int j = warp + W * i;
            acc[i] += j < kg ? __ldcg(counts + (g * kg + j) * n_tiles + tt) : 0;
        }
    }
#pragma unroll
    for (int i = 0; i < kTapsPerWarp; ++i) {
        const int j = warp + W * i;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[i] += __shfl_xor_sync(0xFFFFFFFFu, acc[i], o);
        if (lane == 0 && j < kg) wc[0][j] = acc[i];   // (wc is reused below)
    }
    // ---- place in the group's tile order; nonempty tiles; (block 0, 0) the sum of all union sizes
    const int c = __popc(tile_union[g * n_tiles + t]);
    int32_t greater = 0, equal_before = 0, nonzero = 0, taps_all = 0;
    for (int64_t tt = threadIdx.x; tt < n_tiles; tt += kTileRows) {
        const int cu = __popc(tile_union[g * n_tiles + tt]);
        greater += cu > c ? 1 : 0;
        equal_before += (cu == c && tt < t) ? 1 : 0;
        nonzero += cu > 0 ? 1 : 0;
    }
    if (g == 0 && t == 0)
        for (int64_t tt = threadIdx.x; tt < G * n_tiles; tt += kTileRows) taps_all += __popc(tile_union[tt]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        greater += __shfl_xor_sync(0xFFFFFFFFu, greater, o);
        equal_before += __shfl_xor_sync(0xFFFFFFFFu, equal_before, o);
        nonzero += __shfl_xor_sync(0xFFFFFFFFu, nonzero, o);
        taps_all += __shfl_xor_sync(0xFFFFFFFFu, taps_all, o);
    }
    if (lane == 0) {
        red[0][warp] = greater;
        red[1][warp] = equal_before;
        red[2][warp] = nonzero;
        red[3][warp] = taps_all;
    }
    __syncthreads();
    if (threadIdx.x < kg) seg[threadIdx.x] = tstart[g * kg + threadIdx.x] + wc[0][threadIdx.x];
    if (threadIdx.x == 0) {
        int32_t gs = 0, es = 0, nz = 0, ta = 0;
        for (int w = 0; w < W; ++w) {
            gs += red[0][w];
            es += red[1][w];
            nz += red[2][w];
            ta += red[3][w];
        }
        tile_order[g * n_tiles + gs + es] = static_cast<int32_t>(t);
        if (t == 0) nonempty[g] = nz;
        if (g == 0 && t == 0) {
            totals[0] = tstart[V];
            totals[1] = ta;
        }
    }
    if (g == 0 && t == 0 && threadIdx.x <= V) tap_off[threadIdx.x] = tstart[threadIdx.x];
    __syncthreads();   // seg is complete; wc is rewritten below
    // ---- the pairs and the gather table, as kg_tile_write
    const int64_t s = t * kTileRows + threadIdx.x;
    const bool valid = s < n;
    const int32_t r = valid ? perm[g * n + s] : -1;
    const uint32_t m = valid ? mask[g * n + r] : 0u;
    for (int j = 0; j < kg; ++j) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> j) & 1u);
        if (lane == 0) wc[warp][j] = __popc(b);
    }
    __syncthreads();
    const uint32_t lt = rsort::lanemask_lt();
    // the row's neighbours of the group's present taps, all requested before
    // the first is stored (a load beside each store would wait for each in turn)
    int32_t vv[kMaxGroupTaps];
    const int32_t* nrow = nbr + (r >= 0 ? static_cast<int64_t>(r) * stride : 0) + g * kg;
#pragma unroll
    for (int j = 0; j < kMaxGroupTaps; ++j) vv[j] = (j < kg && ((m >> j) & 1u)) ? __ldcg(nrow + j) : -1;
#pragma unroll
    for (int j = 0; j < kMaxGroupTaps; ++j) {
        if (j >= kg) break;
        const int64_t k = g * kg + j;
        const bool present = (m >> j) & 1u;
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, present);
        if (present) {
            int32_t off = seg[j] + __popc(b & lt);
            for (int w = 0; w < warp; ++w) off += wc[w][j];
            in_rows[off] = vv[j];
            out_rows[off] = r;
        }
        gtab[k * n_pad + s] = vv[j];
    }
}

// kg_tile_write_prefix with four threads a row (used while its blocks fill at
// most two waves of the device: it holds fewer blocks per SM): block (g, t)
// of kGtThreads, thread j of a row takes the
// group's taps j, j + 4, ... (at most kGtSlots of them) and requests their
// neighbours together; ranks within the tile come from ballots masked to the
// lanes of one phase and a scan over the warps (one thread walking all of a
// group's taps was ~25 dependent steps per row).  The pairs of the group's
// taps for the rows of tile t go to the tile's offsets in each tap's list;
// gtab[k][s] = neighbour of the row at position s of the group's order (-1
// when absent or past n).
// As kg_tile_write_prefix, the block finds its own offsets and its place in
// the group's tile order (groups of up to kPrefixTilesG tiles).
constexpr int64_t kPrefixTilesG = 512;
constexpr int kGtThreads = 4 * kTileRows;
constexpr int kGtWarps = kGtThreads / 32;
constexpr int kGtSlots = (kMaxGroupTaps + 3) / 4;   // taps per thread
constexpr int kGtGroupTaps = 8;                     // taps summed by each quarter of the block
static_assert(4 * kGtGroupTaps >= kMaxGroupTaps, "four quarters cover a group's taps");

__global__ void __launch_bounds__(kGtThreads) kg_tile_write4(
    const int32_t* __restrict__ perm, const uint32_t* __restrict__ mask, const int32_t* __restrict__ nbr, int stride,
    int64_t n, int64_t n_tiles, int64_t n_pad, int G, int kg, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ tap_count, const uint32_t* __restrict__ tile_union, int32_t* __restrict__ tap_off,
    int32_t* __restrict__ totals, int32_t* __restrict__ tile_order, int32_t* __restrict__ nonempty,
    int32_t* __restrict__ in_rows, int32_t* __restrict__ out_rows, int32_t* __restrict__ gtab) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t wc[kMaxGroupTaps][kGtWarps];   // rows with each tap per warp, then the warp's first pair
    __shared__ int32_t seg[kMaxGroupTaps];            // the tile's first pair in each of the group's lists
    __shared__ int32_t tstart[kMaxTaps + 1];          // every tap's first pair
    __shared__ int32_t gsum[4][4][kGtGroupTaps];      // [quarter][its warp][tap of the quarter]
    __shared__ int32_t wsum[kGtWarps];
    __shared__ int32_t red[4][kGtWarps];
    const int64_t g = blockIdx.x / n_tiles, t = blockIdx.x % n_tiles;
    const int V = G * kg;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rl = tid >> 2, j = tid & 3;   // row within the tile, tap phase
    const int64_t s = t * kTileRows + rl;
    const bool valid = s < n;
    // the row (two dependent round trips), requested before the sums below
    const int32_t r = valid ? __ldcg(perm + g * n + s) : -1;
    const uint32_t m = valid ? __ldcg(mask + g * n + r) : 0u;
    int32_t vv[kGtSlots];
    const int32_t* nrow = nbr + (r >= 0 ? static_cast<int64_t>(r) * stride : 0) + g * kg;
#pragma unroll
    for (int i = 0; i < kGtSlots; ++i) {
        const int jj = j + 4 * i;
        vv[i] = (jj < kg && ((m >> jj) & 1u)) ? __ldcg(nrow + jj) : -1;
    }
    {
        // tap starts: exclusive prefix of the tap counts (V <= kGtThreads)
        const int32_t tc = tid < V ? __ldcg(tap_count + tid) : 0;
        // the quarter's taps in the tiles before t: thread tid takes tiles tid % 128, + 128, ...
        const int grp = tid / kTileRows;
        int32_t acc[kGtGroupTaps];
#pragma unroll
        for (int i = 0; i < kGtGroupTaps; ++i) acc[i] = 0;
#pragma unroll 4
        for (int64_t tt = tid % kTileRows; tt < t; tt += kTileRows) {
#pragma unroll
            for (int i = 0; i < kGtGroupTaps; ++i) {
                const int jj = kGtGroupTaps * grp + i;
                acc[i] += jj < kg ? __ldcg(counts + (g * kg + jj) * n_tiles + tt) : 0;
            }
        }
        // place in the group's tile order; nonempty tiles; (block 0, 0) the sum of all union sizes
        const int c = __popc(__ldcg(tile_union + g * n_tiles + t));
        int32_t greater = 0, equal_before = 0, nonzero = 0, taps_all = 0;
        for (int64_t tt = tid; tt < n_tiles; tt += kGtThreads) {
            const int cu = __popc(__ldcg(tile_union + g * n_tiles + tt));
            greater += cu > c ? 1 : 0;
            equal_before += (cu == c && tt < t) ? 1 : 0;
            nonzero += cu > 0 ? 1 : 0;
        }
        if (g == 0 && t == 0)
            for (int64_t tt = tid; tt < G * n_tiles; tt += kGtThreads) taps_all += __popc(__ldcg(tile_union + tt));
        int32_t inc = tc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) wsum[warp] = inc;
        // each of the quarter's 8 counters over the warp: three exchanges halve
        // the counters a lane carries, two more add the rest; lane l then holds counter l
#pragma unroll
        for (int h = 4; h >= 1; h >>= 1) {
            const bool upper = (lane & h) != 0;
#pragma unroll
            for (int i = 0; i < h; ++i) {
                const int32_t send = upper ? acc[i] : acc[i + h];
                const int32_t keep = upper ? acc[i + h] : acc[i];
                acc[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, h);
            }
        }
        acc[0] += __shfl_xor_sync(0xFFFFFFFFu, acc[0], 8);
        acc[0] += __shfl_xor_sync(0xFFFFFFFFu, acc[0], 16);
        if (lane < kGtGroupTaps) gsum[grp][warp & 3][lane] = acc[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            greater += __shfl_xor_sync(0xFFFFFFFFu, greater, o);
            equal_before += __shfl_xor_sync(0xFFFFFFFFu, equal_before, o);
            nonzero += __shfl_xor_sync(0xFFFFFFFFu, nonzero, o);
            taps_all += __shfl_xor_sync(0xFFFFFFFFu, taps_all, o);
        }
        if (lane == 0) {
            red[0][warp] = greater;
            red[1][warp] = equal_before;
            red[2][warp] = nonzero;
            red[3][warp] = taps_all;
        }
        __syncthreads();   // wsum
        int32_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kGtWarps; ++w) {
            before += w < warp ? wsum[w] : 0;
            total += wsum[w];
        }
        if (tid <= V) tstart[tid] = tid < V ? before + inc - tc : total;
    }
    // the warp's rows with each of the group's taps: lanes of one phase share their taps
    const uint32_t same = 0x11111111u << j;
#pragma unroll
    for (int i = 0; i < kGtSlots; ++i) {
        const int jj = j + 4 * i;
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, jj < kg && ((m >> jj) & 1u)) & same;
        if (lane == j && jj < kg) wc[jj][warp] = __popc(b);
    }
    __syncthreads();
    // each tap's warp counts -> the warps' first pairs within the tile (two taps per warp)
    if (warp < (kg * kGtWarps + 31) / 32) {   // whole warps: every lane takes part in the shuffles
        const int jj = tid / kGtWarps, w = tid % kGtWarps;
        const int32_t x = jj < kg ? wc[jj][w] : 0;
        int32_t inc = x;
#pragma unroll
        for (int o = 1; o < kGtWarps; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o, kGtWarps);
            if (w >= o) inc += y;
        }
        if (jj < kg) wc[jj][w] = inc - x;
    }
    if (warp == kGtWarps - 1) {
        if (lane < kg) {
            const int q = lane / kGtGroupTaps, i = lane % kGtGroupTaps;
            seg[lane] = tstart[g * kg + lane] + gsum[q][0][i] + gsum[q][1][i] + gsum[q][2][i] + gsum[q][3][i];
        }
        if (lane == 0) {
            int32_t gs = 0, es = 0, nz = 0, ta = 0;
            for (int w = 0; w < kGtWarps; ++w) {
                gs += red[0][w];
                es += red[1][w];
                nz += red[2][w];
                ta += red[3][w];
            }
            tile_order[g * n_tiles + gs + es] = static_cast<int32_t>(t);
            if (t == 0) nonempty[g] = nz;
            if (g == 0 && t == 0) {
                totals[0] = tstart[V];
                totals[1] = ta;
            }
        }
    }
    if (g == 0 && t == 0 && tid <= V) tap_off[tid] = tstart[tid];
    __syncthreads();
    // the pairs and the gather table
    const uint32_t lt = rsort::lanemask_lt();
#pragma unroll
    for (int i = 0; i < kGtSlots; ++i) {
        const int jj = j + 4 * i;
        const bool present = jj < kg && ((m >> jj) & 1u);
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, present) & same;
        if (present) {
            const int32_t off = seg[jj] + wc[jj][warp] + __popc(b & lt);
            in_rows[off] = vv[i];
            out_rows[off] = r;
        }
        if (jj < kg) gtab[(g * kg + jj) * n_pad + s] = vv[i];
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

// The distinct candidates without sorting them all: each input site's up to
// 8 output keys go into a hash set (slot = key + 1, 0 empty, linear probing
// from a multiplicative hash), one thread per candidate (a thread per input
// site and its 8 candidates in turn was 26 us on outdoor, cold); the thread
// whose insertion creates an entry appends the key to uniq[] (the count in
// *n_uniq) and counts its digits for the sort of the distinct keys (the
// passes in d: none where no pass of that sort reads the totals).  The set
// has at least twice as many slots as there can be candidates, so a probe
// always ends.
__device__ __forceinline__ uint64_t set_slot(uint64_t key, int log2) {
    return (key * 0x9E3779B97F4A7C15ull) >> (64 - log2);
}

__global__ void __launch_bounds__(kGBlock) kst_dedupe(const int4* __restrict__ coords, int64_t n, int3 shape,
                                                      int batch, const OutLayout O, uint64_t* __restrict__ set,
                                                      int set_log2, const WideDigits d, uint64_t* __restrict__ uniq,
                                                      int64_t* __restrict__ n_uniq, int32_t* __restrict__ gh) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t h[kWideKeyPassesMax][kWideBins];
    __shared__ uint64_t staged[kGBlock];   // the block's new keys of one round
    __shared__ int32_t n_staged;
    __shared__ unsigned long long base_sh;
    for (int i = threadIdx.x; i < kWideKeyPassesMax * kWideBins; i += kGBlock) (&h[0][0])[i] = 0;
    if (threadIdx.x == 0) n_staged = 0;
    __syncthreads();
    const uint64_t smask = (uint64_t(1) << set_log2) - 1;
    const int lane = threadIdx.x & 31;
    // one candidate a thread: eight lanes share an input site, lane j taking
    // parity choice j (bit a: the second choice on axis a)
    const int64_t m = 8 * n;
    for (int64_t q0 = static_cast<int64_t>(blockIdx.x) * kGBlock; q0 < m; q0 += static_cast<int64_t>(gridDim.x) * kGBlock) {
        const int64_t q = q0 + threadIdx.x;
        const int64_t i = q >> 3;
        const int j = static_cast<int>(q & 7);
        int4 c = make_int4(-1, -1, -1, -1);
        bool v = false;
        if (q < m) {
            c = __ldcg(coords + i);
            v = in_range(c, shape, batch);
        }
        // an even coordinate has o = c / 2 only, an odd one (c - 1) / 2 and (c + 1) / 2
        int o[3];
        const int cc[3] = {c.y, c.z, c.w};
        const int lim[3] = {O.shape.x, O.shape.y, O.shape.z};
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            const int second = (j >> a) & 1;
            const bool odd = cc[a] & 1;
            if (!odd && second) v = false;
            o[a] = odd ? (second ? (cc[a] + 1) >> 1 : (cc[a] - 1) >> 1) : cc[a] >> 1;
            if (o[a] < 0 || o[a] >= lim[a]) v = false;
        }
        const uint64_t key = v ? out_key(c.x, o[0], o[1], o[2], O) : 0ull;
        bool fresh = false;
        if (v) {
            // most probes end at the first slot
            uint64_t slot = set_slot(key, set_log2);
            uint64_t cur = __ldcg(set + slot);
            for (uint64_t probe = 0; probe <= smask; ++probe, slot = (slot + 1) & smask) {
                if (probe > 0) cur = __ldcg(set + slot);
                if (cur == key + 1) break;
                if (cur != 0ull) continue;
                const unsigned long long prev = atomicCAS(reinterpret_cast<unsigned long long*>(set + slot), 0ull,
                                                          static_cast<unsigned long long>(key + 1));
                if (prev == 0ull) {
                    fresh = true;
                    break;
                }
                if (prev == key + 1) break;
            }
        }
        // the block's new keys are staged in shared memory (one shared counter
        // update per warp), then take consecutive slots of uniq with one global
        // counter update per block and round
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, fresh);
        int at = 0;
        if (b && lane == __ffs(b) - 1) at = atomicAdd(&n_staged, __popc(b));
        at = __shfl_sync(0xFFFFFFFFu, at, b ? __ffs(b) - 1 : 0);
        if (fresh) staged[at + __popc(b & ((1u << lane) - 1u))] = key;
        wide_count_digits(key, fresh, d, h);
        __syncthreads();               // the round's keys are staged
        const int cnt = n_staged;
        __syncthreads();               // every thread has read the count
        if (threadIdx.x == 0) {
            if (cnt > 0)
                base_sh = atomicAdd(reinterpret_cast<unsigned long long*>(n_uniq), static_cast<unsigned long long>(cnt));
            n_staged = 0;
        }
        __syncthreads();               // base_sh is set, the counter reset
        for (int e = threadIdx.x; e < cnt; e += kGBlock) uniq[base_sh + e] = staged[e];
        __syncthreads();               // staged is free for the next round
    }
    __syncthreads();
    wide_flush_digits(d, h, gh);
}

// Output row j is the j-th distinct candidate in ascending key order: its
// coordinates and its query site 2o in input coordinates.
__global__ void __launch_bounds__(kGBlock) kst_outputs_sorted(const uint64_t* __restrict__ keys, int64_t m,
                                                              const OutLayout O, int4* __restrict__ out_coords,
                                                              int4* __restrict__ query) {
    pdl_trigger();
    pdl_wait();
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (j >= m) return;
    const uint64_t k = keys[j];
    const int z = static_cast<int>(k & ((uint64_t(1) << O.wz) - 1));
    const int y = static_cast<int>((k >> O.wz) & ((uint64_t(1) << O.wy) - 1));
    const int x = static_cast<int>((k >> (O.wz + O.wy)) & ((uint64_t(1) << O.wx) - 1));
    const int b = static_cast<int>(k >> (O.wz + O.wy + O.wx));
    out_coords[j] = make_int4(b, x, y, z);
    query[j] = make_int4(b, 2 * x, 2 * y, 2 * z);
}

// flags[j] = 1 for the first of each run of equal sorted keys (not no_key).
__global__ void __launch_bounds__(kGBlock) kst_first(const uint64_t* __restrict__ keys, int64_t m, uint64_t no_key,
                                                     int32_t* __restrict__ flags) {
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kGBlock + threadIdx.x;
    if (j >= m) return;
    const uint64_t k = keys[j];
    flags[j] = (k != no_key && (j == 0 || keys[j - 1] != k)) ? 1 : 0;
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

__global__ void k_or_status(int32_t* __restrict__ status, const int32_t* __restrict__ extra) {
    if (threadIdx.x == 0 && *extra) atomicOr(status, *extra);
}

// Inverse map: for every (o, k) of the strided map with input row i,
// inv[i][k] = o (one writer per entry: o is fixed by i and k).
__global__ void __launch_bounds__(kGBlock) kg_inverse_scatter(const int32_t* __restrict__ nbr, int stride, int64_t n,
                                                              int32_t* __restrict__ inv, int inv_stride) {
    pdl_trigger();
    pdl_wait();
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
    // for K = 5, where the hash lookup of 125 taps (75 bucket reads per row, one
    // thread per dx plane) measured no faster on outdoor (map 164 vs 164 us) and
    // slower on 240k rows (631 vs 554 us)
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
    // The sorts run on the whole-GPU pass (one launch per digit of up to 10
    // bits) where the key packs with the row into 64 bits; else on the
    // 8-bit, three-launch passes of rsort.  Mask keys: (g << kg | key) with
    // the row below; coordinate keys (sorted mapper): key_bits + 1 bits.
    const int mrb = std::max(1, bit_len(static_cast<uint64_t>(n > 0 ? n - 1 : 0)));
    const int mbits = kg + bit_len(static_cast<uint64_t>(G) - 1);
    const WideDigits mdig = wide_digits(mrb, mbits);
    const bool wide_mask = mdig.passes > 0 && mbits + mrb <= 64 && G * n <= kWideMaxRows;
    const int ckb = key_bits + 1;
    const WideDigits cdig = wide_digits(mrb, ckb);
    const bool wide_coord = !src && mapper == SPCONV_MAPPER_SORTED && cdig.passes > 0 && ckb + mrb <= 64 &&
                            n <= kWideMaxRows;
    const int64_t look_words = std::max<int64_t>(1, std::max(wide_mask ? wide_sort_look_words(G * n) : 0,
                                                             wide_coord ? wide_sort_look_words(n) : 0));
    const size_t wide_bytes = (wide_mask || wide_coord)
                                  ? (kWideTickets * kWideBins + kWideCounters) * sizeof(int32_t) +
                                        static_cast<size_t>(look_words) * 8
                                  : 0;
    if (wide_mask) {
        add(gn, 8); add(gn, 8); add(gn, 4);           // packed mask keys ping-pong, row orders
    } else {
        add(gn, 4); add(gn, 4); add(gn, 4); add(gn, 4);   // mask keys and row ids, ping-pong
    }
    add(rsort::kBins * nb, 4);                        // radix histograms
    add(wide_bytes, 1);                               // whole-GPU sort: digit totals, tickets, look-back states
    int table_log2 = 11;
    while ((int64_t(1) << table_log2) < kGHashSlotsPerRow * nt1) ++table_log2;
    // Kernel size 5 above kColIndexRows: the sorted search through a column
    // index.  Measured against the lockstep binary searches (map µs): stage
    // (240k rows) 405 -> 363, large (94.5k) 198 -> 191; but outdoor (32k)
    // 116.6 -> 119.6 and three groups of kernel size 3 70.7 -> 81.0, where
    // the index's build and clearing cost more than the searches save.
    const bool col_index = wide_coord && K == 5 && n > kColIndexRows;
    const int col_log2 = col_table_log2(n);
    if (src) {
        // the neighbours come from the strided map
    } else if (wide_coord) {
        add(n1, 8); add(n1, 8);                       // packed coordinate keys, ping-pong
        if (col_index) add(size_t(2) << col_log2, 8);  // column index (2 words an entry)
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
    // the arrays that start at zero come first, cleared by one memset: the
    // status, tap counts, totals, the whole-GPU sort's scratch and the hash table
    char* const zero_begin = p;
    h->status = take<int32_t>(p, 4);
    h->tap_count = take<int32_t>(p, V);
    h->totals = take<int32_t>(p, 2);
    char* wide = take<char>(p, wide_bytes);
    const bool hashed = !src && !wide_coord && mapper == SPCONV_MAPPER_HASH;
    uint64_t* table = hashed ? take<uint64_t>(p, size_t(1) << table_log2) : nullptr;
    uint64_t* col_table = col_index ? take<uint64_t>(p, size_t(2) << col_log2) : nullptr;
    const size_t zero_bytes = static_cast<size_t>(p - zero_begin);
    h->nbr = take<int32_t>(p, n1 * h->nbr_stride);
    h->mask = take<uint32_t>(p, gn);
    h->tap_pos = take<int32_t>(p, V);
    h->tap_off = take<int32_t>(p, V + 1);
    h->in_rows = take<int32_t>(p, V * n1);
    h->out_rows = take<int32_t>(p, V * n1);
    h->gtab = take<int32_t>(p, V * np);
    h->tile_union = take<uint32_t>(p, G * t1);
    h->tile_order = take<int32_t>(p, G * t1);
    int32_t* counts = take<int32_t>(p, V * t1);
    h->seg_off = take<int32_t>(p, V * t1);
    h->tile_nonempty = take<int32_t>(p, G);
    uint32_t *mkey_a = nullptr, *mkey_b = nullptr, *perm_a = nullptr, *perm_b = nullptr;
    uint64_t *mpk_a = nullptr, *mpk_b = nullptr;
    int32_t* perm_w = nullptr;
    if (wide_mask) {
        mpk_a = take<uint64_t>(p, gn);
        mpk_b = take<uint64_t>(p, gn);
        perm_w = take<int32_t>(p, gn);
    } else {
        mkey_a = take<uint32_t>(p, gn);
        mkey_b = take<uint32_t>(p, gn);
        perm_a = take<uint32_t>(p, gn);
        perm_b = take<uint32_t>(p, gn);
    }
    int32_t* hist = take<int32_t>(p, rsort::kBins * nb);
    int32_t* wgh = reinterpret_cast<int32_t*>(wide);                 // [kWideTickets][kWideBins]
    int32_t* wtickets = wgh + kWideTickets * kWideBins;             // [kWideCounters]
    uint64_t* wlook = reinterpret_cast<uint64_t*>(wtickets + kWideCounters);

    SPCONV_CHECK_CUDA(cudaMemsetAsync(zero_begin, 0, zero_bytes, s));
    h->perm = wide_mask ? perm_w : reinterpret_cast<int32_t*>(perm_a);
    if (n == 0) {
        SPCONV_CHECK_CUDA(cudaMemsetAsync(h->tap_off, 0, (V + 1) * sizeof(int32_t), s));
        return cuda_status(cudaGetLastError());
    }
    // the staged search and lookup (kernel size 3 or 5) write every entry of
    // the map's rows; the other mappers fill only the neighbours they find
    // (rows of NbrStride<K> entries: the stride set above for every K)
    const bool staged = (K == 3 || K == 5) && !src && (wide_coord || mapper == SPCONV_MAPPER_HASH);
    if (!staged)
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
    } else if (wide_coord) {
        // packed (key << row bits | row), key_bits + 1 bits of key: an out-of-range
        // row's all-ones key orders it last; the whole-GPU sort, then the search
        uint64_t* ck_a = take<uint64_t>(p, n1);
        uint64_t* ck_b = take<uint64_t>(p, n1);
        // (the digits are counted only for passes that read the totals)
        bool ctot = false;
        SPCONV_CHECK(wide_sort_reads_totals(n, cdig, &ctot));
        kg_pack_keys_packed<<<capped_blocks(n), kGBlock, 0, s>>>(c4, n, shape3, B, L, ckb, mrb,
                                                                 ctot ? cdig : no_counts(cdig), ck_a, wgh, h->status);
        ++launches;
        bool in_b = false;
        SPCONV_CHECK(wide_sort(ck_a, ck_b, n, cdig, wgh, wtickets, 0, wlook, h->status, s, &in_b));
        const uint64_t* sv = in_b ? ck_b : ck_a;
        const uint64_t no_key = (uint64_t(1) << ckb) - 1;
        if (col_index) {
            // each (b, x, y) column's run entered in the column index, then the search through it
            SPCONV_CHECK(launch_chained(kg_col_insert, blocks(n, kGBlock), kGBlock, s, sv, n, mrb, no_key, L.wz, col_log2,
                                        col_table, h->status));
            ++launches;
            SPCONV_CHECK(launch_chained(kg_col_search<5>, blocks(n, LockRows<5>::value), LockRows<5>::value * 5, s, sv, n,
                                        mrb, no_key, L, col_log2, static_cast<const uint64_t*>(col_table), h->nbr,
                                        h->tap_count, h->status));
        } else if (K == 3)
            SPCONV_CHECK(launch_chained(kg_search_lockstep<3>, blocks(n, LockRows<3>::value), LockRows<3>::value * 3, s, sv,
                                        n, mrb, no_key, L, h->nbr, h->tap_count, h->status));
        else if (K == 5)
            SPCONV_CHECK(launch_chained(kg_search_lockstep<5>, blocks(n, LockRows<5>::value), LockRows<5>::value * 5, s, sv,
                                        n, mrb, no_key, L, h->nbr, h->tap_count, h->status));
        else
            SPCONV_CHECK(launch_chained(kg_search<true>, blocks(n, kGBlock), kGBlock, s, sv, nullptr, n, mrb, no_key, L, h->nbr,
                                                                   h->tap_count, h->status));
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
        SPCONV_CHECK(launch_chained(kg_search<false>, blocks(n, kGBlock), kGBlock, s, in_b ? ck_b : ck_a, in_b ? cv_b : cv_a, n, 0, kNoKey,
                                                                L, h->nbr, h->tap_count, h->status));
        ++launches;
    } else if (mapper == SPCONV_MAPPER_HASH) {
        kg_hash_insert<<<blocks(n_table, kGBlock), kGBlock, 0, s>>>(c4, n_table, shape3, B, L, table, table_log2,
                                                                    row_bits, h->status);
        const int4* q4 = query ? reinterpret_cast<const int4*>(query) : c4;
        if (K == 3)
            SPCONV_CHECK(launch_chained(kg_hash_lookup<3>, blocks(n, LookRows<3>::value), 3 * LookRows<3>::value, s, 
                q4, n, shape3, B, L, table, table_log2, row_bits, h->nbr, h->tap_count));
        else
            SPCONV_CHECK(launch_chained(kg_hash_lookup<5>, blocks(n, LookRows<5>::value), 5 * LookRows<5>::value, s, 
                q4, n, shape3, B, L, table, table_log2, row_bits, h->nbr, h->tap_count));
        launches += 2;
    } else {
        int32_t* grid = take<int32_t>(p, static_cast<size_t>(cells));
        SPCONV_CHECK_CUDA(cudaMemsetAsync(grid, 0xFF, static_cast<size_t>(cells) * 4, s));
        kg_grid_scatter<<<blocks(n, kGBlock), kGBlock, 0, s>>>(c4, n, shape3, B, L, grid, h->status);
        SPCONV_CHECK(launch_chained(kg_grid_lookup, blocks(n, kGBlock), kGBlock, s, c4, n, shape3, B, L, grid, h->nbr, h->tap_count));
        launches += 2;
    }
    // the rows' mask-key kernel ranks the taps itself; the others read kg_tap_order's ranks
    const bool rows_keys = wide_mask && ((K == 5 && h->nbr_stride == 128) || (K == 3 && h->nbr_stride == 28));
    const int calibrated = h->bit_order == SPCONV_ORDER_CALIBRATED;
    if (src) {   // (a copy precedes it: a plain launch)
        kg_tap_order<<<1, 128, 0, s>>>(h->tap_count, V, kg, calibrated, h->tap_pos);
        ++launches;
    } else if (!rows_keys) {
        SPCONV_CHECK(launch_chained(kg_tap_order, 1u, 128u, s, static_cast<const int32_t*>(h->tap_count), V, kg,
                                    calibrated, h->tap_pos));
        ++launches;
    }
    const unsigned tiles = static_cast<unsigned>(G * T);
    if (wide_mask) {
        int32_t* mgh = wgh + kWideKeyPassesMax * kWideBins;
        bool mtot = false;
        SPCONV_CHECK(wide_sort_reads_totals(G * n, mdig, &mtot));
        const WideDigits mcnt = mtot ? mdig : no_counts(mdig);   // digits the key kernel counts
        if (K == 5 && h->nbr_stride == 128)
            SPCONV_CHECK(launch_chained(kg_mask_keys_rows<5>, capped_blocks(4 * n), kGBlock, s, h->nbr, n, G, kg, mrb,
                                        static_cast<const int32_t*>(h->tap_count), calibrated, h->tap_pos, mcnt,
                                        h->mask, mpk_a, mgh));
        else if (K == 3 && h->nbr_stride == 28)
            SPCONV_CHECK(launch_chained(kg_mask_keys_rows<3>, capped_blocks(4 * n), kGBlock, s, h->nbr, n, G, kg, mrb,
                                        static_cast<const int32_t*>(h->tap_count), calibrated, h->tap_pos, mcnt,
                                        h->mask, mpk_a, mgh));
        else
            SPCONV_CHECK(launch_chained(kg_mask_keys_packed, capped_blocks(G * n), kGBlock, s, h->nbr, n, h->nbr_stride, G, kg, mrb,
                                                                         h->tap_pos, mcnt, h->mask, mpk_a, mgh));
        launches += 1;
        bool in_b = false;
        SPCONV_CHECK(wide_sort(mpk_a, mpk_b, G * n, mdig, wgh + kWideKeyPassesMax * kWideBins, wtickets,
                               kWideKeyPassesMax, wlook, h->status, s, &in_b));
        SPCONV_CHECK(launch_chained(kg_tile_count<true>, tiles, kTileRows, s, h->perm, in_b ? mpk_b : mpk_a, mrb, h->mask, n, T, kg, counts,
                                                        h->tile_union));
    } else {
        SPCONV_CHECK(launch_chained(kg_mask_keys, blocks(G * n, kGBlock), kGBlock, s, h->nbr, n, h->nbr_stride, G, kg, h->tap_pos, h->mask,
                                                                mkey_a, perm_a));
        launches += 1;
        const bool perm_in_b = rsort::sort_pairs<uint32_t>(mkey_a, perm_a, mkey_b, perm_b, G * n, mbits, hist, s,
                                                           &launches);
        h->perm = reinterpret_cast<int32_t*>(perm_in_b ? perm_b : perm_a);
        SPCONV_CHECK(launch_chained(kg_tile_count<false>, tiles, kTileRows, s, h->perm, nullptr, 0, h->mask, n, T, kg, counts,
                                                         h->tile_union));
    }
    // four threads a row while its blocks fill at most two waves; else one
    // (outdoor maps: strided, 600 blocks, 178.4 -> 168.9 us; three groups,
    // 759 blocks, 64.4 -> 68.7 us and kernel size 5, 1265, 137.0 -> 137.5)
    static int64_t cap4[kMaxDevices] = {};
    int dev = 0;
    SPCONV_CHECK_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return SPCONV_ERR_UNSUPPORTED;
    if (cap4[dev] == 0) {
        int sms = 0, b = 0;
        SPCONV_CHECK_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        SPCONV_CHECK_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kg_tile_write4, kGtThreads, 0));
        cap4[dev] = std::max<int64_t>(1, static_cast<int64_t>(b) * sms);
    }
    if (T <= kPrefixTilesG && V <= kTileRows) {
        if (static_cast<int64_t>(tiles) <= 2 * cap4[dev])
            SPCONV_CHECK(launch_chained(kg_tile_write4, tiles, kGtThreads, s, h->perm, h->mask, h->nbr, h->nbr_stride, n,
                                        T, h->n_pad, G, kg, counts, h->tap_count, h->tile_union, h->tap_off,
                                        h->totals, h->tile_order, h->tile_nonempty, h->in_rows, h->out_rows, h->gtab));
        else
            SPCONV_CHECK(launch_chained(kg_tile_write_prefix, tiles, kTileRows, s, h->perm, h->mask, h->nbr, h->nbr_stride,
                                        n, T, h->n_pad, G, kg, counts, h->tap_count, h->tile_union, h->tap_off,
                                        h->totals, h->tile_order, h->tile_nonempty, h->in_rows, h->out_rows, h->gtab));
        launches -= 1;
    } else {
        SPCONV_CHECK(launch_chained(kg_scan_tiles, static_cast<unsigned>(V + 1), 1024u, s, counts, V, G, kg, T,
                                    static_cast<const int32_t*>(h->tap_count), h->tile_union, h->seg_off, h->tap_off,
                                    h->totals, h->tile_order, h->tile_nonempty, h->status));
        SPCONV_CHECK(launch_chained(kg_tile_write, tiles, kTileRows, s, h->perm, h->mask, h->nbr, h->nbr_stride, n, T,
                                    h->n_pad, kg, h->seg_off, static_cast<const int32_t*>(h->tile_order), h->in_rows,
                                    h->out_rows, h->gtab));
    }
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
    // Where the output key takes at most kWideKeyPassesMax digits, the distinct
    // candidates are found in a hash set and only they are sorted (whole-GPU
    // pass); else every candidate slot is sorted (8-bit passes) and the first
    // of each run kept.
    const WideDigits cdig = wide_digits(0, okey_bits);
    const bool wide_cand = cdig.passes > 0 && m <= kWideMaxRows;
    int set_log2 = 11;
    while ((int64_t(1) << set_log2) < 2 * m) ++set_log2;
    const size_t set_bytes = wide_cand ? (size_t(1) << set_log2) * 8 : 0;
    // digit totals, tickets and barrier counters, a status word (padded to 16 bytes), look-back states
    const size_t wide_bytes = wide_cand ? (kWideTickets * kWideBins + kWideCounters + 4) * sizeof(int32_t) +
                                              static_cast<size_t>(wide_sort_look_words(m)) * 8
                                        : 0;
    add(wide_bytes, 1);
    add(set_bytes, 1);                            // hash set of the candidates
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
    // what starts at zero comes first, cleared by one memset: the output count,
    // the whole-GPU sort's scratch and the hash set
    char* const zero_begin = p;
    int64_t* count = take<int64_t>(p, 1);
    char* wide = take<char>(p, wide_bytes);
    uint64_t* cset = take<uint64_t>(p, set_bytes / 8);
    const size_t zero_bytes = static_cast<size_t>(p - zero_begin);
    int32_t* wgh = reinterpret_cast<int32_t*>(wide);
    int32_t* wtickets = wgh + kWideTickets * kWideBins;
    int32_t* wstatus = wtickets + kWideCounters;
    uint64_t* wlook = reinterpret_cast<uint64_t*>(wstatus + 4);
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
    SPCONV_CHECK_CUDA(cudaMemsetAsync(zero_begin, 0, zero_bytes, s));
    if (n_in > 0) {
        const int3 ishape = make_int3(h->shape[0], h->shape[1], h->shape[2]);
        if (wide_cand) {
            // the distinct sites number at most m: where a sort of m values runs
            // every pass in the count exchange, so does theirs (fewer partitions),
            // and their digits need no counting
            bool stot = false;
            SPCONV_CHECK(wide_sort_reads_totals(m, cdig, &stot));
            kst_dedupe<<<capped_blocks(8 * n_in), kGBlock, 0, s>>>(reinterpret_cast<const int4*>(coords), n_in, ishape,
                                                               h->batch, O, cset, set_log2,
                                                               stot ? cdig : no_counts(cdig), ka, count, wgh);
            ++launches;
            // the one synchronisation: the number of distinct sites sizes the map
            SPCONV_CHECK_CUDA(cudaMemcpyAsync(&n_out, count, 8, cudaMemcpyDeviceToHost, s));
            SPCONV_CHECK_CUDA(cudaStreamSynchronize(s));
            if (n_out > 0) {
                bool in_b = false;
                SPCONV_CHECK(wide_sort(ka, kb, n_out, cdig, wgh, wtickets, 0, wlook, wstatus, s, &in_b, true));
                SPCONV_CHECK(launch_chained(kst_outputs_sorted, blocks(n_out, kGBlock), kGBlock, s, 
                    in_b ? kb : ka, n_out, O, reinterpret_cast<int4*>(h->out_coords), query));
                ++launches;
            }
        } else {
            kst_candidates<<<blocks(n_in, kGBlock), kGBlock, 0, s>>>(reinterpret_cast<const int4*>(coords), n_in,
                                                                      ishape, h->batch, O, ka, va);
            ++launches;
            const bool in_b = rsort::sort_pairs<uint64_t>(ka, va, kb, vb, m, okey_bits + 1, hist, s, &launches);
            const uint64_t* sk = in_b ? kb : ka;
            kst_first<<<blocks(m, kGBlock), kGBlock, 0, s>>>(sk, m, kNoKey, flags);
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
    }
    count_launch(launches);
    h->n = n_out;
    int rc = grouped_core(h, opt, coords, n_in, reinterpret_cast<const int32_t*>(query), nullptr);
    if (rc == SPCONV_OK && wide_cand && h->status) {
        // a stall of the distinct-site sort shows in the map's status
        k_or_status<<<1, 32, 0, s>>>(h->status, wstatus);
        count_launch();
        rc = cuda_status(cudaGetLastError());
    }
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

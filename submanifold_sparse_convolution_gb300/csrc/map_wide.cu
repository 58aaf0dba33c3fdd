// The kernel-map build on the whole GPU, one kernel per step.
//
// The cluster pipeline (map_fused.cu) runs every sort pass on the 16 SMs of
// one thread-block cluster; a pass then costs ~8 us at 32k rows and grows
// with the rows per SM (~40 us at 240k rows).  Here each stable LSD radix
// pass is one kernel over all SMs.  A partition of 1024 keys (2048 from 16k
// rows, 4096 from 128k rows) is ranked stably by
// one CTA, which then needs, per digit, the keys of that digit in the
// partitions before it and in all partitions.  It gets them in one of three
// forms:
//  - up to 64 resident partitions, a count exchange: every partition writes
//    its digit counts as self-validating words (an epoch tag in the high
//    half, two 16-bit counts in the low half), bumps an arrival counter and
//    reads every partition's words in one round.  That gives the digit
//    totals as well, so no histogram kernel runs before the pass, and the
//    first pass of the mask sort makes the mask keys itself;
//  - up to 256 resident partitions, two grid barriers: partitions publish
//    their counts, each CTA scans a few digits across all partitions,
//    partitions read their prefixes back (about seven memory round trips
//    whatever the number of partitions);
//  - otherwise decoupled look-back: a CTA takes its partition from a ticket
//    counter (so it only waits on CTAs already running), publishes its
//    counts, sums those of the CTAs before it up to the first inclusive
//    prefix, publishes its own.  The digit totals then come from the
//    histogram kernel that wrote the keys.
// Kernels follow each other with programmatic dependent launch.
//
// Steps (sorted-key mapper):  pack keys (+ histograms of the key digits
// where a pass reads digit totals) -> key passes -> neighbour search
// (map_search.cu) -> mask keys (inside the first mask pass where the
// exchange runs) -> mask passes -> per-tile pair counts -> (above 1024
// tiles) the scan of the (tap, tile) offsets, one CTA per tap, and the tile
// order -> pair lists, gather table and row order.  The hash mapper
// replaces the first three steps by an insert and a lookup, the dense mapper
// by a presence-grid scatter and a 27-lookup pass.  Results are
// bit-identical to the other pipelines: the same packed keys, the same
// stable order, the same outputs.  Every kernel lets the next one launch as
// soon as all of its CTAs run (the next waits for its completion before
// reading anything).
//
// State and count words carry an epoch: every launch that publishes them
// takes a fresh one, so a word left by an earlier launch in the same memory
// never reads as ready and the buffers need no clearing.  Every wait is
// bounded in time.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "common.cuh"
#include "map_internal.cuh"
#include "ptx_sm100.cuh"

namespace spconv {
namespace {

constexpr int WT = 256;                        // threads per CTA
constexpr int WI = kWideKeysPerCta / WT;       // keys per thread in a sort pass (the smaller partition)
constexpr int WW = WT / 32;                    // warps per CTA
constexpr int kBinsPerThread = kWideBins / WT;
constexpr int kMaskWidth = (kTaps + kWideMaskPasses - 1) / kWideMaskPasses;
// Rows per thread of the key and mask-key kernels (their loads issued
// together): 1 up to kFewRows rows, for parallelism (outdoor 84 -> 80 us per
// build); 4 above, where more CTAs would mean more global atomics for the
// digit counts (stage, 240k rows: 203 vs 210 us).
constexpr int64_t kFewRows = 131072;
static_assert(kBinsPerThread * WT == kWideBins, "digit values split evenly over the threads");
static_assert(WI * WT == kWideKeysPerCta, "keys split evenly over the threads");
static_assert((1 << kMaskWidth) <= kWideBins, "mask digits fit the histogram");

constexpr uint64_t kAgg = 1ull << 30;      // the partition's own count
constexpr uint64_t kPre = 2ull << 30;      // the inclusive prefix up to and including the partition
constexpr uint64_t kFlags = 3ull << 30;
constexpr uint64_t kCount = (1ull << 30) - 1;

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t state(uint32_t epoch, uint64_t flag, int32_t count) {
    return (static_cast<uint64_t>(epoch) << 32) | flag | (static_cast<uint64_t>(count) & kCount);
}

// Decoupled look-back for Q counters of partition c at once: ex[i] = sum of
// counter q[i] over partitions [0, c).  States are look[part * stride + q].
// Each step loads the states of the W partitions below the current one for
// every counter (Q * W independent loads in flight), adds them from the
// nearest down to the first inclusive prefix, and continues below the window
// only if all W were aggregates; a state not yet published ends the step
// early and is read again.  Partitions all publish their aggregates at about
// the same time, so a CTA reaches an inclusive prefix in about c / W steps at
// worst instead of c.  A predecessor that does not publish within the wait
// limit records a timeout and the chain stops (the result is then wrong but
// the kernel ends).
template <int Q, int W>
__device__ void look_back(const uint64_t* look, int64_t stride, int64_t c, const int (&q)[Q], const bool (&act)[Q],
                          uint32_t epoch, int32_t (&ex)[Q], int32_t* status,
                          uint64_t limit_ns = ptx::kWaitLimitNs) {
    int64_t j[Q];   // next partition to read, per counter (-1: done)
    bool all = true;
#pragma unroll
    for (int i = 0; i < Q; ++i) {
        ex[i] = 0;
        j[i] = (act[i] && c > 0) ? c - 1 : -1;
        all &= j[i] < 0;
    }
    if (all) return;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint64_t v[Q][W];
#pragma unroll
        for (int i = 0; i < Q; ++i)
#pragma unroll
            for (int k = 0; k < W; ++k)
                v[i][k] = (j[i] - k >= 0) ? ld_relaxed(look + (j[i] - k) * stride + q[i]) : 0ull;
        all = true;
#pragma unroll
        for (int i = 0; i < Q; ++i) {
            bool go = j[i] >= 0;
#pragma unroll
            for (int k = 0; k < W; ++k) {
                if (!go || j[i] < 0) break;
                const uint64_t x = v[i][k];
                if ((x >> 32) != epoch || (x & kFlags) == 0) {
                    go = false;   // not published yet: read again from here
                    break;
                }
                ex[i] += static_cast<int32_t>(x & kCount);
                j[i] = (x & kFlags) == kPre ? -1 : j[i] - 1;
            }
            all &= j[i] < 0;
        }
        if (all) return;
        if (it == 0) t0 = ptx::globaltimer();
        if ((it & 15u) == 15u && ptx::globaltimer() - t0 > limit_ns) {
            atomicOr(status, kStatusTimeout);
            return;
        }
    }
}

// Exclusive scan over the threads of the CTA (all WT threads call).
__device__ __forceinline__ int32_t block_exclusive(int32_t x, int32_t* wsum) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    int32_t incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    int32_t before = 0;
#pragma unroll
    for (int i = 0; i < WW; ++i) before += i < w ? wsum[i] : 0;
    __syncthreads();
    return before + incl - x;
}

// Barrier over all P CTAs of the grid (every CTA must be resident), for the
// round-th time (0, 1, ...).  bar: kWideBarrierInts counters, zero before
// round 0.  CTA c arrives at counter c % 32; the arrival that completes a
// counter's share of the round bumps the release counter, which every CTA
// polls (with a short sleep between polls) until all used counters have
// completed the round.  Arrivals spread over 32 addresses instead of one.
// Bounded in time.
__device__ void grid_barrier(int32_t* bar, int64_t P, int round, int32_t* status,
                             uint64_t limit_ns = ptx::kWaitLimitNs) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const int nsub = P < 32 ? static_cast<int>(P) : 32;
        const int j = static_cast<int>(blockIdx.x % 32);
        const int share = static_cast<int>(P / 32 + (j < P % 32 ? 1 : 0));
        __threadfence();
        const int old = atomicAdd(bar + j, 1);
        if ((old + 1) % share == 0) {
            __threadfence();
            atomicAdd(bar + 32, 1);
        }
        const int32_t target = (round + 1) * nsub;
        uint64_t t0 = 0;
        for (uint32_t it = 0;; ++it) {
            int32_t v;
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(bar + 32) : "memory");
            if (v >= target) break;
            if (it == 0) t0 = ptx::globaltimer();
            __nanosleep(32);
            if ((it & 63u) == 63u && ptx::globaltimer() - t0 > limit_ns) {
                atomicOr(status, kStatusTimeout);
                break;
            }
        }
        __threadfence();
    }
    __syncthreads();
}

__device__ __forceinline__ bool coord_ok(int4 q, int3 shape, int batch) {
    return q.x >= 0 && q.x < batch && q.y >= 0 && q.y < shape.x && q.z >= 0 && q.z < shape.y && q.w >= 0 &&
           q.w < shape.z;
}

// First kernel of a build: clears the status word, every digit histogram,
// the tickets and barrier counters, the tap counts and totals, the look-back
// states, and the hash table (hash mapper) or the presence grid to -1 (dense
// mapper).  The kernel after it overlaps it and waits for it only before its
// first write to any of these.  The look-back states must start cleared: the
// arena is recycled memory, and a stale word (an old hash entry or packed key)
// can carry the current epoch in its top half and nonzero flag bits.
__global__ void __launch_bounds__(WT) k_wide_clear(const WideArgs a) {
    pdl_trigger();
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * WT + threadIdx.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * WT;
    if (i0 == 0) *a.status = 0;
    for (int64_t i = i0; i < (kWideKeyPassesMax + kWideMaskPasses) * kWideBins; i += stride) a.gh[i] = 0;
    for (int64_t i = i0; i < kWideCounters; i += stride) a.tickets[i] = 0;
    if (i0 < kTaps) a.tap_count[i0] = 0;
    if (i0 < 2) a.totals[i0] = 0;
    {
        ulonglong2* l2 = reinterpret_cast<ulonglong2*>(a.look);
        const int64_t parts = (a.n + kWideKeysPerCta - 1) / kWideKeysPerCta;
        for (int64_t i = i0; i < parts * kWideBins / 2; i += stride) l2[i] = make_ulonglong2(0ull, 0ull);
    }
    if (a.mapper == SPCONV_MAPPER_HASH) {
        ulonglong2* t2 = reinterpret_cast<ulonglong2*>(a.table);
        const int64_t slots2 = (int64_t(1) << a.table_log2) / 2;
        for (int64_t i = i0; i < slots2; i += stride) t2[i] = make_ulonglong2(0ull, 0ull);
    }
    if (a.mapper == SPCONV_MAPPER_DENSE) {
        int4* g4 = reinterpret_cast<int4*>(a.grid);
        const int64_t c4 = a.cells / 4;
        for (int64_t i = i0; i < c4; i += stride) g4[i] = make_int4(-1, -1, -1, -1);
        for (int64_t i = 4 * c4 + i0; i < a.cells; i += stride) a.grid[i] = -1;
    }
}

// The digits of the coordinate sort: the live key bits split into the fewest
// passes of at most kDigitBitsWide bits, as evenly as possible (28 bits:
// 10 + 9 + 9; a 9-bit pass looks back over half the digit values of a
// 10-bit one).
struct KeyDigits {
    int passes;
    int shift[kWideKeyPassesMax];
    int width[kWideKeyPassesMax];
};

// ---------------------------------------------------------------------------
// sorted-key mapper: packed keys and the digit counts of the key passes in
// kd (none where every pass runs in the count exchange)
// ---------------------------------------------------------------------------
template <int kRowsPerThread>
__global__ void __launch_bounds__(WT) k_wide_keys(const WideArgs a, const KeyDigits kd) {
    __shared__ int32_t h[kWideKeyPassesMax][kWideBins];
    const int t = threadIdx.x, lane = t & 31;
    const int passes = kd.passes;
    pdl_trigger();
    for (int i = t; i < kWideKeyPassesMax * kWideBins; i += WT) (&h[0][0])[i] = 0;
    __syncthreads();
    const int rb = a.row_bits;
    const uint64_t invalid = (uint64_t(1) << a.key_bits) - 1;
    int32_t err = 0;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * WT * kRowsPerThread + t;
    int4 qs[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        const int64_t i = row0 + r * WT;
        qs[r] = i < a.n ? a.coords[i] : make_int4(-1, -1, -1, -1);
    }
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        const int64_t i = row0 + r * WT;
        const bool valid = i < a.n;
        uint64_t key = invalid;
        if (valid) {
            const int4 q = qs[r];
            if (coord_ok(q, a.shape, a.batch)) {
                key = (((((static_cast<uint64_t>(q.x) << a.wx) | static_cast<uint64_t>(q.y + 1)) << a.wy) |
                        static_cast<uint64_t>(q.z + 1))
                       << a.wz) |
                      static_cast<uint64_t>(q.w + 1);
            } else {
                err |= kStatusRange;
            }
            a.va[i] = (key << rb) | static_cast<uint64_t>(i);
        }
        for (int p = 0; p < passes; ++p) {
            const uint64_t dmask = (uint64_t(1) << kd.width[p]) - 1;
            const int dg = valid ? static_cast<int>((key >> kd.shift[p]) & dmask) : kWideBins;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, dg);
            if (valid && lane == __ffs(peers) - 1) atomicAdd(&h[p][dg], __popc(peers));
        }
    }
    __syncthreads();
    pdl_wait();   // the histograms and the status word are cleared
    for (int i = t; i < passes * kWideBins; i += WT) {
        const int p = i / kWideBins, b = i % kWideBins;
        const int32_t x = b < (1 << kd.width[p]) ? h[p][b] : 0;
        if (x) atomicAdd(a.gh + p * kWideBins + b, x);
    }
    if (err) atomicOr(a.status, err);
}

// ---------------------------------------------------------------------------
// hash mapper: the packed coordinate keys in an open-addressing table of
// 4-slot buckets (bucketed linear probing), hashed by key >> 1 so that the
// two voxels of a z pair share a bucket; then per row and (dx, dy) column
// two bucket reads cover the three keys of dz = -1, 0, +1.  The packed key's
// arithmetic is the sorted mapper's (neighbour key = key + packed(d)); only
// the lookup structure differs: a probe is a 32-byte bucket read instead of
// a binary search after a sort.  Within a bucket the slots fill in order and
// never empty again, and a pair's entries go to its bucket or the ones after
// it, so a bucket with an empty slot holds every entry of the pairs hashed to
// it; only a full bucket sends a lookup on to the next one.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t hash_bucket(uint64_t key, int log2_buckets) {
    return (key * 0x9E3779B97F4A7C15ull) >> (64 - log2_buckets);   // multiplicative (Fibonacci) hashing
}

// One bucket (4 slots, 32 bytes, 32-byte aligned) in a single 256-bit load
// through L2 (the table was written by the kernel before this one).
__device__ __forceinline__ void load_bucket(const uint64_t* b, ulonglong2& lo, ulonglong2& hi) {
    asm volatile("ld.global.cg.v4.u64 {%0, %1, %2, %3}, [%4];"
                 : "=l"(lo.x), "=l"(lo.y), "=l"(hi.x), "=l"(hi.y)
                 : "l"(b));
}

__device__ __forceinline__ uint64_t packed_key(int4 q, const WideArgs& a) {
    return (((((static_cast<uint64_t>(q.x) << a.wx) | static_cast<uint64_t>(q.y + 1)) << a.wy) |
             static_cast<uint64_t>(q.z + 1))
            << a.wz) |
           static_cast<uint64_t>(q.w + 1);
}

// Table entries: (key << 32 | row) when keys fit 32 bits (kKey32: a slot's key
// and row are its two halves, compared with 32-bit instructions), else
// (key << row_bits | row).  Either way an entry is never 0: keys are >= 1.
template <bool kKey32>
__device__ __forceinline__ uint64_t hash_entry(uint64_t key, int64_t row, int row_bits) {
    return (key << (kKey32 ? 32 : row_bits)) | static_cast<uint64_t>(row);
}

template <bool kKey32>
__global__ void __launch_bounds__(WT) k_wide_hash_insert(const WideArgs a) {
    pdl_trigger();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * WT + threadIdx.x;
    const bool valid = i < a.n;
    const int4 q = valid ? a.coords[i] : make_int4(-1, -1, -1, -1);
    const bool ok = valid && coord_ok(q, a.shape, a.batch);
    const uint64_t key = ok ? packed_key(q, a) : 0ull;
    pdl_wait();   // the table is cleared
    int32_t err = (valid && !ok) ? kStatusRange : 0;
    if (ok) {
        // key >= 1 (every field is offset by one), so an entry is never 0 (empty)
        const uint64_t entry = hash_entry<kKey32>(key, i, a.row_bits);
        const int ks = kKey32 ? 32 : a.row_bits;
        const int lb = a.table_log2 - 2;
        const uint64_t bmask = (uint64_t(1) << lb) - 1;
        uint64_t b = hash_bucket(key >> 1, lb);
        bool placed = false;
        for (uint64_t probe = 0; probe <= bmask && !placed; ++probe, b = (b + 1) & bmask) {
            for (int j = 0; j < kHashBucket; ++j) {
                const unsigned long long prev = atomicCAS(
                    reinterpret_cast<unsigned long long*>(a.table + b * kHashBucket + j), 0ull,
                    static_cast<unsigned long long>(entry));
                if (prev == 0ull || (prev >> ks) == key) {   // placed, or the same voxel twice
                    if (prev != 0ull) err |= kStatusDuplicate;
                    placed = true;
                    break;
                }
            }
        }
        if (!placed) err |= kStatusInternal;   // a full table: cannot happen at load <= 1/16
    }
    if (err) atomicOr(a.status, err);
}

// Scans one bucket (slots lo.x, lo.y, hi.x, hi.y) for the keys kc - 1, kc,
// kc + 1 of a column, recording the rows found in v0, v1, v2; returns whether
// the bucket has an empty slot (then it holds every entry of its pairs).
__device__ __forceinline__ bool bucket_scan(ulonglong2 lo, ulonglong2 hi, uint64_t kc, int row_bits, int32_t& v0,
                                            int32_t& v1, int32_t& v2) {
    const uint64_t s[4] = {lo.x, lo.y, hi.x, hi.y};
    const uint64_t row_mask = (uint64_t(1) << row_bits) - 1;
    bool open = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        open |= s[j] == 0ull;
        const uint64_t d = (s[j] >> row_bits) - (kc - 1);   // 0, 1, 2 for the column's keys
        const int32_t row = static_cast<int32_t>(s[j] & row_mask);
        if (s[j] != 0ull) {
            v0 = d == 0 ? row : v0;
            v1 = d == 1 ? row : v1;
            v2 = d == 2 ? row : v2;
        }
    }
    return open;
}

// bucket_scan for 32-bit keys: key and row are the halves of a slot, and the
// column's keys kc - 1, kc, kc + 1 are the slots whose key minus (kc - 1) is
// 0, 1 or 2 (unsigned); an empty slot is excluded by its zero key.
__device__ __forceinline__ bool bucket_scan32(ulonglong2 lo, ulonglong2 hi, uint64_t kc, int32_t& v0, int32_t& v1,
                                              int32_t& v2) {
    const uint64_t s[4] = {lo.x, lo.y, hi.x, hi.y};
    const uint32_t base = static_cast<uint32_t>(kc) - 1u;
    bool open = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t key = static_cast<uint32_t>(s[j] >> 32);
        const int32_t row = static_cast<int32_t>(static_cast<uint32_t>(s[j]));
        open |= key == 0u;
        const uint32_t d = key == 0u ? 3u : key - base;   // 3 and above: not the column's
        v0 = d == 0u ? row : v0;
        v1 = d == 1u ? row : v1;
        v2 = d == 2u ? row : v2;
    }
    return open;
}

template <bool kKey32>
__device__ __forceinline__ bool scan_bucket(ulonglong2 lo, ulonglong2 hi, uint64_t kc, int row_bits, int32_t& v0,
                                            int32_t& v1, int32_t& v2) {
    return kKey32 ? bucket_scan32(lo, hi, kc, v0, v1, v2) : bucket_scan(lo, hi, kc, row_bits, v0, v1, v2);
}

// Three threads per row, one dx plane each, 128 rows per block: every
// thread's 6 bucket reads are in flight at once (a thread per row with the
// planes in turn had only a third of the reads in flight and waited three
// times as long).  The rows are assembled in shared memory and written whole,
// coalesced.
constexpr int kHashLookupRows = 128;

template <bool kKey32>
__global__ void __launch_bounds__(kHashLookupRows * 3, 2) k_wide_hash_lookup(const WideArgs a) {
    __shared__ int32_t rows_s[kHashLookupRows][kNbrStride + 1];   // +1: conflict-free row and column access
    __shared__ uint32_t mask_s[kHashLookupRows];
    __shared__ int32_t cnt[kTaps];
    const int t = threadIdx.x, lane = t & 31;
    const int p = t / kHashLookupRows;   // this thread's dx plane (warp-uniform)
    const int rl = t % kHashLookupRows;  // its row within the block
    if (t < kTaps) cnt[t] = 0;
    if (t < kHashLookupRows) mask_s[t] = 0;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kHashLookupRows;
    const int64_t i = row0 + rl;
    const bool valid = i < a.n;
    const int4 q = valid ? a.coords[i] : make_int4(-1, -1, -1, -1);
    const bool ok = valid && coord_ok(q, a.shape, a.batch);
    const uint64_t key = ok ? packed_key(q, a) : 0ull;
    pdl_wait();   // every key is in the table
    pdl_trigger();
    int32_t v[9];
#pragma unroll
    for (int k = 0; k < 9; ++k) v[k] = -1;
    const int lb = a.table_log2 - 2;
    const uint64_t bmask = (uint64_t(1) << lb) - 1;
    // the plane's 3 columns, 6 bucket reads (the pairs of kc - 1 and kc + 1);
    // the rare reads that meet a full bucket go on, all of the warp's in the
    // same extra round
    ulonglong2 lo[6], hi[6];
    uint64_t kc[3];
    uint32_t pending = 0;
#pragma unroll
    for (int c = 0; c < 3; ++c) {   // the column's dz = 0 key (32-bit keys: known to fit the low half)
        const uint64_t k64 = key + a.koff[9 * p + 3 * c + 1];
        kc[c] = kKey32 ? static_cast<uint64_t>(static_cast<uint32_t>(k64)) : k64;
    }
#pragma unroll
    for (int r = 0; r < 6; ++r) {
        if (ok) {
            const uint64_t b = hash_bucket((kc[r >> 1] + ((r & 1) ? 1 : -1)) >> 1, lb);
            load_bucket(a.table + b * kHashBucket, lo[r], hi[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < 6; ++r)
        if (ok && !scan_bucket<kKey32>(lo[r], hi[r], kc[r >> 1], a.row_bits, v[3 * (r >> 1)], v[3 * (r >> 1) + 1],
                                       v[3 * (r >> 1) + 2]))
            pending |= 1u << r;
    for (uint64_t step = 1; __any_sync(0xFFFFFFFFu, pending != 0u) && step <= bmask; ++step) {
#pragma unroll
        for (int r = 0; r < 6; ++r) {
            if ((pending >> r) & 1u) {
                const uint64_t b = (hash_bucket((kc[r >> 1] + ((r & 1) ? 1 : -1)) >> 1, lb) + step) & bmask;
                load_bucket(a.table + b * kHashBucket, lo[r], hi[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < 6; ++r)
            if (((pending >> r) & 1u) && scan_bucket<kKey32>(lo[r], hi[r], kc[r >> 1], a.row_bits, v[3 * (r >> 1)],
                                                             v[3 * (r >> 1) + 1], v[3 * (r >> 1) + 2]))
                pending &= ~(1u << r);
    }
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < 9; ++k) {
        rows_s[rl][9 * p + k] = v[k];
        m |= (v[k] >= 0 ? 1u : 0u) << k;
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, v[k] >= 0);
        if (lane == 0 && b) atomicAdd(&cnt[9 * p + k], __popc(b));
    }
    if (p == 0)
        for (int k = kTaps; k < kNbrStride; ++k) rows_s[rl][k] = -1;
    __syncthreads();   // mask_s is cleared
    if (m) atomicOr(&mask_s[rl], m << (9 * p));
    __syncthreads();
    // the block's rows, whole and coalesced
    const int64_t rows = a.n - row0 < kHashLookupRows ? a.n - row0 : kHashLookupRows;
    for (int idx = t; idx < rows * kNbrStride; idx += kHashLookupRows * 3)
        a.nbr[row0 * kNbrStride + idx] = rows_s[idx / kNbrStride][idx % kNbrStride];
    if (t < rows) a.mask[row0 + t] = mask_s[t];
    if (t < kTaps && cnt[t]) atomicAdd(a.tap_count + t, cnt[t]);
}

// ---------------------------------------------------------------------------
// dense mapper: presence grid (cleared to -1 before), then 27 lookups per row
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(WT) k_wide_grid_scatter(const WideArgs a) {
    pdl_trigger();
    pdl_wait();   // the grid is cleared
    int32_t err = 0;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * WT + threadIdx.x; i < a.n;
         i += static_cast<int64_t>(gridDim.x) * WT) {
        const int4 q = a.coords[i];
        if (coord_ok(q, a.shape, a.batch)) {
            const int64_t cell = q.x * a.gsb + static_cast<int64_t>(q.y + 1) * a.gsx +
                                 static_cast<int64_t>(q.z + 1) * a.gsy + (q.w + 1);
            if (atomicCAS(a.grid + cell, -1, static_cast<int32_t>(i)) != -1) err |= kStatusDuplicate;
        } else {
            err |= kStatusRange;
        }
    }
    if (err) atomicOr(a.status, err);
}

__global__ void __launch_bounds__(WT) k_wide_grid_lookup(const WideArgs a) {
    __shared__ int32_t cnt[kTaps];
    const int t = threadIdx.x, lane = t & 31;
    if (t < kTaps) cnt[t] = 0;
    __syncthreads();
    pdl_wait();   // the grid scatter has finished
    pdl_trigger();
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * WT; i0 < a.n; i0 += static_cast<int64_t>(gridDim.x) * WT) {
        const int64_t i = i0 + t;
        uint32_t m = 0;
        if (i < a.n) {
            const int4 q = a.coords[i];
            int32_t v[kNbrStride];
#pragma unroll
            for (int k = 0; k < kNbrStride; ++k) v[k] = -1;
            if (coord_ok(q, a.shape, a.batch)) {
                const int64_t cell = q.x * a.gsb + static_cast<int64_t>(q.y + 1) * a.gsx +
                                     static_cast<int64_t>(q.z + 1) * a.gsy + (q.w + 1);
#pragma unroll
                for (int k = 0; k < kTaps; ++k) {
                    v[k] = __ldcg(a.grid + cell + a.goff[k]);
                    m |= (v[k] >= 0 ? 1u : 0u) << k;
                }
            }
            int4* dst = reinterpret_cast<int4*>(a.nbr + i * kNbrStride);
#pragma unroll
            for (int qq = 0; qq < kNbrStride / 4; ++qq)
                dst[qq] = make_int4(v[4 * qq], v[4 * qq + 1], v[4 * qq + 2], v[4 * qq + 3]);
            a.mask[i] = m;
        }
#pragma unroll
        for (int k = 0; k < kTaps; ++k) {
            const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
            if (lane == 0 && b) atomicAdd(&cnt[k], __popc(b));
        }
    }
    __syncthreads();
    if (t < kTaps && cnt[t]) atomicAdd(a.tap_count + t, cnt[t]);
}

// ---------------------------------------------------------------------------
// mask sort keys: the mask's bits in the tap order (rarest tap in the top bit
// with the calibrated order), packed with the row; digit counts of the passes
// ---------------------------------------------------------------------------
template <int kRowsPerThread>
__global__ void __launch_bounds__(WT) k_wide_mask_keys(const WideArgs a) {
    __shared__ int32_t h[kWideMaskPasses][1 << kMaskWidth];
    __shared__ int32_t taps[kTaps];
    __shared__ int32_t pos[kTaps];
    const int t = threadIdx.x, lane = t & 31;
    constexpr int bins = 1 << kMaskWidth;
    for (int i = t; i < kWideMaskPasses * bins; i += WT) (&h[0][0])[i] = 0;
    pdl_wait();   // masks and tap counts are complete
    pdl_trigger();
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * WT * kRowsPerThread + t;
    uint32_t ms[kRowsPerThread];   // requested with the tap counts: one round trip for both
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        const int64_t i = row0 + r * WT;
        ms[r] = i < a.n ? __ldcg(a.mask + i) : 0u;
    }
    if (t < kTaps) taps[t] = __ldcg(a.tap_count + t);
    __syncthreads();
    if (t < kTaps) {
        int32_t rank = t;
        if (a.calibrated) {
            const int32_t ck = taps[t];
            rank = 0;
            for (int j = 0; j < kTaps; ++j) {
                const int32_t cj = taps[j];
                rank += (cj > ck || (cj == ck && j < t)) ? 1 : 0;
            }
        }
        pos[t] = rank;
    }
    __syncthreads();
    const int rb = a.row_bits;
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        const int64_t i = row0 + r * WT;
        const bool valid = i < a.n;
        uint32_t key = 0;
        if (valid) {
            const uint32_t m = ms[r];
#pragma unroll
            for (int k = 0; k < kTaps; ++k) key |= ((m >> k) & 1u) << pos[k];
            a.va[i] = (static_cast<uint64_t>(key) << rb) | static_cast<uint64_t>(i);
        }
#pragma unroll
        for (int p = 0; p < kWideMaskPasses; ++p) {
            const int dg = valid ? static_cast<int>((key >> (kMaskWidth * p)) & (bins - 1)) : kWideBins;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, dg);
            if (valid && lane == __ffs(peers) - 1) atomicAdd(&h[p][dg], __popc(peers));
        }
    }
    __syncthreads();
    for (int i = t; i < kWideMaskPasses * bins; i += WT) {
        const int p = i / bins, b = i % bins;
        const int32_t x = h[p][b];
        if (x) atomicAdd(a.gh + (kWideKeyPassesMax + p) * kWideBins + b, x);
    }
}

// ---------------------------------------------------------------------------
// one stable LSD pass by the digit of `width` bits at bit `shift` of the
// packed values
// ---------------------------------------------------------------------------
struct PassArgs {
    const uint64_t* in;
    uint64_t* out;
    int64_t n;
    int shift, width;
    const int32_t* gh;     // [kWideBins] digit totals of this pass
    uint64_t* look;        // [partitions][kWideBins] look-back states
    uint32_t epoch;
    int32_t* ticket;       // partition counter, or null: partition = blockIdx.x (the whole grid is resident)
    int32_t* bar;          // non-null: prefixes by two grid barriers instead of look-back (see below)
    uint64_t* words;       // non-null: prefixes and digit totals from every partition's packed counts
    int32_t* arrive;       // with words: the pass's arrival counter (its ticket, zero before the pass)
    int32_t* status;
    // the first pass of the mask sort (kMask): its values are made from the
    // rows' masks, (key << row_bits | row), the key the mask in the tap order
    const uint32_t* mask;
    const int32_t* tap_count;
    int calibrated, row_bits;
};

// Partitions the look-back reads per step.
constexpr int kLookWindow = 8;

// The all-partition form (every partition resident, at most kSumFormParts):
// each partition publishes its digit counts as self-validating 64-bit words
// -- a tag in the high half (the pass's epoch with bit 31 set, which no count
// and no older state word has there) and two 16-bit counts in the low half,
// digits Q t + 2h and Q t + 2h + 1 in word h of thread t -- and reads every
// partition's words until all carry the tag.  No fence, flag or chain of
// prefixes: one store, then one round of loads.  Low halves are added as
// packed pairs over chunks of at most kSumChunk<WI, Q> partitions (chunk x
// keys per partition < 2^16) before they are widened.
constexpr int64_t kSumFormParts = 64;
template <int WI, int Q>
constexpr int kSumChunk = (Q == 2 ? 31 : 15) < 65535 / (WT * WI) ? (Q == 2 ? 31 : 15) : 65535 / (WT * WI);

__device__ __forceinline__ uint64_t word_tag(uint32_t epoch) {
    return static_cast<uint64_t>(0x80000000u | (epoch & 0x7FFFFFFFu)) << 32;
}

// Partition c of P publishes its counts tot and gathers, per digit, the count
// over the partitions before it (ex) and over all of them (all).  Every
// thread of the CTA calls it.  arrive (zero before the pass, or null): a
// counter each partition bumps once its words are out; waiting for it to
// reach P before the first read makes that read find nearly every word
// already published (outdoor map 47.8 -> 45.7 us against reading at once and
// rereading the missing words).  The words alone decide what is read: a
// partition that does not publish within the wait limit records a timeout
// (the sums are then wrong but the kernel ends).
template <int Q, int CH>
__device__ void exchange_counts(uint64_t* words, int64_t P, int64_t c, uint32_t epoch, const int32_t (&tot)[Q],
                                int32_t (&ex)[Q], int32_t (&all)[Q], int32_t* status, int32_t* arrive,
                                uint64_t limit_ns = ptx::kWaitLimitNs) {
    constexpr int NW = Q / 2;
    static_assert(CH >= 1 && CH <= 31, "partitions per chunk");
    const int t = threadIdx.x;
    const uint64_t tag = word_tag(epoch);
#pragma unroll
    for (int h = 0; h < NW; ++h) {
        const uint32_t lo = (static_cast<uint32_t>(tot[2 * h]) & 0xFFFFu) |
                            ((static_cast<uint32_t>(tot[2 * h + 1]) & 0xFFFFu) << 16);
        st_relaxed(words + (c * NW + h) * WT + t, tag | lo);
    }
    if (arrive != nullptr) {
        __syncthreads();
        if (t == 0) {
            atomicAdd(arrive, 1);
            const uint64_t ta = ptx::globaltimer();
            for (uint32_t it = 0;; ++it) {
                int32_t v;
                asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(arrive) : "memory");
                if (v >= P) break;
                __nanosleep(32);
                if ((it & 31u) == 31u && ptx::globaltimer() - ta > limit_ns) break;   // the words' wait reports it
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < Q; ++q) ex[q] = all[q] = 0;
    uint64_t t0 = 0;
    bool gave_up = false;
    for (int64_t p0 = 0; p0 < P; p0 += CH) {
        const int np = P - p0 < CH ? static_cast<int>(P - p0) : CH;
        uint32_t need = gave_up ? 0u : (1u << np) - 1u;
        uint32_t run_all[NW], run_ex[NW];
#pragma unroll
        for (int h = 0; h < NW; ++h) run_all[h] = run_ex[h] = 0;
        while (need != 0u) {
            uint64_t x[CH][NW];
#pragma unroll
            for (int i = 0; i < CH; ++i)
#pragma unroll
                for (int h = 0; h < NW; ++h)
                    x[i][h] = ((need >> i) & 1u) ? ld_relaxed(words + ((p0 + i) * NW + h) * WT + t) : 0ull;
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                if (!((need >> i) & 1u)) continue;
                bool ok = true;
#pragma unroll
                for (int h = 0; h < NW; ++h) ok &= (x[i][h] & 0xFFFFFFFF00000000ull) == tag;
                if (!ok) continue;
                need &= ~(1u << i);
#pragma unroll
                for (int h = 0; h < NW; ++h) {
                    const uint32_t lo = static_cast<uint32_t>(x[i][h]);
                    run_all[h] += lo;
                    run_ex[h] += p0 + i < c ? lo : 0u;
                }
            }
            if (need == 0u) break;
            if (t0 == 0) {
                t0 = ptx::globaltimer();
            } else if (ptx::globaltimer() - t0 > limit_ns) {
                atomicOr(status, kStatusTimeout);
                gave_up = true;
                break;
            }
            __nanosleep(64);
        }
#pragma unroll
        for (int h = 0; h < NW; ++h) {
            all[2 * h] += static_cast<int32_t>(run_all[h] & 0xFFFFu);
            all[2 * h + 1] += static_cast<int32_t>(run_all[h] >> 16);
            ex[2 * h] += static_cast<int32_t>(run_ex[h] & 0xFFFFu);
            ex[2 * h + 1] += static_cast<int32_t>(run_ex[h] >> 16);
        }
    }
}

// Partitions a CTA scans per digit in the barrier form (consecutive, one lane
// each group), and digits a warp scans at once.
constexpr int kScanPerLane = 8;
constexpr int kScanDigitsPerWarp = 4;

// Q: digits per thread (Q WT >= 2^width), consecutive digits Q t .. Q t + Q - 1.
// kMask: the first pass of the mask sort, which makes its values from the
// masks (only with the all-partition form, which needs no digit totals).
// (2048 keys of 10-bit digits need more registers than two CTAs per SM allow)
template <int WI, int Q, bool kMask = false>
__global__ void __launch_bounds__(WT, WI * Q > 16 ? 1 : 2) k_wide_pass(const PassArgs a) {
    static_assert(Q == 2 || Q == 4, "digits per thread");
    // cnt[w][d]: keys of warp w with digit d, then the warp's offset within
    // the CTA's keys of digit d (stable order inside the CTA: warp, item, lane)
    __shared__ uint16_t cnt[WW][kWideBins];
    __shared__ int32_t gbase[kWideBins];   // first output position of each digit
    __shared__ int32_t excl[kWideBins];    // keys of each digit in the partitions before this one
    __shared__ int32_t wsum[WW];
    __shared__ int32_t part_sh, err;
    // kMask: the taps' key bits and, per byte of a mask, the key bits it sets
    __shared__ int32_t mtaps[kMask ? kTaps : 1], mpos[kMask ? kTaps : 1];
    __shared__ uint32_t mtab[kMask ? 4 : 1][kMask ? 256 : 1];
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int bins = 1 << a.width;
    const uint64_t dmask = static_cast<uint64_t>(bins - 1);
    uint32_t* cz = reinterpret_cast<uint32_t*>(&cnt[0][0]);
    for (int i = t; i < WW * kWideBins / 2; i += WT) cz[i] = 0;
    if (t == 0) err = 0;
    pdl_wait();   // the keys and the digit totals are complete
    pdl_trigger();
    int64_t c = blockIdx.x;
    if (a.ticket) {
        if (t == 0) part_sh = atomicAdd(a.ticket, 1);
        __syncthreads();
        c = part_sh;
    }
    // this partition's keys (requested first: their latency overlaps the scan below)
    const int64_t base = c * WT * WI;
    uint64_t v[WI];
    int d[WI], rk[WI];
    if (kMask) {
        // the masks and tap counts; the key of a mask puts tap k at bit pos[k]
        // (calibrated: taps by descending count, ties by index), assembled from
        // four byte tables so that a key costs four shared loads
        uint32_t mk[WI];
#pragma unroll
        for (int j = 0; j < WI; ++j) {
            const int64_t idx = base + static_cast<int64_t>(w) * 32 * WI + 32 * j + lane;
            mk[j] = idx < a.n ? __ldcg(a.mask + idx) : 0u;
        }
        if (t < kTaps) mtaps[t] = __ldcg(a.tap_count + t);
        __syncthreads();
        if (t < kTaps) {
            int32_t rank = t;
            if (a.calibrated) {
                const int32_t ck = mtaps[t];
                rank = 0;
                for (int jj = 0; jj < kTaps; ++jj) {
                    const int32_t cj = mtaps[jj];
                    rank += (cj > ck || (cj == ck && jj < t)) ? 1 : 0;
                }
            }
            mpos[t] = rank;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t x = 0;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int k = 8 * i + b;
                if (k < kTaps && ((t >> b) & 1)) x |= 1u << mpos[k];
            }
            mtab[i][t] = x;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < WI; ++j) {
            const int64_t idx = base + static_cast<int64_t>(w) * 32 * WI + 32 * j + lane;
            const uint32_t m = mk[j];
            const uint32_t key = mtab[0][m & 255u] | mtab[1][(m >> 8) & 255u] | mtab[2][(m >> 16) & 255u] |
                                 mtab[3][m >> 24];
            v[j] = idx < a.n ? (static_cast<uint64_t>(key) << a.row_bits) | static_cast<uint64_t>(idx) : 0ull;
        }
    } else {
#pragma unroll
        for (int j = 0; j < WI; ++j) {
            const int64_t idx = base + static_cast<int64_t>(w) * 32 * WI + 32 * j + lane;
            v[j] = idx < a.n ? __ldcg(a.in + idx) : 0ull;
        }
    }
    // digit totals -> first output position of every digit (thread t: digits Q t .. Q t + Q - 1);
    // the all-partition form takes them from the partitions' published counts instead
    if (a.words == nullptr) {
        int32_t g[Q];
        int32_t gs = 0;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int d = Q * t + q;
            g[q] = d < bins ? __ldcg(a.gh + d) : 0;
            gs += g[q];
        }
        int32_t run = block_exclusive(gs, wsum);   // (synchronises the CTA: cnt is cleared after it)
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            gbase[Q * t + q] = run;
            run += g[q];
        }
    } else {
        __syncthreads();   // cnt is cleared
    }
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int j = 0; j < WI; ++j) {
        const int64_t idx = base + static_cast<int64_t>(w) * 32 * WI + 32 * j + lane;
        d[j] = idx < a.n ? static_cast<int>((v[j] >> a.shift) & dmask) : kWideBins;
    }
#pragma unroll
    for (int j = 0; j < WI; ++j) {
        const bool valid = d[j] < kWideBins;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d[j]);
        const int prior = valid ? cnt[w][d[j]] : 0;
        rk[j] = prior + __popc(peers & lt);
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) cnt[w][d[j]] = static_cast<uint16_t>(prior + __popc(peers));
        __syncwarp();
    }
    __syncthreads();
    // per digit (thread t: digits Q t .. Q t + Q - 1): offsets of the warps,
    // the CTA's count, published as this partition's aggregate
    int qd[Q];
    bool act[Q];
    int32_t tot[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int dd = Q * t + q;
        qd[q] = dd;
        act[q] = dd < bins;
        int32_t x[WW];
#pragma unroll
        for (int ww = 0; ww < WW; ++ww) x[ww] = act[q] ? cnt[ww][dd] : 0;
        int32_t pre = 0;
#pragma unroll
        for (int ww = 0; ww < WW; ++ww) {
            if (act[q]) cnt[ww][dd] = static_cast<uint16_t>(pre);
            pre += x[ww];
        }
        tot[q] = pre;
    }
    int32_t ex[Q];
    if (a.bar != nullptr) {
        // Every partition is resident.  Counts go to pc[digit][partition];
        // after a grid barrier each CTA turns the rows of its own few digits
        // into exclusive prefixes over the partitions (a warp per digit, lane
        // l holding partitions [l K, l K + K)), and after a second barrier
        // each partition reads its prefix of every digit.  About seven
        // dependent memory round trips, whatever the number of partitions.
        const int64_t P = gridDim.x;
        int32_t* pc = reinterpret_cast<int32_t*>(a.look);
#pragma unroll
        for (int q = 0; q < Q; ++q)
            if (act[q]) pc[qd[q] * P + c] = tot[q];
        grid_barrier(a.bar, P, 0, a.status);
        const int per = static_cast<int>((bins + P - 1) / P);       // digits of this CTA
        const int K = static_cast<int>((P + 31) / 32);              // partitions per lane (<= kScanPerLane)
        const int d0 = static_cast<int>(c) * per;
        const int d1 = d0 + per < bins ? d0 + per : bins;
        int32_t x[kScanDigitsPerWarp][kScanPerLane];
#pragma unroll
        for (int i = 0; i < kScanDigitsPerWarp; ++i) {
            const int dd = d0 + w + WW * i;
#pragma unroll
            for (int k = 0; k < kScanPerLane; ++k) {
                const int64_t j = static_cast<int64_t>(lane) * K + k;
                x[i][k] = (dd < d1 && k < K && j < P) ? __ldcg(pc + dd * P + j) : 0;
            }
        }
#pragma unroll
        for (int i = 0; i < kScanDigitsPerWarp; ++i) {
            const int dd = d0 + w + WW * i;
            int32_t sum = 0;
#pragma unroll
            for (int k = 0; k < kScanPerLane; ++k) sum += x[i][k];
            int32_t inc = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += y;
            }
            int32_t run = inc - sum;
#pragma unroll
            for (int k = 0; k < kScanPerLane; ++k) {
                const int64_t j = static_cast<int64_t>(lane) * K + k;
                if (dd < d1 && k < K && j < P) pc[dd * P + j] = run;
                run += x[i][k];
            }
        }
        grid_barrier(a.bar, P, 1, a.status);
#pragma unroll
        for (int q = 0; q < Q; ++q) ex[q] = act[q] ? __ldcg(pc + qd[q] * P + c) : 0;
    } else if (a.words != nullptr) {
        // Every partition is resident and there are at most kSumFormParts:
        // each publishes its counts and reads every partition's, which gives
        // both its prefix and the digit totals (the first output position of
        // every digit, an exclusive scan in digit order).
        int32_t all[Q];
        exchange_counts<Q, kSumChunk<WI, Q>>(a.words, gridDim.x, c, a.epoch, tot, ex, all, a.status, a.arrive);
        int32_t gs = 0;
#pragma unroll
        for (int q = 0; q < Q; ++q) gs += all[q];
        int32_t run = block_exclusive(gs, wsum);
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            gbase[Q * t + q] = run;
            run += all[q];
        }
    } else {
#pragma unroll
        for (int q = 0; q < Q; ++q)
            if (act[q]) st_relaxed(a.look + c * kWideBins + qd[q], state(a.epoch, c == 0 ? kPre : kAgg, tot[q]));
        look_back<Q, kLookWindow>(a.look, kWideBins, c, qd, act, a.epoch, ex, a.status);
#pragma unroll
        for (int q = 0; q < Q; ++q)
            if (act[q] && c > 0) st_relaxed(a.look + c * kWideBins + qd[q], state(a.epoch, kPre, ex[q] + tot[q]));
    }
#pragma unroll
    for (int q = 0; q < Q; ++q)
        if (act[q]) excl[qd[q]] = ex[q];
    __syncthreads();
#pragma unroll
    for (int j = 0; j < WI; ++j) {
        if (d[j] >= kWideBins) continue;
        const int64_t dst = static_cast<int64_t>(gbase[d[j]]) + excl[d[j]] + cnt[w][d[j]] + rk[j];
        if (dst >= 0 && dst < a.n)
            a.out[dst] = v[j];
        else
            atomicOr(&err, kStatusInternal);
    }
    __syncthreads();
    if (t == 0 && err) atomicOr(a.status, err);
}

// ---------------------------------------------------------------------------
// per 128-row tile of the mask-sorted order: pair counts per tap (into
// seg_off, tap-major [27][T]) and the union of the tile's masks
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTileRows) k_wide_tile_count(const WideArgs a, const uint64_t* __restrict__ ms) {
    __shared__ int32_t wc[kTileRows / 32][kTaps];
    __shared__ int32_t taps[kTaps];
    __shared__ int32_t pos[kTaps];
    __shared__ int32_t err;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t T = a.n_tiles, n = a.n;
    const int64_t tile = blockIdx.x;
    const int rb = a.row_bits;
    const uint64_t rmask = (uint64_t(1) << rb) - 1;
    if (t == 0) err = 0;
    pdl_wait();   // the mask sort is complete
    pdl_trigger();
    // the row's mask comes back out of its sort key (the key is the mask in
    // the tap order: tap k at bit pos[k]), not from a second dependent load
    if (t < kTaps) taps[t] = __ldcg(a.tap_count + t);
    const int64_t s = tile * kTileRows + t;
    const uint64_t sv = s < n ? __ldcg(ms + s) : 0ull;
    __syncthreads();
    if (t < kTaps) {
        int32_t rank = t;
        if (a.calibrated) {
            const int32_t ck = taps[t];
            rank = 0;
            for (int j = 0; j < kTaps; ++j) {
                const int32_t cj = taps[j];
                rank += (cj > ck || (cj == ck && j < t)) ? 1 : 0;
            }
        }
        pos[t] = rank;
    }
    __syncthreads();
    int64_t r = s < n ? static_cast<int64_t>(sv & rmask) : -1;
    if (r >= n) {
        atomicOr(&err, kStatusInternal);
        r = -1;
    }
    uint32_t m = 0;
    if (r >= 0) {
        const uint32_t key = static_cast<uint32_t>(sv >> rb);
#pragma unroll
        for (int k = 0; k < kTaps; ++k) m |= ((key >> pos[k]) & 1u) << k;
    }
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
        if (lane == 0) wc[warp][k] = __popc(b);
    }
    __syncthreads();
    if (warp == 0) {
        int32_t x = 0;
        if (lane < kTaps) {
#pragma unroll
            for (int q = 0; q < kTileRows / 32; ++q) x += wc[q][lane];
            a.seg_off[static_cast<int64_t>(lane) * T + tile] = x;
        }
        const uint32_t uni = __ballot_sync(0xFFFFFFFFu, x > 0);
        if (lane == 0) a.tile_union[tile] = uni;
    }
    if (t == 0 && err) atomicOr(a.status, err);
}

// The exclusive scan of the (tap, tile) counts in tap-major order (each
// tap's list starts where the previous tap's ends) in place, the tap offsets
// and totals, and the tiles in descending order of union size, stable in the
// tile index.  One launch of kTaps + 1 CTAs: CTA k < kTaps scans tap k's T
// counts from the tap's start, the exclusive sum of the per-tap pair totals
// the lookup counted (so the taps need nothing from each other; a tap whose
// counts do not add up to its total is reported); CTA kTaps does the tile
// order, a counting sort over the 28 union sizes in which warp w takes a
// contiguous range of tiles, 32 at a time.  (One CTA doing all of it was a
// chain of 27 T / 8192 rounds: 24.8 us on stage's 1,875 tiles.)
constexpr int kScanThreads = 1024;
constexpr int kScanWarps = kScanThreads / 32;
constexpr int kScanPer = 8;                          // values per thread and round
constexpr int kScanRound = kScanThreads * kScanPer;
constexpr int kUnionCache = 2048;                    // unions kept in shared memory

__global__ void __launch_bounds__(kScanThreads) k_wide_tile_scan(const WideArgs a) {
    __shared__ __align__(16) int32_t buf[kScanRound];
    __shared__ uint32_t uc[kUnionCache];
    __shared__ int32_t wsum[kScanWarps];
    __shared__ int32_t wcnt[kScanWarps][kTaps + 1];
    __shared__ int32_t bbase[kTaps + 1];
    __shared__ int32_t tap_sum, tap_start;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int64_t T = a.n_tiles;
    const bool cached = T <= kUnionCache;
    if (t < kScanWarps * (kTaps + 1)) (&wcnt[0][0])[t] = 0;
    if (t == 0) tap_sum = 0;
    pdl_wait();   // counts and unions of every tile are complete
    pdl_trigger();
    if (blockIdx.x < kTaps) {
        const int k = blockIdx.x;
        // the taps' starts: an exclusive scan of the per-tap totals (warp 0)
        if (w == 0) {
            const int32_t tot = lane < kTaps ? __ldcg(a.tap_count + lane) : 0;
            int32_t inc = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += y;
            }
            if (lane == k) tap_start = inc - tot;
            if (k == 0) {   // CTA 0 writes the tap offsets and the pair total
                if (lane < kTaps) a.tap_off[lane] = inc - tot;
                if (lane == kTaps - 1) {
                    a.tap_off[kTaps] = inc;
                    a.totals[0] = inc;
                }
            }
        }
        __syncthreads();
        // tap k's counts, in rounds of kScanRound values: coalesced loads into
        // shared memory, each thread scans kScanPer consecutive values there,
        // a block scan of the thread sums, coalesced stores
        int32_t* seg = a.seg_off + static_cast<int64_t>(k) * T;
        const int32_t first = tap_start;
        int32_t carry = first;
        for (int64_t r0 = 0; r0 < T; r0 += kScanRound) {
#pragma unroll
            for (int q = 0; q < kScanPer; ++q) {
                const int64_t i = r0 + static_cast<int64_t>(q) * kScanThreads + t;
                buf[q * kScanThreads + t] = i < T ? __ldcg(seg + i) : 0;
            }
            __syncthreads();
            int4 v[kScanPer / 4];
#pragma unroll
            for (int q = 0; q < kScanPer / 4; ++q) v[q] = reinterpret_cast<const int4*>(buf)[t * (kScanPer / 4) + q];
            int32_t sum = 0;
#pragma unroll
            for (int q = 0; q < kScanPer / 4; ++q) sum += v[q].x + v[q].y + v[q].z + v[q].w;
            int32_t inc = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += y;
            }
            if (lane == 31) wsum[w] = inc;
            __syncthreads();
            int32_t before = 0, total = 0;
            for (int i = 0; i < kScanWarps; ++i) {
                const int32_t x = wsum[i];
                before += i < w ? x : 0;
                total += x;
            }
            int32_t run = carry + before + inc - sum;
#pragma unroll
            for (int q = 0; q < kScanPer / 4; ++q) {
                int4 o4;
                o4.x = run; run += v[q].x;
                o4.y = run; run += v[q].y;
                o4.z = run; run += v[q].z;
                o4.w = run; run += v[q].w;
                reinterpret_cast<int4*>(buf)[t * (kScanPer / 4) + q] = o4;
            }
            carry += total;
            __syncthreads();
#pragma unroll
            for (int q = 0; q < kScanPer; ++q) {
                const int64_t i = r0 + static_cast<int64_t>(q) * kScanThreads + t;
                if (i < T) seg[i] = buf[q * kScanThreads + t];
            }
            __syncthreads();   // buf and wsum are reused
        }
        if (t == 0 && carry - first != __ldcg(a.tap_count + k)) atomicOr(a.status, kStatusInternal);
        return;
    }
    // ---- tile order (CTA kTaps); the unions up to kUnionCache tiles in shared memory
    if (cached)
        for (int64_t i = t; i < T; i += kScanThreads) uc[i] = __ldcg(a.tile_union + i);
    __syncthreads();
    const int64_t tw = (T + kScanWarps - 1) / kScanWarps;
    const int64_t t0 = w * tw < T ? w * tw : T;
    const int64_t t1 = t0 + tw < T ? t0 + tw : T;
    const uint32_t lt = lanemask_lt();
    int32_t my_taps = 0;
    for (int64_t i0 = t0; i0 < t1; i0 += 32) {
        const int64_t tt = i0 + lane;
        const int c = tt < t1 ? __popc(cached ? uc[tt] : __ldcg(a.tile_union + tt)) : -1;
        const int b = c >= 0 ? kTaps - c : kTaps + 1;
        my_taps += c > 0 ? c : 0;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, b);
        if (b <= kTaps && lane == __ffs(peers) - 1) wcnt[w][b] += __popc(peers);
        __syncwarp();
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) my_taps += __shfl_xor_sync(0xFFFFFFFFu, my_taps, o);
    if (lane == 0) atomicAdd(&tap_sum, my_taps);
    __syncthreads();
    if (t <= kTaps) {   // per size: offsets of the warps, total
        int32_t r = 0;
        for (int q = 0; q < kScanWarps; ++q) {
            const int32_t x = wcnt[q][t];
            wcnt[q][t] = r;
            r += x;
        }
        bbase[t] = r;
    }
    __syncthreads();
    if (t == 0) {
        int32_t r = 0;
        for (int b = 0; b <= kTaps; ++b) {
            const int32_t x = bbase[b];
            bbase[b] = r;
            r += x;
        }
        a.totals[1] = tap_sum;
    }
    __syncthreads();
    for (int64_t i0 = t0; i0 < t1; i0 += 32) {
        const int64_t tt = i0 + lane;
        const int b = tt < t1 ? kTaps - __popc(cached ? uc[tt] : __ldcg(a.tile_union + tt)) : kTaps + 1;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, b);
        if (b <= kTaps) {
            const int64_t at = static_cast<int64_t>(bbase[b]) + wcnt[w][b] + __popc(peers & lt);
            if (at >= 0 && at < T) a.tile_order[at] = static_cast<int32_t>(tt);
        }
        __syncwarp();
        if (b <= kTaps && lane == __ffs(peers) - 1) wcnt[w][b] += __popc(peers);
        __syncwarp();
    }
}

// One CTA of kTwThreads per tile: perm, the per-tap pair lists (from the
// (tap, tile) offsets) and the GEMM gather table (only the taps of the
// tile's union).  Four threads share a row: thread j of the row loads the
// 16-byte quarters j and j + 4 of its neighbour row and handles those eight
// taps (4j .. 4j + 3 and 4j + 16 .. 4j + 19), so each thread's path is a
// quarter of the row's and the SM holds sixteen warps per tile to overlap
// their memory and instruction latencies.
// With kPrefix (up to kPrefixTiles tiles) it also does the tile scan's work,
// so that kernel is not launched: the tile's offset in tap k's list is the
// tap's start (the exclusive sum of the per-tap totals the lookup counted)
// plus the counts of tap k in the tiles before it, which the CTA sums itself
// (the counts are still raw in seg_off); its place in the tile order is the
// number of tiles with a larger union plus those before it with an equal
// one.  CTA 0 writes the tap offsets and totals.
constexpr int64_t kPrefixTiles = 1024;
constexpr int kTwThreads = 4 * kTileRows;
constexpr int kTwWarps = kTwThreads / 32;
constexpr int kTwGroupTaps = 7;   // kPrefix: taps summed by each quarter of the CTA
static_assert(kNbrStride == 32, "a neighbour row is eight 16-byte quarters");
static_assert(4 * kTwGroupTaps >= kTaps, "four tap groups cover the taps");

// The tap of slot i (0 .. 7) of row thread j (0 .. 3); taps 27 .. 31 are padding.
__device__ __forceinline__ int tw_tap(int j, int i) { return (i < 4 ? 4 * j : 4 * j + 12) + i; }

template <bool kPrefix>
__global__ void __launch_bounds__(kTwThreads) k_wide_tile_write(const WideArgs a, const uint64_t* __restrict__ ms) {
    __shared__ int32_t wc[kTaps][kTwWarps];   // present rows of each tap per warp, then the warp's first pair
    __shared__ int32_t seg[kTaps];            // the tile's first pair in every tap's list
    __shared__ int32_t tapc[kTaps];
    __shared__ int32_t gsum[4][4][8];         // kPrefix: [tap group][warp of the group][tap of the group]
    __shared__ int32_t red[3][kTwWarps];
    __shared__ int32_t err;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rl = t >> 2, j = t & 3;         // row within the tile, tap phase
    const int64_t tile = blockIdx.x;
    const int64_t T = a.n_tiles, n = a.n;
    const uint64_t rmask = (uint64_t(1) << a.row_bits) - 1;
    if (t == 0) err = 0;
    pdl_wait();   // the pair offsets (kPrefix: counts) are complete
    pdl_trigger();
    // Loads are issued in the order of their dependences, so that the CTA
    // waits two round trips in all: the row's sort key together with the
    // counts of the earlier tiles and every tile's union, then the row's mask
    // and neighbours (which need the row id) while the sums are reduced.
    const int64_t s = tile * kTileRows + rl;
    const uint64_t sv = s < n ? __ldcg(ms + s) : 0ull;
    if (!kPrefix && t < kTaps) seg[t] = __ldcg(a.seg_off + static_cast<int64_t>(t) * T + tile);
    const uint32_t uni = __ldcg(a.tile_union + tile);
    const int grp = t / kTileRows;   // kPrefix: this thread's tap group (taps 7 grp .. 7 grp + 6)
    int32_t acc[8];
    int32_t greater = 0, equal_before = 0, taps_all = 0;
    if (kPrefix) {
        if (t < kTaps) tapc[t] = __ldcg(a.tap_count + t);
        // the group's taps in the tiles t % 128, t % 128 + 128, ... before this one
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0;
#pragma unroll 4
        for (int64_t tt = t % kTileRows; tt < tile; tt += kTileRows) {
#pragma unroll
            for (int i = 0; i < kTwGroupTaps; ++i) {
                const int k = kTwGroupTaps * grp + i;
                acc[i] += k < kTaps ? __ldcg(a.seg_off + static_cast<int64_t>(k) * T + tt) : 0;
            }
        }
        // place in the tile order (tiles with a larger union, then earlier ones
        // with an equal union), and for CTA 0 the sum of all union sizes
        const int c = __popc(uni);
        for (int64_t tt = t; tt < T; tt += kTwThreads) {
            const int cu = __popc(__ldcg(a.tile_union + tt));
            greater += cu > c ? 1 : 0;
            equal_before += (cu == c && tt < tile) ? 1 : 0;
            taps_all += cu;
        }
    }
    // the row id out of the sort key, then its mask and this thread's two quarters of its neighbours
    bool err_row = false;
    int32_t r = s < n ? static_cast<int32_t>(sv & rmask) : -1;
    if (r >= n) {
        r = -1;
        err_row = true;
    }
    const uint32_t m = r >= 0 ? __ldcg(a.mask + r) : 0u;
    int32_t v[8];
    if (r >= 0) {
        const int4* src = reinterpret_cast<const int4*>(a.nbr + static_cast<int64_t>(r) * kNbrStride);
        const int4 x0 = __ldcg(src + j), x1 = __ldcg(src + j + 4);
        v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
        v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = -1;
    }
    if (kPrefix) {
        // the warp's sum of each of its 8 counters: three exchanges halve the
        // counters a lane carries (4 + 2 + 1 shuffles), after which lane l holds
        // counter l % 8 summed over the lanes l ^ {1, 2, 4}; two more add the rest
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
        if (lane < 8) gsum[grp][warp & 3][lane] = acc[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            greater += __shfl_xor_sync(0xFFFFFFFFu, greater, o);
            equal_before += __shfl_xor_sync(0xFFFFFFFFu, equal_before, o);
            taps_all += __shfl_xor_sync(0xFFFFFFFFu, taps_all, o);
        }
        if (lane == 0) {
            red[0][warp] = greater;
            red[1][warp] = equal_before;
            red[2][warp] = taps_all;
        }
    }
    // the warp's rows with each tap: lanes of one phase (lane % 4 == j) share their taps
    const uint32_t same = 0x11111111u << j;
    uint32_t bal[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int k = tw_tap(j, i);
        bal[i] = __ballot_sync(0xFFFFFFFFu, k < kTaps && ((m >> k) & 1u)) & same;
        if (lane == j && k < kTaps) wc[k][warp] = __popc(bal[i]);
    }
    __syncthreads();
    // each tap's warp counts -> the warps' first pairs within the tile (two taps per warp,
    // a 16-lane scan each)
    if (warp < (kTaps * kTwWarps + 31) / 32) {   // whole warps: every lane takes part in the shuffles
        const int k = t / kTwWarps, w = t % kTwWarps;
        const int32_t x = k < kTaps ? wc[k][w] : 0;
        int32_t inc = x;
#pragma unroll
        for (int o = 1; o < kTwWarps; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o, kTwWarps);
            if (w >= o) inc += y;
        }
        if (k < kTaps) wc[k][w] = inc - x;
    }
    if (kPrefix && warp == kTwWarps - 1) {
        // lane k: tap k's start (an exclusive scan of the tap totals) plus its count in the earlier tiles
        const int32_t x = lane < kTaps ? tapc[lane] : 0;
        int32_t inc = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += y;
        }
        const int32_t start = inc - x;
        if (lane < kTaps) {
            const int g = lane / kTwGroupTaps, i = lane % kTwGroupTaps;
            seg[lane] = start + gsum[g][0][i] + gsum[g][1][i] + gsum[g][2][i] + gsum[g][3][i];
            if (tile == 0) a.tap_off[lane] = start;
        }
        const int32_t pairs = __shfl_sync(0xFFFFFFFFu, inc, 31);
        if (lane == 0) {
            int32_t g2 = 0, e2 = 0, s2 = 0;
#pragma unroll
            for (int w2 = 0; w2 < kTwWarps; ++w2) {
                g2 += red[0][w2];
                e2 += red[1][w2];
                s2 += red[2][w2];
            }
            const int64_t at = static_cast<int64_t>(g2) + e2;
            if (at >= 0 && at < T) a.tile_order[at] = static_cast<int32_t>(tile);
            else atomicOr(&err, kStatusInternal);
            if (tile == 0) {
                a.tap_off[kTaps] = pairs;
                a.totals[0] = pairs;
                a.totals[1] = s2;
            }
        }
    }
    __syncthreads();
    if (j == 0) {
        if (err_row) atomicOr(&err, kStatusInternal);
        a.perm[s] = r;
    }
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int k = tw_tap(j, i);
        if (k >= kTaps || !((uni >> k) & 1u)) continue;
        const bool present = (m >> k) & 1u;
        if (present) {
            const int64_t off = static_cast<int64_t>(seg[k]) + wc[k][warp] + __popc(bal[i] & lt);
            if (off >= 0 && off < kTaps * n) {
                a.in_rows[off] = v[i];
                a.out_rows[off] = r;
            } else {
                atomicOr(&err, kStatusInternal);
            }
        }
        a.gtab[static_cast<int64_t>(k) * a.n_pad + s] = present ? v[i] : -1;
    }
    __syncthreads();
    if (t == 0 && err) atomicOr(a.status, err);
}

// The three bounded waits of the sort passes, each against a state that
// nothing will ever publish, with a short limit: which = 0, the look-back of
// partition 1 over partition 0 (whose state words stay zero); which = 1, the
// grid barrier of a two-CTA grid entered by the only CTA launched; which = 2,
// the count exchange of the all-partition form (a partition that never publishes).
// Each must give up after limit_ns and set kStatusTimeout; nothing else is
// touched.
__global__ void __launch_bounds__(WT) k_wait_probe(int which, const uint64_t* look, int32_t* bar, int32_t* status,
                                                   uint64_t limit_ns) {
    if (which == 0) {
        const int q[1] = {static_cast<int>(threadIdx.x)};
        const bool act[1] = {true};
        int32_t ex[1];
        look_back<1, 8>(look, kWideBins, 1, q, act, 1u, ex, status, limit_ns);
    } else if (which == 1) {
        grid_barrier(bar, 2, 0, status, limit_ns);
    } else {
        // partition 1 of 2: partition 0's words stay zero
        const int32_t tot[2] = {0, 0};
        int32_t ex[2], all[2];
        exchange_counts<2, 31>(const_cast<uint64_t*>(look), 2, 1, 1u, tot, ex, all, status, nullptr, limit_ns);
    }
}

// A fresh nonzero epoch for every launch that publishes look-back states.
uint32_t next_epoch() {
    static std::atomic<uint32_t> counter{0};
    uint32_t e = ++counter;
    if (e == 0) e = ++counter;
    return e;
}

// CTAs of `kernel` (block threads, no dynamic shared memory) the device holds at once.
template <typename Kernel>
int64_t resident_ctas(Kernel kernel, int block, int sms) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, 0) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return static_cast<int64_t>(per_sm) * sms;
}

template <typename Kernel, typename... Args>
int launch_pdl(Kernel kernel, unsigned grid, unsigned block, cudaStream_t s, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    SPCONV_CHECK_CUDA(cudaLaunchKernelEx(&cfg, kernel, args...));
    count_launch();
    return SPCONV_OK;
}

}  // namespace

int wait_probe(int which, uint64_t limit_ns, cudaStream_t s) {
    // look-back states of one partition (zero: never published), barrier counters, status
    const size_t look_bytes = kWideBins * sizeof(uint64_t);
    const size_t bytes = look_bytes + kWideBarrierInts * sizeof(int32_t) + 16;
    void* buf = nullptr;
    SPCONV_CHECK_CUDA(cudaMallocAsync(&buf, bytes, s));
    uint64_t* look = static_cast<uint64_t*>(buf);
    int32_t* bar = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(buf) + look_bytes);
    int32_t* status = bar + kWideBarrierInts;
    int rc = cuda_status(cudaMemsetAsync(buf, 0, bytes, s));
    if (rc == SPCONV_OK) {
        k_wait_probe<<<1, WT, 0, s>>>(which, look, bar, status, limit_ns);
        count_launch();
        rc = cuda_status(cudaGetLastError());
    }
    int32_t st = 0;
    if (rc == SPCONV_OK) rc = cuda_status(cudaMemcpyAsync(&st, status, sizeof(st), cudaMemcpyDeviceToHost, s));
    if (rc == SPCONV_OK) rc = cuda_status(cudaStreamSynchronize(s));
    cudaFreeAsync(buf, s);
    if (rc != SPCONV_OK) return rc;
    return status_from_flags(st);
}

int wide_key_passes(int key_bits) { return (key_bits + kDigitBitsWide - 1) / kDigitBitsWide; }

int hash_table_log2(int64_t n) {
    int l = kHashMinLog2;   // >= 2: whole buckets
    while ((int64_t(1) << l) < kHashSlotsPerRow * n) ++l;
    return l;
}

namespace {

// One pass of the stable sort on stream s: a CTA per partition of
// keys_per_cta values (2 kWideKeysPerCta above kBigPassRows); partitions
// numbered by blockIdx when the device holds the whole grid at once, else by
// the ticket counter tickets[ticket]; offsets by the two-barrier form when
// every partition is resident and the digits spread over them, else by
// decoupled look-back.
// The form a pass over n values with digits of `width` bits takes on this
// device.  Keys per partition: 1024, 2048 above kBigPassRows, 4096 above
// kHugePassRows (fewer partitions: the count exchange reaches 262k rows;
// stage-sized kernel-size-5 maps 523.9 -> 497.3 us with 10-bit digits too).
struct PassPlan {
    int size;   // keys per partition: kWideKeysPerCta << size
    bool narrow, ticket, barrier, all;
    int64_t parts;
};

int plan_wide_pass(int64_t n, int width, PassPlan* pl) {
    // resident CTAs of each form: [device][size][digits per thread: 2, 4]
    static int64_t cap_pass[kMaxDevices][3][2] = {};
    int dev = 0;
    SPCONV_CHECK_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return SPCONV_ERR_UNSUPPORTED;
    if (width < 1 || width > kDigitBitsWide) return SPCONV_ERR_UNSUPPORTED;
    if (cap_pass[dev][0][0] == 0) {
        int sms = 0;
        SPCONV_CHECK_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        // (the mask form of the first mask pass may hold fewer CTAs than its plain form)
        cap_pass[dev][0][0] = std::min(resident_ctas(k_wide_pass<WI, 2>, WT, sms),
                                       resident_ctas(k_wide_pass<WI, 2, true>, WT, sms));
        cap_pass[dev][0][1] = resident_ctas(k_wide_pass<WI, 4>, WT, sms);
        cap_pass[dev][1][0] = std::min(resident_ctas(k_wide_pass<2 * WI, 2>, WT, sms),
                                       resident_ctas(k_wide_pass<2 * WI, 2, true>, WT, sms));
        cap_pass[dev][1][1] = resident_ctas(k_wide_pass<2 * WI, 4>, WT, sms);
        cap_pass[dev][2][0] = std::min(resident_ctas(k_wide_pass<4 * WI, 2>, WT, sms),
                                       resident_ctas(k_wide_pass<4 * WI, 2, true>, WT, sms));
        cap_pass[dev][2][1] = resident_ctas(k_wide_pass<4 * WI, 4>, WT, sms);
    }
    pl->narrow = (1 << width) <= 2 * WT;   // two digits per thread cover the digit values
    pl->size = n > kHugePassRows ? 2 : n > kBigPassRows ? 1 : 0;
    const int64_t keys_per_cta = static_cast<int64_t>(kWideKeysPerCta) << pl->size;
    pl->parts = (n + keys_per_cta - 1) / keys_per_cta;
    if (pl->parts > 0x7FFFFFFF) return SPCONV_ERR_UNSUPPORTED;
    pl->ticket = pl->parts > cap_pass[dev][pl->size][pl->narrow ? 0 : 1];
    // the barrier form when every partition is resident, each warp scans at
    // most kScanDigitsPerWarp digits and each lane at most kScanPerLane partitions
    const int64_t bins = int64_t(1) << width;
    pl->barrier = !pl->ticket && pl->parts > kSumFormParts && bins <= pl->parts * WW * kScanDigitsPerWarp &&
                  pl->parts <= 32 * kScanPerLane;
    // a few resident partitions: each reads every partition's packed counts
    // (parts x Q / 2 x WT words of the look-back buffer)
    pl->all = !pl->ticket && !pl->barrier && pl->parts <= kSumFormParts;
    return SPCONV_OK;
}

// One pass of the stable sort on stream s, in the form plan_wide_pass gives.
// mask_src: the first pass of the mask sort, its values made from the masks
// (the all-partition form and 9-bit digits only).
int launch_wide_pass(const uint64_t* in, uint64_t* out, int64_t n, int shift, int width, const int32_t* gh,
                     uint64_t* look, int32_t* tickets, int ticket, int32_t* status, cudaStream_t s, bool pdl = true,
                     const WideArgs* mask_src = nullptr) {
    PassPlan pl;
    SPCONV_CHECK(plan_wide_pass(n, width, &pl));
    if (mask_src && (!pl.all || !pl.narrow)) return SPCONV_ERR_INTERNAL;
    PassArgs pa = {};
    pa.in = in;
    pa.out = out;
    pa.n = n;
    pa.shift = shift;
    pa.width = width;
    pa.gh = gh;
    pa.look = look;
    pa.epoch = next_epoch();
    pa.ticket = pl.ticket ? tickets + ticket : nullptr;
    pa.bar = pl.barrier ? tickets + kWideTickets + ticket * kWideBarrierInts : nullptr;
    pa.words = pl.all ? look : nullptr;
    pa.arrive = pl.all ? tickets + ticket : nullptr;
    pa.status = status;
    if (mask_src) {
        pa.mask = mask_src->mask;
        pa.tap_count = mask_src->tap_count;
        pa.calibrated = mask_src->calibrated;
        pa.row_bits = mask_src->row_bits;
    }
    const unsigned grid = static_cast<unsigned>(pl.parts);
    if (mask_src)
        return pl.size == 2 ? launch_pdl(k_wide_pass<4 * WI, 2, true>, grid, WT, s, pdl, pa)
             : pl.size == 1 ? launch_pdl(k_wide_pass<2 * WI, 2, true>, grid, WT, s, pdl, pa)
                            : launch_pdl(k_wide_pass<WI, 2, true>, grid, WT, s, pdl, pa);
    if (pl.size == 2)
        return pl.narrow ? launch_pdl(k_wide_pass<4 * WI, 2>, grid, WT, s, pdl, pa)
                         : launch_pdl(k_wide_pass<4 * WI, 4>, grid, WT, s, pdl, pa);
    if (pl.size == 1)
        return pl.narrow ? launch_pdl(k_wide_pass<2 * WI, 2>, grid, WT, s, pdl, pa)
                         : launch_pdl(k_wide_pass<2 * WI, 4>, grid, WT, s, pdl, pa);
    return pl.narrow ? launch_pdl(k_wide_pass<WI, 2>, grid, WT, s, pdl, pa)
                     : launch_pdl(k_wide_pass<WI, 4>, grid, WT, s, pdl, pa);
}

}  // namespace

WideDigits wide_digits(int lo, int bits) {
    WideDigits d = {};
    const int passes = (bits + kDigitBitsWide - 1) / kDigitBitsWide;
    if (passes > kWideKeyPassesMax) return d;
    d.passes = passes;
    for (int p = 0, at = lo; p < passes; ++p) {
        d.width[p] = bits / passes + (p < bits % passes ? 1 : 0);
        d.shift[p] = at;
        at += d.width[p];
    }
    return d;
}

int64_t wide_sort_look_words(int64_t n) {
    const int64_t keys_per_cta = n > kBigPassRows ? 2 * kWideKeysPerCta : kWideKeysPerCta;   // (at least the parts of any pass)
    return (n + keys_per_cta - 1) / keys_per_cta * kWideBins;
}

int wide_sort_reads_totals(int64_t n, const WideDigits& d, bool* reads) {
    *reads = false;
    for (int p = 0; p < d.passes; ++p) {
        PassPlan pl;
        SPCONV_CHECK(plan_wide_pass(std::max<int64_t>(1, n), d.width[p], &pl));
        if (!pl.all) *reads = true;
    }
    return SPCONV_OK;
}

int wide_sort(uint64_t* a, uint64_t* b, int64_t n, const WideDigits& d, const int32_t* gh, int32_t* tickets,
              int ticket0, uint64_t* look, int32_t* status, cudaStream_t s, bool* in_b, bool first_plain) {
    *in_b = false;
    if (d.passes < 1 || ticket0 < 0 || ticket0 + d.passes > kWideTickets) return SPCONV_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(look) % 16 != 0 || reinterpret_cast<uintptr_t>(a) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(b) % 8 != 0)
        return SPCONV_ERR_INTERNAL;   // 64-bit words throughout
    if (n > kWideMaxRows) return SPCONV_ERR_UNSUPPORTED;
    for (int p = 0; p < d.passes; ++p) {
        const bool odd = p & 1;
        SPCONV_CHECK(launch_wide_pass(odd ? b : a, odd ? a : b, n, d.shift[p], d.width[p], gh + p * kWideBins, look,
                                      tickets, ticket0 + p, status, s, !(first_plain && p == 0)));
    }
    *in_b = (d.passes & 1) != 0;
    return SPCONV_OK;
}

int launch_map_wide(const WideArgs& a, int sms, cudaStream_t s) {
    const int64_t n = a.n;
    if (reinterpret_cast<uintptr_t>(a.look) % 16 != 0 || reinterpret_cast<uintptr_t>(a.va) % 8 != 0 ||
        reinterpret_cast<uintptr_t>(a.vb) % 8 != 0)
        return SPCONV_ERR_INTERNAL;   // 64-bit words throughout
    // keys per sort CTA: 1024, or 2048 above kBigPassRows (fewer partitions
    // whose counts every partition reads: 32k rows 52.9 -> 50.8 us per build)
    const bool big_pass = n > kBigPassRows;
    const int64_t keys_per_cta = big_pass ? 2 * kWideKeysPerCta : kWideKeysPerCta;
    const unsigned parts = static_cast<unsigned>((n + keys_per_cta - 1) / keys_per_cta);
    const bool few = n <= kFewRows;
    const int rpt = few ? 1 : 4;
    const unsigned key_blocks = static_cast<unsigned>((n + WT * rpt - 1) / (WT * rpt));
    const unsigned row_blocks = static_cast<unsigned>((n + WT - 1) / WT);
    // every thread clears ~8 16-byte words of the largest array
    const int64_t look16 = static_cast<int64_t>(parts) * kWideBins / 2;
    int64_t clear16 = a.mapper == SPCONV_MAPPER_DENSE ? a.cells / 4
                    : a.mapper == SPCONV_MAPPER_HASH ? (int64_t(1) << a.table_log2) / 2
                                                     : 0;
    if (look16 > clear16) clear16 = look16;
    int64_t clear_blocks = (clear16 + WT * 8 - 1) / (WT * 8);
    if (clear_blocks > 4 * sms) clear_blocks = 4 * sms;
    SPCONV_CHECK(launch_pdl(k_wide_clear, static_cast<unsigned>(clear_blocks < 1 ? 1 : clear_blocks), WT, s, false, a));
    auto pass = [&](const uint64_t* in, uint64_t* out, int shift, int width, const int32_t* gh, int ticket) {
        return launch_wide_pass(in, out, n, shift, width, gh, a.look, a.tickets, ticket, a.status, s);
    };
    if (a.mapper == SPCONV_MAPPER_HASH) {
        const unsigned look_blocks = static_cast<unsigned>((n + kHashLookupRows - 1) / kHashLookupRows);
        if (a.key_bits <= 32) {
            SPCONV_CHECK(launch_pdl(k_wide_hash_insert<true>, row_blocks, WT, s, true, a));
            SPCONV_CHECK(launch_pdl(k_wide_hash_lookup<true>, look_blocks, 3 * kHashLookupRows, s, true, a));
        } else {
            SPCONV_CHECK(launch_pdl(k_wide_hash_insert<false>, row_blocks, WT, s, true, a));
            SPCONV_CHECK(launch_pdl(k_wide_hash_lookup<false>, look_blocks, 3 * kHashLookupRows, s, true, a));
        }
    } else if (a.mapper == SPCONV_MAPPER_SORTED) {
        const int passes = wide_key_passes(a.key_bits);
        if (passes > kWideKeyPassesMax) return SPCONV_ERR_UNSUPPORTED;
        KeyDigits kd = {};
        kd.passes = passes;
        for (int p = 0, at = 0; p < passes; ++p) {
            kd.width[p] = a.key_bits / passes + (p < a.key_bits % passes ? 1 : 0);
            kd.shift[p] = at;
            at += kd.width[p];
        }
        // (no digit counts where every key pass runs in the count exchange)
        KeyDigits kc = kd;
        bool reads = false;
        for (int p = 0; p < passes; ++p) {
            PassPlan pl;
            SPCONV_CHECK(plan_wide_pass(n, kd.width[p], &pl));
            reads |= !pl.all;
        }
        if (!reads) kc.passes = 0;
        SPCONV_CHECK(few ? launch_pdl(k_wide_keys<1>, key_blocks, WT, s, true, a, kc)
                         : launch_pdl(k_wide_keys<4>, key_blocks, WT, s, true, a, kc));
        for (int p = 0; p < passes; ++p)
            SPCONV_CHECK(pass((p & 1) ? a.vb : a.va, (p & 1) ? a.va : a.vb, a.row_bits + kd.shift[p], kd.width[p],
                              a.gh + p * kWideBins, p));
        SPCONV_CHECK(launch_search_window((passes & 1) ? a.vb : a.va, n, a.row_bits, a.key_bits, a.koff, a.nbr, a.mask,
                                          a.tap_count, a.status, s));
        count_launch();
    } else {
        SPCONV_CHECK(launch_pdl(k_wide_grid_scatter, row_blocks, WT, s, true, a));
        SPCONV_CHECK(launch_pdl(k_wide_grid_lookup, row_blocks, WT, s, true, a));
    }
    // the mask sort: when its passes read every partition's counts (few rows),
    // the first pass makes the keys from the masks itself; otherwise a kernel
    // makes them with the digit totals the other forms need
    PassPlan mp;
    SPCONV_CHECK(plan_wide_pass(n, kMaskWidth, &mp));
    if (mp.all) {
        SPCONV_CHECK(launch_wide_pass(nullptr, a.vb, n, a.row_bits, kMaskWidth, nullptr, a.look, a.tickets,
                                      kWideKeyPassesMax, a.status, s, true, &a));
    } else {
        SPCONV_CHECK(few ? launch_pdl(k_wide_mask_keys<1>, key_blocks, WT, s, true, a)
                         : launch_pdl(k_wide_mask_keys<4>, key_blocks, WT, s, true, a));
        SPCONV_CHECK(pass(a.va, a.vb, a.row_bits, kMaskWidth, a.gh + kWideKeyPassesMax * kWideBins, kWideKeyPassesMax));
    }
    for (int p = 1; p < kWideMaskPasses; ++p)
        SPCONV_CHECK(pass((p & 1) ? a.vb : a.va, (p & 1) ? a.va : a.vb, a.row_bits + kMaskWidth * p, kMaskWidth,
                          a.gh + (kWideKeyPassesMax + p) * kWideBins, kWideKeyPassesMax + p));
    const uint64_t* ms = (kWideMaskPasses & 1) ? a.vb : a.va;
    const unsigned tiles = static_cast<unsigned>(a.n_tiles);
    SPCONV_CHECK(launch_pdl(k_wide_tile_count, tiles, kTileRows, s, true, a, ms));
    if (a.n_tiles <= kPrefixTiles) {
        SPCONV_CHECK(launch_pdl(k_wide_tile_write<true>, tiles, kTwThreads, s, true, a, ms));
    } else {
        SPCONV_CHECK(launch_pdl(k_wide_tile_scan, static_cast<unsigned>(kTaps + 1), static_cast<unsigned>(kScanThreads), s,
                                true, a));
        SPCONV_CHECK(launch_pdl(k_wide_tile_write<false>, tiles, kTwThreads, s, true, a, ms));
    }
    return SPCONV_OK;
}

}  // namespace spconv

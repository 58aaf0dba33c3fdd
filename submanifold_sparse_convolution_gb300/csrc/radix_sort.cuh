// Stable LSD radix sort of (key, value) pairs on the device, 8 bits per pass.
//
// Each pass is reduce-then-scan with no atomics on global memory and no
// inter-block waiting: an upsweep writes per-tile digit counts, one block
// scans them (digit-major, so the scan yields every tile's output offset for
// every digit), and a downsweep ranks each tile's keys stably and scatters
// them.  Used for the packed coordinate keys (mapper) and for the 27-bit mask
// keys (row order for the output tiles).
//
// The three kernels of every pass are launched with programmatic dependent
// launch: each lets its successor be scheduled as soon as it starts, then
// waits for its predecessor before its first global access, so a kernel's
// launch latency hides behind the tail of the one before.  Data an earlier
// kernel wrote is read through L2 (ld.global.cg), never the read-only path.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"

namespace spconv {
namespace rsort {

constexpr int kThreads = 256;
constexpr int kItems = 8;
constexpr int kTile = kThreads * kItems;  // 2048 keys per block
constexpr int kBins = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kScanThreads = 1024;

inline int64_t num_tiles(int64_t n) { return (n + kTile - 1) / kTile; }

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

template <typename K>
__global__ void __launch_bounds__(kThreads) upsweep(const K* __restrict__ keys, int64_t n, int shift,
                                                   int32_t* __restrict__ hist, int64_t nb) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t h[kBins];
    for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = 0;
    __syncthreads();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kTile;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int64_t idx = base + j * kThreads + threadIdx.x;
        const bool valid = idx < n;
        const int d = valid ? static_cast<int>((__ldcg(keys + idx) >> shift) & 0xFF) : kBins;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, d);
        if (valid && lane == __ffs(peers) - 1) atomicAdd(&h[d], __popc(peers));
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[static_cast<int64_t>(i) * nb + blockIdx.x] = h[i];
}

// Exclusive scan of m int32 values from src to dst (the same array or
// disjoint ones) by one block of kScanThreads threads.  Each round takes 16
// consecutive values per thread (four 16-byte loads where both arrays are
// 16-byte aligned), scans them in registers, then across the warp and across
// the block's 32 warp sums; every load of a round is issued before its first
// barrier.  on(i0, v) is called once per round by every thread whose run
// starts inside the array, after it stored dst[i0 + j] = v[j] for the j with
// i0 + j < m.  The scan starts from carry0 (dst[0] = carry0); returns
// carry0 plus the total, in every thread.
constexpr int kScanPer = 16;
static_assert(kScanThreads == 1024, "the block scan holds one warp sum per lane");

template <typename F>
__device__ __forceinline__ int32_t block_scan_exclusive(const int32_t* src, int32_t* dst, int64_t m, F on,
                                                        int32_t carry0 = 0) {
    __shared__ int32_t wsum[2][kScanThreads / 32];
    constexpr int64_t kRound = static_cast<int64_t>(kScanPer) * kScanThreads;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
    int32_t carry = carry0;
    int buf = 0;
    for (int64_t base = 0; base < m; base += kRound, buf ^= 1) {
        const int64_t i0 = base + static_cast<int64_t>(kScanPer) * t;
        const bool whole = vec && i0 + kScanPer <= m;
        int32_t v[kScanPer];
        if (whole) {
#pragma unroll
            for (int q = 0; q < kScanPer / 4; ++q) {
                const int4 x = __ldcg(reinterpret_cast<const int4*>(src + i0) + q);
                v[4 * q] = x.x;
                v[4 * q + 1] = x.y;
                v[4 * q + 2] = x.z;
                v[4 * q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kScanPer; ++j) v[j] = i0 + j < m ? __ldcg(src + i0 + j) : 0;
        }
        int32_t s = 0;
#pragma unroll
        for (int j = 0; j < kScanPer; ++j) s += v[j];
        int32_t inc = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += y;
        }
        // two buffers: a warp writes this round's sum only after every warp
        // has passed the barrier that follows its reads of the same buffer
        // two rounds back
        if (lane == 31) wsum[buf][w] = inc;
        __syncthreads();
        const int32_t ws = wsum[buf][lane];
        int32_t winc = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, winc, o);
            if (lane >= o) winc += y;
        }
        const int32_t before = __shfl_sync(0xFFFFFFFFu, winc - ws, w);
        const int32_t total = __shfl_sync(0xFFFFFFFFu, winc, 31);
        int32_t run = carry + before + inc - s;
#pragma unroll
        for (int j = 0; j < kScanPer; ++j) {
            const int32_t x = v[j];
            v[j] = run;
            run += x;
        }
        if (whole) {
#pragma unroll
            for (int q = 0; q < kScanPer / 4; ++q)
                reinterpret_cast<int4*>(dst + i0)[q] = make_int4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < kScanPer; ++j)
                if (i0 + j < m) dst[i0 + j] = v[j];
        }
        if (i0 < m) on(i0, v);
        carry += total;
    }
    return carry;
}

struct NoVisit {
    __device__ void operator()(int64_t, const int32_t (&)[kScanPer]) const {}
};

// Exclusive scan, in place, of m int32 values (one block).
static __global__ void __launch_bounds__(kScanThreads) scan_exclusive(int32_t* __restrict__ a, int64_t m) {
    pdl_trigger();
    pdl_wait();
    block_scan_exclusive(a, a, m, NoVisit());
}

template <typename K>
__global__ void __launch_bounds__(kThreads) downsweep(const K* __restrict__ keys_in,
                                                     const uint32_t* __restrict__ vals_in,
                                                     K* __restrict__ keys_out,
                                                     uint32_t* __restrict__ vals_out, int64_t n,
                                                     int shift, const int32_t* __restrict__ hist,
                                                     int64_t nb) {
    pdl_trigger();
    pdl_wait();
    // cnt[j][w][d]: keys of item slot j in warp w with digit d; then the
    // exclusive prefix of those counts in tile order (j, w, lane).
    __shared__ uint16_t cnt[kItems][kWarps][kBins];
    __shared__ int32_t gbase[kBins];
    uint32_t* cz = reinterpret_cast<uint32_t*>(&cnt[0][0][0]);
    for (int i = threadIdx.x; i < kItems * kWarps * kBins / 2; i += kThreads) cz[i] = 0;
    for (int i = threadIdx.x; i < kBins; i += kThreads) gbase[i] = __ldcg(hist + static_cast<int64_t>(i) * nb + blockIdx.x);
    __syncthreads();

    const int64_t base = static_cast<int64_t>(blockIdx.x) * kTile;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    K key[kItems];
    uint32_t val[kItems];
    int dig[kItems];
    int rank[kItems];
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int64_t idx = base + j * kThreads + threadIdx.x;
        const bool valid = idx < n;
        key[j] = valid ? __ldcg(keys_in + idx) : K(0);
        val[j] = valid ? __ldcg(vals_in + idx) : 0u;
        dig[j] = valid ? static_cast<int>((key[j] >> shift) & 0xFF) : kBins;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, dig[j]);
        rank[j] = __popc(peers & lanemask_lt());
        if (valid && lane == __ffs(peers) - 1) cnt[j][warp][dig[j]] = static_cast<uint16_t>(__popc(peers));
    }
    __syncthreads();
    for (int d = threadIdx.x; d < kBins; d += kThreads) {
        uint32_t run = 0;
        for (int j = 0; j < kItems; ++j)
            for (int w = 0; w < kWarps; ++w) {
                const uint32_t c = cnt[j][w][d];
                cnt[j][w][d] = static_cast<uint16_t>(run);
                run += c;
            }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        if (dig[j] < kBins) {
            const int64_t dst = static_cast<int64_t>(gbase[dig[j]]) + cnt[j][warp][dig[j]] + rank[j];
            keys_out[dst] = key[j];
            vals_out[dst] = val[j];
        }
    }
}

template <typename Kernel, typename... Args>
void launch_chained(Kernel kernel, unsigned grid, unsigned block, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a failed launch stays in cudaGetLastError, which every caller checks
    (void)cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Sort (keys, vals) of length n on the live low `bits` of the key.  Returns
// true if the result ended in (keys_b, vals_b), false if in (keys_a, vals_a).
// hist needs kBins * num_tiles(n) int32.
template <typename K>
bool sort_pairs(K* keys_a, uint32_t* vals_a, K* keys_b, uint32_t* vals_b, int64_t n, int bits,
                int32_t* hist, cudaStream_t s, int* launches) {
    if (n <= 1 || bits <= 0) return false;
    const int64_t nb = num_tiles(n);
    const int passes = (bits + 7) / 8;
    bool in_b = false;
    for (int p = 0; p < passes; ++p) {
        const K* kin = in_b ? keys_b : keys_a;
        const uint32_t* vin = in_b ? vals_b : vals_a;
        K* kout = in_b ? keys_a : keys_b;
        uint32_t* vout = in_b ? vals_a : vals_b;
        launch_chained(upsweep<K>, static_cast<unsigned>(nb), kThreads, s, kin, n, 8 * p, hist, nb);
        launch_chained(scan_exclusive, 1u, kScanThreads, s, hist, static_cast<int64_t>(kBins) * nb);
        launch_chained(downsweep<K>, static_cast<unsigned>(nb), kThreads, s, kin, vin, kout, vout, n, 8 * p,
                       static_cast<const int32_t*>(hist), nb);
        *launches += 3;
        in_b = !in_b;
    }
    return in_b;
}

}  // namespace rsort
}  // namespace spconv

// Declarations shared by the two kernel-map pipelines (map.cu: one kernel per
// step, any size; map_fused.cu: one cluster launch for up to kFusedMaxRows).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace spconv {

// Largest row count the single-launch pipeline takes, and the per-CTA radix
// histogram width it uses (digits of up to 10 bits).
constexpr int64_t kFusedMaxRows = int64_t(1) << 20;
constexpr int kFusedBins = 1024;

struct FusedArgs {
    const int4* coords;
    int64_t n;
    int3 shape;
    int batch;
    int mapper;                 // SPCONV_MAPPER_DENSE or SPCONV_MAPPER_SORTED
    int calibrated;             // mask key bit order
    // sorted-key layout: key = (((b << wx | x+1) << wy | y+1) << wz | z+1), key_bits live bits,
    // packed with the row below it: value = key << row_bits | row
    int wz, wy, wx, key_bits, row_bits;
    uint64_t koff[kTaps];       // packed(d_k), two's complement
    // dense grid layout
    int64_t gsb, gsx, gsy, cells;
    int64_t goff[kTaps];
    int32_t* grid;
    // scratch
    uint64_t* va;               // [n]
    uint64_t* vb;               // [n]
    int32_t* hist;              // [3][cluster][kFusedBins]
    int32_t* cta_tot;           // [cluster][27]
    int32_t* cta_bkt;           // [cluster][28]
    // outputs (see MapHandle)
    int32_t* nbr;
    uint32_t* mask;
    int32_t* tap_count;
    int32_t* perm;
    int32_t* tap_off;
    int32_t* totals;
    int32_t* in_rows;
    int32_t* out_rows;
    int32_t* gtab;
    uint32_t* tile_union;
    int32_t* tile_order;
    int32_t* seg_off;           // [27][n_tiles] first pair of (tap, tile)
    int32_t* status;
    int64_t n_tiles, n_pad;
};

// Lower bounds of 9 targets in a sorted array a[0..n) (first index with
// a[i] >= t[c], n if none), searched in lockstep: the branch-free halving
// below takes the same steps for every target, so each step issues 9
// independent loads instead of one.
__device__ __forceinline__ void lower_bound9(const uint64_t* __restrict__ a, int64_t n, const uint64_t (&t)[9],
                                             int64_t (&out)[9]) {
    int64_t base[9];
#pragma unroll
    for (int c = 0; c < 9; ++c) base[c] = 0;
    int64_t len = n;
    while (len > 1) {
        const int64_t half = len >> 1;
#pragma unroll
        for (int c = 0; c < 9; ++c) base[c] += __ldg(a + base[c] + half - 1) < t[c] ? half : 0;
        len -= half;
    }
#pragma unroll
    for (int c = 0; c < 9; ++c) out[c] = n == 0 ? 0 : base[c] + (__ldg(a + base[c]) < t[c] ? 1 : 0);
}

// Lower bound of t in a[0..n) given that it is >= from: probe from, from+1,
// from+2, from+4, ... then halve inside the bracket.
__device__ __forceinline__ int64_t lower_bound_from(const uint64_t* __restrict__ a, int64_t n, int64_t from,
                                                    uint64_t t) {
    if (from >= n || __ldg(a + from) >= t) return from;
    int64_t lo = from;          // a[lo] < t
    int64_t step = 1;
    int64_t hi = from + 1;
    while (hi < n && __ldg(a + hi) < t) {
        lo = hi;
        step <<= 1;
        hi = from + step;
    }
    if (hi > n) hi = n;         // answer in (lo, hi]
    int64_t first = lo + 1, count = hi - first;
    while (count > 0) {
        const int64_t st = count >> 1;
        if (__ldg(a + first + st) < t) {
            first += st + 1;
            count -= st + 1;
        } else {
            count = st;
        }
    }
    return first;
}

// Cluster size the fused kernel can be launched with on this device (16 or
// 8), or 0 if none.
int fused_cluster_size(cudaStream_t s);
int launch_map_fused(const FusedArgs& a, int cluster, cudaStream_t s);

}  // namespace spconv

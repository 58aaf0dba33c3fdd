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

// Cluster size the fused kernel can be launched with on this device (16 or
// 8), or 0 if none.
int fused_cluster_size(cudaStream_t s);
int launch_map_fused(const FusedArgs& a, int cluster, cudaStream_t s);

}  // namespace spconv

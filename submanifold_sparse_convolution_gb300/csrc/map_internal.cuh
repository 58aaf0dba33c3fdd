// Declarations shared by the kernel-map pipelines (map.cu: one kernel per
// step, any size; map_fused.cu: one cluster launch for up to kFusedMaxRows;
// map_wide.cu: whole-GPU passes; map_groups.cu: offset groups, kernel size 5
// and strided maps).
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

// ---- whole-GPU pipeline (map_wide.cu) --------------------------------------
constexpr int kWideKeysPerCta = 1024;    // keys per CTA (look-back partition) of a sort pass
constexpr int64_t kBigPassRows = 16384;  // above this, twice as many keys per sort CTA
constexpr int64_t kHugePassRows = 131072;  // above this, four times as many
constexpr int kWideBins = 1024;          // histogram width: digits of up to 10 bits
constexpr int kDigitBitsWide = 10;
constexpr int kWideKeyPassesMax = 4;     // coordinate keys of up to 40 bits
constexpr int kWideMaskPasses = 3;       // 27-bit mask keys, 9-bit digits
constexpr int kWideTickets = kWideKeyPassesMax + kWideMaskPasses;   // one per sort pass
constexpr int kWideBarrierInts = 33;                // a grid barrier: 32 arrival counters + a release counter
// the tickets, then a grid barrier per sort pass
// rounded up to 16 bytes: callers place 64-bit arrays right after the counters
constexpr int kWideCounters = (kWideTickets + kWideTickets * kWideBarrierInts + 3) / 4 * 4;
static_assert(kWideCounters % 4 == 0, "the counters keep what follows them 16-byte aligned");
constexpr int64_t kWideMaxRows = int64_t(1) << 26;
// Hash mapper table: the smallest power of two >= kHashSlotsPerRow * n
// entries, in buckets of kHashBucket (one 32-byte sector).  At a load of at
// most 1/16 a bucket is almost never full, so nearly every probe ends in the
// first bucket: one round trip per lookup.
constexpr int kHashSlotsPerRow = 16;
constexpr int kHashBucket = 4;
constexpr int kHashMinLog2 = 11;
int hash_table_log2(int64_t n);

struct WideArgs {
    const int4* coords;
    int64_t n;
    int3 shape;
    int batch;
    int mapper;
    int calibrated;
    int wz, wy, wx, key_bits, row_bits;   // as in FusedArgs
    uint64_t koff[kTaps];
    int64_t gsb, gsx, gsy, cells;         // dense grid layout
    int64_t goff[kTaps];
    int32_t* grid;
    // hash mapper: open-addressing table of (key << row_bits | row), 0 = empty
    uint64_t* table;       // [1 << table_log2]
    int table_log2;
    // scratch
    uint64_t* va;          // [n] packed (key << row_bits | row), ping-pong
    uint64_t* vb;          // [n]
    int32_t* gh;           // [kWideKeyPassesMax + kWideMaskPasses][kWideBins] digit totals
    int32_t* tickets;      // [kWideCounters]
    uint64_t* look;        // [ceil(n / kWideKeysPerCta)][kWideBins] look-back states (or counts) of a sort pass
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
    int32_t* seg_off;
    int32_t* status;
    int64_t n_tiles, n_pad;
};

// Coordinate sort passes the whole-GPU pipeline takes for a key width.
int wide_key_passes(int key_bits);

// ---- the whole-GPU stable sort on its own, for the other map builders -----
// Digits of a sort of packed 64-bit values by their bits [lo, lo + bits):
// the fewest passes of at most kDigitBitsWide bits, as even as possible.
struct WideDigits {
    int passes;
    int shift[kWideKeyPassesMax];   // lowest bit of pass p's digit in the packed value
    int width[kWideKeyPassesMax];   // its width
};
// passes = 0 when bits needs more than kWideKeyPassesMax passes.
WideDigits wide_digits(int lo, int bits);
// Look-back state words a sort of n values needs (zeroed by the caller).
int64_t wide_sort_look_words(int64_t n);
// Stable LSD sort of the n packed values in a by the digits d, one
// whole-GPU pass per digit (a and b ping-pong), each launched with
// programmatic dependent launch.  gh[p][kWideBins] holds pass p's digit
// totals over all n values (counted by the kernel that wrote a; a pass in the
// count-exchange form derives them itself and does not read them); tickets
// (kWideCounters ints; passes use the ticket indices ticket0, ticket0 + 1,
// ... as tickets or arrival counters) and look are zero before the first
// pass; look is 16-byte aligned.  *in_b: the result is in b.
// first_plain: the first pass waits for the whole stream before it (a copy
// or memset precedes it) rather than overlapping a kernel's tail.
int wide_sort(uint64_t* a, uint64_t* b, int64_t n, const WideDigits& d, const int32_t* gh, int32_t* tickets,
              int ticket0, uint64_t* look, int32_t* status, cudaStream_t s, bool* in_b, bool first_plain = false);
// Whether a sort of up to n values by the digits d reads digit totals
// counted beforehand (gh): not when every pass runs in the count exchange,
// whose partitions derive the totals from each other's counts.  The kernel
// that writes the values then need not count them: it gets no_counts(d).
int wide_sort_reads_totals(int64_t n, const WideDigits& d, bool* reads);
inline WideDigits no_counts(WideDigits d) {
    d.passes = 0;
    return d;
}

// In a kernel whose every thread calls it together (whole warps): adds the
// digits of v under d to the block's histograms h[pass][digit] when valid.
__device__ __forceinline__ void wide_count_digits(uint64_t v, bool valid, const WideDigits& d,
                                                  int32_t (*h)[kWideBins]) {
    const int lane = threadIdx.x & 31;
    for (int p = 0; p < d.passes; ++p) {
        const int dg = valid ? static_cast<int>((v >> d.shift[p]) & ((1u << d.width[p]) - 1u)) : kWideBins;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, dg);
        if (valid && lane == __ffs(peers) - 1) atomicAdd(&h[p][dg], __popc(peers));
    }
}

// Adds a block's histograms h (cleared before) into gh[pass][digit] (all
// threads of the block call it after their counts, behind a barrier).
__device__ __forceinline__ void wide_flush_digits(const WideDigits& d, int32_t (*h)[kWideBins], int32_t* gh) {
    for (int i = threadIdx.x; i < d.passes * kWideBins; i += blockDim.x) {
        const int32_t x = h[i / kWideBins][i % kWideBins];
        if (x) atomicAdd(gh + i, x);
    }
}
// The whole build on stream s; sms = multiprocessors of the device.
int launch_map_wide(const WideArgs& a, int sms, cudaStream_t s);

// Neighbour search (map_search.cu) over sv, the n packed values (key <<
// row_bits | row) in ascending order: writes nbr (original row order), mask
// and adds the per-tap counts to tap_count.  Launched with programmatic
// dependent launch: it waits for the kernels before it.
int launch_search_window(const uint64_t* sv, int64_t n, int row_bits, int key_bits, const uint64_t* koff,
                         int32_t* nbr, uint32_t* mask, int32_t* tap_count, int32_t* status, cudaStream_t s);

}  // namespace spconv

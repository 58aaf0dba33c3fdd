// bf16 gather implicit GEMM on the 5th-generation tensor cores (tcgen05 +
// TMEM), fp32 accumulation, output written back in the original row order.
//
// Work decomposition ("Sparse convolution in FP32", "Neighbour masks and sorted
// rows"): rows are in mask-sorted order and cut into 128-row tiles; a tile
// visits only the taps in the union of its rows' masks.  For each such tap
// the tile's input rows are gathered (a row without that neighbour is filled
// with zeros and costs no memory traffic) and multiplied by that tap's
// weights, accumulating all taps of the tile in tensor memory; the
// accumulator is rounded to bf16 once and each row is stored to its original
// position (FlyDSL PR #942: fp32 accumulation, gather fused into the GEMM).
//
// Per CTA (persistent, one per SM), warp-specialised:
//   warps 0-3   epilogue: tcgen05.ld of the accumulator, the optional
//               scale / bias / residual / ReLU in fp32, bf16 convert, store
//   warp 4      TMEM allocation + MMA issue (the whole warp runs the loop,
//               lane 0 issues)
//   warp 5      scheduler: walks this CTA's work items (tile, output block)
//               and bulk-copies each tile's gather indices for every tap of
//               its union into shared memory, two items ahead of the
//               producers.  Items come largest tap union first and are dealt
//               to the CTAs in snake order (CTA c takes item c of the first
//               round, item 2G-1-c of the second, ...), which keeps the
//               largest and smallest items together and the SMs balanced.
//   warps 6..   one producer warp per pipeline stage: cp.async 16-byte row
//               gathers of A into the 128-byte-swizzled layout (a row
//               without the neighbour is written as zeros, with no memory
//               request), plus one bulk async copy of the pre-packed weight
//               tile B.  Warp w runs on scheduler partition w % 4; no
//               producer is placed on partition 0, where the MMA warp runs,
//               so the MMA issue never queues behind a burst of gathers
//               (warps 8, 12 are left idle).
// The accumulator is double-buffered in TMEM so the epilogue of one tile
// overlaps the main loop of the next.
//
// Two work decompositions share this kernel ("Compaction is the largest
// single win", FlyDSL PR #942; "Offset-group partitioning", "Sparse
// convolution in FP32"):
//   tile-union (TM = false)  an item is a 128-row tile of the mask-sorted
//       rows and one output block; it visits every tap of the tile's union,
//       accumulates them all in TMEM and stores each row once, in bf16.
//       Rows lacking a tap of the union multiply zeros.
//   tap-major (TM = true)    an item is 128 consecutive pairs of one tap's
//       compacted pair list (the last item of a tap is ragged), so no MMA
//       row is wasted; each row's product is added in fp32 into an
//       accumulation buffer (vector red.global.add), which a final pass
//       rounds to bf16.  It trades the zero rows for reduction traffic of
//       4 bytes per pair and output channel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx_sm100.cuh"

namespace spconv {
namespace {

constexpr int BM = 128;          // tile rows (MMA M)
constexpr int BK = 64;           // input channels per stage (one 128-byte row)
constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kSchedWarp = 5;
constexpr int kProdWarp0 = 6;

// Warp of producer slot s: the s-th warp id >= kProdWarp0 that is not a
// multiple of 4, and the inverse (-1 for a warp that is not a producer).
__host__ __device__ constexpr int producer_warp(int s) { return kProdWarp0 + s + (s + 1) / 3; }
__device__ __forceinline__ int producer_slot(int w) {
    return (w < kProdWarp0 || (w & 3) == 0) ? -1 : w - kProdWarp0 - ((w - 1) / 4 - 1);
}
constexpr int kStageA = BM * BK * 2;   // 16 KB
constexpr int kIdxBytes = kTaps * BM * 4;   // one item's gather indices, 13.5 KB
constexpr int kMetaRing = 4;                // items in flight between scheduler and epilogue
constexpr int kLayerMark = -2;              // a meta entry that closes a layer of a fused stack

struct TcParams {
    const __nv_bfloat16* feats;   // [n][c_in], the input of layer 0
    const int32_t* gtab;          // [27][n_pad]
    const uint32_t* tile_union;   // [n_tiles]
    const int32_t* tile_order;    // [n_tiles]
    const int32_t* perm;          // [n_pad]
    const int32_t* tap_off;       // [28]  tap-major: CSR offsets of the pair lists
    const int32_t* in_rows;       // [P]   tap-major: input row of each pair
    const int32_t* out_rows;      // [P]   tap-major: output row of each pair
    float* acc;                   // [n][c_out] tap-major: fp32 sums (zero at launch)
    int32_t* status;
    int64_t n, n_pad;
    int64_t n_in;                 // rows of feats (gather bound)
    int32_t n_items;              // n_tiles * n_nb
    int32_t c_in, c_out;
    int32_t k_chunks;             // ceil(c_in / 64)
    int32_t n_tile;               // output channels per item (multiple of 16, <= NTMAX)
    int32_t n_nb;                 // c_out / n_tile
    // offset groups: this launch covers the group's taps [k0, k0 + taps of the
    // union bits); gtab, tile_union, tile_order and perm point at the group's
    // slices, the packed weights hold taps_w taps per output block
    int32_t k0, taps_w;
    int32_t mode;                 // kModeStore, or the partial-sum modes of a grouped forward
    float* ws;                    // [n][c_out] fp32 partial sums of the groups before the last
    const int32_t* tiles_dev;     // device count of the leading tiles of tile_order to visit, or null (all)
    // Layer l multiplies the output of layer l - 1 (layer 0: feats) by its
    // packed weights wpacks[l] (see k_pack_weights), applies epis[l] to each
    // fp32 sum before the rounding (when epi_ons[l]) and stores outs[l]
    // ([n][c_out]).  One layer is the plain forward.  A stack of layers over
    // the same map runs in one launch (tile-union only): between two layers
    // every CTA counts itself into layer_done[l] once its stores are visible,
    // and no gather of layer l + 1 starts before all have.
    int32_t n_layers;
    const uint8_t* wpacks[kMaxFusedLayers];
    __nv_bfloat16* outs[kMaxFusedLayers];
    Epilogue epis[kMaxFusedLayers];
    int32_t epi_ons[kMaxFusedLayers];
    int32_t* layer_done;          // [kMaxFusedLayers], zero at launch
};

// Output modes.  One group: the tile's sum, rounded once, to out.  G groups,
// one launch each, ws zeroed first: every group but the centre one adds its
// sums to ws, visiting only the tiles whose union is not empty; the centre
// group (every row has the centre tap, so every tile is visited) goes last,
// adds ws to its own sums and rounds once to out.  Items with no tap are
// never scheduled: two of them in a row could stall the stage ring, whose
// MMA waits span consecutive items.
enum : int32_t { kModeStore = 0, kModeWsAdd = 2, kModeWsFinish = 3 };

template <int NTMAX>
struct TcConfig {
    static constexpr int kStageB = NTMAX * 128;
    static constexpr int kStage = kStageA + kStageB;
    static constexpr int kStages = (NTMAX == 256) ? 4 : (NTMAX == 128 ? 6 : 8);
    // The MMA thread waits once per group of kGroup stages: a barrier wait
    // stalls its issue for ~100-200 cycles, which only hides behind at least
    // ~500 cycles of queued MMA work (4 MMAs of N=256, or 8 of N=128).
    static constexpr int kGroup = (NTMAX == 256) ? 1 : 2;
    static_assert(kStages % kGroup == 0, "stages come in whole groups");
    // Producer warps per stage.  With N = 256 the tensor pipe spends 512 cycles
    // on a stage, and one warp's ~1,600-cycle gather round trip across four
    // stages cannot keep up, so two warps share each stage (64 rows each).
    static constexpr int kProdPerStage = (NTMAX == 256) ? 2 : 1;
    static_assert(kProdPerStage == 1 || kGroup == 1, "shared stages are not grouped");
    static constexpr int kProducers = kStages * kProdPerStage;
    static constexpr int kThreads = 32 * (producer_warp(kProducers - 1) + 1);
    static constexpr int kTmemCols = 2 * NTMAX < 32 ? 32 : 2 * NTMAX;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmem = kStages * kStage + 2 * kIdxBytes + 1024 + kBarBytes;
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

// Item that CTA `cta` of `grid` takes in its round L (snake order).
__device__ __forceinline__ int snake_item(int L, int cta, int grid) {
    return L * grid + ((L & 1) ? grid - 1 - cta : cta);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// The epilogue on 8 consecutive sums v[0..7] of output row `row`, channels
// o .. o+7 (o a multiple of 8; scale, bias and residual 16-byte aligned).
__device__ __forceinline__ void epilogue8(uint32_t* v, const Epilogue& e, int64_t row, int c_out, int o) {
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = __uint_as_float(v[j]);
    if (e.scale) {
        const float4 a = *reinterpret_cast<const float4*>(e.scale + o);
        const float4 b = *reinterpret_cast<const float4*>(e.scale + o + 4);
        y[0] *= a.x; y[1] *= a.y; y[2] *= a.z; y[3] *= a.w;
        y[4] *= b.x; y[5] *= b.y; y[6] *= b.z; y[7] *= b.w;
    }
    if (e.bias) {
        const float4 a = *reinterpret_cast<const float4*>(e.bias + o);
        const float4 b = *reinterpret_cast<const float4*>(e.bias + o + 4);
        y[0] += a.x; y[1] += a.y; y[2] += a.z; y[3] += a.w;
        y[4] += b.x; y[5] += b.y; y[6] += b.z; y[7] += b.w;
    }
    if (e.residual) {
        const uint4 q = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(e.residual) +
                                                        row * c_out + o);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            y[2 * j] += __uint_as_float(w[j] << 16);
            y[2 * j + 1] += __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
    if (e.relu) {
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = fmaxf(y[j], 0.0f);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __float_as_uint(y[j]);
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

template <int NTMAX, bool TM>
__global__ void __launch_bounds__(TcConfig<NTMAX>::kThreads, 1) k_tc_gemm(const TcParams p) {
    using Cfg = TcConfig<NTMAX>;
    constexpr int S = Cfg::kStages;
    constexpr int G = Cfg::kGroup;
    constexpr int P = Cfg::kProdPerStage;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int32_t* idx = reinterpret_cast<int32_t*>(smem + S * Cfg::kStage);   // [2][27][128]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStage + 2 * kIdxBytes);
    uint64_t* full = bars;                       // [S / G], one per group of G stages
    uint64_t* empty = full + S;                  // [S]
    uint64_t* acc_full = empty + S;              // [2]
    uint64_t* acc_empty = acc_full + 2;          // [2]
    uint64_t* idx_full = acc_empty + 2;          // [2] indices + item landed
    uint64_t* idx_empty = idx_full + 2;          // [2] producers and MMA done with the item
    uint64_t* meta_full = idx_empty + 2;         // [kMetaRing] item published (epilogue side)
    uint64_t* meta_empty = meta_full + kMetaRing;// [kMetaRing] epilogue has read it
    uint64_t* exit_bar = meta_empty + kMetaRing;
    uint64_t* layer_bar = exit_bar + 1;          // the epilogue warps have stored a layer
    int32_t* m_item = reinterpret_cast<int32_t*>(layer_bar + 1);   // [kMetaRing], -1 = no more work
    int32_t* m_tile = m_item + kMetaRing;
    uint32_t* m_uni = reinterpret_cast<uint32_t*>(m_tile + kMetaRing);
    int32_t* m_layer = reinterpret_cast<int32_t*>(m_uni + kMetaRing);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(m_layer + kMetaRing);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // tap-major: the output rows of the items in the meta ring, in the last
    // kMetaRing x 128 entries of the index area (only rank 0 of each index
    // buffer is used in that mode)
    int32_t* m_orow = idx + 2 * kTaps * BM - kMetaRing * BM;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            if (s < S / G) ptx::mbar_init(&full[s], 2 * G * P);   // two arrivals per producer warp of the group
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], kEpiWarps);
            ptx::mbar_init(&idx_full[b], 1);
            ptx::mbar_init(&idx_empty[b], Cfg::kProducers + 1);
        }
        for (int r = 0; r < kMetaRing; ++r) {
            ptx::mbar_init(&meta_full[r], 1);
            ptx::mbar_init(&meta_empty[r], kEpiWarps);
        }
        ptx::mbar_init(exit_bar, 1);
        ptx::mbar_init(layer_bar, kEpiWarps);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(tmem_slot, Cfg::kTmemCols);
        ptx::tmem_relinquish();
    }
    // launched early (programmatic dependent launch): the map and inputs are
    // read only after the kernels before this one have finished
    pdl_wait();
    // Scheduler state.  Tile-union items come from the tile order; tap-major
    // items are numbered tap by tap: lane k < 27 holds t_excl, the number of
    // 128-pair tiles of taps before k, and the item count is derived here.
    int n_items = p.n_items;
    if (p.tiles_dev && warp == kSchedWarp) n_items = *p.tiles_dev * p.n_nb;
    int32_t t_excl = 0, t_off = 0, t_end = 0;
    if (TM && warp == kSchedWarp) {
        t_off = lane <= kTaps ? p.tap_off[lane] : 0;
        const int32_t nxt = __shfl_down_sync(0xFFFFFFFFu, t_off, 1);
        const int32_t tiles = lane < kTaps ? (nxt - t_off + BM - 1) / BM : 0;
        int32_t incl = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        t_excl = incl - tiles;
        t_end = nxt;
        n_items = __shfl_sync(0xFFFFFFFFu, incl, kTaps - 1) * p.n_nb;
    }
    // the scheduler looks up its first item while the CTA sets up:
    // tile-union (tile, union); tap-major (pair base, pair count in s_tile, tap bit in s_uni)
    int s_layer = 0, s_round = 0;   // the scheduler's layer and its round in that layer
    int s_it = snake_item(0, blockIdx.x, gridDim.x), s_tile = 0, s_cnt = 0;
    uint32_t s_uni = 0;
    auto lookup = [&](int it) {
        if (TM) {
            const int pt = it / p.n_nb;
            const uint32_t le = __ballot_sync(0xFFFFFFFFu, lane < kTaps && t_excl <= pt);
            const int k = __popc(le) - 1;
            const int32_t ex = __shfl_sync(0xFFFFFFFFu, t_excl, k);
            const int32_t off = __shfl_sync(0xFFFFFFFFu, t_off, k);
            const int32_t end = __shfl_sync(0xFFFFFFFFu, t_end, k);
            s_tile = off + (pt - ex) * BM;
            s_cnt = end - s_tile < BM ? end - s_tile : BM;
            s_uni = 1u << k;
        } else {
            s_tile = p.tile_order[it / p.n_nb];
            s_uni = p.tile_union[s_tile];
        }
    };
    if (warp == kSchedWarp && s_it < n_items) lookup(s_it);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t smem_base = ptx::smem_u32(smem);
    const uint32_t idx_base = ptx::smem_u32(idx);

    auto fail = [&]() {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
    };
    // every lane polls (warp-uniform control flow); the warp goes on only if all saw the phase
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        const bool ok = ptx::mbar_wait(bar, parity, abort_flag);
        return __all_sync(0xFFFFFFFFu, ok);
    };

    if (warp == kSchedWarp) {
        // ---------------- scheduler: item L goes to index buffer L % 2 and
        // meta slot L % kMetaRing
        int pend[2] = {-1, -1};   // item issued into each index buffer, not yet known consumed
        for (int L = 0;; ++L) {
            const int b = L & 1, r = L % kMetaRing;
            if (L >= kMetaRing && !warp_wait(&meta_empty[r], ((L / kMetaRing) - 1) & 1)) {
                if (lane == 0) fail();
                break;
            }
            if (L >= 2) {
                if (!warp_wait(&idx_empty[b], ((L >> 1) - 1) & 1)) {
                    if (lane == 0) fail();
                    break;
                }
                pend[b] = -1;   // consumed, so its copies have landed
            }
            const int it = s_it;
            const int tile = s_tile;
            const uint32_t uni = s_uni;
            if (it >= n_items && s_layer + 1 < p.n_layers) {
                // this CTA's items of the layer are published: a marker tells the
                // epilogue to count the CTA in once they are stored, and the next
                // layer's items wait until every CTA has
                if (lane == 0) {
                    m_item[r] = kLayerMark;
                    m_layer[r] = s_layer;
                    ptx::mbar_arrive(&idx_full[b]);
                    ptx::mbar_arrive(&meta_full[r]);
                }
                bool ok = true;
                if (lane == 0) {
                    const uint64_t t0 = ptx::globaltimer();
                    for (uint32_t spin = 0;; ++spin) {
                        int32_t v;
                        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];"
                                     : "=r"(v)
                                     : "l"(p.layer_done + s_layer)
                                     : "memory");
                        if (v >= static_cast<int32_t>(gridDim.x)) break;
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        __nanosleep(64);
                        if ((spin & 63u) == 63u && ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
                    if (lane == 0) fail();
                    break;
                }
                ++s_layer;
                s_round = 0;
                s_it = snake_item(0, blockIdx.x, gridDim.x);
                if (s_it < n_items) lookup(s_it);
                continue;
            }
            if (it >= n_items) {   // no more work: publish the end marker
                if (lane == 0) {
                    m_item[r] = -1;
                    ptx::mbar_arrive(&idx_full[b]);
                    ptx::mbar_arrive(&meta_full[r]);
                }
                break;
            }
            if (TM) {
                // the item's input rows (rank 0 of index buffer b) and output rows
                // (meta slot r), -1 past the end of the tap's list
                const int32_t cnt = s_cnt;
#pragma unroll
                for (int q = 0; q < BM / 32; ++q) {
                    const int i = lane + 32 * q;
                    idx[b * kTaps * BM + i] = i < cnt ? p.in_rows[tile + i] : -1;
                    m_orow[r * BM + i] = i < cnt ? p.out_rows[tile + i] : -1;
                }
                __syncwarp();
                if (lane == 0) {
                    m_item[r] = it;
                    m_tile[r] = tile;
                    m_uni[r] = uni;
                    m_layer[r] = s_layer;
                    ptx::mbar_arrive(&idx_full[b]);
                }
            } else {
                if (lane == 0) {
                    m_item[r] = it;
                    m_tile[r] = tile;
                    m_uni[r] = uni;
                    m_layer[r] = s_layer;
                    ptx::mbar_arrive_expect_tx(&idx_full[b], static_cast<uint32_t>(__popc(uni)) * (BM * 4));
                }
                __syncwarp();
                // lane k copies tap k's 128 indices to the tap's rank in the union
                if (lane < kTaps && ((uni >> lane) & 1u)) {
                    const int rank = __popc(uni & ((1u << lane) - 1u));
                    ptx::bulk_copy_g2s(idx_base + static_cast<uint32_t>((b * kTaps + rank) * BM * 4),
                                       p.gtab + static_cast<int64_t>(lane) * p.n_pad + static_cast<int64_t>(tile) * BM,
                                       BM * 4, &idx_full[b]);
                }
                pend[b] = L;
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&meta_full[r]);
            // look up the next item now: the loads overlap the waits above
            s_it = snake_item(++s_round, blockIdx.x, gridDim.x);
            if (s_it < n_items) lookup(s_it);
        }
        // copies still in flight (only after an abort) land before the CTA exits
        if (lane == 0)
            for (int b = 0; b < 2; ++b)
                if (pend[b] >= 0 && !ptx::mbar_wait(&idx_full[b], (pend[b] >> 1) & 1, nullptr))
                    atomicOr(p.status, kStatusTimeout);
        __syncwarp();
    } else if (producer_slot(warp) >= 0) {
        // ---------------- producers: warp producer_warp(P s + h) fills rows
        // [h 128/P, (h + 1) 128/P) of stage s and arrives on the barrier of the
        // stage's group; part h = 0 also brings the stage's weight tile
        const int slot = producer_slot(warp) / P, part = producer_slot(warp) % P;
        uint64_t* gfull = &full[slot / G];
        const uint32_t a_smem = smem_base + slot * Cfg::kStage;
        const uint32_t b_smem = a_smem + kStageA;
        const uint32_t b_bytes = static_cast<uint32_t>(p.n_tile) * 128u;
        uint32_t f = 0;
        int64_t last = -1;   // last fill this warp issued
        bool stop = false;
        // lane group g (8 lanes) gathers RG consecutive rows of this warp's part,
        // one 16-byte chunk per lane, so each instruction reads four whole 128-byte rows
        constexpr int RG = BM / P / 4;
        const int grp = lane >> 3, chunk = lane & 7;
        const int row0 = part * (BM / P) + grp * RG;   // a multiple of 8: the swizzle phase of row0 + i is i & 7
        // The MMA waits for whole groups of G stages: an incomplete group (at
        // the end, or before a layer boundary, where the next stage waits for
        // every CTA) is completed with empty stages, two arrivals each.
        auto pad_group = [&]() {
            const uint32_t padded = (f + G - 1) / G * G;
            for (uint32_t d = f; d < padded && !stop; ++d) {
                if (static_cast<int>(d % S) != slot) continue;
                const uint32_t u = d / S;
                if (u > 0 && !warp_wait(&empty[slot], (u - 1) & 1)) {
                    if (lane == 0) fail();
                    stop = true;
                    break;
                }
                if (lane == 0) {
                    ptx::mbar_arrive(gfull);
                    ptx::mbar_arrive(gfull);
                }
                last = d;
            }
            f = padded;
        };
        for (int L = 0; !stop; ++L) {
            const int b = L & 1;
            if (!warp_wait(&idx_full[b], (L >> 1) & 1)) {
                if (lane == 0) fail();
                break;
            }
            const int it = m_item[L % kMetaRing];
            if (it == kLayerMark) {   // a layer boundary: nothing to gather
                pad_group();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&idx_empty[b]);
                continue;
            }
            if (it < 0) break;
            const int nb = it % p.n_nb;
            const int layer = m_layer[L % kMetaRing];
            uint32_t uni = m_uni[L % kMetaRing];
            const int32_t* gidx = idx + b * kTaps * BM;
            const __nv_bfloat16* lin = layer == 0 ? p.feats : p.outs[layer - 1];
            const uint8_t* lw = p.wpacks[layer];
            // this warp's stages of the item: fs in [f, f + stages) with fs % S == slot;
            // stage fs is chunk kc of the union's j-th tap (taps in ascending order)
            const uint32_t f_end = f + static_cast<uint32_t>(__popc(uni) * p.k_chunks);
            uint32_t ucur = uni;   // the union without its first jcur taps
            int jcur = 0;
            for (uint32_t fs = f + static_cast<uint32_t>((slot - static_cast<int>(f % S) + S) % S); fs < f_end && !stop;
                 fs += S) {
                const int j = static_cast<int>((fs - f) / static_cast<uint32_t>(p.k_chunks));
                const int kc = static_cast<int>(fs - f) - j * p.k_chunks;
                for (; jcur < j; ++jcur) ucur &= ucur - 1;
                const int k = __ffs(ucur) - 1;
                // all RG source rows of this lane group, read before any copy is issued
                int32_t sr[RG];
                const int4* gsrc = reinterpret_cast<const int4*>(gidx + j * BM + row0);
#pragma unroll
                for (int q = 0; q < RG / 4; ++q) {
                    const int4 v4 = gsrc[q];
                    sr[4 * q] = v4.x;
                    sr[4 * q + 1] = v4.y;
                    sr[4 * q + 2] = v4.z;
                    sr[4 * q + 3] = v4.w;
                }
                const uint32_t u = fs / S;
                if (u > 0 && !warp_wait(&empty[slot], (u - 1) & 1)) {
                    if (lane == 0) fail();
                    stop = true;
                    break;
                }
                if (lane == 0) {
                    if (part == 0) {
                        ptx::mbar_arrive_expect_tx(gfull, b_bytes);
                        const uint8_t* src =
                            lw + (static_cast<int64_t>(nb * p.taps_w + p.k0 + k) * p.k_chunks + kc) * b_bytes;
                        ptx::bulk_copy_g2s(b_smem, src, b_bytes, gfull);
                    } else {
                        ptx::mbar_arrive(gfull);
                    }
                }
                const int kcol = kc * BK + chunk * 8;
                // rows below lim are copied: n, or none when this lane's channels lie past c_in
                const uint32_t lim = kcol < p.c_in ? static_cast<uint32_t>(p.n_in) : 0u;
                const char* fcol = reinterpret_cast<const char*>(lin + kcol);
                const uint32_t row_bytes = static_cast<uint32_t>(p.c_in) * 2u;
                const uint32_t dst0 = a_smem + static_cast<uint32_t>(row0) * 128;
                // Each row is one predicated copy or zero store: the producer's
                // instruction count per row is on the kernel's critical path, so
                // absent (-1) and out-of-range indices are caught by one unsigned
                // compare, and a row index past n (skipped: a zero row) is reported
                // from one 16-byte word of the indices per lane (the eight lanes of
                // a group cover its rows) rather than per row.
#pragma unroll
                for (int i = 0; i < RG; ++i) {
                    const int32_t src_row = sr[i];
                    const uint32_t dst = dst0 + i * 128 + ((chunk ^ (i & 7)) << 4);
                    if (static_cast<uint32_t>(src_row) < lim)
                        ptx::cp_async_16(dst, fcol + static_cast<uint64_t>(static_cast<uint32_t>(src_row)) * row_bytes, 16u);
                    else
                        ptx::st_shared_zero16(dst);   // absent neighbour: no memory request
                }
                bool past = false;
                if (chunk < RG / 4) {
                    const int4 w4 = gsrc[chunk];
                    past = max(max(w4.x, w4.y), max(w4.z, w4.w)) >= p.n_in;
                }
                if (__any_sync(0xFFFFFFFFu, past) && lane == 0) atomicOr(p.status, kStatusInternal);
                ptx::cp_async_commit();
                ptx::cp_async_wait_all();
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(gfull);
                last = fs;
            }
            if (!stop) f = f_end;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&idx_empty[b]);
        }
        // the last group may be incomplete: its remaining stages arrive empty
        if (!stop) pad_group();
        // every copy this warp issued has landed before the CTA may exit
        if (lane == 0 && last >= 0 && !ptx::mbar_wait(gfull, (static_cast<uint32_t>(last) / S) & 1, nullptr))
            atomicOr(p.status, kStatusTimeout);
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer: the warp runs the loop, lane 0 issues
        const uint32_t leader = lane == 0;
        const uint32_t idesc = ptx::idesc_bf16_f32(BM, static_cast<uint32_t>(p.n_tile));
        const uint64_t desc0 = ptx::sdesc_k128(smem_base);   // stage 0's A operand
        uint32_t f = 0;
        int ai = 0;   // items accumulated so far: item ai uses TMEM buffer ai & 1
        bool stop = false;
        for (int L = 0; !stop; ++L) {
            const int b = L & 1;
            if (!warp_wait(&idx_full[b], (L >> 1) & 1)) {
                if (lane == 0) fail();
                break;
            }
            const int it = m_item[L % kMetaRing];
            const int n_taps = __popc(m_uni[L % kMetaRing]);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&idx_empty[b]);
            if (it == kLayerMark) {
                // the producers completed the open group with empty stages (its
                // barrier was waited for at its first stage): release them
                for (; f % G != 0; ++f) ptx::mma_commit_if(leader, &empty[f % S]);
                continue;
            }
            if (it < 0) break;
            const int buf = ai & 1;
            const uint32_t v = static_cast<uint32_t>(ai >> 1);
            ++ai;
            if (v > 0 && !warp_wait(&acc_empty[buf], (v - 1) & 1)) {
                if (lane == 0) fail();
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * NTMAX);
            bool first = true;
            for (int t = 0; t < n_taps && !stop; ++t) {
                for (int kc = 0; kc < p.k_chunks; ++kc, ++f) {
                    const int slot = static_cast<int>(f % S);
                    if (slot % G == 0 && !warp_wait(&full[slot / G], (f / S) & 1)) {
                        if (lane == 0) fail();
                        stop = true;
                        break;
                    }
                    // the stage's descriptors: the base one plus the stage's offset / 16 in
                    // the start-address field (shared addresses stay below 2^18: no carry)
                    const uint64_t a_desc = desc0 + static_cast<uint64_t>((slot * Cfg::kStage) >> 4);
                    const uint64_t b_desc = a_desc + static_cast<uint64_t>(kStageA >> 4);
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j) {
                        ptx::mma_bf16_if(leader, d_tmem, a_desc + 2 * j, b_desc + 2 * j, idesc,
                                         (first && j == 0) ? 0u : 1u);   // K step 16 bf16 = 32 bytes
                    }
                    first = false;
                    ptx::mma_commit_if(leader, &empty[slot]);
                }
            }
            if (!stop) ptx::mma_commit_if(leader, &acc_full[buf]);
        }
        // all MMAs issued by this warp have completed once exit_bar flips
        ptx::mma_commit_if(leader, exit_bar);
        // (no early exit on abort here: TMEM is freed only after this)
        const bool done = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(exit_bar, 0, nullptr));
        if (!done && lane == 0) atomicOr(p.status, kStatusTimeout);
    } else if (warp < kEpiWarps) {
        // ---------------- epilogue: warp w reads TMEM lanes [32w, 32w + 32)
        int ai = 0;      // items stored so far: item ai sits in TMEM buffer ai & 1
        int marks = 0;   // layer markers seen
        for (int L = 0;; ++L) {
            const int r = L % kMetaRing;
            if (!warp_wait(&meta_full[r], (L / kMetaRing) & 1)) {
                if (lane == 0) fail();
                break;
            }
            const int it = m_item[r];
            const int tile = m_tile[r];
            // a tile none of whose rows has a tap of this group: no MMA ran, the sums are zero
            const bool none = m_uni[r] == 0u;
            // the row this thread writes: tile-union, perm of the sorted position;
            // tap-major, the pair's output row
            int32_t orig = -1;
            if (TM) {
                orig = m_orow[r * BM + warp * 32 + lane];
            } else if (it >= 0) {
                const int64_t s = static_cast<int64_t>(tile) * BM + warp * 32 + lane;
                orig = s < p.n ? p.perm[s] : -1;
            }
            const int layer = m_layer[r];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&meta_empty[r]);
            if (it == kLayerMark) {
                // every store of this CTA's items of the layer has been issued:
                // each thread makes its own visible GPU-wide, the warps meet on
                // layer_bar, and warp 0 counts the CTA in
                __threadfence();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(layer_bar);
                if (warp == 0) {
                    if (!warp_wait(layer_bar, static_cast<uint32_t>(marks) & 1u)) {
                        if (lane == 0) fail();
                        break;
                    }
                    if (lane == 0) atomicAdd(p.layer_done + layer, 1);
                }
                ++marks;
                continue;
            }
            if (it < 0) break;
            const int nb = it % p.n_nb;
            const int buf = ai & 1;
            const uint32_t par = static_cast<uint32_t>(ai >> 1) & 1u;
            ++ai;
            __nv_bfloat16* lout = p.outs[layer];
            const Epilogue& lepi = p.epis[layer];
            const int32_t lepi_on = p.epi_ons[layer];
            if (!warp_wait(&acc_full[buf], par)) {
                if (lane == 0) fail();
                break;
            }
            ptx::tc_fence_after();
            const bool to_out = p.mode == kModeStore || p.mode == kModeWsFinish;
            __nv_bfloat16* dst_row = (!TM && orig >= 0 && to_out)
                                         ? lout + static_cast<int64_t>(orig) * p.c_out + nb * p.n_tile
                                         : nullptr;
            float* ws_row = (!TM && orig >= 0 && p.mode != kModeStore)
                                ? p.ws + static_cast<int64_t>(orig) * p.c_out + nb * p.n_tile
                                : nullptr;
            const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(buf * NTMAX);
            // n_tile is a multiple of 16; columns go 32 at a time (two loads per wait)
            for (int c = 0; c < p.n_tile; c += 32) {
                const bool two = c + 16 < p.n_tile;
                uint32_t v[32];
                if (!none) {
                    ptx::tmem_ld_32x32b_x16_at(t_addr + c, v);
                    if (two) ptx::tmem_ld_32x32b_x16_at(t_addr + c + 16, v + 16);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0u;
                }
                if (ws_row) {
                    // partial sums of a grouped forward (one thread per row: no races)
                    float4* w4 = reinterpret_cast<float4*>(ws_row + c);
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        if (h >= 4 && !two) break;
                        float4 a = make_float4(__uint_as_float(v[4 * h]), __uint_as_float(v[4 * h + 1]),
                                               __uint_as_float(v[4 * h + 2]), __uint_as_float(v[4 * h + 3]));
                        if (none && p.mode == kModeWsAdd) continue;
                        const float4 b = w4[h];
                        a.x += b.x;
                        a.y += b.y;
                        a.z += b.z;
                        a.w += b.w;
                        if (p.mode == kModeWsAdd) {
                            w4[h] = a;
                        } else {
                            v[4 * h] = __float_as_uint(a.x);
                            v[4 * h + 1] = __float_as_uint(a.y);
                            v[4 * h + 2] = __float_as_uint(a.z);
                            v[4 * h + 3] = __float_as_uint(a.w);
                        }
                    }
                }
                if (TM) {
                    if (orig >= 0) {
                        float* dacc = p.acc + static_cast<int64_t>(orig) * p.c_out + nb * p.n_tile + c;
#pragma unroll
                        for (int h = 0; h < 8; ++h) {
                            if (h >= 4 && !two) break;
                            red_add_v4(dacc + 4 * h, __uint_as_float(v[4 * h]), __uint_as_float(v[4 * h + 1]),
                                       __uint_as_float(v[4 * h + 2]), __uint_as_float(v[4 * h + 3]));
                        }
                    }
                } else if (dst_row) {
                    if (lepi_on) {
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            if (h >= 2 && !two) break;
                            epilogue8(v + 8 * h, lepi, orig, p.c_out, nb * p.n_tile + c + 8 * h);
                        }
                    }
                    uint4* d = reinterpret_cast<uint4*>(dst_row + c);
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (h >= 2 && !two) break;
                        uint4 q;
                        q.x = pack_bf16x2(__uint_as_float(v[8 * h + 0]), __uint_as_float(v[8 * h + 1]));
                        q.y = pack_bf16x2(__uint_as_float(v[8 * h + 2]), __uint_as_float(v[8 * h + 3]));
                        q.z = pack_bf16x2(__uint_as_float(v[8 * h + 4]), __uint_as_float(v[8 * h + 5]));
                        q.w = pack_bf16x2(__uint_as_float(v[8 * h + 6]), __uint_as_float(v[8 * h + 7]));
                        d[h] = q;
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&acc_empty[buf]);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kMmaWarp) ptx::tmem_dealloc(tmem_base, Cfg::kTmemCols);
    pdl_trigger();
}

// Packed weight image: for each (output block nb, tap k, 64-channel input
// chunk kc) a block of n_tile rows x 128 bytes; row n holds
// W[k][kc*64 .. kc*64+63][nb*n_tile + n] (zero past c_in), its 16-byte chunk c
// stored at chunk position c ^ (n & 7) -- the K-major 128-byte-swizzled
// shared-memory layout that the MMA reads directly after one bulk copy.
__global__ void k_pack_weights(const __nv_bfloat16* __restrict__ w, int c_in, int c_out, int taps, int n_tile,
                               int k_chunks, int n_nb, uint4* __restrict__ dst) {
    const int64_t total = static_cast<int64_t>(n_nb) * taps * k_chunks * n_tile * 8;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // idx enumerates (nb, k, kc, c, n) with n fastest so reads of W rows coalesce
        int64_t q = idx;
        const int n = static_cast<int>(q % n_tile);
        q /= n_tile;
        const int c = static_cast<int>(q % 8);
        q /= 8;
        const int kc = static_cast<int>(q % k_chunks);
        q /= k_chunks;
        const int k = static_cast<int>(q % taps);
        const int nb = static_cast<int>(q / taps);
        const int o = nb * n_tile + n;
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const int i0 = kc * BK + c * 8 + e;
            const __nv_bfloat16 z = __float2bfloat16(0.0f);
            const __nv_bfloat16 a = i0 < c_in ? w[(static_cast<int64_t>(k) * c_in + i0) * c_out + o] : z;
            const __nv_bfloat16 b = i0 + 1 < c_in ? w[(static_cast<int64_t>(k) * c_in + i0 + 1) * c_out + o] : z;
            __nv_bfloat162 v;
            v.x = a;
            v.y = b;
            h[e / 2] = *reinterpret_cast<uint32_t*>(&v);
        }
        const int64_t blk = (static_cast<int64_t>(nb) * taps + k) * k_chunks + kc;
        const int64_t off16 = blk * n_tile * 8 + static_cast<int64_t>(n) * 8 + (c ^ (n & 7));
        dst[off16] = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

int num_sms() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

// fp32 sums of the tap-major variant -> bf16 output (round to nearest even),
// four values per thread and step.
// Rounds the tap-major sums to bf16, 8 channels per thread, applying the
// epilogue on the way (c_out is a multiple of 16, so 8 never straddle rows).
__global__ void __launch_bounds__(256) k_acc_to_bf16(const float4* __restrict__ acc, uint4* __restrict__ out,
                                                     int64_t count8, int c_out, Epilogue epi, int epi_on) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < count8;
         i += static_cast<int64_t>(gridDim.x) * 256) {
        const float4 a = acc[2 * i], b = acc[2 * i + 1];
        uint32_t v[8] = {__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(a.z), __float_as_uint(a.w),
                         __float_as_uint(b.x), __float_as_uint(b.y), __float_as_uint(b.z), __float_as_uint(b.w)};
        if (epi_on) {
            const int64_t e0 = 8 * i;
            epilogue8(v, epi, e0 / c_out, c_out, static_cast<int>(e0 % c_out));
        }
        out[i] = make_uint4(pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                            pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                            pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                            pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
    }
}

// grid: one persistent CTA per SM, or fewer when the item count is known and smaller
// cooperative: every CTA resident at once (a fused stack waits across CTAs
// between layers), launched without programmatic dependent launch
template <int NTMAX, bool TM>
int launch_tc(const TcParams& p, int grid, cudaStream_t s, bool cooperative) {
    using Cfg = TcConfig<NTMAX>;
    static bool smem_set[kMaxDevices] = {};   // once per device
    int dev = 0;
    SPCONV_CHECK_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return SPCONV_ERR_UNSUPPORTED;
    if (!smem_set[dev]) {
        SPCONV_CHECK_CUDA(
            cudaFuncSetAttribute(k_tc_gemm<NTMAX, TM>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem));
        smem_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    if (cooperative) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    SPCONV_CHECK_CUDA(cudaLaunchKernelEx(&cfg, k_tc_gemm<NTMAX, TM>, p));
    count_launch();
    return SPCONV_OK;
}

template <bool TM>
int launch_tc_n(const TcParams& p, int grid, cudaStream_t s, bool cooperative = false) {
    if (p.n_tile > 128) return launch_tc<256, TM>(p, grid, s, cooperative);
    if (p.n_tile > 64) return launch_tc<128, TM>(p, grid, s, cooperative);
    return launch_tc<64, TM>(p, grid, s, cooperative);
}

}  // namespace

// Output channels per tensor-core item: c_out split into ceil(c_out/256)
// equal blocks, each a multiple of 16.
int tc_tile_n(int32_t c_out) {
    if (c_out <= 0 || c_out % 16 != 0) return 0;
    const int nb = (c_out + 255) / 256;
    if (c_out % nb != 0 || (c_out / nb) % 16 != 0) return 0;
    return c_out / nb;
}

bool tc_supported(int32_t c_in, int32_t c_out) {
    return c_in > 0 && c_in % 8 == 0 && c_in <= 65536 && tc_tile_n(c_out) > 0;
}

size_t tc_pack_bytes(int32_t c_in, int32_t c_out, int32_t taps) {
    const int nt = tc_tile_n(c_out);
    const int kcs = (c_in + BK - 1) / BK;
    return static_cast<size_t>(c_out / nt) * taps * kcs * nt * 128;
}

int tc_pack_weights(const void* w, int32_t c_in, int32_t c_out, int32_t taps, void* dst, cudaStream_t s) {
    const int nt = tc_tile_n(c_out);
    const int kcs = (c_in + BK - 1) / BK;
    const int n_nb = c_out / nt;
    const int64_t total = static_cast<int64_t>(n_nb) * taps * kcs * nt * 8;
    const int threads = 256;
    const int64_t blocks64 = (total + threads - 1) / threads;
    const unsigned blocks = static_cast<unsigned>(blocks64 < 65535 * 16 ? blocks64 : 65535 * 16);
    k_pack_weights<<<blocks, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(w), c_in, c_out, taps, nt, kcs,
                                              n_nb, static_cast<uint4*>(dst));
    count_launch();
    return cuda_status(cudaGetLastError());
}

namespace {

// The launch parameters shared by every forward of map h (one layer, the
// plain store mode, all tiles).
TcParams base_params(const MapHandle* h, const void* feats, int32_t c_in, int32_t c_out) {
    TcParams p = {};
    p.feats = static_cast<const __nv_bfloat16*>(feats);
    p.gtab = h->gtab;
    p.tile_union = h->tile_union;
    p.tile_order = h->tile_order;
    p.perm = h->perm;
    p.tap_off = h->tap_off;
    p.in_rows = h->in_rows;
    p.out_rows = h->out_rows;
    p.acc = nullptr;
    p.status = h->status;
    p.n = h->n;
    p.n_pad = h->n_pad;
    p.n_in = h->n_in >= 0 ? h->n_in : h->n;
    p.c_in = c_in;
    p.c_out = c_out;
    p.k_chunks = (c_in + BK - 1) / BK;
    p.n_tile = tc_tile_n(c_out);
    p.n_nb = c_out / p.n_tile;
    p.k0 = 0;
    p.taps_w = h->taps;
    p.mode = kModeStore;
    p.ws = nullptr;
    p.tiles_dev = nullptr;
    p.n_layers = 1;
    p.layer_done = nullptr;
    return p;
}

}  // namespace

int tc_forward(MapHandle* h, const void* feats, const void* wpack, void* out, int32_t c_in,
               int32_t c_out, const Epilogue& epi, cudaStream_t s) {
    if (h->n == 0) return SPCONV_OK;
    TcParams p = base_params(h, feats, c_in, c_out);
    p.wpacks[0] = static_cast<const uint8_t*>(wpack);
    p.outs[0] = static_cast<__nv_bfloat16*>(out);
    p.epis[0] = epi;
    p.epi_ons[0] = epi.active() ? 1 : 0;
    const int64_t items = h->n_tiles * p.n_nb;
    if (items > 0x7FFFFFFF) return SPCONV_ERR_UNSUPPORTED;
    p.n_items = static_cast<int32_t>(items);
    const int sms = num_sms();
    const int grid = p.n_items < sms ? p.n_items : sms;
    auto ensure_acc = [&](size_t need) -> int {
        if (h->acc_bytes >= need) return SPCONV_OK;
        if (h->acc) cudaFreeAsync(h->acc, s);
        h->acc = nullptr;
        h->acc_bytes = 0;
        if (pool_alloc(&h->acc, need, s) != cudaSuccess) {
            cudaGetLastError();
            h->acc = nullptr;
            return SPCONV_ERR_OOM;
        }
        h->acc_bytes = need;
        return SPCONV_OK;
    };
    if (h->groups > 1) {
        // offset groups ("Offset-group partitioning", "Sparse convolution in FP32"):
        // one tile-union pass per group over that group's row order, the
        // partial sums carried in fp32 between the passes, one rounding at the end
        const size_t ws_bytes = static_cast<size_t>(h->n) * c_out * sizeof(float);
        SPCONV_CHECK(ensure_acc(ws_bytes));
        p.ws = static_cast<float*>(h->acc);
        SPCONV_CHECK_CUDA(cudaMemsetAsync(p.ws, 0, ws_bytes, s));
        const int centre = (h->groups - 1) / 2;   // the group of the centre tap
        for (int j = 0; j < h->groups; ++j) {
            const int g = j < centre ? j : (j + 1 < h->groups ? j + 1 : centre);
            p.k0 = g * h->group_taps;
            p.gtab = h->gtab + static_cast<int64_t>(p.k0) * h->n_pad;
            p.tile_union = h->tile_union + g * h->n_tiles;
            p.tile_order = h->tile_order + g * h->n_tiles;
            p.perm = h->perm + g * h->n;
            p.mode = g == centre ? kModeWsFinish : kModeWsAdd;
            p.tiles_dev = g == centre ? nullptr : h->tile_nonempty + g;
            SPCONV_CHECK(launch_tc_n<false>(p, grid, s));
        }
        return SPCONV_OK;
    }
    if (h->gemm != SPCONV_GEMM_TAP_MAJOR) return launch_tc_n<false>(p, grid, s);

    // tap-major: zeroed fp32 sums, the GEMM adds every pair's product, one rounding pass
    // (at most 27n pairs: the item count fits in int32 when 27n/128 * n_nb does)
    if (static_cast<int64_t>(kTaps) * h->n / BM * p.n_nb > 0x7FFFFFFF) return SPCONV_ERR_UNSUPPORTED;
    const size_t need = static_cast<size_t>(h->n) * c_out * sizeof(float);
    SPCONV_CHECK(ensure_acc(need));
    p.acc = static_cast<float*>(h->acc);
    SPCONV_CHECK_CUDA(cudaMemsetAsync(p.acc, 0, need, s));
    SPCONV_CHECK(launch_tc_n<true>(p, sms, s));
    const int64_t count8 = static_cast<int64_t>(h->n) * c_out / 8;
    const int64_t blocks = (count8 + 255) / 256;
    k_acc_to_bf16<<<static_cast<unsigned>(blocks < 8 * sms ? blocks : 8 * sms), 256, 0, s>>>(
        reinterpret_cast<const float4*>(p.acc), reinterpret_cast<uint4*>(out), count8, c_out, epi, p.epi_ons[0]);
    count_launch();
    return cuda_status(cudaGetLastError());
}

int tc_forward_layers(MapHandle* h, const void* feats, const void* const* wpacks, void* const* outs,
                      const Epilogue* epis, int32_t n_layers, int32_t c_in, int32_t c_out, cudaStream_t s) {
    if (h->n == 0) return SPCONV_OK;
    if (n_layers < 1 || n_layers > kMaxFusedLayers) return SPCONV_ERR_INVALID_ARG;
    if (h->groups > 1 || h->gemm == SPCONV_GEMM_TAP_MAJOR) return SPCONV_ERR_UNSUPPORTED;
    TcParams p = base_params(h, feats, c_in, c_out);
    p.n_layers = n_layers;
    for (int l = 0; l < n_layers; ++l) {
        p.wpacks[l] = static_cast<const uint8_t*>(wpacks[l]);
        p.outs[l] = static_cast<__nv_bfloat16*>(outs[l]);
        p.epis[l] = epis[l];
        p.epi_ons[l] = epis[l].active() ? 1 : 0;
    }
    const int64_t items = h->n_tiles * p.n_nb;
    if (items > 0x7FFFFFFF) return SPCONV_ERR_UNSUPPORTED;
    p.n_items = static_cast<int32_t>(items);
    const int sms = num_sms();
    const int grid = p.n_items < sms ? p.n_items : sms;
    if (n_layers == 1) return launch_tc_n<false>(p, grid, s);
    if (!h->layer_done) {
        void* buf = nullptr;
        if (pool_alloc(&buf, kMaxFusedLayers * sizeof(int32_t), s) != cudaSuccess) {
            cudaGetLastError();
            return SPCONV_ERR_OOM;
        }
        h->layer_done = static_cast<int32_t*>(buf);
    }
    SPCONV_CHECK_CUDA(cudaMemsetAsync(h->layer_done, 0, kMaxFusedLayers * sizeof(int32_t), s));
    p.layer_done = h->layer_done;
    // one CTA per SM, all resident together: the kernel's shared memory admits one per SM
    return launch_tc_n<false>(p, grid, s, true);
}

}  // namespace spconv

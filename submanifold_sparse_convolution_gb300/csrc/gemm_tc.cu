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
//   warps 0-3   epilogue: tcgen05.ld of the accumulator, bf16 convert, store
//   warp 4      TMEM allocation + MMA issue (one thread)
//   warps 5..   one producer warp per pipeline stage: cp.async 16-byte row
//               gathers of A into the 128-byte-swizzled layout (a row
//               without the neighbour is written as zeros, with no memory
//               request), plus one bulk async copy of the pre-packed weight
//               tile B
// The accumulator is double-buffered in TMEM so the epilogue of one tile
// overlaps the main loop of the next.
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
constexpr int kProdWarp0 = 5;
constexpr int kStageA = BM * BK * 2;   // 16 KB

struct TcParams {
    const __nv_bfloat16* feats;   // [n][c_in]
    const uint8_t* wpack;         // packed weights, see k_pack_weights
    __nv_bfloat16* out;           // [n][c_out]
    const int32_t* gtab;          // [27][n_pad]
    const uint32_t* tile_union;   // [n_tiles]
    const int32_t* tile_order;    // [n_tiles]
    const int32_t* perm;          // [n_pad]
    int32_t* status;
    int64_t n, n_pad;
    int32_t n_items;              // n_tiles * n_nb
    int32_t c_in, c_out;
    int32_t k_chunks;             // ceil(c_in / 64)
    int32_t n_tile;               // output channels per item (multiple of 16, <= NTMAX)
    int32_t n_nb;                 // c_out / n_tile
};

template <int NTMAX>
struct TcConfig {
    static constexpr int kStageB = NTMAX * 128;
    static constexpr int kStage = kStageA + kStageB;
    static constexpr int kStages = (NTMAX == 256) ? 4 : (NTMAX == 128 ? 6 : 8);
    static constexpr int kThreads = 32 * (kProdWarp0 + kStages);
    static constexpr int kTmemCols = 2 * NTMAX < 32 ? 32 : 2 * NTMAX;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmem = kStages * kStage + 1024 + kBarBytes;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int NTMAX>
__global__ void __launch_bounds__(TcConfig<NTMAX>::kThreads, 1) k_tc_gemm(const TcParams p) {
    using Cfg = TcConfig<NTMAX>;
    constexpr int S = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStage);
    uint64_t* full = bars;             // [S]
    uint64_t* empty = bars + S;        // [S]
    uint64_t* acc_full = bars + 2 * S; // [2]
    uint64_t* acc_empty = acc_full + 2;// [2]
    uint64_t* exit_bar = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(exit_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 2);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], kEpiWarps);
        }
        ptx::mbar_init(exit_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(tmem_slot, Cfg::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t smem_base = ptx::smem_u32(smem);

    auto fail = [&]() {
        atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
    };
    // lane 0 waits, the warp follows its verdict
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        int ok = 1;
        if (lane == 0) ok = ptx::mbar_wait(bar, parity, abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        return ok != 0;
    };

    if (warp >= kProdWarp0) {
        // ---------------- producers: warp (kProdWarp0 + s) owns stage s
        const int slot = warp - kProdWarp0;
        const uint32_t a_smem = smem_base + slot * Cfg::kStage;
        const uint32_t b_smem = a_smem + kStageA;
        const uint32_t b_bytes = static_cast<uint32_t>(p.n_tile) * 128u;
        uint32_t f = 0;
        bool stop = false;
        for (int it = blockIdx.x; it < p.n_items && !stop; it += gridDim.x) {
            const int tile = p.tile_order[it / p.n_nb];
            const int nb = it % p.n_nb;
            uint32_t uni = p.tile_union[tile];
            while (uni && !stop) {
                const int k = __ffs(uni) - 1;
                uni &= uni - 1;
                const int32_t* g = p.gtab + static_cast<int64_t>(k) * p.n_pad + static_cast<int64_t>(tile) * BM;
                int32_t gr[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) gr[q] = g[lane + 32 * q];
                for (int kc = 0; kc < p.k_chunks; ++kc, ++f) {
                    if (static_cast<int>(f % S) != slot) continue;
                    const uint32_t u = f / S;
                    if (u > 0 && !warp_wait(&empty[slot], (u - 1) & 1)) {
                        if (lane == 0) fail();
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(&full[slot], b_bytes);
                        const uint8_t* src = p.wpack + (static_cast<int64_t>(nb * kTaps + k) * p.k_chunks + kc) * b_bytes;
                        ptx::bulk_copy_g2s(b_smem, src, b_bytes, &full[slot]);
                    }
                    const int chunk = lane & 7;
                    const int kcol = kc * BK + chunk * 8;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int row = 4 * i + (lane >> 3);
                        const int32_t src_row = __shfl_sync(0xFFFFFFFFu, gr[i >> 3], row & 31);
                        const uint32_t dst = a_smem + row * 128 + ((chunk ^ (row & 7)) << 4);
                        if (src_row >= 0 && kcol < p.c_in)
                            ptx::cp_async_16(dst, p.feats + static_cast<int64_t>(src_row) * p.c_in + kcol, 16u);
                        else
                            ptx::st_shared_zero16(dst);   // absent neighbour: no memory request
                    }
                    ptx::cp_async_commit();
                    ptx::cp_async_wait_all();
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&full[slot]);
                }
            }
        }
        ptx::cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(BM, static_cast<uint32_t>(p.n_tile));
            uint32_t f = 0;
            int local = 0;
            bool stop = false;
            for (int it = blockIdx.x; it < p.n_items && !stop; it += gridDim.x, ++local) {
                const int tile = p.tile_order[it / p.n_nb];
                const int buf = local & 1;
                const uint32_t v = static_cast<uint32_t>(local >> 1);
                if (v > 0 && !ptx::mbar_wait(&acc_empty[buf], (v - 1) & 1, abort_flag)) {
                    fail();
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * NTMAX);
                uint32_t uni = p.tile_union[tile];
                bool first = true;
                while (uni && !stop) {
                    uni &= uni - 1;
                    for (int kc = 0; kc < p.k_chunks; ++kc, ++f) {
                        const int slot = static_cast<int>(f % S);
                        if (!ptx::mbar_wait(&full[slot], (f / S) & 1, abort_flag)) {
                            fail();
                            stop = true;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t a_addr = smem_base + slot * Cfg::kStage;
                        const uint32_t b_addr = a_addr + kStageA;
#pragma unroll
                        for (int j = 0; j < BK / 16; ++j) {
                            ptx::mma_bf16(d_tmem, ptx::sdesc_k128(a_addr + 32 * j),
                                          ptx::sdesc_k128(b_addr + 32 * j), idesc,
                                          (first && j == 0) ? 0u : 1u);
                        }
                        first = false;
                        ptx::mma_commit(&empty[slot]);
                    }
                }
                if (!stop) ptx::mma_commit(&acc_full[buf]);
            }
            // all MMAs issued by this thread have completed once exit_bar flips
            ptx::mma_commit(exit_bar);
            if (!ptx::mbar_wait(exit_bar, 0, nullptr)) atomicOr(p.status, kStatusTimeout);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warp w reads TMEM lanes [32w, 32w + 32)
        int local = 0;
        for (int it = blockIdx.x; it < p.n_items; it += gridDim.x, ++local) {
            const int tile = p.tile_order[it / p.n_nb];
            const int nb = it % p.n_nb;
            const int buf = local & 1;
            const uint32_t v = static_cast<uint32_t>(local >> 1);
            if (!warp_wait(&acc_full[buf], v & 1)) {
                if (lane == 0) fail();
                break;
            }
            ptx::tc_fence_after();
            const int64_t s = static_cast<int64_t>(tile) * BM + warp * 32 + lane;
            const int32_t orig = s < p.n ? p.perm[s] : -1;
            __nv_bfloat16* dst_row = orig >= 0 ? p.out + static_cast<int64_t>(orig) * p.c_out + nb * p.n_tile : nullptr;
            const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(buf * NTMAX);
            for (int c = 0; c < p.n_tile; c += 16) {
                uint32_t r[16];
                ptx::tmem_ld_32x32b_x16(t_addr + c, r);
                ptx::tmem_ld_wait();
                if (dst_row) {
                    uint4 lo, hi;
                    lo.x = pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1]));
                    lo.y = pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3]));
                    lo.z = pack_bf16x2(__uint_as_float(r[4]), __uint_as_float(r[5]));
                    lo.w = pack_bf16x2(__uint_as_float(r[6]), __uint_as_float(r[7]));
                    hi.x = pack_bf16x2(__uint_as_float(r[8]), __uint_as_float(r[9]));
                    hi.y = pack_bf16x2(__uint_as_float(r[10]), __uint_as_float(r[11]));
                    hi.z = pack_bf16x2(__uint_as_float(r[12]), __uint_as_float(r[13]));
                    hi.w = pack_bf16x2(__uint_as_float(r[14]), __uint_as_float(r[15]));
                    uint4* d = reinterpret_cast<uint4*>(dst_row + c);
                    d[0] = lo;
                    d[1] = hi;
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
}

// Packed weight image: for each (output block nb, tap k, 64-channel input
// chunk kc) a block of n_tile rows x 128 bytes; row n holds
// W[k][kc*64 .. kc*64+63][nb*n_tile + n] (zero past c_in), its 16-byte chunk c
// stored at chunk position c ^ (n & 7) -- the K-major 128-byte-swizzled
// shared-memory layout that the MMA reads directly after one bulk copy.
__global__ void k_pack_weights(const __nv_bfloat16* __restrict__ w, int c_in, int c_out, int n_tile,
                               int k_chunks, int n_nb, uint4* __restrict__ dst) {
    const int64_t total = static_cast<int64_t>(n_nb) * kTaps * k_chunks * n_tile * 8;
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
        const int k = static_cast<int>(q % kTaps);
        const int nb = static_cast<int>(q / kTaps);
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
        const int64_t blk = (static_cast<int64_t>(nb) * kTaps + k) * k_chunks + kc;
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

template <int NTMAX>
int launch_tc(const TcParams& p, cudaStream_t s) {
    using Cfg = TcConfig<NTMAX>;
    SPCONV_CHECK_CUDA(cudaFuncSetAttribute(k_tc_gemm<NTMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem));
    const int grid = p.n_items < num_sms() ? p.n_items : num_sms();
    k_tc_gemm<NTMAX><<<grid, Cfg::kThreads, Cfg::kSmem, s>>>(p);
    count_launch();
    return cuda_status(cudaGetLastError());
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

size_t tc_pack_bytes(int32_t c_in, int32_t c_out) {
    const int nt = tc_tile_n(c_out);
    const int kcs = (c_in + BK - 1) / BK;
    return static_cast<size_t>(c_out / nt) * kTaps * kcs * nt * 128;
}

int tc_pack_weights(const void* w, int32_t c_in, int32_t c_out, void* dst, cudaStream_t s) {
    const int nt = tc_tile_n(c_out);
    const int kcs = (c_in + BK - 1) / BK;
    const int n_nb = c_out / nt;
    const int64_t total = static_cast<int64_t>(n_nb) * kTaps * kcs * nt * 8;
    const int threads = 256;
    const int64_t blocks64 = (total + threads - 1) / threads;
    const unsigned blocks = static_cast<unsigned>(blocks64 < 65535 * 16 ? blocks64 : 65535 * 16);
    k_pack_weights<<<blocks, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(w), c_in, c_out, nt, kcs,
                                              n_nb, static_cast<uint4*>(dst));
    count_launch();
    return cuda_status(cudaGetLastError());
}

int tc_forward(const MapHandle* h, const void* feats, const void* wpack, void* out, int32_t c_in,
               int32_t c_out, cudaStream_t s) {
    if (h->n == 0) return SPCONV_OK;
    TcParams p;
    p.feats = static_cast<const __nv_bfloat16*>(feats);
    p.wpack = static_cast<const uint8_t*>(wpack);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.gtab = h->gtab;
    p.tile_union = h->tile_union;
    p.tile_order = h->tile_order;
    p.perm = h->perm;
    p.status = h->status;
    p.n = h->n;
    p.n_pad = h->n_pad;
    p.c_in = c_in;
    p.c_out = c_out;
    p.k_chunks = (c_in + BK - 1) / BK;
    p.n_tile = tc_tile_n(c_out);
    p.n_nb = c_out / p.n_tile;
    const int64_t items = h->n_tiles * p.n_nb;
    if (items > 0x7FFFFFFF) return SPCONV_ERR_UNSUPPORTED;
    p.n_items = static_cast<int32_t>(items);
    if (p.n_tile > 128) return launch_tc<256>(p, s);
    if (p.n_tile > 64) return launch_tc<128>(p, s);
    return launch_tc<64>(p, s);
}

}  // namespace spconv

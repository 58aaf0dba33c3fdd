// SIMT path: fp32 exact mode and bf16 for channel counts the tensor-core path
// does not take (C = 1, C not a multiple of 8 or 16).
//
// One thread per (row, group of VEC output channels), rows visited in the
// mask-sorted order so that a warp's rows share their taps.  Each output
// element is a plain FMA chain in fp32 over taps 0..V-1 and input channels in
// ascending order, skipping absent taps ("Sparse convolution in FP32":
// weights read as [offset][input][output] with consecutive output channels per
// thread), so the result does not depend on the launch shape.  The optional
// epilogue (scale, bias, residual, ReLU) is applied to the fp32 sum before
// the store.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace spconv {
namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <typename T, int VEC>
__global__ void __launch_bounds__(256) k_simt(const T* __restrict__ feats, const T* __restrict__ w,
                                              T* __restrict__ out, const int32_t* __restrict__ perm,
                                              const int32_t* __restrict__ nbr, int taps, int stride,
                                              int64_t n, int c_in, int c_out, Epilogue epi) {
    const int groups = (c_out + VEC - 1) / VEC;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t s = idx / groups;
    if (s >= n) return;
    const int g = static_cast<int>(idx % groups);
    const int o0 = g * VEC;
    const int32_t r = perm[s];
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.0f;
    const int32_t* nrow = nbr + static_cast<int64_t>(r) * stride;
    for (int k = 0; k < taps; ++k) {
        const int32_t j = nrow[k];
        if (j < 0) continue;
        const T* f = feats + static_cast<int64_t>(j) * c_in;
        const T* wk = w + static_cast<int64_t>(k) * c_in * c_out + o0;
        for (int c = 0; c < c_in; ++c) {
            const float fv = to_f(f[c]);
            const T* wr = wk + static_cast<int64_t>(c) * c_out;
#pragma unroll
            for (int v = 0; v < VEC; ++v)
                if (o0 + v < c_out) acc[v] = fmaf(fv, to_f(wr[v]), acc[v]);
        }
    }
    T* dst = out + static_cast<int64_t>(r) * c_out + o0;
    const T* res = epi.residual ? static_cast<const T*>(epi.residual) + static_cast<int64_t>(r) * c_out + o0 : nullptr;
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        if (o0 + v >= c_out) continue;
        float y = acc[v];
        if (epi.scale) y *= epi.scale[o0 + v];
        if (epi.bias) y += epi.bias[o0 + v];
        if (res) y += to_f(res[v]);
        if (epi.relu) y = fmaxf(y, 0.0f);
        dst[v] = from_f<T>(y);
    }
}

// ---------------------------------------------------------------------------
// fp32 exact mode, tiled: one CTA per (128-row tile of the mask-sorted order,
// 64 output channels).  It visits the taps of the tile's mask union in
// ascending order, 32 input channels at a time ("Neighbour masks and sorted
// rows": rows of a tile share their taps); for each (tap, channel chunk) the
// weight slab W[k][c0 .. c0+31][o0 .. o0+63] and the tile's 128 gathered
// input rows (through the map's gather table; a row without the tap is
// zeros) are staged in shared memory by cp.async, double-buffered, and each
// thread accumulates an 8 x 8 block of outputs in registers.  A row without
// the tap adds fma(0, w, acc) = acc, so every output element is the same FMA
// chain as in k_simt (taps ascending, channels ascending, absent taps
// skipped) and the result has the same bits.
// ---------------------------------------------------------------------------
constexpr int kFRows = kTileRows;     // rows per tile
constexpr int kFCols = 64;            // output channels per CTA
constexpr int kFK = 32;               // input channels per stage (3 CTAs per SM fit; 64 admitted 2)
constexpr int kFThreads = 128;        // 16 row groups x 8 column groups
constexpr int kFRowStride = kFK + 4;  // floats per staged feature row (16-byte aligned, conflict-free)
constexpr int kFStageFloats = kFRows * kFRowStride + kFK * kFCols;
constexpr int kFSmem = 2 * kFStageFloats * 4;

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

__global__ void __launch_bounds__(kFThreads, 3) k_fp32_tiled(const float* __restrict__ feats,
                                                             const float* __restrict__ w,
                                                             float* __restrict__ out,
                                                             const int32_t* __restrict__ perm,
                                                             const int32_t* __restrict__ gtab,
                                                             const uint32_t* __restrict__ tile_union,
                                                             const int32_t* __restrict__ tile_order,
                                                             int64_t n, int64_t n_pad, int64_t n_in, int c_in,
                                                             int c_out, Epilogue epi, int32_t* __restrict__ status) {
    extern __shared__ float fsm[];
    const int t = threadIdx.x;
    const int cg = t & 7, rg = t >> 3;        // columns 8 cg .. + 7; rows rg + 16 i
    // CTAs start in blockIdx order: taking the tiles by descending union size
    // (their cost) puts the cheapest last, where they fill the final wave
    const int64_t tile = tile_order ? tile_order[blockIdx.x] : blockIdx.x;
    const int o0 = blockIdx.y * kFCols;
    const uint32_t uni = tile_union[tile];
    const int kcs = (c_in + kFK - 1) / kFK;
    const int n_stages = __popc(uni) * kcs;
    // stage st: its weight slab and the tile's gathered rows (thread t loads
    // rows t / (kFK / 4) + q kFThreads / (kFK / 4), 16-byte chunk t % (kFK / 4))
    constexpr int kCh = kFK / 4;                           // 16-byte chunks of a staged row
    constexpr int kRowsPer = kFRows / (kFThreads / kCh);   // rows each thread stages
    // st-th (tap, chunk) of the tile: the tap is the (st / kcs)-th set bit of the union
    auto tap_of = [&](int st) {
        uint32_t u = uni;
        for (int j = st / kcs; j > 0; --j) u &= u - 1;
        return __ffs(u) - 1;
    };
    // the source rows of stage st for this thread's staged rows, loaded a stage
    // ahead of their copies so that their latency hides behind the compute
    auto load_idx = [&](int st, int32_t (&jr)[kRowsPer]) {
        const int k = tap_of(st);
#pragma unroll
        for (int q = 0; q < kRowsPer; ++q)
            jr[q] = __ldg(gtab + static_cast<int64_t>(k) * n_pad + tile * kFRows + t / kCh + q * (kFThreads / kCh));
    };
    auto stage = [&](int st, float* buf, const int32_t (&jr)[kRowsPer]) {
        const int k = tap_of(st);
        const int c0 = (st % kcs) * kFK;
        float* fs = buf;
        float* ws = buf + kFRows * kFRowStride;
        // weights: kFK rows of kFCols floats, 16 chunks of 16 bytes each
        for (int i = t; i < kFK * (kFCols / 4); i += kFThreads) {
            const int c = i / (kFCols / 4), q = i % (kFCols / 4);
            float* d = ws + c * kFCols + 4 * q;
            if (c0 + c < c_in)
                cp_async16(d, w + (static_cast<int64_t>(k) * c_in + c0 + c) * c_out + o0 + 4 * q);
            else
                *reinterpret_cast<float4*>(d) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // gathered rows: 128 rows of kFK floats (kFK / 4 16-byte chunks per row)
        const int ch = t % kCh;
#pragma unroll
        for (int q = 0; q < kRowsPer; ++q) {
            const int r = t / kCh + q * (kFThreads / kCh);
            const int32_t j = jr[q];
            float* d = fs + r * kFRowStride + 4 * ch;
            if (j >= 0 && j < n_in && c0 + 4 * ch < c_in)
                cp_async16(d, feats + static_cast<int64_t>(j) * c_in + c0 + 4 * ch);
            else
                *reinterpret_cast<float4*>(d) = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j >= n_in) atomicOr(status, kStatusInternal);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[i][v] = 0.0f;
    int32_t jn[kRowsPer];   // the source rows of the next stage to issue
    if (n_stages > 0) {
        load_idx(0, jn);
        stage(0, fsm, jn);
    }
    if (n_stages > 1) load_idx(1, jn);
    for (int st = 0; st < n_stages; ++st) {
        float* buf = fsm + (st & 1) * kFStageFloats;
        if (st + 1 < n_stages) {
            stage(st + 1, fsm + ((st + 1) & 1) * kFStageFloats, jn);
            if (st + 2 < n_stages) load_idx(st + 2, jn);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        const float* fs = buf;
        const float* ws = buf + kFRows * kFRowStride;
        const int cmax = c_in - (st % kcs) * kFK < kFK ? c_in - (st % kcs) * kFK : kFK;
        // channels c .. c + 3 of the stage into the 8 x 8 block (cc < lim of them)
        auto step4 = [&](int c, int lim) {
            float4 f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = *reinterpret_cast<const float4*>(fs + (rg + 16 * i) * kFRowStride + c);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                if (cc >= lim) break;
                const float4 w0 = *reinterpret_cast<const float4*>(ws + (c + cc) * kFCols + 8 * cg);
                const float4 w1 = *reinterpret_cast<const float4*>(ws + (c + cc) * kFCols + 8 * cg + 4);
                const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float fv = cc == 0 ? f[i].x : cc == 1 ? f[i].y : cc == 2 ? f[i].z : f[i].w;
#pragma unroll
                    for (int v = 0; v < 8; ++v) acc[i][v] = fmaf(fv, wv[v], acc[i][v]);
                }
            }
        };
        if (cmax == kFK) {
            // a full stage: every offset is a compile-time constant
#pragma unroll
            for (int c = 0; c < kFK; c += 4) step4(c, 4);
        } else {
            for (int c = 0; c < cmax; c += 4) step4(c, cmax - c);
        }
        __syncthreads();   // the buffer is refilled by the next iteration's stage
    }
    // store: thread owns rows rg + 16 i, columns o0 + 8 cg .. + 7
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t s = tile * kFRows + rg + 16 * i;
        const int32_t r = s < n ? perm[s] : -1;
        if (r < 0) continue;
        const int o = o0 + 8 * cg;
        float y[8];
#pragma unroll
        for (int v = 0; v < 8; ++v) y[v] = acc[i][v];
        if (epi.scale || epi.bias || epi.residual || epi.relu) {
            const float* res = epi.residual ? static_cast<const float*>(epi.residual) + static_cast<int64_t>(r) * c_out + o
                                            : nullptr;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                if (epi.scale) y[v] *= epi.scale[o + v];
                if (epi.bias) y[v] += epi.bias[o + v];
                if (res) y[v] += res[v];
                if (epi.relu) y[v] = fmaxf(y[v], 0.0f);
            }
        }
        float4* d = reinterpret_cast<float4*>(out + static_cast<int64_t>(r) * c_out + o);
        d[0] = make_float4(y[0], y[1], y[2], y[3]);
        d[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
}

int launch_fp32_tiled(const MapHandle* h, const void* feats, const void* w, void* out, int32_t c_in,
                      int32_t c_out, const Epilogue& epi, cudaStream_t s) {
    static bool smem_set[kMaxDevices] = {};
    int dev = 0;
    SPCONV_CHECK_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return SPCONV_ERR_UNSUPPORTED;
    if (!smem_set[dev]) {
        SPCONV_CHECK_CUDA(cudaFuncSetAttribute(k_fp32_tiled, cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmem));
        smem_set[dev] = true;
    }
    if (h->n_tiles > 0x7FFFFFFF) return SPCONV_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(h->n_tiles), static_cast<unsigned>(c_out / kFCols));
    k_fp32_tiled<<<grid, kFThreads, kFSmem, s>>>(
        static_cast<const float*>(feats), static_cast<const float*>(w), static_cast<float*>(out), h->perm, h->gtab,
        h->tile_union, h->tile_order, h->n, h->n_pad, h->n_in >= 0 ? h->n_in : h->n, c_in, c_out, epi, h->status);
    count_launch();
    return cuda_status(cudaGetLastError());
}

bool fp32_tiled_ok(const MapHandle* h, const void* feats, const void* w, const void* out, int32_t c_in,
                   int32_t c_out, const Epilogue& epi) {
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    return h->groups == 1 && c_in % 4 == 0 && c_out % kFCols == 0 && al(feats) && al(w) && al(out) &&
           al(epi.scale) && al(epi.bias) && al(epi.residual);
}

template <typename T>
int launch(const MapHandle* h, const void* feats, const void* w, void* out, int32_t c_in,
           int32_t c_out, const Epilogue& epi, cudaStream_t s) {
    const int vec = c_out % 4 == 0 ? 4 : 1;
    const int64_t groups = (c_out + vec - 1) / vec;
    const int64_t threads = h->n * groups;
    const int64_t blocks = (threads + 255) / 256;
    if (blocks > 0x7FFFFFFF) return SPCONV_ERR_UNSUPPORTED;
    if (vec == 4)
        k_simt<T, 4><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            static_cast<const T*>(feats), static_cast<const T*>(w), static_cast<T*>(out), h->perm, h->nbr,
            h->taps, h->nbr_stride, h->n, c_in, c_out, epi);
    else
        k_simt<T, 1><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
            static_cast<const T*>(feats), static_cast<const T*>(w), static_cast<T*>(out), h->perm, h->nbr,
            h->taps, h->nbr_stride, h->n, c_in, c_out, epi);
    count_launch();
    return cuda_status(cudaGetLastError());
}

}  // namespace

int simt_forward(const MapHandle* h, const void* feats, const void* w, void* out, int32_t c_in,
                 int32_t c_out, int32_t dtype, const Epilogue& epi, cudaStream_t s) {
    if (h->n == 0) return SPCONV_OK;
    if (dtype == SPCONV_FP32) {
        if (fp32_tiled_ok(h, feats, w, out, c_in, c_out, epi))
            return launch_fp32_tiled(h, feats, w, out, c_in, c_out, epi, s);
        return launch<float>(h, feats, w, out, c_in, c_out, epi, s);
    }
    return launch<__nv_bfloat16>(h, feats, w, out, c_in, c_out, epi, s);
}

}  // namespace spconv

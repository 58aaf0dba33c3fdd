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
    if (dtype == SPCONV_FP32) return launch<float>(h, feats, w, out, c_in, c_out, epi, s);
    return launch<__nv_bfloat16>(h, feats, w, out, c_in, c_out, epi, s);
}

}  // namespace spconv

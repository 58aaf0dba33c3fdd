// C ABI of libspconv (declared in include/spconv.h): argument checks, handle
// lifetime, dispatch between the tensor-core and SIMT paths.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "common.cuh"

namespace spconv {

namespace {
thread_local int g_launches = 0;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

int read_status(const MapHandle* h) {
    int32_t st = 0;
    SPCONV_CHECK_CUDA(cudaStreamSynchronize(h->stream));
    SPCONV_CHECK_CUDA(cudaMemcpy(&st, h->status, sizeof(st), cudaMemcpyDeviceToHost));
    return status_from_flags(st);
}

int check_forward_args(const MapHandle* h, const void* feats, const void* out, int32_t c_in,
                       int32_t c_out, int32_t dtype) {
    if (!h) return SPCONV_ERR_INVALID_ARG;
    if (dtype != SPCONV_BF16 && dtype != SPCONV_FP32) return SPCONV_ERR_INVALID_ARG;
    if (c_in < 1 || c_out < 1 || c_in > 65536 || c_out > 65536) return SPCONV_ERR_INVALID_ARG;
    if (h->n == 0) return SPCONV_OK;
    if (!feats || !out) return SPCONV_ERR_INVALID_ARG;
    const size_t es = dtype == SPCONV_FP32 ? 4 : 2;
    if (!aligned(feats, es) || !aligned(out, es)) return SPCONV_ERR_INVALID_ARG;
    const int64_t n_in = h->n_in >= 0 ? h->n_in : h->n;
    if (overlaps(feats, static_cast<size_t>(n_in) * c_in * es, out, static_cast<size_t>(h->n) * c_out * es))
        return SPCONV_ERR_ALIAS;
    return SPCONV_OK;
}

// Validates an epilogue against the forward's output and fills *e.
int check_epilogue(const MapHandle* h, const spconv_epilogue_t* epi, const void* out, int32_t c_out,
                   int32_t dtype, Epilogue* e) {
    *e = Epilogue();
    if (!epi) return SPCONV_OK;
    if (epi->relu != 0 && epi->relu != 1) return SPCONV_ERR_INVALID_ARG;
    if (!aligned(epi->scale_dev, 16) || !aligned(epi->bias_dev, 16) || !aligned(epi->residual_dev, 16))
        return SPCONV_ERR_INVALID_ARG;
    if (epi->residual_dev && epi->residual_dev != out) {
        const size_t bytes = static_cast<size_t>(h->n) * c_out * (dtype == SPCONV_FP32 ? 4 : 2);
        if (overlaps(epi->residual_dev, bytes, out, bytes)) return SPCONV_ERR_ALIAS;
    }
    e->scale = epi->scale_dev;
    e->bias = epi->bias_dev;
    e->residual = epi->residual_dev;
    e->relu = epi->relu;
    return SPCONV_OK;
}

bool use_tensor_path(int32_t c_in, int32_t c_out, int32_t dtype, const void* feats, const void* out) {
    return dtype == SPCONV_BF16 && tc_supported(c_in, c_out) && aligned(feats, 16) && aligned(out, 16);
}

}  // namespace

cudaError_t pool_alloc(void** p, size_t bytes, cudaStream_t s) {
    static cudaMemPool_t pools[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaMallocAsync(p, bytes, s);
    if (pools[dev] == nullptr) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = ~0ull;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        pools[dev] = pool;
    }
    return cudaMallocFromPoolAsync(p, bytes, pools[dev], s);
}

void count_launch(int n) { g_launches += n; }
void reset_launch_count() { g_launches = 0; }

}  // namespace spconv

using namespace spconv;

struct spconv_map_s : MapHandle {};
struct spconv_wpack_s : WPackHandle {};

extern "C" {

int spconv_build_map(const int32_t* coords_dev, int64_t n, const int32_t* spatial_shape,
                     int32_t batch_size, int32_t kernel_size, const spconv_options_t* opt,
                     void* stream, spconv_map_t* out_map) {
    reset_launch_count();
    if (!out_map) return SPCONV_ERR_INVALID_ARG;
    *out_map = nullptr;
    if (n < 0 || n >= (int64_t(1) << 30)) return SPCONV_ERR_INVALID_ARG;
    if (n > 0 && (!coords_dev || !aligned(coords_dev, 16))) return SPCONV_ERR_INVALID_ARG;
    if (kernel_size != 3 && kernel_size != 5) return SPCONV_ERR_UNSUPPORTED;
    if (batch_size < 0) return SPCONV_ERR_INVALID_ARG;
    if (opt) {
        if (opt->mapper < SPCONV_MAPPER_AUTO || opt->mapper > SPCONV_MAPPER_HASH) return SPCONV_ERR_INVALID_ARG;
        if (opt->bit_order != SPCONV_ORDER_CALIBRATED && opt->bit_order != SPCONV_ORDER_PLAIN)
            return SPCONV_ERR_INVALID_ARG;
        if (opt->dense_max_cells < 0) return SPCONV_ERR_INVALID_ARG;
        if (opt->pipeline < SPCONV_PIPELINE_AUTO || opt->pipeline > SPCONV_PIPELINE_WIDE) return SPCONV_ERR_INVALID_ARG;
        if (opt->gemm < SPCONV_GEMM_AUTO || opt->gemm > SPCONV_GEMM_TAP_MAJOR) return SPCONV_ERR_INVALID_ARG;
    }
    // offset groups: one (K = 3 only: 27 taps fit one mask) or K (the taps of each dx)
    int32_t groups = (opt && opt->groups > 0) ? opt->groups : (kernel_size == 3 ? 1 : kernel_size);
    if (opt && opt->groups < 0) return SPCONV_ERR_INVALID_ARG;
    if (groups != kernel_size && !(groups == 1 && kernel_size == 3)) return SPCONV_ERR_UNSUPPORTED;
    if (groups > 1 && opt) {
        if (opt->pipeline != SPCONV_PIPELINE_AUTO && opt->pipeline != SPCONV_PIPELINE_MULTI)
            return SPCONV_ERR_UNSUPPORTED;
        if (opt->gemm == SPCONV_GEMM_TAP_MAJOR) return SPCONV_ERR_UNSUPPORTED;
    }
    int32_t shape[3] = {1, 1, 1};
    int32_t batch = batch_size;
    if (spatial_shape) {
        for (int a = 0; a < 3; ++a) {
            if (spatial_shape[a] < 1 || spatial_shape[a] >= (1 << 30)) return SPCONV_ERR_INVALID_ARG;
            shape[a] = spatial_shape[a];
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!spatial_shape || batch <= 0) {
        int32_t dshape[3], dbatch = 1;
        SPCONV_CHECK(derive_shape(coords_dev, n, s, dshape, &dbatch));
        if (!spatial_shape) std::memcpy(shape, dshape, sizeof(shape));
        if (batch <= 0) batch = dbatch;
    }
    spconv_map_s* h = new (std::nothrow) spconv_map_s();
    if (!h) return SPCONV_ERR_OOM;
    h->stream = s;
    cudaGetDevice(&h->device);
    h->n = n;
    std::memcpy(h->shape, shape, sizeof(shape));
    h->batch = batch;
    h->kernel_size = kernel_size;
    h->taps = kernel_size * kernel_size * kernel_size;
    h->groups = groups;
    const int rc = build_map_impl(h, coords_dev, opt);
    if (rc != SPCONV_OK) {
        if (h->arena) cudaFreeAsync(h->arena, s);
        delete h;
        return rc;
    }
    *out_map = h;
    return SPCONV_OK;
}

int spconv_build_map_strided(const int32_t* coords_dev, int64_t n, const int32_t* spatial_shape,
                             int32_t batch_size, int32_t kernel_size, int32_t stride, const spconv_options_t* opt,
                             void* stream, spconv_map_t* out_map) {
    reset_launch_count();
    if (!out_map) return SPCONV_ERR_INVALID_ARG;
    *out_map = nullptr;
    if (n < 0 || n >= (int64_t(1) << 27)) return SPCONV_ERR_INVALID_ARG;   // 8 n candidates in int32 ranks
    if (n > 0 && (!coords_dev || !aligned(coords_dev, 16))) return SPCONV_ERR_INVALID_ARG;
    if (kernel_size != 3 || stride != 2) return SPCONV_ERR_UNSUPPORTED;
    if (batch_size < 0) return SPCONV_ERR_INVALID_ARG;
    if (opt) {
        if (opt->mapper != SPCONV_MAPPER_AUTO && opt->mapper != SPCONV_MAPPER_HASH) return SPCONV_ERR_UNSUPPORTED;
        if (opt->bit_order != SPCONV_ORDER_CALIBRATED && opt->bit_order != SPCONV_ORDER_PLAIN)
            return SPCONV_ERR_INVALID_ARG;
        if (opt->pipeline != SPCONV_PIPELINE_AUTO && opt->pipeline != SPCONV_PIPELINE_MULTI)
            return SPCONV_ERR_UNSUPPORTED;
        if (opt->gemm == SPCONV_GEMM_TAP_MAJOR) return SPCONV_ERR_UNSUPPORTED;
        if (opt->gemm < SPCONV_GEMM_AUTO || opt->gemm > SPCONV_GEMM_TAP_MAJOR) return SPCONV_ERR_INVALID_ARG;
        if (opt->groups != 0 && opt->groups != 1) return SPCONV_ERR_UNSUPPORTED;
    }
    int32_t shape[3] = {1, 1, 1};
    int32_t batch = batch_size;
    if (spatial_shape) {
        for (int a = 0; a < 3; ++a) {
            if (spatial_shape[a] < 1 || spatial_shape[a] >= (1 << 30)) return SPCONV_ERR_INVALID_ARG;
            shape[a] = spatial_shape[a];
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!spatial_shape || batch <= 0) {
        int32_t dshape[3], dbatch = 1;
        SPCONV_CHECK(derive_shape(coords_dev, n, s, dshape, &dbatch));
        if (!spatial_shape) std::memcpy(shape, dshape, sizeof(shape));
        if (batch <= 0) batch = dbatch;
    }
    spconv_map_s* h = new (std::nothrow) spconv_map_s();
    if (!h) return SPCONV_ERR_OOM;
    h->stream = s;
    cudaGetDevice(&h->device);
    std::memcpy(h->shape, shape, sizeof(shape));
    h->batch = batch;
    h->kernel_size = 3;
    h->taps = kTaps;
    h->groups = 1;
    const int rc = build_map_strided(h, coords_dev, n, opt);
    if (rc != SPCONV_OK) {
        if (h->arena) cudaFreeAsync(h->arena, s);
        if (h->out_alloc) cudaFreeAsync(h->out_alloc, s);
        delete h;
        return rc;
    }
    *out_map = h;
    return SPCONV_OK;
}

int spconv_build_map_inverse(spconv_map_t strided, const spconv_options_t* opt, spconv_map_t* out_map) {
    reset_launch_count();
    if (!out_map) return SPCONV_ERR_INVALID_ARG;
    *out_map = nullptr;
    if (!strided || strided->conv != kConvStrided) return SPCONV_ERR_INVALID_ARG;
    if (opt) {
        if (opt->bit_order != SPCONV_ORDER_CALIBRATED && opt->bit_order != SPCONV_ORDER_PLAIN)
            return SPCONV_ERR_INVALID_ARG;
        if (opt->gemm == SPCONV_GEMM_TAP_MAJOR) return SPCONV_ERR_UNSUPPORTED;
    }
    spconv_map_s* h = new (std::nothrow) spconv_map_s();
    if (!h) return SPCONV_ERR_OOM;
    h->stream = strided->stream;
    h->device = strided->device;
    h->kernel_size = 3;
    h->taps = kTaps;
    h->groups = 1;
    const int rc = build_map_inverse(h, strided, opt);
    if (rc != SPCONV_OK) {
        if (h->arena) cudaFreeAsync(h->arena, h->stream);
        delete h;
        return rc;
    }
    *out_map = h;
    return SPCONV_OK;
}

int spconv_map_out_coords(spconv_map_t map, int32_t* out_coords_dev, void* stream) {
    if (!map || !map->out_coords) return SPCONV_ERR_INVALID_ARG;
    if (map->n == 0) return SPCONV_OK;
    if (!out_coords_dev) return SPCONV_ERR_INVALID_ARG;
    return cuda_status(cudaMemcpyAsync(out_coords_dev, map->out_coords, static_cast<size_t>(map->n) * 16,
                                       cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)));
}

int spconv_subm_forward(spconv_map_t map, const void* feats_dev, const void* weights_dev, void* out_dev,
                        int32_t c_in, int32_t c_out, int32_t dtype, void* stream) {
    return spconv_subm_forward_ex(map, feats_dev, weights_dev, out_dev, c_in, c_out, dtype, nullptr, stream);
}

int spconv_subm_forward_ex(spconv_map_t map, const void* feats_dev, const void* weights_dev, void* out_dev,
                           int32_t c_in, int32_t c_out, int32_t dtype, const spconv_epilogue_t* epi,
                           void* stream) {
    reset_launch_count();
    SPCONV_CHECK(check_forward_args(map, feats_dev, out_dev, c_in, c_out, dtype));
    Epilogue e;
    SPCONV_CHECK(check_epilogue(map, epi, out_dev, c_out, dtype, &e));
    if (map->n == 0) return SPCONV_OK;
    if (!weights_dev) return SPCONV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (use_tensor_path(c_in, c_out, dtype, feats_dev, out_dev) && aligned(weights_dev, 2)) {
        const size_t need = tc_pack_bytes(c_in, c_out, map->taps);
        if (map->wspace_bytes < need) {
            if (map->wspace) cudaFreeAsync(map->wspace, s);
            map->wspace = nullptr;
            map->wspace_bytes = 0;
            if (pool_alloc(&map->wspace, need, s) != cudaSuccess) {
                cudaGetLastError();
                map->wspace = nullptr;
                return SPCONV_ERR_OOM;
            }
            map->wspace_bytes = need;
        }
        SPCONV_CHECK(tc_pack_weights(weights_dev, c_in, c_out, map->taps, map->wspace, s));
        return tc_forward(map, feats_dev, map->wspace, out_dev, c_in, c_out, e, s);
    }
    return simt_forward(map, feats_dev, weights_dev, out_dev, c_in, c_out, dtype, e, s);
}

int spconv_wpack_create(const void* weights_dev, int32_t c_in, int32_t c_out, int32_t dtype, void* stream,
                        spconv_wpack_t* out_wpack) {
    return spconv_wpack_create_ex(weights_dev, 3, c_in, c_out, dtype, stream, out_wpack);
}

int spconv_wpack_create_ex(const void* weights_dev, int32_t kernel_size, int32_t c_in, int32_t c_out,
                           int32_t dtype, void* stream, spconv_wpack_t* out_wpack) {
    reset_launch_count();
    if (!out_wpack) return SPCONV_ERR_INVALID_ARG;
    *out_wpack = nullptr;
    if (kernel_size != 3 && kernel_size != 5) return SPCONV_ERR_UNSUPPORTED;
    const int32_t taps = kernel_size * kernel_size * kernel_size;
    if (!weights_dev || c_in < 1 || c_out < 1 || c_in > 65536 || c_out > 65536) return SPCONV_ERR_INVALID_ARG;
    if (dtype != SPCONV_BF16 && dtype != SPCONV_FP32) return SPCONV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    spconv_wpack_s* w = new (std::nothrow) spconv_wpack_s();
    if (!w) return SPCONV_ERR_OOM;
    w->c_in = c_in;
    w->c_out = c_out;
    w->dtype = dtype;
    w->taps = taps;
    w->stream = s;
    w->tensor_path = (dtype == SPCONV_BF16 && tc_supported(c_in, c_out)) ? 1 : 0;
    const size_t es = dtype == SPCONV_FP32 ? 4 : 2;
    w->bytes = w->tensor_path ? tc_pack_bytes(c_in, c_out, taps) : static_cast<size_t>(taps) * c_in * c_out * es;
    if (pool_alloc(&w->data, w->bytes, s) != cudaSuccess) {
        cudaGetLastError();
        delete w;
        return SPCONV_ERR_OOM;
    }
    int rc = SPCONV_OK;
    if (w->tensor_path) {
        w->n_tile = tc_tile_n(c_out);
        rc = tc_pack_weights(weights_dev, c_in, c_out, taps, w->data, s);
    } else {
        rc = cuda_status(cudaMemcpyAsync(w->data, weights_dev, w->bytes, cudaMemcpyDeviceToDevice, s));
    }
    if (rc != SPCONV_OK) {
        cudaFreeAsync(w->data, s);
        delete w;
        return rc;
    }
    *out_wpack = w;
    return SPCONV_OK;
}

int spconv_subm_forward_packed(spconv_map_t map, const void* feats_dev, spconv_wpack_t wpack, void* out_dev,
                               void* stream) {
    return spconv_subm_forward_packed_ex(map, feats_dev, wpack, out_dev, nullptr, stream);
}

int spconv_subm_forward_packed_ex(spconv_map_t map, const void* feats_dev, spconv_wpack_t wpack, void* out_dev,
                                  const spconv_epilogue_t* epi, void* stream) {
    reset_launch_count();
    if (!wpack) return SPCONV_ERR_INVALID_ARG;
    SPCONV_CHECK(check_forward_args(map, feats_dev, out_dev, wpack->c_in, wpack->c_out, wpack->dtype));
    if (wpack->taps != map->taps) return SPCONV_ERR_INVALID_ARG;
    Epilogue e;
    SPCONV_CHECK(check_epilogue(map, epi, out_dev, wpack->c_out, wpack->dtype, &e));
    if (map->n == 0) return SPCONV_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (wpack->tensor_path) {
        if (!aligned(feats_dev, 16) || !aligned(out_dev, 16)) return SPCONV_ERR_INVALID_ARG;
        return tc_forward(map, feats_dev, wpack->data, out_dev, wpack->c_in, wpack->c_out, e, s);
    }
    return simt_forward(map, feats_dev, wpack->data, out_dev, wpack->c_in, wpack->c_out, wpack->dtype, e, s);
}

int spconv_subm_forward_layers(spconv_map_t map, const void* feats_dev, const spconv_wpack_t* wpacks,
                               void* const* outs_dev, int32_t n_layers, const spconv_epilogue_t* epis,
                               void* stream) {
    reset_launch_count();
    if (!map || !wpacks || !outs_dev || n_layers < 1 || n_layers > kMaxFusedLayers) return SPCONV_ERR_INVALID_ARG;
    for (int l = 0; l < n_layers; ++l)
        if (!wpacks[l]) return SPCONV_ERR_INVALID_ARG;
    const int32_t c_in = wpacks[0]->c_in, c_out = wpacks[0]->c_out;
    for (int l = 0; l < n_layers; ++l) {
        const WPackHandle* w = wpacks[l];
        if (w->c_in != c_in || w->c_out != c_out || w->taps != map->taps) return SPCONV_ERR_INVALID_ARG;
        if (!w->tensor_path || w->dtype != SPCONV_BF16) return SPCONV_ERR_UNSUPPORTED;
    }
    if (n_layers > 1 && c_in != c_out) return SPCONV_ERR_INVALID_ARG;
    // later layers gather the previous output through the same map: its rows
    // must be the sites it indexes (a submanifold map, one offset group)
    if (n_layers > 1 && (map->conv != kConvSubmanifold || map->groups > 1 || map->gemm == SPCONV_GEMM_TAP_MAJOR))
        return SPCONV_ERR_UNSUPPORTED;
    Epilogue e[kMaxFusedLayers];
    const void* wp[kMaxFusedLayers];
    for (int l = 0; l < n_layers; ++l) {
        const void* in = l == 0 ? feats_dev : outs_dev[l - 1];
        SPCONV_CHECK(check_forward_args(map, in, outs_dev[l], c_in, c_out, SPCONV_BF16));
        SPCONV_CHECK(check_epilogue(map, epis ? &epis[l] : nullptr, outs_dev[l], c_out, SPCONV_BF16, &e[l]));
        if (map->n > 0 && (!aligned(in, 16) || !aligned(outs_dev[l], 16))) return SPCONV_ERR_INVALID_ARG;
        wp[l] = wpacks[l]->data;
    }
    if (map->n == 0) return SPCONV_OK;
    return tc_forward_layers(map, feats_dev, wp, outs_dev, e, n_layers, c_in, c_out, static_cast<cudaStream_t>(stream));
}

void spconv_wpack_destroy(spconv_wpack_t wpack) {
    if (!wpack) return;
    if (wpack->data) cudaFreeAsync(wpack->data, wpack->stream);
    delete wpack;
}

int spconv_map_status(spconv_map_t map) {
    if (!map) return SPCONV_ERR_INVALID_ARG;
    return read_status(map);
}

int spconv_map_info(spconv_map_t map, spconv_map_info_t* info) {
    if (!map || !info) return SPCONV_ERR_INVALID_ARG;
    int32_t totals[2] = {0, 0};
    SPCONV_CHECK_CUDA(cudaStreamSynchronize(map->stream));
    SPCONV_CHECK_CUDA(cudaMemcpy(totals, map->totals, sizeof(totals), cudaMemcpyDeviceToHost));
    info->n = map->n;
    info->pairs = totals[0];
    info->n_tiles = map->n_tiles;
    info->tile_taps = totals[1];
    info->mapper = map->mapper;
    info->pipeline = map->pipeline;
    info->key_bits = map->key_bits;
    std::memcpy(info->shape, map->shape, sizeof(info->shape));
    info->batch_size = map->batch;
    info->gemm = map->gemm;
    info->kernel_size = map->kernel_size;
    info->groups = map->groups;
    info->n_in = map->n_in >= 0 ? map->n_in : map->n;
    info->conv = map->conv;
    std::memcpy(info->out_shape, map->conv == kConvStrided ? map->out_shape : map->shape, sizeof(info->out_shape));
    return SPCONV_OK;
}

int spconv_map_rows(spconv_map_t map, int64_t* n, int64_t* n_in) {
    if (!map) return SPCONV_ERR_INVALID_ARG;
    if (n) *n = map->n;
    if (n_in) *n_in = map->n_in >= 0 ? map->n_in : map->n;
    return SPCONV_OK;
}

int spconv_map_export(spconv_map_t map, int32_t* nbr_dev, uint32_t* mask_dev, int32_t* perm_dev,
                      int32_t* tap_off_dev, int32_t* in_rows_dev, int32_t* out_rows_dev, void* stream) {
    reset_launch_count();
    if (!map) return SPCONV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t n = map->n;
    const size_t V = static_cast<size_t>(map->taps), G = static_cast<size_t>(map->groups);
    if (n > 0 && nbr_dev)
        SPCONV_CHECK_CUDA(cudaMemcpy2DAsync(nbr_dev, V * sizeof(int32_t), map->nbr, map->nbr_stride * sizeof(int32_t),
                                            V * sizeof(int32_t), static_cast<size_t>(n), cudaMemcpyDeviceToDevice, s));
    if (n > 0 && mask_dev)
        SPCONV_CHECK_CUDA(cudaMemcpyAsync(mask_dev, map->mask, G * n * sizeof(uint32_t), cudaMemcpyDeviceToDevice, s));
    if (n > 0 && perm_dev)
        SPCONV_CHECK_CUDA(cudaMemcpyAsync(perm_dev, map->perm, G * n * sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
    if (tap_off_dev)
        SPCONV_CHECK_CUDA(cudaMemcpyAsync(tap_off_dev, map->tap_off, (V + 1) * sizeof(int32_t),
                                          cudaMemcpyDeviceToDevice, s));
    if (in_rows_dev || out_rows_dev) {
        spconv_map_info_t info;
        SPCONV_CHECK(spconv_map_info(map, &info));
        if (info.pairs > 0 && in_rows_dev)
            SPCONV_CHECK_CUDA(cudaMemcpyAsync(in_rows_dev, map->in_rows, info.pairs * sizeof(int32_t),
                                              cudaMemcpyDeviceToDevice, s));
        if (info.pairs > 0 && out_rows_dev)
            SPCONV_CHECK_CUDA(cudaMemcpyAsync(out_rows_dev, map->out_rows, info.pairs * sizeof(int32_t),
                                              cudaMemcpyDeviceToDevice, s));
    }
    return SPCONV_OK;
}

void spconv_map_destroy(spconv_map_t map) {
    if (!map) return;
    if (map->arena) cudaFreeAsync(map->arena, map->stream);
    if (map->wspace) cudaFreeAsync(map->wspace, map->stream);
    if (map->acc) cudaFreeAsync(map->acc, map->stream);
    if (map->layer_done) cudaFreeAsync(map->layer_done, map->stream);
    if (map->out_alloc) cudaFreeAsync(map->out_alloc, map->stream);
    delete map;
}

int32_t spconv_last_launch_count(void) { return g_launches; }

int spconv_selftest_wait_timeout(int32_t which, int64_t limit_ns, void* stream) {
    reset_launch_count();
    if (which < 0 || which > 2 || limit_ns < 1000000 || limit_ns > 100000000) return SPCONV_ERR_INVALID_ARG;
    return wait_probe(which, static_cast<uint64_t>(limit_ns), static_cast<cudaStream_t>(stream));
}

const char* spconv_status_string(int status) {
    switch (status) {
        case SPCONV_OK: return "ok";
        case SPCONV_ERR_INVALID_ARG: return "invalid argument";
        case SPCONV_ERR_UNSUPPORTED: return "unsupported";
        case SPCONV_ERR_OOM: return "out of device memory";
        case SPCONV_ERR_CUDA: return "CUDA runtime error";
        case SPCONV_ERR_DUPLICATE_COORD: return "duplicate coordinate";
        case SPCONV_ERR_COORD_RANGE: return "coordinate out of range";
        case SPCONV_ERR_ALIAS: return "output overlaps input";
        case SPCONV_ERR_TIMEOUT: return "kernel wait timed out";
        case SPCONV_ERR_INTERNAL: return "internal consistency check failed";
        default: return "unknown status";
    }
}

}  // extern "C"

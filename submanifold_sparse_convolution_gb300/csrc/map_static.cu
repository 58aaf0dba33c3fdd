// spconv_kernel_map_static: the kernel map nbr[n][27] with no device
// allocation at all.
//
// Some callers cannot allocate device memory when they run this code: a
// plugin's enqueue step inside an inference runtime that plans every device
// buffer at initialisation and forbids cudaMalloc afterwards, or runtimes
// certified to never allocate after start-up.  For them this
// entry point keeps its working buffers (packed keys, row ids, radix
// histograms, a status word) in one file-scope device array of fixed size,
// kStaticScratchBytes, which every GPU that loads the library holds until the
// process exits.  It runs the sorted-key mapper: pack keys, stable LSD radix
// sort, then one lower_bound per (dx, dy) column written straight into the
// caller's [n][27] buffer.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "radix_sort.cuh"

namespace spconv {
namespace {

constexpr int64_t kStaticMaxRows = 65536;
constexpr int64_t kStaticHistTiles = (kStaticMaxRows + rsort::kTile - 1) / rsort::kTile;
// keys ping-pong (u64), row ids ping-pong (u32), radix histograms, status
constexpr size_t kKeysBytes = static_cast<size_t>(kStaticMaxRows) * sizeof(uint64_t);
constexpr size_t kValsBytes = static_cast<size_t>(kStaticMaxRows) * sizeof(uint32_t);
constexpr size_t kHistBytes = static_cast<size_t>(rsort::kBins) * kStaticHistTiles * sizeof(int32_t);
constexpr size_t kStaticScratchBytes = 2 * kKeysBytes + 2 * kValsBytes + kHistBytes + 256;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr uint64_t kInvalid = ~0ull;

__global__ void __launch_bounds__(256) k_pack_keys_static(const int4* __restrict__ coords, int64_t n, int3 shape,
                                                          int batch, int wz, int wy, int wx,
                                                          uint64_t* __restrict__ keys,
                                                          uint32_t* __restrict__ vals,
                                                          int32_t* __restrict__ status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    uint64_t key = kInvalid;
    if (c.x >= 0 && c.x < batch && c.y >= 0 && c.y < shape.x && c.z >= 0 && c.z < shape.y && c.w >= 0 &&
        c.w < shape.z) {
        key = ((((static_cast<uint64_t>(c.x) << wx) | static_cast<uint64_t>(c.y + 1)) << wy |
                static_cast<uint64_t>(c.z + 1))
               << wz) |
              static_cast<uint64_t>(c.w + 1);
    } else {
        atomicOr(status, kStatusRange);
    }
    keys[i] = key;
    vals[i] = static_cast<uint32_t>(i);
}

struct Offsets27 {
    uint64_t off[kTaps];
};

// One thread per sorted position: the 27 neighbours of that voxel written as
// row (b, x, y, z)'s entry of the caller's [n][27] table.
__global__ void __launch_bounds__(256) k_search_static(const uint64_t* __restrict__ skeys,
                                                       const uint32_t* __restrict__ svals, int64_t n,
                                                       Offsets27 o, int32_t* __restrict__ nbr,
                                                       int32_t* __restrict__ status) {
    const int64_t s = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
    if (s >= n) return;
    const uint64_t q = skeys[s];
    int32_t* row = nbr + static_cast<int64_t>(svals[s]) * kTaps;
    if (q == kInvalid) {
        for (int k = 0; k < kTaps; ++k) row[k] = -1;
        return;
    }
    if (s > 0 && skeys[s - 1] == q) atomicOr(status, kStatusDuplicate);
    for (int c = 0; c < 9; ++c) {
        const uint64_t lo_t = q + o.off[3 * c];
        const uint64_t hi_t = q + o.off[3 * c + 2];
        int64_t first = 0, count = n;
        while (count > 0) {
            const int64_t st = count >> 1;
            if (__ldg(skeys + first + st) < lo_t) {
                first += st + 1;
                count -= st + 1;
            } else {
                count = st;
            }
        }
        int32_t v[3] = {-1, -1, -1};
        for (int j = 0; j < 3; ++j) {
            const int64_t p = first + j;
            if (p < n) {
                const uint64_t kk = __ldg(skeys + p);
                if (kk <= hi_t) v[kk - lo_t] = static_cast<int32_t>(__ldg(svals + p));
            }
        }
        row[3 * c] = v[0];
        row[3 * c + 1] = v[1];
        row[3 * c + 2] = v[2];
    }
}

int bit_len(uint64_t v) {
    int b = 0;
    while (v) {
        ++b;
        v >>= 1;
    }
    return b;
}

// Device address of g_static_scratch per device, looked up on the first call
// with that device current.
void* scratch_address() {
    constexpr int kMaxDevices = 64;
    static void* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace
}  // namespace spconv

using namespace spconv;

extern "C" int spconv_kernel_map_static(const int32_t* coords_dev, int64_t n, const int32_t* spatial_shape,
                                        int32_t batch_size, int32_t* nbr_dev, void* stream) {
    reset_launch_count();
    if (n < 0 || n > kStaticMaxRows) return SPCONV_ERR_INVALID_ARG;   // beyond the static scratch
    if (!spatial_shape || batch_size < 1) return SPCONV_ERR_INVALID_ARG;
    if (n > 0 && (!coords_dev || !nbr_dev || (reinterpret_cast<uintptr_t>(coords_dev) & 15) != 0 ||
                  (reinterpret_cast<uintptr_t>(nbr_dev) & 3) != 0))
        return SPCONV_ERR_INVALID_ARG;
    for (int a = 0; a < 3; ++a)
        if (spatial_shape[a] < 1 || spatial_shape[a] >= (1 << 30)) return SPCONV_ERR_INVALID_ARG;
    const int X = spatial_shape[0], Y = spatial_shape[1], Z = spatial_shape[2];
    const int wz = bit_len(static_cast<uint64_t>(Z) + 1), wy = bit_len(static_cast<uint64_t>(Y) + 1);
    const int wx = bit_len(static_cast<uint64_t>(X) + 1), wb = bit_len(static_cast<uint64_t>(batch_size) - 1);
    const int key_bits = wz + wy + wx + wb;
    if (key_bits > 63) return SPCONV_ERR_UNSUPPORTED;
    if (n == 0) return SPCONV_OK;

    unsigned char* base = static_cast<unsigned char*>(scratch_address());
    if (base == nullptr) return SPCONV_ERR_CUDA;
    uint64_t* keys_a = reinterpret_cast<uint64_t*>(base);
    uint64_t* keys_b = reinterpret_cast<uint64_t*>(base + kKeysBytes);
    uint32_t* vals_a = reinterpret_cast<uint32_t*>(base + 2 * kKeysBytes);
    uint32_t* vals_b = reinterpret_cast<uint32_t*>(base + 2 * kKeysBytes + kValsBytes);
    int32_t* hist = reinterpret_cast<int32_t*>(base + 2 * kKeysBytes + 2 * kValsBytes);
    int32_t* status = reinterpret_cast<int32_t*>(base + 2 * kKeysBytes + 2 * kValsBytes + kHistBytes);

    Offsets27 o;
    for (int dx = -1; dx <= 1; ++dx)
        for (int dy = -1; dy <= 1; ++dy)
            for (int dz = -1; dz <= 1; ++dz)
                o.off[9 * (dx + 1) + 3 * (dy + 1) + (dz + 1)] = static_cast<uint64_t>(
                    static_cast<int64_t>(dx) * (int64_t(1) << (wy + wz)) + static_cast<int64_t>(dy) * (int64_t(1) << wz) + dz);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status word keeps the previous call's value: clear it
    SPCONV_CHECK_CUDA(cudaMemsetAsync(status, 0, sizeof(int32_t), s));
    const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
    k_pack_keys_static<<<blocks, 256, 0, s>>>(reinterpret_cast<const int4*>(coords_dev), n, make_int3(X, Y, Z),
                                              batch_size, wz, wy, wx, keys_a, vals_a, status);
    int launches = 1;
    const bool in_b = rsort::sort_pairs<uint64_t>(keys_a, vals_a, keys_b, vals_b, n, key_bits + 1, hist, s, &launches);
    k_search_static<<<blocks, 256, 0, s>>>(in_b ? keys_b : keys_a, in_b ? vals_b : vals_a, n, o, nbr_dev, status);
    ++launches;
    count_launch(launches);
    SPCONV_CHECK_CUDA(cudaGetLastError());
    int32_t st = 0;
    SPCONV_CHECK_CUDA(cudaMemcpyAsync(&st, status, sizeof(st), cudaMemcpyDeviceToHost, s));
    SPCONV_CHECK_CUDA(cudaStreamSynchronize(s));
    if (st & kStatusRange) return SPCONV_ERR_COORD_RANGE;
    if (st & kStatusDuplicate) return SPCONV_ERR_DUPLICATE_COORD;
    return SPCONV_OK;
}

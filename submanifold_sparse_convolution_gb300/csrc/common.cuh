// Internal declarations shared by the translation units of libspconv.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/spconv.h"

namespace spconv {

constexpr int kTaps = 27;           // taps of a 3x3x3 kernel
constexpr int kMaxKernel = 5;       // largest kernel size (5x5x5, 125 taps)
constexpr int kMaxTaps = kMaxKernel * kMaxKernel * kMaxKernel;
constexpr int kMaxGroupTaps = 27;   // taps of one offset group (mask bits, GEMM index buffer)
constexpr int kMaxDevices = 64;    // per-device one-time settings are kept for device ids below this
constexpr int kTileRows = 128;      // rows per output tile (tensor-core M)
constexpr int kNbrStride = 32;      // padded width of the internal kernel-map rows
constexpr int kMaxFusedLayers = 8;  // layers of one fused forward launch

// Device status word bits (set with atomicOr by kernels).
enum : int32_t {
    kStatusDuplicate = 1,
    kStatusRange = 2,
    kStatusTimeout = 4,
    kStatusInternal = 8,   // an internal consistency guard fired (a would-be out-of-range store was skipped)
};

// Programmatic dependent launch.  A kernel launched with
// pdl_attr() may start while the previous kernel of its stream is finishing;
// before its first read of anything an earlier kernel wrote it must call
// pdl_wait(), which returns once every earlier kernel has completed and its
// writes are visible.  pdl_trigger() lets the next such kernel be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

inline cudaLaunchAttribute pdl_attr() {
    cudaLaunchAttribute at = {};
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    return at;
}

// Counts launches of the current host thread (reported by
// spconv_last_launch_count).
void count_launch(int n = 1);
void reset_launch_count();

// A stream-ordered device buffer.
struct DevBuf {
    void* ptr = nullptr;
    size_t bytes = 0;
};

// What a map's rows and neighbours are: a submanifold map (rows and
// neighbours are the same sites), a strided map (rows are the output sites of
// a kernel-3, stride-2, padding-1 convolution, neighbours the input sites), or
// the inverse of a strided map (rows the strided map's input sites,
// neighbours its output sites).
enum : int32_t { kConvSubmanifold = 0, kConvStrided = 1, kConvInverse = 2 };

struct MapHandle {
    cudaStream_t stream = nullptr;
    int device = 0;
    int64_t n = 0;            // rows (output sites)
    int64_t n_in = -1;        // sites the neighbours index (feature rows of a forward); -1: n
    int32_t conv = kConvSubmanifold;
    int32_t out_shape[3] = {0, 0, 0};   // spatial shape of the row sites (strided: the output grid)
    int32_t* out_coords = nullptr;      // strided and inverse maps: [n][4] (b, x, y, z) of the rows
    void* out_alloc = nullptr;          // the allocation holding out_coords
    int64_t n_tiles = 0;
    int64_t n_pad = 0;        // n_tiles * kTileRows
    int32_t shape[3] = {0, 0, 0};
    int32_t batch = 0;
    int32_t mapper = 0;       // spconv_mapper_t used
    int32_t pipeline = 0;     // spconv_pipeline_t used
    int32_t bit_order = 0;
    int32_t gemm = 0;         // spconv_gemm_t used by the bf16 forward (TILE_UNION or TAP_MAJOR)
    int32_t key_bits = 0;
    int32_t kernel_size = 3;  // K: the kernel is K x K x K
    int32_t taps = kTaps;     // V = K^3
    int32_t groups = 1;       // G offset groups of V / G consecutive taps, each with its own row order
    int32_t group_taps = kTaps;     // V / G
    int32_t nbr_stride = kNbrStride;   // width of an nbr row (>= V, a multiple of 4)
    // device arrays
    int32_t* status = nullptr;     // [1]
    // (with G groups: masks, orders, unions and tile orders per group, group-major)
    int32_t* nbr = nullptr;        // [n][nbr_stride], original row order
    uint32_t* mask = nullptr;      // [G][n] bit j: tap g V/G + j present
    int32_t* perm = nullptr;       // one group: [n_pad] (rows >= n: -1); G groups: [G][n]
    int32_t* tap_count = nullptr;  // [V]
    int32_t* tap_pos = nullptr;    // [V] key bit of each tap within its group
    int32_t* tap_off = nullptr;    // [V + 1]
    int32_t* in_rows = nullptr;    // [V n]
    int32_t* out_rows = nullptr;   // [V n]
    int32_t* gtab = nullptr;       // [V][n_pad]: nbr[perm_g[s]][k] or -1 (g the group of tap k)
    uint32_t* tile_union = nullptr;  // [G][n_tiles]
    int32_t* tile_order = nullptr;   // [G][n_tiles], each group's tiles by descending union size
    int32_t* seg_off = nullptr;      // [V][n_tiles] pair count of (tap, tile), scanned into offsets where a scan runs
    int32_t* tile_nonempty = nullptr;  // [G] tiles with a nonempty union (the first ones of each tile order)
    int32_t* totals = nullptr;       // [2]: pairs, sum of union sizes
    void* arena = nullptr;           // one allocation holding the arrays above
    size_t arena_bytes = 0;
    // weight workspace for spconv_subm_forward
    void* wspace = nullptr;
    size_t wspace_bytes = 0;
    // fp32 sums of the tap-major forward ([n][c_out])
    void* acc = nullptr;
    size_t acc_bytes = 0;
    // per-layer CTA counters of a fused layer stack ([kMaxFusedLayers] int32)
    int32_t* layer_done = nullptr;
};

struct WPackHandle {
    int32_t c_in = 0, c_out = 0, dtype = 0;
    int32_t taps = kTaps;      // kernel volume the weights are for
    int32_t tensor_path = 0;   // 1: tcgen05 shared-memory image, 0: row-major copy for SIMT
    int32_t n_tile = 0;        // output channels per tensor-core tile
    int32_t k_chunks = 0;      // 64-wide input-channel chunks
    void* data = nullptr;
    size_t bytes = 0;
    cudaStream_t stream = nullptr;
};

// What the forward does to each fp32 sum before its one rounding to the
// output dtype: y = sum * scale[o] + bias[o] + residual[row][o], then
// max(y, 0) if relu.  Null pointers stand for 1, 0 and 0.  Device pointers;
// residual is in the output dtype with the output's [n][c_out] layout.
struct Epilogue {
    const float* scale = nullptr;
    const float* bias = nullptr;
    const void* residual = nullptr;
    int32_t relu = 0;
    bool active() const { return scale || bias || residual || relu; }
};

// ---- map building (map.cu) -----------------------------------------------
int build_map_impl(MapHandle* h, const int32_t* coords, const spconv_options_t* opt);
// K != 3 or more than one offset group (map_groups.cu)
int build_map_grouped(MapHandle* h, const int32_t* coords, const spconv_options_t* opt);
// strided (kernel 3, stride 2, padding 1) map of coords [n_in][4]; synchronises once (the
// number of output sites sizes the map); h->shape is the input shape
int build_map_strided(MapHandle* h, const int32_t* coords, int64_t n_in, const spconv_options_t* opt);
// the inverse of strided map src, into h (same device and stream)
int build_map_inverse(MapHandle* h, const MapHandle* src, const spconv_options_t* opt);
int derive_shape(const int32_t* coords, int64_t n, cudaStream_t stream, int32_t shape[3],
                 int32_t* batch);

// ---- tensor-core GEMM (gemm_tc.cu) ------------------------------------------
bool tc_supported(int32_t c_in, int32_t c_out);
int tc_tile_n(int32_t c_out);
size_t tc_pack_bytes(int32_t c_in, int32_t c_out, int32_t taps);
int tc_pack_weights(const void* w, int32_t c_in, int32_t c_out, int32_t taps, void* dst, cudaStream_t s);
int tc_forward(MapHandle* h, const void* feats, const void* wpack, void* out, int32_t c_in,
               int32_t c_out, const Epilogue& epi, cudaStream_t s);
// n_layers layers of c_in -> c_out (c_in == c_out when n_layers > 1) in one
// cooperative launch: layer l reads outs[l - 1] (layer 0: feats), stores outs[l]
int tc_forward_layers(MapHandle* h, const void* feats, const void* const* wpacks, void* const* outs,
                      const Epilogue* epis, int32_t n_layers, int32_t c_in, int32_t c_out, cudaStream_t s);

// ---- SIMT path (gemm_simt.cu) ----------------------------------------------
int simt_forward(const MapHandle* h, const void* feats, const void* w, void* out, int32_t c_in,
                 int32_t c_out, int32_t dtype, const Epilogue& epi, cudaStream_t s);

// One bounded wait of the sort passes run against a state nothing publishes
// (which = 0: look-back, 1: grid barrier); the status it ends with (map_wide.cu).
int wait_probe(int which, uint64_t limit_ns, cudaStream_t s);

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? SPCONV_OK : SPCONV_ERR_CUDA; }

// The status code of a device status word (kStatus* flags), the most specific first.
inline int status_from_flags(int32_t st) {
    if (st & kStatusRange) return SPCONV_ERR_COORD_RANGE;
    if (st & kStatusDuplicate) return SPCONV_ERR_DUPLICATE_COORD;
    if (st & kStatusTimeout) return SPCONV_ERR_TIMEOUT;
    if (st & kStatusInternal) return SPCONV_ERR_INTERNAL;
    return SPCONV_OK;
}

// Stream-ordered allocation from the library's memory pool on the current
// device.  The pool keeps freed memory for reuse (no release threshold), so
// a map rebuilt every frame does not map and unmap device memory each time.
cudaError_t pool_alloc(void** p, size_t bytes, cudaStream_t s);

}  // namespace spconv

#define SPCONV_CHECK_CUDA(call)                             \
    do {                                                    \
        cudaError_t e_ = (call);                            \
        if (e_ != cudaSuccess) return SPCONV_ERR_CUDA;      \
    } while (0)

#define SPCONV_CHECK(call)                                  \
    do {                                                    \
        int s_ = (call);                                    \
        if (s_ != SPCONV_OK) return s_;                     \
    } while (0)

// Neighbour search over the sorted packed (key << row_bits | row) array, on
// the whole GPU: the kernel map rows, the 27-bit masks and the per-tap pair
// counts.  Shared by the cluster pipeline (map_fused.cu) and the whole-GPU
// pipeline (map_wide.cu), between their coordinate sort and their mask sort.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "map_internal.cuh"

namespace spconv {
namespace {

// Adds this warp's tap counts to the CTA's shared counters.
__device__ __forceinline__ void add_tap_counts(uint32_t m, int32_t* cta_taps) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> k) & 1u);
        if (lane == 0 && b) atomicAdd(cta_taps + k, __popc(b));
    }
}

// Neighbour search on the whole GPU, between the two cluster launches.  One
// thread per sorted position s of the packed (key << rb | row) array finds
// the 27 neighbours of the voxel there: one lower bound per (dx, dy) column
// for key + packed(dx, dy, -1), then a look at the next three keys for
// dz = -1, 0, +1.
//
// The targets of one column are the block's own sorted keys plus a constant,
// so they are sorted too and their lower bounds fall in one short run of the
// array (a sorted search).  A block of kSearchRows rows loads every
// 2^sample_shift-th packed key (at most kSampleMax of them), brackets each
// column's run from that sample, copies the 9 runs into shared memory and
// searches there; the only global loads are the sample and the runs, all
// independent.  A run longer than wcap entries (a block whose neighbouring
// columns are much denser than itself) is searched in global memory instead.
// The 9 searches of a row advance in lockstep (independent shared-memory
// loads).  The block's kernel-map rows (128 bytes each, at their original row
// index) are staged in shared memory and written 8 lanes per row, so every
// store instruction writes four whole rows.
constexpr int kSearchRows = 256;
constexpr int kSampleMax = 2048;

struct SearchArgs {
    const uint64_t* sv;
    int64_t n;
    int rb, key_bits;
    int sample_shift;          // sample stride = 2^sample_shift
    int wcap;                  // shared-memory run capacity per column
    uint64_t koff[kTaps];
    int32_t* nbr;
    uint32_t* mask;
    int32_t* tap_count;
    int32_t* status;
};

// First index i in a[0, len) with a[i] >= t (len if none), shared or global.
__device__ __forceinline__ int64_t lower_bound_in(const uint64_t* a, int64_t len, uint64_t t) {
    int64_t base = 0;
    while (len > 1) {
        const int64_t half = len >> 1;
        base += a[base + half - 1] < t ? half : 0;
        len -= half;
    }
    return len == 1 && a[base] < t ? base + 1 : base;
}

__global__ void __launch_bounds__(kSearchRows) k_search_window(const SearchArgs a) {
    extern __shared__ uint64_t sh_search[];
    uint64_t* samp = sh_search;                  // [kSampleMax]
    uint64_t* win = sh_search + kSampleMax;      // [9][wcap]
    __shared__ int64_t wlo[9];
    __shared__ int32_t wlen[9];                  // -1: search this column in global memory
    __shared__ int32_t wsteps;                   // halving steps that cover the longest run
    __shared__ int32_t cnt[kTaps];
    __shared__ int32_t err;
    const int t = threadIdx.x;
    const int64_t n = a.n;
    const int rb = a.rb;
    const uint64_t rmask = (uint64_t(1) << rb) - 1;
    const uint64_t invalid_key = (uint64_t(1) << a.key_bits) - 1;
    const int64_t ns = ((n - 1) >> a.sample_shift) + 1;
    const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kSearchRows;
    const int64_t s_end = s0 + kSearchRows < n ? s0 + kSearchRows : n;
    if (t < kTaps) cnt[t] = 0;
    if (t == 0) err = 0;
    pdl_wait();   // the coordinate sort must have finished
    pdl_trigger();
    for (int64_t j = t; j < ns; j += kSearchRows) samp[j] = __ldcg(a.sv + (j << a.sample_shift));
    const int64_t s = s0 + t;
    const uint64_t vs = s < n ? __ldg(a.sv + s) : ~uint64_t(0);
    __syncthreads();
    // ---- bracket each column's run of lower bounds from the sample
    if (t < 9) {
        const uint64_t qf = __ldg(a.sv + s0) >> rb;
        const uint64_t ql = __ldg(a.sv + s_end - 1) >> rb;
        int64_t lo = 0, len = 0;
        if (qf == invalid_key) {
            len = 0;                              // no valid row in this block
        } else if (ql == invalid_key) {
            len = -1;                             // invalid rows at the end: plain search
        } else {
            const int64_t jf = lower_bound_in(samp, ns, (qf + a.koff[3 * t]) << rb);
            const int64_t jl = lower_bound_in(samp, ns, (ql + a.koff[3 * t]) << rb);
            lo = jf > 0 ? ((jf - 1) << a.sample_shift) + 1 : 0;
            int64_t hi = (jl << a.sample_shift) + 3;
            if (hi > n) hi = n;
            len = hi - lo;
            if (len > a.wcap) len = -1;
        }
        wlo[t] = lo;
        wlen[t] = static_cast<int32_t>(len);
    }
    __syncthreads();
    if (t == 0) {
        int32_t most = 0;
        for (int c = 0; c < 9; ++c) most = wlen[c] > most ? wlen[c] : most;
        wsteps = 32 - __clz(most);
    }
    // ---- copy the runs (independent loads, several in flight per thread)
    for (int c = 0; c < 9; ++c) {
        const int32_t len = wlen[c];
        const uint64_t* src = a.sv + wlo[c];
        uint64_t* dst = win + c * a.wcap;
        for (int32_t i0 = t; i0 < len; i0 += 4 * kSearchRows) {
            uint64_t v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int32_t i = i0 + u * kSearchRows;
                v[u] = i < len ? __ldg(src + i) : 0ull;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (i0 + u * kSearchRows < len) dst[i0 + u * kSearchRows] = v[u];
        }
    }
    __syncthreads();
    uint32_t m = 0;
    int32_t x27[kTaps];
#pragma unroll
    for (int k = 0; k < kTaps; ++k) x27[k] = -1;
    int64_t r = -1;
    if (s < n) {
        const uint64_t q = vs >> rb;
        r = static_cast<int64_t>(vs & rmask);
        if (r >= n) {
            atomicOr(&err, kStatusInternal);
            r = -1;
        }
        if (q != invalid_key) {
            if (s > 0 && (__ldg(a.sv + s - 1) >> rb) == q) atomicOr(&err, kStatusDuplicate);
            // lower bounds of the 9 targets in the shared runs, in lockstep and
            // branch-free (every step issues its 9 loads together; a finished
            // column re-reads a valid slot and ignores it)
            uint64_t tl[9];
            int32_t base[9], len[9];
#pragma unroll
            for (int cc = 0; cc < 9; ++cc) {
                tl[cc] = (q + a.koff[3 * cc]) << rb;
                base[cc] = 0;
                len[cc] = wlen[cc] > 0 ? wlen[cc] : 0;
            }
            for (int it = 0; it < wsteps; ++it) {
#pragma unroll
                for (int cc = 0; cc < 9; ++cc) {
                    const int32_t half = len[cc] >> 1;
                    const int32_t probe = base[cc] + (half > 0 ? half - 1 : 0);
                    const uint64_t v = win[cc * a.wcap + probe];
                    base[cc] += (half > 0 && v < tl[cc]) ? half : 0;
                    len[cc] -= half;
                }
            }
            int32_t pos[9];
#pragma unroll
            for (int cc = 0; cc < 9; ++cc) {
                const uint64_t v = win[cc * a.wcap + base[cc]];
                pos[cc] = base[cc] + ((len[cc] == 1 && v < tl[cc]) ? 1 : 0);
            }
            // the three candidates after each lower bound (clamped reads, masked)
#pragma unroll
            for (int cc = 0; cc < 9; ++cc) {
                const uint64_t hi_k = q + a.koff[3 * cc + 2];
                const int32_t wl = wlen[cc];
                uint64_t cand[3];
                int32_t avail;
                if (wl >= 0) {
                    avail = wl - pos[cc];
#pragma unroll
                    for (int j = 0; j < 3; ++j) {
                        const int32_t pp = pos[cc] + j < a.wcap ? pos[cc] + j : a.wcap - 1;
                        cand[j] = win[cc * a.wcap + pp];
                    }
                } else {   // a run too long for shared memory: search the array
                    const int64_t gp = lower_bound_in(a.sv, n, tl[cc]);
                    avail = static_cast<int32_t>(n - gp < 3 ? n - gp : 3);
#pragma unroll
                    for (int j = 0; j < 3; ++j) cand[j] = gp + j < n ? __ldg(a.sv + gp + j) : 0ull;
                }
                int32_t x[3] = {-1, -1, -1};
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const uint64_t kk = cand[j] >> rb;
                    const bool hit = j < avail && kk <= hi_k;
                    const uint64_t dz = kk - (tl[cc] >> rb);
                    const int64_t rr = static_cast<int64_t>(cand[j] & rmask);
                    const int32_t nr = rr < n ? static_cast<int32_t>(rr) : -1;
                    x[0] = (hit && dz == 0) ? nr : x[0];
                    x[1] = (hit && dz == 1) ? nr : x[1];
                    x[2] = (hit && dz == 2) ? nr : x[2];
                }
                m |= ((x[0] >= 0 ? 1u : 0u) | (x[1] >= 0 ? 2u : 0u) | (x[2] >= 0 ? 4u : 0u)) << (3 * cc);
                x27[3 * cc] = x[0];
                x27[3 * cc + 1] = x[1];
                x27[3 * cc + 2] = x[2];
            }
        }
        if (r >= 0) a.mask[r] = m;
    }
    // ---- stage the rows in shared memory (the runs are no longer needed) and
    // write each 128-byte row with 8 lanes
    __syncthreads();
    int32_t* stage = reinterpret_cast<int32_t*>(sh_search);          // [kSearchRows][kNbrStride]
    int64_t* stage_row = reinterpret_cast<int64_t*>(stage + kSearchRows * kNbrStride);   // [kSearchRows]
    {
        int4* mine = reinterpret_cast<int4*>(stage + t * kNbrStride);
#pragma unroll
        for (int qq = 0; qq < kNbrStride / 4; ++qq) {
            int4 v4;
            v4.x = 4 * qq < kTaps ? x27[4 * qq] : -1;
            v4.y = 4 * qq + 1 < kTaps ? x27[4 * qq + 1] : -1;
            v4.z = 4 * qq + 2 < kTaps ? x27[4 * qq + 2] : -1;
            v4.w = 4 * qq + 3 < kTaps ? x27[4 * qq + 3] : -1;
            mine[(qq + t) & 7] = v4;   // rotated by row: the 8 lanes of a row hit distinct banks when read
        }
        stage_row[t] = r;
    }
    __syncthreads();
    for (int j = t >> 3; j < kSearchRows; j += kSearchRows / 8) {
        const int64_t rr = stage_row[j];
        if (rr >= 0) {
            const int qq = t & 7;
            reinterpret_cast<int4*>(a.nbr + rr * kNbrStride)[qq] =
                reinterpret_cast<const int4*>(stage + j * kNbrStride)[(qq + j) & 7];
        }
    }
    add_tap_counts(m, cnt);
    __syncthreads();
    if (t < kTaps && cnt[t]) atomicAdd(a.tap_count + t, cnt[t]);
    if (t == 0 && err) atomicOr(a.status, err);
}

}  // namespace

int launch_search_window(const uint64_t* sv, int64_t n, int row_bits, int key_bits, const uint64_t* koff,
                         int32_t* nbr, uint32_t* mask, int32_t* tap_count, int32_t* status, cudaStream_t s) {
    SearchArgs sa;
    sa.sv = sv;
    sa.n = n;
    sa.rb = row_bits;
    sa.key_bits = key_bits;
    for (int k = 0; k < kTaps; ++k) sa.koff[k] = koff[k];
    sa.nbr = nbr;
    sa.mask = mask;
    sa.tap_count = tap_count;
    sa.status = status;
    // sample stride: the smallest power of two >= 64 giving at most kSampleMax samples
    int sh = 6;
    while (((n - 1) >> sh) + 1 > kSampleMax) ++sh;
    sa.sample_shift = sh;
    // run capacity: what a block needs at this stride, at most what the shared
    // memory attribute below covers (longer runs are searched in global memory)
    const int wcap_max = kSearchRows + 2 * static_cast<int>(kFusedMaxRows / kSampleMax) + 64;
    const int64_t want = kSearchRows + 2 * (int64_t(1) << sh) + 64;
    sa.wcap = static_cast<int>(want < wcap_max ? want : wcap_max);
    // the sample and runs, then (reusing them) the staged kernel-map rows and their row ids
    const size_t smem_search = (static_cast<size_t>(kSampleMax) + 9 * static_cast<size_t>(sa.wcap)) * sizeof(uint64_t);
    const size_t smem_stage = static_cast<size_t>(kSearchRows) * (kNbrStride * sizeof(int32_t) + sizeof(int64_t));
    const size_t smem = smem_search > smem_stage ? smem_search : smem_stage;
    // once per device, for the largest run buffer
    static bool smem_set[kMaxDevices] = {};
    int dev = 0;
    SPCONV_CHECK_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return SPCONV_ERR_UNSUPPORTED;
    if (!smem_set[dev]) {
        const int most = static_cast<int>((kSampleMax + 9 * static_cast<size_t>(wcap_max)) * sizeof(uint64_t));
        SPCONV_CHECK_CUDA(cudaFuncSetAttribute(k_search_window, cudaFuncAttributeMaxDynamicSharedMemorySize, most));
        smem_set[dev] = true;
    }
    cudaLaunchConfig_t scfg = {};
    scfg.gridDim = dim3(static_cast<unsigned>((n + kSearchRows - 1) / kSearchRows));
    scfg.blockDim = dim3(kSearchRows);
    scfg.dynamicSmemBytes = smem;
    scfg.stream = s;
    cudaLaunchAttribute sattr[1] = {pdl_attr()};
    scfg.attrs = sattr;
    scfg.numAttrs = 1;
    SPCONV_CHECK_CUDA(cudaLaunchKernelEx(&scfg, k_search_window, sa));
    return SPCONV_OK;
}

}  // namespace spconv

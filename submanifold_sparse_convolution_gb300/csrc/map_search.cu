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

// Neighbour search on the whole GPU, between the coordinate sort and the
// mask sort.  For each sorted position s of the packed (key << rb | row)
// array it finds the 27 neighbours of the voxel there: one lower bound per (dx, dy) column
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
// columns are much denser than itself) is searched in global memory instead,
// within the same bracket; wcap leaves a block's own rows plus two sample
// strides plus 256 entries of slack, so that stays rare.
// Three threads serve each row, three (dx, dy) columns each, in warp-uniform
// groups: one row's 9 searches on one thread left ~2 warps per scheduler on
// 32k rows, issue-bound at ~180 instructions per halving step.  A thread's 3
// searches advance in lockstep (independent shared-memory loads).  The
// block's kernel-map rows (128 bytes each, at their original row index) are
// combined in shared memory and written 8 lanes per row, so every store
// instruction writes four whole rows.
// Block shapes: on small arrays (at most kSearchBigRows rows, about one wave
// of blocks) 128 rows x 3 threads per row, for parallelism within the wave;
// above that 256 rows x 1 thread per row, so several blocks share an SM and
// one block's loads overlap another's search (stage, 240k rows: 57 us, vs 66
// with 128 x 3 and 80 with 256 x 3).
constexpr int kSampleMax = 2048;
constexpr int64_t kSearchBigRows = 65536;

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

// Runs are stored in shared memory with one 8-byte gap after every 16
// entries: entry i at i + i / 16.  The lanes of a warp search the targets of
// consecutive rows, so after a few halving steps they probe entries spaced by
// the current half-length, often a multiple of 16 entries (128 bytes, one
// pass over the 32 banks); unpadded, those probes all hit one bank (a 16- to
// 32-way conflict on every load, ~5 us of the kernel on 32k rows).
__device__ __forceinline__ int32_t pad_idx(int32_t i) { return i + (i >> 4); }
__host__ __device__ constexpr int64_t padded_cap(int64_t wcap) { return wcap + (wcap >> 4) + 1; }

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

// The same over global memory written by the kernel before this one (which
// may still have been running when this kernel started): L2 loads only.
__device__ __forceinline__ int64_t lower_bound_global(const uint64_t* a, int64_t len, uint64_t t) {
    int64_t base = 0;
    while (len > 1) {
        const int64_t half = len >> 1;
        base += __ldcg(a + base + half - 1) < t ? half : 0;
        len -= half;
    }
    return len == 1 && __ldcg(a + base) < t ? base + 1 : base;
}

template <int kSearchRows, int kSearchGroups>
__global__ void __launch_bounds__(kSearchRows * kSearchGroups) k_search_window(const SearchArgs a) {
    constexpr int kSearchThreads = kSearchRows * kSearchGroups;
    constexpr int CPT = 9 / kSearchGroups;    // (dx, dy) columns per thread
    static_assert(kSearchRows % 32 == 0 && CPT * kSearchGroups == 9, "a column group is whole warps");
    extern __shared__ uint64_t sh_search[];
    uint64_t* samp = sh_search;                  // [kSampleMax]
    uint64_t* win = sh_search + kSampleMax;      // [9][padded_cap(wcap)], padded (pad_idx)
    __shared__ int64_t wlo[9];
    __shared__ int32_t wlen[9];                  // -1: search this column in global memory
    __shared__ int64_t glen[9];                  // for those: the run [wlo, wlo + glen) searched there
    __shared__ int32_t wofs[10];                 // start of each column's run in the flat copy order
    __shared__ uint64_t qkey[kSearchRows + 1];   // the block's packed keys, [0] = the one before the block
    __shared__ uint32_t mpart[kSearchGroups][kSearchRows];   // each column group's mask bits of a row
    __shared__ int32_t wsteps;                   // halving steps that cover the longest run
    __shared__ int32_t cnt[kTaps];
    __shared__ int32_t err;
    const int t = threadIdx.x;
    const int g = t / kSearchRows;               // column group: (dx, dy) columns CPT g .. (warp-uniform)
    const int i = t % kSearchRows;               // the block's row this thread serves
    const int64_t n = a.n;
    const int rb = a.rb;
    const uint64_t rmask = (uint64_t(1) << rb) - 1;
    const uint64_t invalid_key = (uint64_t(1) << a.key_bits) - 1;
    const int64_t ns = ((n - 1) >> a.sample_shift) + 1;
    const int32_t wst = static_cast<int32_t>(padded_cap(a.wcap));   // column stride in win
    const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kSearchRows;
    const int64_t s_end = s0 + kSearchRows < n ? s0 + kSearchRows : n;
    if (t < kTaps) cnt[t] = 0;
    if (t == 0) err = 0;
    pdl_wait();   // the coordinate sort must have finished
    pdl_trigger();
    // every load of this phase is issued before any is used: the sample, this
    // block's keys and the key before the block
    constexpr int kSampPerThread = (kSampleMax + kSearchThreads - 1) / kSearchThreads;
    uint64_t sv8[kSampPerThread];
#pragma unroll
    for (int u = 0; u < kSampPerThread; ++u) {
        const int64_t j = t + static_cast<int64_t>(u) * kSearchThreads;
        sv8[u] = j < ns ? __ldcg(a.sv + (j << a.sample_shift)) : 0ull;
    }
    const int64_t s = s0 + i;
    const uint64_t vs = (g == 0 && s < n) ? __ldcg(a.sv + s) : ~uint64_t(0);
    const uint64_t before = (t == 0 && s0 > 0) ? __ldcg(a.sv + s0 - 1) : ~uint64_t(0);
#pragma unroll
    for (int u = 0; u < kSampPerThread; ++u) {
        const int64_t j = t + static_cast<int64_t>(u) * kSearchThreads;
        if (j < ns) samp[j] = sv8[u];
    }
    if (g == 0) qkey[i + 1] = vs;
    if (t == 0) qkey[0] = before;
    __syncthreads();
    // ---- bracket each column's run of lower bounds from the sample
    if (t < 9) {
        const uint64_t qf = qkey[1] >> rb;
        const uint64_t ql = qkey[s_end - s0] >> rb;
        int64_t lo = 0, len = 0, glob = n;
        if (qf == invalid_key) {
            len = 0;                              // no valid row in this block
        } else if (ql == invalid_key) {
            len = -1;                             // invalid rows at the end: search the whole array
        } else {
            const int64_t jf = lower_bound_in(samp, ns, (qf + a.koff[3 * t]) << rb);
            const int64_t jl = lower_bound_in(samp, ns, (ql + a.koff[3 * t]) << rb);
            lo = jf > 0 ? ((jf - 1) << a.sample_shift) + 1 : 0;
            int64_t hi = (jl << a.sample_shift) + 3;
            if (hi > n) hi = n;
            len = hi - lo;
            if (len > a.wcap) {                   // too long for shared memory: search the run in place
                glob = len;
                len = -1;
            }
        }
        glen[t] = glob;
        wlo[t] = lo;
        wlen[t] = static_cast<int32_t>(len);
    }
    __syncthreads();
    if (t == 0) {
        int32_t most = 0, at = 0;
        for (int c = 0; c < 9; ++c) {
            most = wlen[c] > most ? wlen[c] : most;
            wofs[c] = at;
            at += wlen[c] > 0 ? wlen[c] : 0;
        }
        wofs[9] = at;
        wsteps = 32 - __clz(most);
    }
    __syncthreads();
    // ---- copy the 9 runs as one flat list, kCopyBatch loads in flight per thread
    constexpr int kCopyBatch = 8;
    const int32_t total = wofs[9];
    for (int32_t e0 = t; e0 < total; e0 += kCopyBatch * kSearchThreads) {
        uint64_t v[kCopyBatch];
        int32_t slot[kCopyBatch];
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u) {
            const int32_t e = e0 + u * kSearchThreads;
            int c = 0;
#pragma unroll
            for (int q = 1; q < 9; ++q) c += e >= wofs[q] ? 1 : 0;
            const int32_t i = e - wofs[c];
            slot[u] = e < total ? c * wst + pad_idx(i) : -1;
            v[u] = e < total ? __ldcg(a.sv + wlo[c] + i) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u)
            if (slot[u] >= 0) win[slot[u]] = v[u];
    }
    __syncthreads();
    // ---- search: thread (g, i) finds row i's neighbours in columns CPT g ..
    // CPT g + CPT - 1 (taps 3 CPT g ..): lower bounds of its targets in the
    // shared runs, in lockstep and branch-free (a finished column re-reads a
    // valid slot)
    const uint64_t vrow = qkey[i + 1];
    uint32_t mp = 0;
    int32_t x9[3 * CPT];
#pragma unroll
    for (int k = 0; k < 3 * CPT; ++k) x9[k] = -1;
    int64_t r = -1;
    if (s < n) {
        const uint64_t q = vrow >> rb;
        r = static_cast<int64_t>(vrow & rmask);
        if (r >= n) {
            if (g == 0) atomicOr(&err, kStatusInternal);
            r = -1;
        }
        if (q != invalid_key) {
            if (g == 0 && s > 0 && (qkey[i] >> rb) == q) atomicOr(&err, kStatusDuplicate);
            uint64_t tl[CPT];
            int32_t base[CPT], len[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                const int cc = CPT * g + c;
                tl[c] = (q + a.koff[3 * cc]) << rb;
                base[c] = 0;
                len[c] = wlen[cc] > 0 ? wlen[cc] : 0;
            }
            for (int it = 0; it < wsteps; ++it) {
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    const int32_t half = len[c] >> 1;
                    const int32_t probe = base[c] + (half > 0 ? half - 1 : 0);
                    const uint64_t v = win[(CPT * g + c) * wst + pad_idx(probe)];
                    base[c] += (half > 0 && v < tl[c]) ? half : 0;
                    len[c] -= half;
                }
            }
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                const int cc = CPT * g + c;
                const uint64_t vb = win[cc * wst + pad_idx(base[c])];
                const int32_t pos = base[c] + ((len[c] == 1 && vb < tl[c]) ? 1 : 0);
                // the three candidates after the lower bound (clamped reads, masked)
                const uint64_t hi_k = q + a.koff[3 * cc + 2];
                const int32_t wl = wlen[cc];
                uint64_t cand[3];
                int32_t avail;
                if (wl >= 0) {
                    avail = wl - pos;
#pragma unroll
                    for (int j = 0; j < 3; ++j) {
                        const int32_t pp = pos + j < a.wcap ? pos + j : a.wcap - 1;
                        cand[j] = win[cc * wst + pad_idx(pp)];
                    }
                } else {   // a run too long for shared memory: search it in global memory
                    const int64_t gp = wlo[cc] + lower_bound_global(a.sv + wlo[cc], glen[cc], tl[c]);
                    avail = static_cast<int32_t>(n - gp < 3 ? n - gp : 3);
#pragma unroll
                    for (int j = 0; j < 3; ++j) cand[j] = gp + j < n ? __ldcg(a.sv + gp + j) : 0ull;
                }
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const uint64_t kk = cand[j] >> rb;
                    const bool hit = j < avail && kk <= hi_k;
                    const uint64_t dz = kk - (tl[c] >> rb);
                    const int64_t rr = static_cast<int64_t>(cand[j] & rmask);
                    const int32_t nr = rr < n ? static_cast<int32_t>(rr) : -1;
#pragma unroll
                    for (int d = 0; d < 3; ++d) x9[3 * c + d] = (hit && dz == static_cast<uint64_t>(d)) ? nr : x9[3 * c + d];
                }
#pragma unroll
                for (int d = 0; d < 3; ++d) mp |= (x9[3 * c + d] >= 0 ? 1u : 0u) << (3 * c + d);
            }
        }
    }
    mpart[g][i] = mp;
    // ---- stage the rows in shared memory (the runs are no longer needed):
    // chunk q (taps 4q .. 4q+3) of row j at chunk slot (q + j) & 7, so the 8
    // lanes that read a row hit distinct banks; then write each 128-byte row
    // with 8 lanes
    __syncthreads();
    int32_t* stage = reinterpret_cast<int32_t*>(sh_search);          // [kSearchRows][kNbrStride]
    int64_t* stage_row = reinterpret_cast<int64_t*>(stage + kSearchRows * kNbrStride);   // [kSearchRows]
    auto slot = [&](int tap) { return i * kNbrStride + (((tap >> 2) + i) & 7) * 4 + (tap & 3); };
#pragma unroll
    for (int k = 0; k < 3 * CPT; ++k) stage[slot(3 * CPT * g + k)] = x9[k];
    if (g == kSearchGroups - 1)
        for (int tap = kTaps; tap < kNbrStride; ++tap) stage[slot(tap)] = -1;
    uint32_t m = 0;
    if (g == 0) {
        stage_row[i] = r;
#pragma unroll
        for (int gg = 0; gg < kSearchGroups; ++gg) m |= mpart[gg][i] << (3 * CPT * gg);
        if (r >= 0) a.mask[r] = m;
        add_tap_counts(m, cnt);   // (warps 0 .. kSearchRows/32 - 1: whole warps)
    }
    __syncthreads();
    for (int j = t >> 3; j < kSearchRows; j += kSearchThreads / 8) {
        const int64_t rr = stage_row[j];
        if (rr >= 0) {
            const int qq = t & 7;
            reinterpret_cast<int4*>(a.nbr + rr * kNbrStride)[qq] =
                reinterpret_cast<const int4*>(stage + j * kNbrStride)[(qq + j) & 7];
        }
    }
    __syncthreads();
    if (t < kTaps && cnt[t]) atomicAdd(a.tap_count + t, cnt[t]);
    if (t == 0 && err) atomicOr(a.status, err);
}

}  // namespace

namespace {

template <int ROWS, int GROUPS>
int launch_search_rows(SearchArgs sa, int64_t n, cudaStream_t s) {
    // sample stride: the smallest power of two >= 64 giving at most kSampleMax samples
    int sh = 6;
    while (((n - 1) >> sh) + 1 > kSampleMax) ++sh;
    sa.sample_shift = sh;
    // run capacity: what a block needs at this stride, at most what the shared
    // memory attribute below covers (longer runs are searched in global memory)
    const int wcap_max = 2 * ROWS + 2 * static_cast<int>(kFusedMaxRows / kSampleMax);
    const int64_t want = 2 * ROWS + 2 * (int64_t(1) << sh);
    sa.wcap = static_cast<int>(want < wcap_max ? want : wcap_max);
    // the sample and runs, then (reusing them) the staged kernel-map rows and their row ids
    const size_t smem_search = (static_cast<size_t>(kSampleMax) + 9 * static_cast<size_t>(padded_cap(sa.wcap))) * sizeof(uint64_t);
    const size_t smem_stage = static_cast<size_t>(ROWS) * (kNbrStride * sizeof(int32_t) + sizeof(int64_t));
    const size_t smem = smem_search > smem_stage ? smem_search : smem_stage;
    // once per device, for the largest run buffer
    static bool smem_set[kMaxDevices] = {};
    int dev = 0;
    SPCONV_CHECK_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return SPCONV_ERR_UNSUPPORTED;
    if (!smem_set[dev]) {
        const int most = static_cast<int>((kSampleMax + 9 * static_cast<size_t>(padded_cap(wcap_max))) * sizeof(uint64_t));
        SPCONV_CHECK_CUDA(cudaFuncSetAttribute(k_search_window<ROWS, GROUPS>, cudaFuncAttributeMaxDynamicSharedMemorySize, most));
        smem_set[dev] = true;
    }
    cudaLaunchConfig_t scfg = {};
    scfg.gridDim = dim3(static_cast<unsigned>((n + ROWS - 1) / ROWS));
    scfg.blockDim = dim3(ROWS * GROUPS);
    scfg.dynamicSmemBytes = smem;
    scfg.stream = s;
    cudaLaunchAttribute sattr[1] = {pdl_attr()};
    scfg.attrs = sattr;
    scfg.numAttrs = 1;
    SPCONV_CHECK_CUDA(cudaLaunchKernelEx(&scfg, k_search_window<ROWS, GROUPS>, sa));
    return SPCONV_OK;
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
    return n > kSearchBigRows ? launch_search_rows<256, 1>(sa, n, s) : launch_search_rows<128, 3>(sa, n, s);
}

}  // namespace spconv

// Plain, slow CPU oracle for submanifold sparse convolution (K x K x K
// kernels, K odd: 3 and 5).
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of the
// build entry module and the CPU-baseline leg of the benchmark may load or
// call this code.  The product path never does, and the two share no code.
//
// What it computes (each function names the passage it follows):
//   * the kernel map: for every active voxel and each of the K^3 offsets, the
//     row of the neighbour at that offset, or -1 -- an exact set lookup
//     through a hash map ("Sparse convolution in FP32", section "The starting
//     point": the work is finding which neighbours exist);
//   * the neighbour mask of each row over a group of taps and the rows
//     sorted by it (same page, "Neighbour masks and sorted rows"; the bit
//     order may be the plain one or calibrated, same page, "Calibrated bit
//     order").  With one group (K = 3) the mask has all 27 bits; with the
//     taps partitioned into groups, each group has its own masks and its own
//     row order (same page, "Offset-group partitioning");
//   * the per-tap pair lists, each in the row order of its tap's group
//     (FlyDSL PR #942 summary, "Compaction is the largest single win": only
//     the valid pairs, grouped by tap);
//   * the convolution itself, out[i][o] = sum_k sum_c f[nbr[i][k]][c] W[k][c][o],
//     in fp64 ("Sparse convolution in FP32", "The starting point").
//
// Conventions (the pages leave them open; this is the reading used
// throughout):
//   r = (K-1)/2, tap k = K*K*(dx+r) + K*(dy+r) + (dz+r), offset
//   d = (dx,dy,dz) in {-r..r}^3, V = K^3 taps (k = 9(dx+1) + 3(dy+1) + (dz+1)
//   for K = 3);
//   nbr[i][k] = row of the voxel at coords[i] + d_k in the same batch, else -1;
//   weights are [V][C_in][C_out]; out = sum_k W[k]^T f(p + d_k)
//   (cross-correlation, as torch conv3d with padding r);
//   a group is a run of consecutive taps [k0, k0 + kg): with G groups of
//   V / G taps, group g holds the taps with dx = g - r when G = K.
#include <algorithm>
#include <array>
#include <cstdint>
#include <cstring>
#include <unordered_map>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

struct Voxel {
    int32_t b, x, y, z;
    bool operator==(const Voxel& o) const {
        return b == o.b && x == o.x && y == o.y && z == o.z;
    }
};

struct VoxelHash {
    size_t operator()(const Voxel& v) const {
        uint64_t h = 1469598103934665603ull;
        const int32_t f[4] = {v.b, v.x, v.y, v.z};
        for (int i = 0; i < 4; ++i) {
            h ^= static_cast<uint32_t>(f[i]);
            h *= 1099511628211ull;
        }
        return static_cast<size_t>(h);
    }
};

inline int tap_index(int K, int dx, int dy, int dz) {
    const int r = (K - 1) / 2;
    return K * K * (dx + r) + K * (dy + r) + (dz + r);
}

}  // namespace

extern "C" {

// Error codes match the meaning (not the implementation) of the library's.
enum { ORACLE_OK = 0, ORACLE_ERR_DUPLICATE = -5, ORACLE_ERR_RANGE = -6 };

// Kernel map by hash lookup.  coords: [n][4] (b,x,y,z).  shape: {X,Y,Z}.
// A coordinate outside 0 <= b < batch_size, 0 <= x < X, ... is an error, and
// so is a repeated coordinate.  K: odd kernel size.  nbr: [n][K^3].
int oracle_kernel_map(const int32_t* coords, int64_t n, const int32_t* shape,
                      int32_t batch_size, int32_t K, int32_t* nbr) {
    const int r = (K - 1) / 2;
    const int64_t V = static_cast<int64_t>(K) * K * K;
    std::unordered_map<Voxel, int32_t, VoxelHash> where;
    where.reserve(static_cast<size_t>(n) * 2 + 1);
    for (int64_t i = 0; i < n; ++i) {
        Voxel v{coords[4 * i], coords[4 * i + 1], coords[4 * i + 2], coords[4 * i + 3]};
        if (v.b < 0 || v.b >= batch_size || v.x < 0 || v.x >= shape[0] || v.y < 0 ||
            v.y >= shape[1] || v.z < 0 || v.z >= shape[2])
            return ORACLE_ERR_RANGE;
        if (!where.emplace(v, static_cast<int32_t>(i)).second) return ORACLE_ERR_DUPLICATE;
    }
    for (int64_t i = 0; i < n; ++i) {
        const int32_t* c = coords + 4 * i;
        for (int dx = -r; dx <= r; ++dx)
            for (int dy = -r; dy <= r; ++dy)
                for (int dz = -r; dz <= r; ++dz) {
                    Voxel q{c[0], c[1] + dx, c[2] + dy, c[3] + dz};
                    auto it = where.find(q);
                    nbr[V * i + tap_index(K, dx, dy, dz)] = it == where.end() ? -1 : it->second;
                }
    }
    return ORACLE_OK;
}

// Mask over the group of taps [k0, k0 + kg) (kg <= 32): mask[i] bit j set
// iff nbr[i][k0 + j] >= 0.  nbr rows have V entries.
void oracle_masks(const int32_t* nbr, int64_t n, int32_t V, int32_t k0, int32_t kg, uint32_t* mask) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t m = 0;
        for (int j = 0; j < kg; ++j)
            if (nbr[V * i + k0 + j] >= 0) m |= 1u << j;
        mask[i] = m;
    }
}

// Bit order of the sort key of one group of kg taps (masks as above).
// order[j] is the group's tap (bit of the mask) whose presence sets key bit j.
// calibrated == 0: plain order, order[j] = j.
// calibrated != 0: taps by descending number of rows that have them (ties by
// ascending tap index), so the rarest tap is the most significant key bit and
// rows that share rare taps end up next to each other.
void oracle_tap_order(const uint32_t* mask, int64_t n, int32_t kg, int calibrated, int32_t* order) {
    std::vector<int64_t> count(static_cast<size_t>(kg), 0);
    for (int64_t i = 0; i < n; ++i)
        for (int k = 0; k < kg; ++k) count[k] += (mask[i] >> k) & 1u;
    std::vector<int32_t> taps(static_cast<size_t>(kg));
    for (int k = 0; k < kg; ++k) taps[k] = k;
    if (calibrated)
        std::stable_sort(taps.begin(), taps.end(),
                         [&](int32_t a, int32_t b) { return count[a] > count[b]; });
    for (int j = 0; j < kg; ++j) order[j] = taps[j];
}

// key[i] = sum_j [tap order[j] present in row i] << j, j < kg.
void oracle_sort_keys(const uint32_t* mask, int64_t n, int32_t kg, const int32_t* order, uint32_t* key) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t k = 0;
        for (int j = 0; j < kg; ++j)
            if ((mask[i] >> order[j]) & 1u) k |= 1u << j;
        key[i] = k;
    }
}

// perm: rows in ascending key order; equal keys keep ascending row order.
void oracle_perm(const uint32_t* key, int64_t n, int32_t* perm) {
    std::vector<int32_t> rows(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) rows[i] = static_cast<int32_t>(i);
    std::stable_sort(rows.begin(), rows.end(),
                     [&](int32_t a, int32_t b) { return key[a] < key[b]; });
    std::memcpy(perm, rows.data(), sizeof(int32_t) * static_cast<size_t>(n));
}

// Per-tap pair lists, tap k in the row order of its group: perms holds G
// orders of n rows ([G][n]), the taps split into G groups of V / G
// consecutive taps.  tap_off: [V + 1], CSR offsets.  in_rows / out_rows: room
// for every pair (V n at most).  Returns the pair count P.
int64_t oracle_pair_lists(const int32_t* nbr, const int32_t* perms, int64_t n, int32_t V, int32_t G,
                          int32_t* tap_off, int32_t* in_rows, int32_t* out_rows) {
    int64_t p = 0;
    for (int k = 0; k < V; ++k) {
        tap_off[k] = static_cast<int32_t>(p);
        const int32_t* perm = perms + static_cast<int64_t>(k / (V / G)) * n;
        for (int64_t s = 0; s < n; ++s) {
            int32_t r = perm[s];
            int32_t j = nbr[static_cast<int64_t>(V) * r + k];
            if (j >= 0) {
                in_rows[p] = j;
                out_rows[p] = r;
                ++p;
            }
        }
    }
    tap_off[V] = static_cast<int32_t>(p);
    return p;
}

// out[r][o] = sum_{k<V} sum_c feats[nbr[r][k]][c] * weights[k][c][o] in fp64, for
// the rows listed in rows[0..n_rows) (all rows when rows == NULL, then
// n_rows == n).  out is [n_rows][c_out], in the order of rows.
void oracle_conv_f64(const int32_t* nbr, int32_t V, const int32_t* rows, int64_t n_rows,
                     const double* feats, const double* weights, int32_t c_in, int32_t c_out,
                     double* out, int32_t threads) {
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 64) num_threads(threads)
#endif
    for (int64_t t = 0; t < n_rows; ++t) {
        int64_t r = rows ? rows[t] : t;
        double* o = out + t * c_out;
        for (int32_t q = 0; q < c_out; ++q) o[q] = 0.0;
        for (int k = 0; k < V; ++k) {
            int32_t j = nbr[static_cast<int64_t>(V) * r + k];
            if (j < 0) continue;
            const double* f = feats + static_cast<int64_t>(j) * c_in;
            const double* w = weights + static_cast<int64_t>(k) * c_in * c_out;
            for (int32_t c = 0; c < c_in; ++c) {
                const double fc = f[c];
                const double* wr = w + static_cast<int64_t>(c) * c_out;
                for (int32_t q = 0; q < c_out; ++q) o[q] += fc * wr[q];
            }
        }
    }
}

// Strided (downsampling) convolution, kernel 3, stride 2, padding 1 ("Sparse
// convolution in FP32", "Calibrated bit order": the strided kernels change
// the coordinate set).  Output shape X' = (X - 1) / 2 + 1 per axis (torch
// conv3d with kernel 3, stride 2, padding 1).  The output sites are every o
// in [0, X') x [0, Y') x [0, Z') of a batch whose window {2o + d : d in
// {-1,0,1}^3} holds an input site, in ascending (b, x, y, z) order;
// nbr[o][k] = the input row at 2o + d_k, else -1 (tap k as above, K = 3).
// out_coords: room for 8 n rows (an input site lies in at most 8 windows).
// Returns the number of output sites.
int64_t oracle_strided_map(const int32_t* coords, int64_t n, const int32_t* shape, int32_t batch_size,
                           int32_t* out_coords, int32_t* nbr) {
    std::unordered_map<Voxel, int32_t, VoxelHash> where;
    where.reserve(static_cast<size_t>(n) * 2 + 1);
    for (int64_t i = 0; i < n; ++i) {
        Voxel v{coords[4 * i], coords[4 * i + 1], coords[4 * i + 2], coords[4 * i + 3]};
        if (v.b < 0 || v.b >= batch_size || v.x < 0 || v.x >= shape[0] || v.y < 0 ||
            v.y >= shape[1] || v.z < 0 || v.z >= shape[2])
            return ORACLE_ERR_RANGE;
        if (!where.emplace(v, static_cast<int32_t>(i)).second) return ORACLE_ERR_DUPLICATE;
    }
    const int32_t os[3] = {(shape[0] - 1) / 2 + 1, (shape[1] - 1) / 2 + 1, (shape[2] - 1) / 2 + 1};
    // every output whose window holds an input: o = (c - d) / 2 with c - d even, inside the output shape
    std::vector<std::array<int32_t, 4>> outs;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t* c = coords + 4 * i;
        for (int dx = -1; dx <= 1; ++dx)
            for (int dy = -1; dy <= 1; ++dy)
                for (int dz = -1; dz <= 1; ++dz) {
                    const int32_t px = c[1] - dx, py = c[2] - dy, pz = c[3] - dz;
                    if (px < 0 || py < 0 || pz < 0 || px % 2 || py % 2 || pz % 2) continue;
                    const std::array<int32_t, 4> o = {c[0], px / 2, py / 2, pz / 2};
                    if (o[1] < os[0] && o[2] < os[1] && o[3] < os[2]) outs.push_back(o);
                }
    }
    std::sort(outs.begin(), outs.end());
    outs.erase(std::unique(outs.begin(), outs.end()), outs.end());
    for (size_t j = 0; j < outs.size(); ++j) {
        for (int a = 0; a < 4; ++a) out_coords[4 * j + a] = outs[j][a];
        for (int dx = -1; dx <= 1; ++dx)
            for (int dy = -1; dy <= 1; ++dy)
                for (int dz = -1; dz <= 1; ++dz) {
                    Voxel q{outs[j][0], 2 * outs[j][1] + dx, 2 * outs[j][2] + dy, 2 * outs[j][3] + dz};
                    auto it = where.find(q);
                    nbr[27 * j + tap_index(3, dx, dy, dz)] = it == where.end() ? -1 : it->second;
                }
    }
    return static_cast<int64_t>(outs.size());
}

// The map of the inverse (transposed) convolution of a strided map: rows are
// the strided map's input sites, inv[i][k] = the output site o with
// 2o + d_k = the site of row i (there is at most one), else -1.
void oracle_inverse_map(const int32_t* nbr, int64_t n_out, int64_t n_in, int32_t* inv) {
    for (int64_t i = 0; i < 27 * n_in; ++i) inv[i] = -1;
    for (int64_t o = 0; o < n_out; ++o)
        for (int k = 0; k < 27; ++k) {
            const int32_t i = nbr[27 * o + k];
            if (i >= 0) inv[27 * static_cast<int64_t>(i) + k] = static_cast<int32_t>(o);
        }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

}  // extern "C"

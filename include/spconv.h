/*
 * spconv.h -- C ABI of the GB300 (sm_103a) submanifold sparse convolution
 * (3x3x3 and 5x5x5 kernels, stride 1).
 *
 * The operation (FlyDSL PR #942, "Add submanifold sparse 3D convolution",
 * Summary: raw voxel coordinates in, output features out, the kernel map built
 * internally; "Sparse convolution in FP32", section "The starting point": for
 * every active voxel, the sum over its 27 neighbours of the neighbour's
 * features times the weights of that kernel offset; FlyDSL PR #942, "Test
 * plan": kernel sizes 3 and 5):
 *
 *     out[i][o] = sum_{k=0..V-1} sum_{c} f[nbr[i][k]][c] * W[k][c][o]
 *
 * over the rows i of the input, where nbr[i][k] is the row of the voxel at
 * coords[i] + d_k (same batch index), the term skipped when there is none.
 * Kernel size K (3 or 5), radius r = (K-1)/2, V = K^3 taps; tap order
 * k = K*K*(dx+r) + K*(dy+r) + (dz+r) for d = (dx,dy,dz) in {-r..r}^3, i.e.
 * k = 9*(dx+1) + 3*(dy+1) + (dz+1) for K = 3 (cross-correlation, as torch
 * conv3d with padding r).  Outputs live at the input sites, in the input row
 * order.
 *
 * Memory: every pointer argument named *_dev is a device pointer that the
 * caller owns; host pointers are marked host.  The library allocates only map
 * handles and packed-weight handles (stream-ordered, on the stream passed to
 * the creating call) and frees them in the matching destroy call.
 *
 * Streams: all work is enqueued on the caller's stream; nothing synchronises
 * the device except where a function says it does.
 *
 * Errors: functions return SPCONV_OK (0) or a negative spconv_status_t.
 * Argument errors are detected on the host before any work is enqueued.
 * Data errors found on the device (duplicate or out-of-range coordinates) are
 * recorded in the map handle and reported by spconv_map_status(); the map's
 * contents are then unspecified, but every kernel stays within its buffers.
 * No kernel traps; bounded waits inside kernels report SPCONV_ERR_TIMEOUT.
 */
#ifndef SPCONV_H_
#define SPCONV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPCONV_OK = 0,
    SPCONV_ERR_INVALID_ARG = -1,   /* null pointer, bad size, bad enum, misaligned buffer */
    SPCONV_ERR_UNSUPPORTED = -2,   /* valid request outside what this build implements    */
    SPCONV_ERR_OOM = -3,           /* device allocation failed                             */
    SPCONV_ERR_CUDA = -4,          /* a CUDA runtime call failed                            */
    SPCONV_ERR_DUPLICATE_COORD = -5,
    SPCONV_ERR_COORD_RANGE = -6,   /* b, x, y or z outside [0, batch) x [0, shape)          */
    SPCONV_ERR_ALIAS = -7,         /* out overlaps feats                                     */
    SPCONV_ERR_TIMEOUT = -8,       /* a bounded wait inside a kernel ran out                 */
    SPCONV_ERR_INTERNAL = -9       /* a kernel's consistency guard fired (a library bug)     */
} spconv_status_t;

typedef enum { SPCONV_BF16 = 0, SPCONV_FP32 = 1 } spconv_dtype_t;

typedef enum {
    SPCONV_MAPPER_AUTO = 0,   /* dense grid iff padded cells <= dense_max_cells, else HASH when
                                 the WIDE pipeline or a grouped K = 3 build makes the map, else
                                 SORTED                                                           */
    SPCONV_MAPPER_DENSE = 1,  /* presence grid over the padded bounding box                       */
    SPCONV_MAPPER_SORTED = 2, /* sorted 64-bit keys + binary search, memory O(N)                   */
    SPCONV_MAPPER_HASH = 3    /* the same packed keys in an open-addressing hash table, one
                                 bucket read per pair of z neighbours; memory O(N).  The WIDE
                                 pipeline and grouped builds only (the FUSED and MULTI
                                 pipelines with one group: SPCONV_ERR_UNSUPPORTED)                 */
} spconv_mapper_t;

typedef enum {
    SPCONV_ORDER_CALIBRATED = 0, /* sort key bits by descending tap frequency (rarest tap = MSB) */
    SPCONV_ORDER_PLAIN = 1       /* sort key = the mask itself                                    */
} spconv_bit_order_t;

typedef enum {
    SPCONV_PIPELINE_AUTO = 0,  /* WIDE when it applies, else FUSED when it applies, else MULTI    */
    SPCONV_PIPELINE_FUSED = 1, /* whole build in one thread-block-cluster launch (n <= 2^20)     */
    SPCONV_PIPELINE_MULTI = 2, /* one kernel per step, three per 8-bit sort pass (any n)          */
    SPCONV_PIPELINE_WIDE = 3   /* one kernel per step on the whole GPU, look-back sort passes     */
                               /* (n <= 2^26; sorted mapper: coordinate keys of at most 40 bits) */
} spconv_pipeline_t;

/* Work decomposition of the bf16 tensor-core forward ("Compaction is the
 * largest single win", FlyDSL PR #942; "Offset-group partitioning", "Sparse
 * convolution in FP32").  Both give the same sums up to fp32 rounding order. */
typedef enum {
    SPCONV_GEMM_AUTO = 0,        /* TILE_UNION (measured faster on every tested workload)      */
    SPCONV_GEMM_TILE_UNION = 1,  /* output-stationary: 128 mask-sorted rows per tile, all taps of
                                    the tile's mask union accumulated on chip, one bf16 store;
                                    deterministic                                             */
    SPCONV_GEMM_TAP_MAJOR = 2    /* 128 pairs of one tap per tile (compacted pair lists, no
                                    zero rows), fp32 sums added in an [n][c_out] workspace,
                                    then rounded to bf16; summation order varies run to run   */
} spconv_gemm_t;

/* Options of spconv_build_map.  Pass NULL for the defaults.  None of them
 * changes any result beyond fp32 rounding order; they select how the same
 * map is built and used. */
typedef struct {
    int32_t mapper;          /* spconv_mapper_t, default AUTO                          */
    int32_t bit_order;       /* spconv_bit_order_t, default CALIBRATED                 */
    int64_t dense_max_cells; /* AUTO threshold on B*(X+2)*(Y+2)*(Z+2); default 1<<24   */
    int32_t pipeline;        /* spconv_pipeline_t, default AUTO                        */
    int32_t gemm;            /* spconv_gemm_t for the bf16 forward on this map, default AUTO */
    int32_t groups;          /* offset groups ("Sparse convolution in FP32", "Offset-group
                                partitioning"): the V taps split into G runs of V/G
                                consecutive taps (G = K: the taps of one dx each), every
                                group with its own masks, row order and tiles, the forward
                                one GEMM pass per group.  0: default (1 for K = 3, 5 for
                                K = 5); 1 (K = 3 only) or K.  G > 1 builds with the MULTI
                                pipeline and the TILE_UNION forward; other choices of
                                pipeline or gemm return SPCONV_ERR_UNSUPPORTED.           */
} spconv_options_t;

typedef struct spconv_map_s* spconv_map_t;
typedef struct spconv_wpack_s* spconv_wpack_t;

/*
 * Epilogue of a forward: what happens to each fp32 sum of output row i,
 * channel o before its one rounding to the output dtype.  The inference form
 * of a layer's batch norm (a per-channel scale and shift), its bias, a
 * residual branch and the ReLU between layers, fused into the store so that
 * they cost no extra pass over [n][c_out].  The pages' networks are stacks of
 * such layers (FlyDSL PR #942, "Open questions": a layer stack with
 * normalisation and residuals; "Sparse convolution in FP32", "Offset-group
 * partitioning": the convolution's last launch applies the ReLU to every row):
 *
 *   y = sum * scale[o] + bias[o] + residual[i][o];   out[i][o] = relu ? max(y, 0) : y
 *
 *   scale_dev     fp32 [c_out], device, 16-byte aligned; NULL means 1.
 *   bias_dev      fp32 [c_out], device, 16-byte aligned; NULL means 0.
 *   residual_dev  [n][c_out] in the forward's dtype, device, 16-byte aligned,
 *                 row-major in the original row order; NULL means 0.  It may
 *                 be out_dev itself (an in-place add) or feats_dev, but must
 *                 not partly overlap out_dev (SPCONV_ERR_ALIAS).
 *   relu          0: none, 1: max(y, 0).  Other values: SPCONV_ERR_INVALID_ARG.
 * The caller owns every buffer; the library only reads them, in stream order.
 */
typedef struct {
    const float* scale_dev;
    const float* bias_dev;
    const void* residual_dev;
    int32_t relu;
} spconv_epilogue_t;

/* Summary of a built map.  Filling it synchronises the map's stream. */
typedef struct {
    int64_t n;           /* active voxels (rows)                                  */
    int64_t pairs;       /* P = number of (row, tap) with a neighbour (>= n)      */
    int64_t n_tiles;     /* 128-row tiles of the mask-sorted order (per group)    */
    int64_t tile_taps;   /* sum over tiles (all groups) of the taps in the tile's mask union */
    int32_t mapper;      /* spconv_mapper_t actually used (DENSE, SORTED or HASH) */
    int32_t pipeline;    /* spconv_pipeline_t actually used (FUSED, MULTI, WIDE)  */
    int32_t key_bits;    /* live bits of the packed coordinate key                */
    int32_t shape[3];    /* spatial shape used                                    */
    int32_t batch_size;  /* batch size used                                       */
    int32_t gemm;        /* spconv_gemm_t the bf16 forward uses (TILE_UNION or TAP_MAJOR) */
    int32_t kernel_size; /* K                                                     */
    int32_t groups;      /* G offset groups                                       */
    int64_t n_in;        /* rows of the features a forward reads (n but for strided and inverse maps) */
    int32_t conv;        /* 0 submanifold, 1 strided, 2 inverse of a strided map  */
    int32_t out_shape[3];/* spatial shape of the map's rows (a strided map: the output grid) */
} spconv_map_info_t;

/*
 * Build the kernel map of a coordinate set (FlyDSL PR #942, "Two mappers, both
 * required"; "Sparse convolution in FP32", "Neighbour masks and sorted rows";
 * FlyDSL PR #942, "Compaction is the largest single win").
 *
 *   coords_dev     int32 [n][4] rows (b, x, y, z), device, row-major.  Must stay
 *                  valid until the stream has passed this call; the handle
 *                  keeps what it needs.
 *   n              number of rows, 0 <= n < 2^30.
 *   spatial_shape  host int32[3] {X, Y, Z}, each >= 1; NULL derives max+1 per
 *                  axis on the device (synchronises the stream).
 *   batch_size     frames, >= 1; 0 derives max(b)+1 (synchronises the stream).
 *   kernel_size    3 or 5 (others return SPCONV_ERR_UNSUPPORTED).
 *   opt            options, NULL for defaults.
 *   stream         CUDA stream (cudaStream_t) the work is enqueued on.
 *   out_map        receives the handle; free it with spconv_map_destroy.
 *
 * Device-side results (all in the handle): the kernel map nbr[n][V]; per
 * offset group its masks (bit j: the group's tap j present), perm (rows in
 * ascending sort-key order, ties by row) and 128-row tile work list; the
 * per-tap pair lists, each in the order of its tap's group.
 */
int spconv_build_map(const int32_t* coords_dev, int64_t n, const int32_t* spatial_shape,
                     int32_t batch_size, int32_t kernel_size, const spconv_options_t* opt,
                     void* stream, spconv_map_t* out_map);

/*
 * The map of a strided (downsampling) sparse convolution: kernel 3, stride 2,
 * padding 1 per axis ("Sparse convolution in FP32", "Calibrated bit order":
 * the strided kernels, which change the coordinate set).  Its rows are the
 * output sites: every o of the output grid, X' = (X - 1) / 2 + 1 per axis,
 * whose window {2o + d : d in {-1,0,1}^3} holds an input site of the same
 * batch, in ascending (b, x, y, z) order; tap k of row o is the input row at
 * 2o + d_k.  A forward on it computes out[o] = sum_k W[k]^T f(2o + d_k):
 * feats [n][c_in] on the input sites, out [n_out][c_out] (torch conv3d with
 * stride 2 and padding 1, read at the output sites).
 *
 *   coords_dev, n, spatial_shape, batch_size: as spconv_build_map (n < 2^27).
 *   kernel_size 3 and stride 2 only (else SPCONV_ERR_UNSUPPORTED).
 *   opt: mapper AUTO or HASH, pipeline AUTO or MULTI, gemm not TAP_MAJOR,
 *        groups 0 or 1 (else SPCONV_ERR_UNSUPPORTED).
 * Synchronises the stream once: the number of output sites sizes the map.
 * spconv_map_rows gives n (output sites) and n_in without a second
 * synchronisation; spconv_map_info also out_shape;
 * spconv_map_out_coords copies the output sites' coordinates.
 */
int spconv_build_map_strided(const int32_t* coords_dev, int64_t n, const int32_t* spatial_shape,
                             int32_t batch_size, int32_t kernel_size, int32_t stride, const spconv_options_t* opt,
                             void* stream, spconv_map_t* out_map);

/*
 * The map of the inverse (transposed) convolution of a strided map: rows are
 * the strided map's input sites (its n_in), tap k of row i is the output site
 * o with 2o + d_k at site i, or none.  A forward on it computes
 * out[i] = sum_k W[k]^T g(o_k(i)) with g [n_out][c_in] on the strided map's
 * output sites and out [n_in][c_out] (torch conv_transpose3d, stride 2,
 * padding 1, read at the input sites).  Enqueued on the strided map's stream,
 * which the strided map must outlive until then; no synchronisation.
 * opt: bit_order and gemm (not TAP_MAJOR) are used; NULL for defaults.
 */
int spconv_build_map_inverse(spconv_map_t strided, const spconv_options_t* opt, spconv_map_t* out_map);

/* Copy a strided map's output sites, int32 [n][4] (b, x, y, z), to caller
 * device memory, enqueued on stream.  SPCONV_ERR_INVALID_ARG for other maps. */
int spconv_map_out_coords(spconv_map_t map, int32_t* out_coords_dev, void* stream);

/*
 * out = subm_conv(feats, weights) over the map's sites (the definition at the
 * top of this file).
 *
 *   feats_dev    [n_in][c_in] row-major, dtype elements, 16-byte aligned
 *                (n_in = n but for strided and inverse maps, spconv_map_info).
 *   weights_dev  [V][c_in][c_out] row-major, dtype elements (V = K^3 of the map).
 *   out_dev      [n][c_out] row-major, dtype elements, 16-byte aligned; must
 *                not overlap feats (SPCONV_ERR_ALIAS).
 *   dtype        SPCONV_BF16: bf16 in/out, fp32 accumulation, one rounding to
 *                bf16 at the store (tensor cores when c_in % 8 == 0 and
 *                c_out % 16 == 0, else a SIMT kernel).  SPCONV_FP32: fp32
 *                in/out with fp32 FMA on the SIMT path (exact mode).
 * Packs the weights into a workspace owned by the map on every call; use
 * spconv_wpack_create + spconv_subm_forward_packed to pack once.
 */
int spconv_subm_forward(spconv_map_t map, const void* feats_dev, const void* weights_dev,
                        void* out_dev, int32_t c_in, int32_t c_out, int32_t dtype, void* stream);

/* spconv_subm_forward with an epilogue (spconv_epilogue_t above; NULL is the
 * plain forward).  Same arguments, layouts and errors otherwise. */
int spconv_subm_forward_ex(spconv_map_t map, const void* feats_dev, const void* weights_dev,
                           void* out_dev, int32_t c_in, int32_t c_out, int32_t dtype,
                           const spconv_epilogue_t* epi, void* stream);

/*
 * Pre-pack weights [27][c_in][c_out] of a 3x3x3 kernel for repeated forwards (FlyDSL PR #942,
 * "Weight layout is [kv, t, k_outer, u, k_inner]": a packed tile layout; here
 * the tensor-core shared-memory image).  The handle owns a copy; the source
 * may be freed once the stream has passed this call.
 */
int spconv_wpack_create(const void* weights_dev, int32_t c_in, int32_t c_out, int32_t dtype,
                        void* stream, spconv_wpack_t* out_wpack);
int spconv_subm_forward_packed(spconv_map_t map, const void* feats_dev, spconv_wpack_t wpack,
                               void* out_dev, void* stream);
/* spconv_subm_forward_packed with an epilogue (NULL: none). */
int spconv_subm_forward_packed_ex(spconv_map_t map, const void* feats_dev, spconv_wpack_t wpack,
                                  void* out_dev, const spconv_epilogue_t* epi, void* stream);
/* spconv_wpack_create for a kernel of size kernel_size (3 or 5): weights
 * [K^3][c_in][c_out].  A packed forward on a map of another kernel size returns
 * SPCONV_ERR_INVALID_ARG. */
int spconv_wpack_create_ex(const void* weights_dev, int32_t kernel_size, int32_t c_in, int32_t c_out,
                           int32_t dtype, void* stream, spconv_wpack_t* out_wpack);
void spconv_wpack_destroy(spconv_wpack_t wpack);

/*
 * A stack of n_layers submanifold convolutions over one kernel map in a single
 * launch ("Sparse convolution in FP32", "Offset-group partitioning": the
 * convolution's last step applies the ReLU to every output row; layers that
 * share one coordinate set share one map, FlyDSL PR #942, "API style").
 * Layer l computes out_l = epilogue_l(conv(in_l, W_l)) with in_0 = feats and
 * in_l = out_{l-1}; every layer visits the same mask-sorted tiles and gather
 * table.  A layer's gathers start only after every CTA has stored the layer
 * before it, so each layer's result equals that of a separate
 * spconv_subm_forward_packed_ex call, bit for bit.
 *
 *   map        a submanifold map with one offset group and the tile-union GEMM
 *              (else SPCONV_ERR_UNSUPPORTED when n_layers > 1).
 *   feats_dev  bf16 [n][c_in], 16-byte aligned.
 *   wpacks     n_layers bf16 tensor-core weight packs (spconv_wpack_create),
 *              all c_in -> c_out with c_in == c_out when n_layers > 1.
 *   outs_dev   n_layers bf16 [n][c_out] outputs, 16-byte aligned, caller-owned;
 *              outs_dev[l] must not overlap its own input (feats_dev for l = 0,
 *              else outs_dev[l - 1]): SPCONV_ERR_ALIAS.  outs_dev[l] may equal
 *              outs_dev[l - 2] (two buffers ping-pong).
 *   n_layers   1 .. 8.
 *   epis       n_layers epilogues (each as in spconv_subm_forward_ex), or NULL.
 *   stream     CUDA stream; with n_layers > 1 the launch is cooperative (one
 *              CTA per SM, all resident) and uses a small per-map counter array.
 * Device-side waits between layers are bounded: a stall sets
 * SPCONV_ERR_TIMEOUT in the map's status (spconv_map_status).
 */
int spconv_subm_forward_layers(spconv_map_t map, const void* feats_dev, const spconv_wpack_t* wpacks,
                               void* const* outs_dev, int32_t n_layers, const spconv_epilogue_t* epis,
                               void* stream);

/* Synchronise the map's stream and return the first device-detected error
 * (duplicate or out-of-range coordinates, kernel timeouts), else SPCONV_OK. */
int spconv_map_status(spconv_map_t map);

/* Fill *info (synchronises the map's stream). */
int spconv_map_info(spconv_map_t map, spconv_map_info_t* info);

/*
 * The map's row count (output sites) and the count of the sites its
 * neighbours index (n_in; = rows but for strided and inverse maps), both
 * known on the host once the build call has returned: no synchronisation
 * and no device access.  Either pointer may be NULL.  Returns
 * SPCONV_ERR_INVALID_ARG for a NULL map.
 */
int spconv_map_rows(spconv_map_t map, int64_t* n, int64_t* n_in);

/*
 * Copy the map's arrays into caller device buffers (any may be NULL):
 *   nbr_dev int32 [n][V]; mask_dev uint32 [G][n]; perm_dev int32 [G][n];
 *   tap_off_dev int32 [V + 1]; in_rows_dev, out_rows_dev int32 [pairs].
 * Enqueued on stream; no synchronisation.
 */
int spconv_map_export(spconv_map_t map, int32_t* nbr_dev, uint32_t* mask_dev, int32_t* perm_dev,
                      int32_t* tap_off_dev, int32_t* in_rows_dev, int32_t* out_rows_dev,
                      void* stream);

/* Free the handle (stream-ordered on the stream of the build). */
void spconv_map_destroy(spconv_map_t map);

/*
 * The kernel map nbr[n][27] of a coordinate set without allocating any device
 * memory.  The pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate at the point where they run this code (a
 * plugin's enqueue step in an inference runtime that plans all device memory
 * up front, runtimes that forbid allocation after start-up).
 *
 *   coords_dev     int32 [n][4] rows (b, x, y, z), device, 16-byte aligned.
 *   n              0 <= n <= 65536; larger n returns SPCONV_ERR_INVALID_ARG
 *                  (the working buffers live in a fixed 1.6 MB device array).
 *   spatial_shape  host int32[3] {X, Y, Z} (required).
 *   batch_size     >= 1 (required).
 *   nbr_dev        int32 [n][27] output, caller-owned: the same values as the
 *                  nbr that spconv_map_export returns for this input.
 *   stream         CUDA stream; the call synchronises it before returning and
 *                  returns SPCONV_ERR_DUPLICATE_COORD / SPCONV_ERR_COORD_RANGE
 *                  for bad coordinates.
 *
 * No cudaMalloc, cudaFree or allocating library routine is called.  The
 * working buffers are one file-scope device array that every GPU loading this
 * library holds until the process exits; the first call on a device looks up
 * its address (make that first call before any stream capture).  All calls
 * share the array, so calls whose work overlaps on the GPU (different streams
 * or threads) race; serialise them.
 */
int spconv_kernel_map_static(const int32_t* coords_dev, int64_t n, const int32_t* spatial_shape,
                             int32_t batch_size, int32_t* nbr_dev, void* stream);

/* Number of kernel launches enqueued by the last call on this thread. */
int32_t spconv_last_launch_count(void);

/*
 * Diagnostics: runs one of the bounded device waits of the sort passes
 * against a state that nothing will ever publish, so that it must give up.
 * The pages have no counterpart; every device wait of the library ends after
 * a time limit (2 s in the product path) with SPCONV_ERR_TIMEOUT instead of
 * hanging the GPU, and this call shows that path working with a short limit.
 *
 *   which     0: the decoupled look-back of a sort pass, waiting for a
 *             predecessor partition whose state stays unpublished;
 *             1: the grid barrier of a two-CTA grid of which only one CTA
 *             runs;
 *             2: the flag wait of a pass that sums its predecessors'
 *             counts, on a flag that stays unset.
 *   limit_ns  the wait's limit, 1 ms .. 100 ms.
 *   stream    CUDA stream; the call allocates a few hundred bytes
 *             stream-ordered, synchronises the stream and frees them.
 *
 * Returns SPCONV_ERR_TIMEOUT when the wait ran out as designed (the GPU
 * context stays usable), SPCONV_ERR_INVALID_ARG for a bad argument, or
 * SPCONV_ERR_CUDA.
 */
int spconv_selftest_wait_timeout(int32_t which, int64_t limit_ns, void* stream);

const char* spconv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPCONV_H_ */

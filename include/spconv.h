/*
 * spconv.h - C ABI of the GB300 (sm_103a) submanifold sparse 3-D convolution.
 *
 * The operation is the one defined on the page "sparse_conv_metal.py"
 * (trellis-2-mrp-mlx, mlx_backend):
 *
 *     out[n, co] = bias[co] + sum_k sum_ci feats[nmap[k, n], ci] * w[k, ci, co]
 *
 * (module docstring: the fused gather-GEMM-accumulate formula; kernel body:
 * an entry that is not a valid row contributes nothing and accumulation is in
 * fp32; wrapper: the (K, N) int32 map with N marking a missing neighbour,
 * weights laid out (K, Ci, Co), output (N, Co) in the weights' type, bias
 * added to the result).  The page takes the neighbour map as given; this
 * library also builds it from voxel coordinates with a GPU hash table.
 *
 * Conventions for every call:
 *  - Pointers named *_dev are device pointers; *_host are host pointers.  The
 *    caller owns all memory; no call allocates or frees device memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued on it; only spconv_build_nmap and
 *    spconv_device_status wait for the stream (they read back a flag).
 *  - Arrays are dense, row-major, with no padding: coords (N, 3) int32 in
 *    (z, y, x) order; offsets (K, 3) int32 in (dz, dy, dx) order; nmap (K, N)
 *    int32, nmap[k * N + n]; feats (N, Ci); w (K, Ci, Co); bias (Co); out
 *    (N, Co).
 *  - Return value: SPCONV_OK (0) or a negative spconv_status.  On error a
 *    message is available from spconv_last_error() in the calling thread, and
 *    nothing has been enqueued unless the status is SPCONV_ERR_CUDA.
 *  - Every call needs a GPU of compute capability 10.3 (GB300) as the current
 *    device; other devices get SPCONV_ERR_UNSUPPORTED.
 */
#ifndef SPCONV_H
#define SPCONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPCONV_VERSION 1

/* A maximum on the number of offsets spconv_build_nmap accepts (7^3). */
#define SPCONV_MAX_BUILD_OFFSETS 343

/* Coordinates must satisfy 0 <= c < SPCONV_COORD_LIMIT in every component. */
#define SPCONV_COORD_LIMIT (1 << 20)

typedef enum spconv_status {
    SPCONV_OK = 0,
    SPCONV_ERR_INVALID_ARG = -1,      /* null pointer, bad size, misaligned pointer, coord range */
    SPCONV_ERR_UNSUPPORTED = -2,      /* shape/dtype/device combination not implemented */
    SPCONV_ERR_WORKSPACE = -3,        /* workspace smaller than the size query returned */
    SPCONV_ERR_DUPLICATE_COORD = -4,  /* two voxels share a coordinate */
    SPCONV_ERR_CUDA = -5,             /* a CUDA runtime call or launch failed */
    SPCONV_ERR_DEVICE = -6            /* a kernel reported an internal error (see spconv_device_status) */
} spconv_status;

typedef enum spconv_dtype {
    SPCONV_F32 = 0,   /* fp32 storage, fp32 products and fp32 accumulation (CUDA cores) */
    SPCONV_TF32 = 1,  /* fp32 storage, tf32 tensor-core products (the MMA reads each fp32
                         operand's sign, exponent and top 10 mantissa bits), fp32
                         accumulation, fp32 output; within 4e-3 * sum|terms| */
    SPCONV_BF16 = 2   /* bf16 storage, bf16 tensor-core products, fp32 accumulation, bf16 output */
} spconv_dtype;

/* SPCONV_VERSION of the loaded library. */
int spconv_version(void);

/* Message for the last failing call in this thread ("" if none). The
 * pointer stays valid until the thread's next spconv call. */
const char* spconv_last_error(void);

/*
 * Bytes of device workspace spconv_build_nmap needs for N voxels: a hash table
 * of the next power of two >= 2N slots (16 bytes each, at least 64 slots)
 * plus 256 bytes of flags.  Returns 0 if N < 0.
 */
size_t spconv_build_nmap_workspace_size(int64_t N);

/*
 * Build the neighbour map the convolution consumes (the (K, N) int32 map of
 * the page's wrapper docstring, missing neighbours marked with N):
 *
 *     nmap[k, n] = m   if coords[m] == coords[n] + offsets[k] (componentwise)
 *     nmap[k, n] = N   otherwise (including neighbours outside [0, 2^20)^3)
 *
 *  coords_dev     (N, 3) int32, device, any order; indices in nmap refer to it.
 *                 Components must lie in [0, SPCONV_COORD_LIMIT) and rows
 *                 must be distinct.
 *  N              number of voxels, 0 <= N < 2^31 - 1.  N == 0 is a no-op.
 *  offsets_host   (K, 3) int32, host; read during the call only.
 *  K              1 <= K <= SPCONV_MAX_BUILD_OFFSETS.
 *  nmap_dev       (K, N) int32, device, written.
 *  workspace_dev  device scratch of at least spconv_build_nmap_workspace_size(N)
 *                 bytes, 256-byte aligned; contents on entry are ignored and
 *                 undefined on exit.  It must not be used by another call
 *                 until this one returns.
 *  stream         cudaStream_t (as void*).
 *
 * The call enqueues its kernels and then waits for the stream once to read
 * the error flags, so it cannot be captured into a CUDA graph.  A first
 * kernel checks the coordinate range and whether the coordinates are
 * strictly increasing in (z, y, x) order and finds their bounding box; the
 * device then takes one of three paths (the other paths' kernels return at
 * once).  Strictly increasing input, as a voxeliser emits it, whose box's
 * rows fit the workspace lays the box out as words of 32 cells (an
 * occupancy bit per cell and the index of the word's first voxel), so a
 * neighbour is one word load; other strictly increasing input builds a
 * hash of (z, y) rows and finds neighbours by searching rows; any other
 * order builds a hash of voxels.  All give the same map.  Returns SPCONV_ERR_DUPLICATE_COORD if two
 * voxels share a coordinate and SPCONV_ERR_INVALID_ARG if a coordinate is
 * out of range; nmap is then undefined.
 */
spconv_status spconv_build_nmap(const int32_t* coords_dev, int64_t N, const int32_t* offsets_host,
                                int32_t K, int32_t* nmap_dev, void* workspace_dev,
                                size_t workspace_bytes, void* stream);

/*
 * The map build without the host wait: identical to spconv_build_nmap
 * except that the verdict of the device-side checks (coordinate range,
 * duplicates, table overflow) is written as an spconv_status (0 = OK) to
 * status_dev, an int32 in device memory, on `stream`.  The call returns
 * after enqueueing; argument errors found on the host are still returned
 * directly.  For pipelines that keep several steps in flight (copies of
 * the next step overlapping this step's kernels); check status_dev before
 * trusting nmap.  With N == 0 it writes 0.  No counterpart on the page.
 */
spconv_status spconv_build_nmap_async(const int32_t* coords_dev, int64_t N,
                                      const int32_t* offsets_host, int32_t K, int32_t* nmap_dev,
                                      void* workspace_dev, size_t workspace_bytes,
                                      int32_t* status_dev, void* stream);

/* Largest N spconv_build_nmap_noalloc accepts (its fixed table holds
 * 2 * SPCONV_NOALLOC_MAX_VOXELS slots). */
#define SPCONV_NOALLOC_MAX_VOXELS (1 << 20)

/*
 * spconv_build_nmap without a workspace: the same map, built in a fixed
 * device array that belongs to the library, so the call needs no device
 * memory from the caller.  The page has no counterpart of this call.
 *
 * It is for callers that cannot allocate device memory where they need a
 * map: code inside a host framework that owns every device allocation (its
 * own allocator, no raw cudaMalloc allowed), or a deployment with a fixed
 * memory budget that forbids allocations after start-up.  Nothing is
 * allocated or freed by the call itself.
 *
 * Arguments are those of spconv_build_nmap without the workspace; coords
 * and nmap are still the caller's.  Limits and behaviour:
 *  - N must not exceed SPCONV_NOALLOC_MAX_VOXELS; larger N returns
 *    SPCONV_ERR_UNSUPPORTED before any device work.
 *  - The array is a static device variable of 32 MiB + 256 B: it takes that
 *    much on each device where this library's module is loaded, until the
 *    process exits.
 *  - Each call looks up the array's device address on the current device
 *    (the runtime's symbol lookup; nothing is cached between calls).
 *  - Every call on a device shares the one array and clears what it needs
 *    (table keys and flags) at its start; the previous call's contents are
 *    otherwise left in place.  Calls whose work overlaps on the GPU (other
 *    streams, other host threads) race on the array and must be ordered by
 *    the caller.
 *  - Like spconv_build_nmap, it waits for `stream` once at the end to read
 *    the duplicate / range flags.
 */
spconv_status spconv_build_nmap_noalloc(const int32_t* coords_dev, int64_t N,
                                        const int32_t* offsets_host, int32_t K, int32_t* nmap_dev,
                                        void* stream);

/*
 * Fused submanifold convolution: gathers the neighbour rows tile by tile in
 * on-chip memory (the (K, N, Ci) gather is never written to device memory),
 * multiplies them with w[k] and accumulates over k in fp32, then adds the
 * bias and casts once to the storage type.
 *
 *  feats_dev  (N, Ci) in the storage type of `dtype`.  No pad row is needed.
 *  nmap_dev   (K, N) int32.  Entry v is a neighbour row iff 0 <= v < N; every
 *             other value (N, the page's marker, negative or larger values)
 *             contributes nothing.
 *  w_dev      (K, Ci, Co) storage type.
 *  bias_dev   (Co,) storage type, or NULL for no bias.
 *  out_dev    (N, Co) storage type, written (must not overlap the inputs).
 *  N, K, Ci, Co   N >= 0 (0 is a no-op), K >= 1, Ci >= 1, Co >= 1.
 *             SPCONV_BF16 / SPCONV_TF32 need Ci and Co multiples of 16 and
 *             16-byte aligned feats, w and out.  SPCONV_F32 needs 4-byte
 *             alignment only.
 *  dtype      SPCONV_F32, SPCONV_TF32 or SPCONV_BF16.
 *  stream     cudaStream_t (as void*).
 *
 * Asynchronous: no host wait, no allocation, no workspace; safe to capture
 * in a CUDA graph.  Tensor-core paths multiply the zero rows that stand for
 * missing neighbours inside a partly valid tile, so a non-finite weight can
 * turn such an output into NaN where an exact skip would not; offsets that
 * are missing for every voxel of a tile (256 voxels on the tensor-core
 * path, 64 on the fp32 path) are skipped outright.
 * Internal kernel errors (a pipeline wait that timed out) are reported by
 * spconv_device_status().
 */
spconv_status spconv_submconv3d(const void* feats_dev, const int32_t* nmap_dev, const void* w_dev,
                                const void* bias_dev, void* out_dev, int64_t N, int32_t K,
                                int32_t Ci, int32_t Co, spconv_dtype dtype, void* stream);

/* Activation applied by spconv_submconv3d_ex (after bias and residual). */
typedef enum spconv_activation {
    SPCONV_ACT_NONE = 0,
    SPCONV_ACT_RELU = 1, /* max(x, 0) */
    SPCONV_ACT_SILU = 2  /* x / (1 + exp(-x)), evaluated in fp32 with expf */
} spconv_activation;

/*
 * The convolution with a fused epilogue for chaining layers:
 *
 *     out[n, co] = act(conv[n, co] + bias[co] + residual[n, co])
 *
 * where conv[n, co] = sum_k sum_ci feats[nmap[k, n], ci] * w[k, ci, co] is
 * the sum of spconv_submconv3d.  The page ("sparse_conv_metal.py", module
 * docstring) runs this convolution layer after layer inside decoders; it
 * defines no epilogue beyond the bias (wrapper), so the residual add and the
 * activation are an extension: they are applied in fp32 to the accumulator
 * before the single cast to the storage type, instead of by separate passes
 * over (N, Co) in device memory.
 *
 *  residual_dev  (N, Co) storage type, or NULL for none, aligned like
 *                out_dev.  It may be the same buffer as out_dev (an in-place
 *                residual update); it must not overlap feats_dev.
 *  act           SPCONV_ACT_NONE, SPCONV_ACT_RELU or SPCONV_ACT_SILU; any
 *                other value gives SPCONV_ERR_INVALID_ARG.
 *  Every other argument, requirement and property is as for
 *  spconv_submconv3d; with residual_dev == NULL and SPCONV_ACT_NONE the two
 *  calls compute the same result.
 */
spconv_status spconv_submconv3d_ex(const void* feats_dev, const int32_t* nmap_dev,
                                   const void* w_dev, const void* bias_dev,
                                   const void* residual_dev, void* out_dev, int64_t N, int32_t K,
                                   int32_t Ci, int32_t Co, spconv_dtype dtype,
                                   spconv_activation act, void* stream);

/*
 * Gradient of the convolution with respect to its input features:
 *
 *     dfeats[m, ci] = sum over entries nmap[k, n] == m of
 *                     sum_co dout[n, co] * w[k, ci, co]
 *
 * (the chain rule applied to the formula of spconv_submconv3d; the page
 * computes the forward pass only).  The map must come from a point-symmetric
 * offset list in mirrored order, offsets[K-1-k] == -offsets[k] (true of the
 * lexicographic 3x3x3 list and of every cube list): then nmap[k, n] == m
 * exactly when nmap[K-1-k, m] == n, and the gradient is the forward
 * convolution of dout over the same map with the weights of offset k taken
 * as w[K-1-k] transposed.  Those weights are read in place from w's forward
 * (K, Ci, Co) layout; nothing is copied.
 *
 *  dout_dev    (N, Co) storage type.
 *  nmap_dev    (K, N) int32, as for spconv_submconv3d (built from a
 *              point-symmetric, mirrored offset list).
 *  w_dev       (K, Ci, Co) storage type: the forward weights.
 *  dfeats_dev  (N, Ci) storage type, written (must not overlap the inputs).
 *  N, K, Ci, Co, dtype, stream   the forward layer's sizes; requirements,
 *              tolerance and asynchrony as for spconv_submconv3d (bf16 and
 *              tf32 on the tensor cores, f32 exact fp32 on CUDA cores).
 */
spconv_status spconv_submconv3d_dgrad(const void* dout_dev, const int32_t* nmap_dev,
                                      const void* w_dev, void* dfeats_dev, int64_t N, int32_t K,
                                      int32_t Ci, int32_t Co, spconv_dtype dtype, void* stream);

/*
 * Gradients with respect to the weights and the bias:
 *
 *     dw[k, ci, co] = sum over valid entries m = nmap[k, n] of feats[m, ci] * dout[n, co]
 *     dbias[co]     = sum_n dout[n, co]
 *
 * (the chain rule applied to the formula of spconv_submconv3d and to the
 * wrapper's bias add; the page computes the forward pass only).  Any offset
 * list.  Computed exactly in fp32 on CUDA cores from the stored values
 * (bf16 widened exactly); dw and dbias are fp32 and are overwritten.
 * Partial sums of voxel slices are combined with fp32 atomic adds, so the
 * last bits may differ from run to run.
 *
 *  feats_dev  (N, Ci) storage type: the forward input.
 *  dout_dev   (N, Co) storage type: the gradient of the forward output.
 *  nmap_dev   (K, N) int32, as for spconv_submconv3d.
 *  dw_dev     (K, Ci, Co) float32, written.
 *  dbias_dev  (Co,) float32, written, or NULL to skip it.
 *  N >= 0, K, Ci, Co >= 1; dtype SPCONV_F32, SPCONV_TF32 (same as F32) or
 *  SPCONV_BF16; feats and dout aligned to their element, dw and dbias to 4
 *  bytes.  Asynchronous; no allocation, no workspace.
 */
spconv_status spconv_submconv3d_wgrad(const void* feats_dev, const void* dout_dev,
                                      const int32_t* nmap_dev, float* dw_dev, float* dbias_dev,
                                      int64_t N, int32_t K, int32_t Ci, int32_t Co, spconv_dtype dtype,
                                      void* stream);

/*
 * Count the entries v of a (K, N) map with 0 <= v < N (the valid pairs that
 * define the FLOP count 2 * pairs * Ci * Co).  Writes one int64 to count_dev
 * (device) asynchronously.
 */
spconv_status spconv_count_valid_pairs(const int32_t* nmap_dev, int64_t N, int32_t K,
                                       int64_t* count_dev, void* stream);

/*
 * A tile order for spconv_submconv3d_ordered: a permutation of 0..N-1
 * written to order_dev ((N,) int32, device).  Within each chunk of 4096
 * consecutive voxels, the voxels are sorted by their neighbour mask (which
 * of the first 32 offsets have a neighbour in nmap), ties by index.
 *
 * The page's kernel skips missing neighbours one element at a time (kernel
 * body).  A tile here skips an offset only when none of its 256 voxels has
 * that neighbour, and otherwise gathers zero rows for the missing ones.
 * Grouping voxels with like masks into tiles leaves fewer such rows; the
 * chunks keep tiles spatially local.  Measured by row-slot count: 24% fewer
 * kept (tile, offset) pairs on the channel workload (30% scattered voxels),
 * 3% on the decoder shells.
 *
 *  nmap_dev  (K, N) int32 map (entries outside [0, N) are missing).
 *  K         >= 1 (offsets beyond the 32nd do not enter the mask).
 *  order_dev (N,) int32, device, written.
 *
 * Asynchronous on `stream`; no workspace, no allocation.
 */
spconv_status spconv_tile_order(const int32_t* nmap_dev, int64_t N, int32_t K, int32_t* order_dev,
                                void* stream);

/*
 * spconv_submconv3d with the voxels taken in the given tile order: tile
 * slot s gathers the map column order[s] and writes output row order[s].
 * The result equals spconv_submconv3d's, bit for bit (each voxel's sums are
 * formed in the same order).  Only the grouping of voxels into tiles
 * changes, and with it how many empty rows the tiles gather.
 *
 *  order_dev  (N,) int32, device: a permutation of 0..N-1, for example from
 *             spconv_tile_order.  Entries outside [0, N) are treated as
 *             empty slots.  If order is not a permutation, rows it omits
 *             are not written and rows it repeats are written more than
 *             once.
 *
 * Other arguments, layouts and errors as spconv_submconv3d.  For SPCONV_F32
 * the order does not change how the exact fp32 kernel works, and it is
 * ignored.
 */
spconv_status spconv_submconv3d_ordered(const void* feats_dev, const int32_t* nmap_dev,
                                        const int32_t* order_dev, const void* w_dev,
                                        const void* bias_dev, void* out_dev, int64_t N, int32_t K,
                                        int32_t Ci, int32_t Co, spconv_dtype dtype, void* stream);

/*
 * x-run slot layout for spconv_submconv3d_xrun.
 *
 * A run is a maximal sequence of consecutive voxel indices whose cells are
 * consecutive in x on one (z, y) line.  The layout lists the voxels in index
 * order as slots, with separator slots between runs, so that for every voxel
 * slot s and dx in {-1, 0, +1}, slot s + dx stands for the cell (z, y, x + dx).
 * A separator stands for the cell just outside its run.  Slot codes (int32):
 * n >= 0 is voxel n; -2 - 2n is the cell right of voxel n (a run end);
 * -3 - 2n is the cell left of voxel n (a run start).  Between two runs there
 * is one separator when the first run's right cells and the next run's left
 * cells have the same map entries for all nine (dz, dy), else two.  Any
 * voxel order gives a valid layout; sorted (z, y, x) order gives long runs.
 *
 *  coords_dev      (N, 3) int32 (z, y, x), device.
 *  nmap_dev        (K, N) int32 map built from these coordinates with the
 *                  default lexicographic 3x3x3 offsets (K = 27).
 *  slots_dev       int32, device, written: S slot codes.
 *  slots_capacity  entries of slots_dev, >= spconv_xrun_slot_capacity(N)
 *                  (3N + 1, the most a layout can need).
 *  slot_count_dev  (1,) int64, device, written: S.
 *  workspace_dev   device scratch of >= spconv_xrun_workspace_size(N)
 *                  bytes, 8-byte aligned.
 *
 * Asynchronous on `stream`; no allocation.  Errors: SPCONV_ERR_INVALID_ARG
 * (N outside [1, 2^30), NULL or misaligned pointers, small capacity),
 * SPCONV_ERR_UNSUPPORTED (K != 27), SPCONV_ERR_WORKSPACE.
 */
size_t spconv_xrun_workspace_size(int64_t N);
int64_t spconv_xrun_slot_capacity(int64_t N);
spconv_status spconv_xrun_layout(const int32_t* coords_dev, const int32_t* nmap_dev, int64_t N, int32_t K,
                                 int32_t* slots_dev, int64_t slots_capacity, int64_t* slot_count_dev,
                                 void* workspace_dev, size_t workspace_bytes, void* stream);

/*
 * The map and the x-run layout in one call, for the lexicographic 3x3x3
 * offsets: the same nmap as spconv_build_nmap (K = 27) and the same slots
 * and slot count as spconv_xrun_layout on that map.  When the build takes
 * its dense-row path (sorted coordinates whose bounding box fits the
 * workspace), the map query also writes the layout's per-voxel flags from
 * the map entries it holds, so the layout reads neither the map nor the
 * coordinates again (measured at decoder scale: map then layout as two
 * calls 0.85 ms, this call 0.70 ms); on the build's other paths the layout
 * reads the map as spconv_xrun_layout does.  No counterpart on the page.
 *
 *  coords_dev, N     as spconv_build_nmap; 1 <= N < 2^30.
 *  nmap_dev          (27, N) int32, device, written.
 *  slots_dev, slots_capacity, slot_count_dev   as spconv_xrun_layout.
 *  workspace_dev     device scratch of >= spconv_build_nmap_xrun_workspace_size(N)
 *                    bytes, 256-byte aligned.
 *  status_dev        NULL: the call waits for `stream` once after the map
 *                    build and returns its verdict (as spconv_build_nmap);
 *                    else an int32 in device memory that receives the
 *                    verdict, and the call returns without waiting (as
 *                    spconv_build_nmap_async).
 */
size_t spconv_build_nmap_xrun_workspace_size(int64_t N);
spconv_status spconv_build_nmap_xrun(const int32_t* coords_dev, int64_t N, int32_t* nmap_dev, int32_t* slots_dev,
                                     int64_t slots_capacity, int64_t* slot_count_dev, void* workspace_dev,
                                     size_t workspace_bytes, int32_t* status_dev, void* stream);

/*
 * spconv_submconv3d over an x-run slot layout (spconv_xrun_layout).  For
 * each (dz, dy) a 256-slot tile gathers one operand of 258 rows (the
 * neighbour rows of the slots from one before the tile to one after it) and
 * reads its three dx offsets as the same rows shifted by one: a tile gathers
 * 9 x 258 rows instead of 27 x 256.  Separator slots cost MMA work; their
 * outputs are dropped.  Same sum as spconv_submconv3d, within the same
 * tolerance (products in bf16, fp32 accumulation, one rounding to bf16 after
 * the bias); the order of the fp32 additions differs.
 *
 *  slots_dev, slot_count_dev  from spconv_xrun_layout on the same map; the
 *                             kernel reads S from slot_count_dev and clamps
 *                             it to slots_capacity (the entries of
 *                             slots_dev), so no read leaves the buffer.
 *                             Slot codes naming no voxel of [0, N) are
 *                             treated as empty.
 *  dtype                      SPCONV_BF16 only; K = 27, Ci = 128, Co a
 *                             multiple of 16 in [16, 128].
 *
 * Other arguments, layouts and errors as spconv_submconv3d.  Other shapes
 * return SPCONV_ERR_UNSUPPORTED.
 */
spconv_status spconv_submconv3d_xrun(const void* feats_dev, const int32_t* nmap_dev, const int32_t* slots_dev,
                                     int64_t slots_capacity, const int64_t* slot_count_dev, const void* w_dev,
                                     const void* bias_dev, void* out_dev, int64_t N, int32_t K, int32_t Ci,
                                     int32_t Co, spconv_dtype dtype, void* stream);

/*
 * spconv_submconv3d_xrun with the fused epilogue of spconv_submconv3d_ex:
 *
 *     out[n, co] = act(conv[n, co] + bias[co] + residual[n, co])
 *
 * in fp32 on the accumulator, then one rounding to bf16.  An extension for
 * chaining decoder layers (the page runs the convolution layer after layer,
 * "sparse_conv_metal.py" module docstring, and defines no epilogue beyond
 * the bias).
 *
 *  residual_dev  (N, Co) bf16, 16-byte aligned, or NULL for none.  It may
 *                be the same buffer as out_dev (an in-place residual
 *                update); it must not overlap feats_dev.
 *  act           SPCONV_ACT_NONE, SPCONV_ACT_RELU or SPCONV_ACT_SILU; any
 *                other value gives SPCONV_ERR_INVALID_ARG.
 *
 * Other arguments, shapes and errors as spconv_submconv3d_xrun; with
 * residual_dev == NULL and SPCONV_ACT_NONE the two calls are the same.
 */
spconv_status spconv_submconv3d_xrun_ex(const void* feats_dev, const int32_t* nmap_dev, const int32_t* slots_dev,
                                        int64_t slots_capacity, const int64_t* slot_count_dev, const void* w_dev,
                                        const void* bias_dev, const void* residual_dev, void* out_dev, int64_t N,
                                        int32_t K, int32_t Ci, int32_t Co, spconv_dtype dtype,
                                        spconv_activation act, void* stream);

/*
 * spconv_submconv3d_dgrad over an x-run slot layout: dfeats (N, Ci) from
 * dout (N, Co), dfeats[n] = sum_k dout[nmap[k, n]] . w[K-1-k]^T (the map of
 * the 3x3x3 offsets is symmetric), with the row-shifted operands of
 * spconv_submconv3d_xrun gathered from dout.
 *
 *  dtype  SPCONV_BF16 only; K = 27, Co = 128 (the reduced channels), Ci a
 *         multiple of 16 in [16, 128] (the output channels).
 *
 * Other arguments as spconv_submconv3d_xrun and spconv_submconv3d_dgrad.
 */
spconv_status spconv_submconv3d_dgrad_xrun(const void* dout_dev, const int32_t* nmap_dev, const int32_t* slots_dev,
                                           int64_t slots_capacity, const int64_t* slot_count_dev,
                                           const void* w_dev, void* dfeats_dev, int64_t N, int32_t K, int32_t Ci,
                                           int32_t Co, spconv_dtype dtype, void* stream);

/*
 * Wait for `stream`, then read and clear the current device's sticky kernel
 * error word.  Returns SPCONV_OK if no kernel of this library has reported
 * an internal error since the last call, else SPCONV_ERR_DEVICE with the
 * error bits in the message.
 */
spconv_status spconv_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPCONV_H */

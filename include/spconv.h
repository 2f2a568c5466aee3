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
    SPCONV_TF32 = 1,  /* fp32 storage, results within the tf32 tolerance (4e-3 * sum|terms|);
                         currently computed with fp32 products on CUDA cores */
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
 * The call enqueues three kernels (table clear, insert, query) and then
 * waits for the stream once to read the error flags, so it cannot be
 * captured into a CUDA graph.  Returns SPCONV_ERR_DUPLICATE_COORD if two
 * voxels share a coordinate and SPCONV_ERR_INVALID_ARG if a coordinate is
 * out of range; nmap is then undefined.
 */
spconv_status spconv_build_nmap(const int32_t* coords_dev, int64_t N, const int32_t* offsets_host,
                                int32_t K, int32_t* nmap_dev, void* workspace_dev,
                                size_t workspace_bytes, void* stream);

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
 *  - The array (32 MiB + 256 B) is a static device variable: every GPU that
 *    loads this library holds it until the process exits.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
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
 * are missing for every voxel of a 128-voxel tile are skipped outright.
 * Internal kernel errors (a pipeline wait that timed out) are reported by
 * spconv_device_status().
 */
spconv_status spconv_submconv3d(const void* feats_dev, const int32_t* nmap_dev, const void* w_dev,
                                const void* bias_dev, void* out_dev, int64_t N, int32_t K,
                                int32_t Ci, int32_t Co, spconv_dtype dtype, void* stream);

/*
 * Count the entries v of a (K, N) map with 0 <= v < N (the valid pairs that
 * define the FLOP count 2 * pairs * Ci * Co).  Writes one int64 to count_dev
 * (device) asynchronously.
 */
spconv_status spconv_count_valid_pairs(const int32_t* nmap_dev, int64_t N, int32_t K,
                                       int64_t* count_dev, void* stream);

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

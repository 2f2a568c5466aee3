// Weight and bias gradients of the submanifold convolution, exact fp32 on
// CUDA cores:
//
//     dw[k, ci, co] = sum over valid entries m = nmap[k, n] of feats[m, ci] * dout[n, co]
//     dbias[co]     = sum_n dout[n, co]
//
// (the chain rule applied to the formula of page "sparse_conv_metal.py",
// trellis-2-mrp-mlx: module docstring, and to the wrapper's bias add; the
// page computes the forward pass only).  A CTA owns one offset k, a 64 x 64
// (ci, co) tile and a slice of kSlice voxels: per 16-voxel step it stages the
// neighbour indices (a step with none valid is skipped), the gathered feature
// rows and the dout rows in shared memory and accumulates 4 x 4 outputs per
// thread with FFMA; at the end it adds its partial tile to dw with fp32
// atomics (dw is zeroed first).  Inputs are fp32 or bf16 storage, widened
// exactly to fp32; the sums are fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace spconv {
namespace {

constexpr int kTile = 64;      // ci and co tile
constexpr int kStep = 16;      // voxels per step
constexpr int kSlice = 16384;  // voxels per CTA
constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float widen(T v);
template <>
__device__ __forceinline__ float widen<float>(float v) { return v; }
template <>
__device__ __forceinline__ float widen<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__global__ void __launch_bounds__(kThreads)
    wgrad_simt_kernel(const T* __restrict__ feats, const T* __restrict__ dout,
                      const int32_t* __restrict__ nmap, float* __restrict__ dw, int64_t n,
                      int32_t ci, int32_t co, int32_t slices) {
  __shared__ int32_t idx[kStep];
  __shared__ float as[kStep][kTile];
  __shared__ float bs[kStep][kTile];
  const int tid = threadIdx.x;
  const int k = blockIdx.z / slices;
  const int64_t v0 = static_cast<int64_t>(blockIdx.z % slices) * kSlice;
  const int64_t v1 = v0 + kSlice < n ? v0 + kSlice : n;
  const int ci0 = blockIdx.x * kTile;
  const int co0 = blockIdx.y * kTile;
  const int tr = tid / 16;  // ci rows tr*4 .. +3
  const int tc = tid % 16;  // co cols tc*4 .. +3
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int64_t s0 = v0; s0 < v1; s0 += kStep) {
    int valid = 0;
    if (tid < kStep) {
      const int64_t v = s0 + tid;
      int32_t m = -1;
      if (v < v1) m = nmap[static_cast<int64_t>(k) * n + v];
      if (m < 0 || m >= n) m = -1;
      idx[tid] = m;
      valid = m >= 0;
    }
    if (!__syncthreads_or(valid)) continue;
    for (int e = tid; e < kStep * kTile; e += kThreads) {
      const int r = e / kTile, c = e % kTile;
      const int32_t m = idx[r];
      // a voxel without this neighbour contributes nothing: its row is zero
      as[r][c] = (m >= 0 && ci0 + c < ci) ? widen(feats[static_cast<int64_t>(m) * ci + ci0 + c]) : 0.0f;
      bs[r][c] = (m >= 0 && co0 + c < co) ? widen(dout[(s0 + r) * co + co0 + c]) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kStep; ++r) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = as[r][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = bs[r][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c_in = ci0 + tr * 4 + i;
    if (c_in >= ci) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c_out = co0 + tc * 4 + j;
      if (c_out < co && acc[i][j] != 0.0f)
        atomicAdd(dw + (static_cast<int64_t>(k) * ci + c_in) * co + c_out, acc[i][j]);
    }
  }
}

// dbias[co] = sum_n dout[n, co]: a CTA sums a slice of rows per column.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    dbias_kernel(const T* __restrict__ dout, float* __restrict__ dbias, int64_t n, int32_t co) {
  const int c = blockIdx.x * kThreads + threadIdx.x;
  if (c >= co) return;
  const int64_t v0 = static_cast<int64_t>(blockIdx.y) * kSlice;
  const int64_t v1 = v0 + kSlice < n ? v0 + kSlice : n;
  float s = 0.0f;
  for (int64_t v = v0; v < v1; ++v) s += widen(dout[v * co + c]);
  atomicAdd(dbias + c, s);
}

// dbias[co] = sum_n dout[n, co], vectorised: a CTA sums a slab of kDbRows
// rows; each thread takes one 16-byte piece (kVec channels) of every
// (kThreads / pieces)-th row, so a warp reads whole rows, coalesced, with
// many independent loads in flight; the CTA combines its threads' partial
// sums in shared memory and adds one value per channel with an atomic.
// (The per-column loop above reads 2 bytes a thread per row, one row after
// another: at 1.0 M rows x 128 channels it took ~0.9 ms, longer than the
// weight gradient itself.)
constexpr int64_t kDbRows = 4096;

template <typename T, int kVec>
__global__ void __launch_bounds__(kThreads)
    dbias_vec_kernel(const T* __restrict__ dout, float* __restrict__ dbias, int64_t n, int32_t co) {
  __shared__ float part[kThreads * kVec];
  const int pieces = co / kVec;  // <= kThreads (checked by the launcher)
  const int rps = kThreads / pieces;
  const int t = static_cast<int>(threadIdx.x);
  const int g = t % pieces, r0 = t / pieces;
  float acc[kVec];
#pragma unroll
  for (int j = 0; j < kVec; ++j) acc[j] = 0.0f;
  if (r0 < rps) {
    const int64_t v0 = static_cast<int64_t>(blockIdx.x) * kDbRows;
    const int64_t v1 = v0 + kDbRows < n ? v0 + kDbRows : n;
#pragma unroll 4
    for (int64_t v = v0 + r0; v < v1; v += rps) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(dout + v * co) + g);
      const T* e = reinterpret_cast<const T*>(&q);
#pragma unroll
      for (int j = 0; j < kVec; ++j) acc[j] += widen(e[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < kVec; ++j) part[t * kVec + j] = acc[j];
  __syncthreads();
  for (int c = t; c < co; c += kThreads) {
    const int gc = c / kVec, j = c - gc * kVec;
    float s = 0.0f;
    for (int r = 0; r < rps; ++r) s += part[(r * pieces + gc) * kVec + j];
    atomicAdd(dbias + c, s);
  }
}

template <typename T>
spconv_status launch_typed(const T* feats, const T* dout, const int32_t* nmap, float* dw, float*,
                           int64_t n, int32_t k, int32_t ci, int32_t co, cudaStream_t stream) {
  spconv_status st = SPCONV_OK;
  const size_t dw_bytes = static_cast<size_t>(k) * ci * co * sizeof(float);
  if (!cuda_ok(cudaMemsetAsync(dw, 0, dw_bytes, stream), "cudaMemsetAsync(dw)", &st)) return st;
  const int64_t slices = (n + kSlice - 1) / kSlice;
  const int64_t gz = slices * k;
  const int gx = (ci + kTile - 1) / kTile, gy = (co + kTile - 1) / kTile;
  if (gz > 65535 || gy > 65535) return fail(SPCONV_ERR_UNSUPPORTED, "problem too large for the wgrad grid");
  wgrad_simt_kernel<T><<<dim3(gx, gy, static_cast<unsigned>(gz)), kThreads, 0, stream>>>(
      feats, dout, nmap, dw, n, ci, co, static_cast<int32_t>(slices));
  if (!cuda_ok(cudaGetLastError(), "wgrad_simt_kernel launch", &st)) return st;
  return SPCONV_OK;
}

}  // namespace

spconv_status launch_dbias(spconv_dtype dtype, const void* dout, float* dbias, int64_t n, int32_t co,
                           cudaStream_t stream) {
  spconv_status st = SPCONV_OK;
  if (!cuda_ok(cudaMemsetAsync(dbias, 0, static_cast<size_t>(co) * sizeof(float), stream),
               "cudaMemsetAsync(dbias)", &st))
    return st;
  const size_t esz = dtype == SPCONV_BF16 ? 2u : 4u;
  const int vec = static_cast<int>(16u / esz);
  if (co % vec == 0 && co / vec <= kThreads && reinterpret_cast<uintptr_t>(dout) % 16u == 0u) {
    const int64_t blocks = (n + kDbRows - 1) / kDbRows;
    if (blocks > 0x7fffffff) return fail(SPCONV_ERR_UNSUPPORTED, "problem too large for the dbias grid");
    if (dtype == SPCONV_BF16)
      dbias_vec_kernel<__nv_bfloat16, 8><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(dout), dbias, n, co);
    else
      dbias_vec_kernel<float, 4><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
          static_cast<const float*>(dout), dbias, n, co);
    if (!cuda_ok(cudaGetLastError(), "dbias_vec_kernel launch", &st)) return st;
    return SPCONV_OK;
  }
  const int64_t slices = (n + kSlice - 1) / kSlice;
  if (slices > 65535) return fail(SPCONV_ERR_UNSUPPORTED, "problem too large for the dbias grid");
  const dim3 grid((co + kThreads - 1) / kThreads, static_cast<unsigned>(slices));
  if (dtype == SPCONV_BF16)
    dbias_kernel<<<grid, kThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(dout), dbias, n, co);
  else
    dbias_kernel<<<grid, kThreads, 0, stream>>>(static_cast<const float*>(dout), dbias, n, co);
  if (!cuda_ok(cudaGetLastError(), "dbias_kernel launch", &st)) return st;
  return SPCONV_OK;
}

spconv_status launch_wgrad_simt(spconv_dtype dtype, const void* feats, const void* dout,
                                const int32_t* nmap, float* dw, float* dbias, int64_t n, int32_t k,
                                int32_t ci, int32_t co, cudaStream_t stream) {
  spconv_status st =
      dtype == SPCONV_BF16
          ? launch_typed(static_cast<const __nv_bfloat16*>(feats), static_cast<const __nv_bfloat16*>(dout),
                         nmap, dw, dbias, n, k, ci, co, stream)
          : launch_typed(static_cast<const float*>(feats), static_cast<const float*>(dout), nmap, dw, dbias,
                         n, k, ci, co, stream);
  if (st != SPCONV_OK || dbias == nullptr) return st;
  return launch_dbias(dtype, dout, dbias, n, co, stream);
}

}  // namespace spconv

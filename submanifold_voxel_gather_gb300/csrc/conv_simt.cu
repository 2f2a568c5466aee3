// Exact-fp32 submanifold convolution on CUDA cores.
//
// Same operation as the tensor-core path (page "sparse_conv_metal.py",
// trellis-2-mrp-mlx: module docstring formula, kernel-body sentinel skip,
// wrapper bias), for fp32 storage with fp32 products: tf32 products would
// miss the fp32 tolerance.  A CTA computes a 64-voxel x 64-channel output
// tile; for each offset k it stages the 64 neighbour indices, skips k when
// none is valid, gathers the rows chunk by chunk into shared memory (rows
// that are not valid become zeros) and accumulates with FFMA, 4 x 4 outputs
// per thread.  Each output accumulates over k, then ci, in order.  The
// epilogue adds the bias and, for the fused-epilogue entry point, a residual
// row and an activation, in fp32.  With `dgrad` set the same loop computes
// the input gradient: the gathered rows are dout rows and the weights of
// offset k are w[K-1-k] transposed, read in place from the (K, Ci, Co)
// forward layout (here ci counts dout channels and co dfeats channels).
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "internal.h"

namespace spconv {
namespace {

constexpr int kBM = 64;
constexpr int kBN = 64;
constexpr int kBK = 16;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    submconv_simt_f32_kernel(const float* __restrict__ feats, const int32_t* __restrict__ nmap,
                             const float* __restrict__ w, const float* __restrict__ bias,
                             const float* residual, float* out, int64_t n, int32_t k_count,
                             int32_t ci, int32_t co, int act, int dgrad) {
  __shared__ int32_t idx[kBM];
  __shared__ float as[kBK][kBM + 4];
  __shared__ float bs[kBK][kBN];

  const int tid = threadIdx.x;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kBM;
  const int col0 = blockIdx.y * kBN;
  const int tr = tid / 16;  // 16 x 16 thread grid, 4 x 4 outputs each
  const int tc = tid % 16;

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int32_t k = 0; k < k_count; ++k) {
    int valid = 0;
    if (tid < kBM) {
      const int64_t r = row0 + tid;
      int32_t v = -1;
      if (r < n) v = nmap[static_cast<int64_t>(k) * n + r];
      if (v < 0 || v >= n) v = -1;
      idx[tid] = v;
      valid = v >= 0;
    }
    if (!__syncthreads_or(valid)) continue;  // no neighbour under this offset in the tile

    for (int c0 = 0; c0 < ci; c0 += kBK) {
      // A: 64 rows x 16 channels, stored transposed; zero for invalid rows.
      for (int e = tid; e < kBM * kBK; e += kThreads) {
        const int r = e / kBK;
        const int c = e % kBK;
        const int32_t src = idx[r];
        float v = 0.0f;
        if (src >= 0 && c0 + c < ci) v = feats[static_cast<int64_t>(src) * ci + c0 + c];
        as[c][r] = v;
      }
      // B: 16 channels x 64 output channels of w[k].
      for (int e = tid; e < kBK * kBN; e += kThreads) {
        const int r = e / kBN;
        const int c = e % kBN;
        float v = 0.0f;
        if (c0 + r < ci && col0 + c < co)
          v = dgrad ? w[(static_cast<int64_t>(k_count - 1 - k) * co + col0 + c) * ci + c0 + r]
                    : w[(static_cast<int64_t>(k) * ci + c0 + r) * co + col0 + c];
        bs[r][c] = v;
      }
      __syncthreads();
#pragma unroll
      for (int c = 0; c < kBK; ++c) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = as[c][tr * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = bs[c][tc * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      __syncthreads();
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = row0 + tr * 4 + i;
    if (r >= n) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = col0 + tc * 4 + j;
      if (c >= co) continue;
      // residual may be the same buffer as out: each element is read and
      // then written by this thread only.
      float x = acc[i][j] + (bias != nullptr ? bias[c] : 0.0f);
      if (residual != nullptr) x += residual[r * co + c];
      out[r * co + c] = apply_activation(x, act);
    }
  }
}

}  // namespace

spconv_status launch_conv_simt_f32(const float* feats, const int32_t* nmap, const float* w,
                                   const float* bias, const float* residual, float* out,
                                   int64_t n, int32_t k, int32_t ci, int32_t co,
                                   spconv_activation act, bool dgrad, cudaStream_t stream) {
  const int64_t gx = (n + kBM - 1) / kBM;
  const int gy = (co + kBN - 1) / kBN;
  if (gx > 0x7fffffff || gy > 65535)
    return fail(SPCONV_ERR_UNSUPPORTED, "problem too large for the fp32 grid");
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  submconv_simt_f32_kernel<<<grid, kThreads, 0, stream>>>(feats, nmap, w, bias, residual, out, n, k, ci,
                                                          co, static_cast<int>(act), dgrad ? 1 : 0);
  spconv_status st = SPCONV_OK;
  if (!cuda_ok(cudaGetLastError(), "submconv_simt_f32_kernel launch", &st)) return st;
  return SPCONV_OK;
}

}  // namespace spconv

// C ABI of the library (declared in include/spconv.h): argument validation,
// device checks and dispatch to the kernels.  Validation comes first and
// nothing is enqueued when it fails.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"
#include "spconv.h"

namespace spconv {

namespace {

thread_local std::string t_last_error;

constexpr int kMaxDevices = 64;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The kernels are built for sm_103a only; anything else fails loudly here
// rather than with a missing-image launch error.
spconv_status check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return fail(SPCONV_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  static int checked[kMaxDevices] = {0};  // 0 unknown, 1 ok, -1 unsupported
  if (dev >= 0 && dev < kMaxDevices && checked[dev] == 1) return SPCONV_OK;
  int major = 0, minor = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess)
    return fail(SPCONV_ERR_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
  if (major != 10 || minor != 3) {
    if (dev >= 0 && dev < kMaxDevices) checked[dev] = -1;
    return fail(SPCONV_ERR_UNSUPPORTED, "device " + std::to_string(dev) + " has compute capability " +
                                            std::to_string(major) + "." + std::to_string(minor) +
                                            "; this library is built for 10.3 (sm_103a) only");
  }
  if (dev >= 0 && dev < kMaxDevices) checked[dev] = 1;
  return SPCONV_OK;
}

spconv_status ok() {
  t_last_error.clear();
  return SPCONV_OK;
}

}  // namespace

spconv_status fail(spconv_status code, const std::string& msg) {
  t_last_error = msg;
  return code;
}

bool cuda_ok(cudaError_t err, const char* what, spconv_status* out) {
  if (err == cudaSuccess) return true;
  *out = fail(SPCONV_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(err));
  return false;
}

int sm_count() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < kMaxDevices) cache[dev] = n;
  return n;
}

}  // namespace spconv

using spconv::fail;

extern "C" {

int spconv_version(void) { return SPCONV_VERSION; }

const char* spconv_last_error(void) { return spconv::t_last_error.c_str(); }

size_t spconv_build_nmap_workspace_size(int64_t N) {
  if (N < 0) return 0;
  return 256 + spconv::hash_capacity(N) * 16;
}

namespace spconv {
namespace {

spconv_status build_nmap_impl(const int32_t* coords_dev, int64_t N, const int32_t* offsets_host,
                              int32_t K, int32_t* nmap_dev, void* workspace_dev, size_t workspace_bytes,
                              int32_t* status_dev, void* stream) {
  if (N < 0 || N >= INT32_MAX) return fail(SPCONV_ERR_INVALID_ARG, "N must satisfy 0 <= N < 2^31-1");
  if (K < 1 || K > SPCONV_MAX_BUILD_OFFSETS)
    return fail(SPCONV_ERR_INVALID_ARG, "K must satisfy 1 <= K <= SPCONV_MAX_BUILD_OFFSETS");
  if (offsets_host == nullptr) return fail(SPCONV_ERR_INVALID_ARG, "offsets_host is NULL");
  if (status_dev != nullptr && !aligned(status_dev, 4))
    return fail(SPCONV_ERR_INVALID_ARG, "status must be 4-byte aligned");
  spconv_status st = SPCONV_OK;
  if (N == 0) {
    if (status_dev == nullptr) return ok();
    st = check_device();
    if (st != SPCONV_OK) return st;
    if (!cuda_ok(cudaMemsetAsync(status_dev, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)),
                 "cudaMemsetAsync(status)", &st))
      return st;
    return ok();
  }
  if (coords_dev == nullptr || nmap_dev == nullptr || workspace_dev == nullptr)
    return fail(SPCONV_ERR_INVALID_ARG, "coords, nmap and workspace must be non-NULL");
  if (!aligned(coords_dev, 4) || !aligned(nmap_dev, 4))
    return fail(SPCONV_ERR_INVALID_ARG, "coords and nmap must be 4-byte aligned");
  if (!aligned(workspace_dev, 256))
    return fail(SPCONV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < spconv_build_nmap_workspace_size(N))
    return fail(SPCONV_ERR_WORKSPACE, "workspace smaller than spconv_build_nmap_workspace_size(N)");
  for (int32_t i = 0; i < 3 * K; ++i) {
    const int32_t d = offsets_host[i];
    if (d <= -SPCONV_COORD_LIMIT || d >= SPCONV_COORD_LIMIT)
      return fail(SPCONV_ERR_INVALID_ARG, "offset component out of range");
  }
  st = check_device();
  if (st != SPCONV_OK) return st;
  BuildOffsets offs;
  std::memset(&offs, 0, sizeof offs);
  std::memcpy(offs.d, offsets_host, sizeof(int32_t) * 3 * static_cast<size_t>(K));
  st = launch_build_nmap(coords_dev, N, offs, K, nmap_dev, workspace_dev, static_cast<cudaStream_t>(stream),
                         status_dev);
  return st == SPCONV_OK ? ok() : st;
}

}  // namespace
}  // namespace spconv

spconv_status spconv_build_nmap(const int32_t* coords_dev, int64_t N, const int32_t* offsets_host,
                                int32_t K, int32_t* nmap_dev, void* workspace_dev,
                                size_t workspace_bytes, void* stream) {
  return spconv::build_nmap_impl(coords_dev, N, offsets_host, K, nmap_dev, workspace_dev, workspace_bytes,
                                 nullptr, stream);
}

spconv_status spconv_build_nmap_async(const int32_t* coords_dev, int64_t N,
                                      const int32_t* offsets_host, int32_t K, int32_t* nmap_dev,
                                      void* workspace_dev, size_t workspace_bytes,
                                      int32_t* status_dev, void* stream) {
  if (status_dev == nullptr) return fail(SPCONV_ERR_INVALID_ARG, "status must be non-NULL");
  return spconv::build_nmap_impl(coords_dev, N, offsets_host, K, nmap_dev, workspace_dev, workspace_bytes,
                                 status_dev, stream);
}

spconv_status spconv_build_nmap_noalloc(const int32_t* coords_dev, int64_t N,
                                        const int32_t* offsets_host, int32_t K, int32_t* nmap_dev,
                                        void* stream) {
  if (N < 0) return fail(SPCONV_ERR_INVALID_ARG, "N must be >= 0");
  if (N > SPCONV_NOALLOC_MAX_VOXELS)
    return fail(SPCONV_ERR_UNSUPPORTED,
                "N exceeds SPCONV_NOALLOC_MAX_VOXELS (" + std::to_string(SPCONV_NOALLOC_MAX_VOXELS) +
                    "); use spconv_build_nmap with a workspace");
  if (K < 1 || K > SPCONV_MAX_BUILD_OFFSETS)
    return fail(SPCONV_ERR_INVALID_ARG, "K must satisfy 1 <= K <= SPCONV_MAX_BUILD_OFFSETS");
  if (offsets_host == nullptr) return fail(SPCONV_ERR_INVALID_ARG, "offsets_host is NULL");
  if (N == 0) return spconv::ok();
  if (coords_dev == nullptr || nmap_dev == nullptr)
    return fail(SPCONV_ERR_INVALID_ARG, "coords and nmap must be non-NULL");
  if (!spconv::aligned(coords_dev, 4) || !spconv::aligned(nmap_dev, 4))
    return fail(SPCONV_ERR_INVALID_ARG, "coords and nmap must be 4-byte aligned");
  for (int32_t i = 0; i < 3 * K; ++i) {
    const int32_t d = offsets_host[i];
    if (d <= -SPCONV_COORD_LIMIT || d >= SPCONV_COORD_LIMIT)
      return fail(SPCONV_ERR_INVALID_ARG, "offset component out of range");
  }
  spconv_status st = spconv::check_device();
  if (st != SPCONV_OK) return st;
  void* scratch = nullptr;
  st = spconv::noalloc_scratch(&scratch);
  if (st != SPCONV_OK) return st;
  spconv::BuildOffsets offs;
  std::memset(&offs, 0, sizeof offs);
  std::memcpy(offs.d, offsets_host, sizeof(int32_t) * 3 * static_cast<size_t>(K));
  st = spconv::launch_build_nmap(coords_dev, N, offs, K, nmap_dev, scratch,
                                 static_cast<cudaStream_t>(stream));
  return st == SPCONV_OK ? spconv::ok() : st;
}

namespace spconv {
namespace {

// Shared validation and dispatch of spconv_submconv3d, _ex and _dgrad.  Ci
// and Co are the widths of the gathered input rows and of the output rows
// (for the input gradient: the forward Co and Ci).
spconv_status submconv3d_impl(const void* feats_dev, const int32_t* nmap_dev, const void* w_dev,
                              const void* bias_dev, const void* residual_dev, void* out_dev, int64_t N,
                              int32_t K, int32_t Ci, int32_t Co, spconv_dtype dtype,
                              spconv_activation act, bool dgrad, void* stream,
                              const int32_t* order = nullptr) {
  if (N < 0 || N >= INT32_MAX) return fail(SPCONV_ERR_INVALID_ARG, "N must satisfy 0 <= N < 2^31-1");
  if (K < 1 || Ci < 1 || Co < 1) return fail(SPCONV_ERR_INVALID_ARG, "K, Ci and Co must be >= 1");
  if (dtype != SPCONV_F32 && dtype != SPCONV_TF32 && dtype != SPCONV_BF16)
    return fail(SPCONV_ERR_INVALID_ARG, "unknown dtype");
  if (act != SPCONV_ACT_NONE && act != SPCONV_ACT_RELU && act != SPCONV_ACT_SILU)
    return fail(SPCONV_ERR_INVALID_ARG, "unknown activation");
  if (N == 0) return ok();
  if (feats_dev == nullptr || nmap_dev == nullptr || w_dev == nullptr || out_dev == nullptr)
    return fail(SPCONV_ERR_INVALID_ARG, "feats, nmap, w and out must be non-NULL");
  if (!aligned(nmap_dev, 4)) return fail(SPCONV_ERR_INVALID_ARG, "nmap must be 4-byte aligned");
  const size_t elem = dtype == SPCONV_BF16 ? 2 : 4;
  if (static_cast<uint64_t>(N) * static_cast<uint64_t>(K) > (1ull << 40))
    return fail(SPCONV_ERR_UNSUPPORTED, "K * N too large");
  if (residual_dev != nullptr && !aligned(residual_dev, dtype == SPCONV_F32 ? 4 : 16))
    return fail(SPCONV_ERR_INVALID_ARG, "residual is misaligned (needs the alignment of out)");
  if (dtype == SPCONV_F32) {
    if (!aligned(feats_dev, 4) || !aligned(w_dev, 4) || !aligned(out_dev, 4) ||
        (bias_dev != nullptr && !aligned(bias_dev, 4)))
      return fail(SPCONV_ERR_INVALID_ARG, "fp32 arrays must be 4-byte aligned");
  } else {
    if (Ci % 16 != 0 || Co % 16 != 0)
      return fail(SPCONV_ERR_UNSUPPORTED, "bf16/tf32 need Ci and Co to be multiples of 16");
    if (!aligned(feats_dev, 16) || !aligned(w_dev, 16) || !aligned(out_dev, 16))
      return fail(SPCONV_ERR_INVALID_ARG, "feats, w and out must be 16-byte aligned");
    if (bias_dev != nullptr && !aligned(bias_dev, elem))
      return fail(SPCONV_ERR_INVALID_ARG, "bias is misaligned");
  }
  spconv_status st = check_device();
  if (st != SPCONV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // SPCONV_F32: exact fp32 products on CUDA cores; SPCONV_TF32 and
  // SPCONV_BF16: the tensor-core kernel (kind::tf32 / kind::f16 MMAs).
  if (dtype == SPCONV_F32)
    st = launch_conv_simt_f32(static_cast<const float*>(feats_dev), nmap_dev,
                              static_cast<const float*>(w_dev), static_cast<const float*>(bias_dev),
                              static_cast<const float*>(residual_dev), static_cast<float*>(out_dev), N,
                              K, Ci, Co, act, dgrad, s);
  else
    st = launch_conv_tc(dtype, feats_dev, nmap_dev, w_dev, bias_dev, residual_dev, out_dev, N, K, Ci,
                        Co, act, dgrad, s, order);
  return st == SPCONV_OK ? ok() : st;
}

}  // namespace
}  // namespace spconv

spconv_status spconv_submconv3d(const void* feats_dev, const int32_t* nmap_dev, const void* w_dev,
                                const void* bias_dev, void* out_dev, int64_t N, int32_t K,
                                int32_t Ci, int32_t Co, spconv_dtype dtype, void* stream) {
  return spconv::submconv3d_impl(feats_dev, nmap_dev, w_dev, bias_dev, nullptr, out_dev, N, K, Ci, Co,
                                 dtype, SPCONV_ACT_NONE, false, stream);
}

spconv_status spconv_submconv3d_ordered(const void* feats_dev, const int32_t* nmap_dev,
                                        const int32_t* order_dev, const void* w_dev,
                                        const void* bias_dev, void* out_dev, int64_t N, int32_t K,
                                        int32_t Ci, int32_t Co, spconv_dtype dtype, void* stream) {
  if (N > 0 && (order_dev == nullptr || !spconv::aligned(order_dev, 4)))
    return fail(SPCONV_ERR_INVALID_ARG, "order must be non-NULL and 4-byte aligned");
  return spconv::submconv3d_impl(feats_dev, nmap_dev, w_dev, bias_dev, nullptr, out_dev, N, K, Ci, Co,
                                 dtype, SPCONV_ACT_NONE, false, stream, order_dev);
}

spconv_status spconv_tile_order(const int32_t* nmap_dev, int64_t N, int32_t K, int32_t* order_dev,
                                void* stream) {
  if (N < 0 || N >= INT32_MAX || K < 1) return fail(SPCONV_ERR_INVALID_ARG, "bad N or K");
  if (N == 0) return spconv::ok();
  if (nmap_dev == nullptr || order_dev == nullptr)
    return fail(SPCONV_ERR_INVALID_ARG, "nmap and order must be non-NULL");
  if (!spconv::aligned(nmap_dev, 4) || !spconv::aligned(order_dev, 4))
    return fail(SPCONV_ERR_INVALID_ARG, "nmap and order must be 4-byte aligned");
  spconv_status st = spconv::check_device();
  if (st != SPCONV_OK) return st;
  st = spconv::launch_tile_order(nmap_dev, N, K, order_dev, static_cast<cudaStream_t>(stream));
  return st == SPCONV_OK ? spconv::ok() : st;
}

size_t spconv_xrun_workspace_size(int64_t N) { return N < 0 ? 0 : spconv::xrun_workspace_bytes(N); }

int64_t spconv_xrun_slot_capacity(int64_t N) { return N < 0 ? 0 : spconv::xrun_slot_capacity(N); }

spconv_status spconv_xrun_layout(const int32_t* coords_dev, const int32_t* nmap_dev, int64_t N, int32_t K,
                                 int32_t* slots_dev, int64_t slots_capacity, int64_t* slot_count_dev,
                                 void* workspace_dev, size_t workspace_bytes, void* stream) {
  if (N < 1 || N >= (int64_t{1} << 30)) return fail(SPCONV_ERR_INVALID_ARG, "N must be in [1, 2^30)");
  if (K != 27) return fail(SPCONV_ERR_UNSUPPORTED, "the x-run layout needs the 27 lexicographic 3x3x3 offsets");
  if (coords_dev == nullptr || nmap_dev == nullptr || slots_dev == nullptr || slot_count_dev == nullptr ||
      workspace_dev == nullptr)
    return fail(SPCONV_ERR_INVALID_ARG, "coords, nmap, slots, slot_count and workspace must be non-NULL");
  if (!spconv::aligned(coords_dev, 4) || !spconv::aligned(nmap_dev, 4) || !spconv::aligned(slots_dev, 4) ||
      !spconv::aligned(slot_count_dev, 8) || !spconv::aligned(workspace_dev, 8))
    return fail(SPCONV_ERR_INVALID_ARG, "misaligned pointer (coords, nmap, slots: 4 bytes; slot_count, workspace: 8)");
  if (slots_capacity < spconv::xrun_slot_capacity(N))
    return fail(SPCONV_ERR_INVALID_ARG, "slots_capacity below spconv_xrun_slot_capacity(N)");
  if (workspace_bytes < spconv::xrun_workspace_bytes(N))
    return fail(SPCONV_ERR_WORKSPACE, "workspace smaller than spconv_xrun_workspace_size(N)");
  spconv_status st = spconv::check_device();
  if (st != SPCONV_OK) return st;
  st = spconv::launch_xrun_layout(coords_dev, nmap_dev, N, slots_dev, slots_capacity, slot_count_dev,
                                  workspace_dev, static_cast<cudaStream_t>(stream));
  return st == SPCONV_OK ? spconv::ok() : st;
}

size_t spconv_build_nmap_xrun_workspace_size(int64_t N) {
  if (N < 0) return 0;
  return (spconv_build_nmap_workspace_size(N) + 255) / 256 * 256 + spconv::xrun_workspace_bytes(N);
}

spconv_status spconv_build_nmap_xrun(const int32_t* coords_dev, int64_t N, int32_t* nmap_dev, int32_t* slots_dev,
                                     int64_t slots_capacity, int64_t* slot_count_dev, void* workspace_dev,
                                     size_t workspace_bytes, int32_t* status_dev, void* stream) {
  if (N < 1 || N >= (int64_t{1} << 30)) return fail(SPCONV_ERR_INVALID_ARG, "N must be in [1, 2^30)");
  if (coords_dev == nullptr || nmap_dev == nullptr || slots_dev == nullptr || slot_count_dev == nullptr ||
      workspace_dev == nullptr)
    return fail(SPCONV_ERR_INVALID_ARG, "coords, nmap, slots, slot_count and workspace must be non-NULL");
  if (!spconv::aligned(coords_dev, 4) || !spconv::aligned(nmap_dev, 4) || !spconv::aligned(slots_dev, 4) ||
      !spconv::aligned(slot_count_dev, 8) || !spconv::aligned(workspace_dev, 256) ||
      (status_dev != nullptr && !spconv::aligned(status_dev, 4)))
    return fail(SPCONV_ERR_INVALID_ARG,
                "misaligned pointer (coords, nmap, slots, status: 4 bytes; slot_count: 8; workspace: 256)");
  if (slots_capacity < spconv::xrun_slot_capacity(N))
    return fail(SPCONV_ERR_INVALID_ARG, "slots_capacity below spconv_xrun_slot_capacity(N)");
  if (workspace_bytes < spconv_build_nmap_xrun_workspace_size(N))
    return fail(SPCONV_ERR_WORKSPACE, "workspace smaller than spconv_build_nmap_xrun_workspace_size(N)");
  spconv_status st = spconv::check_device();
  if (st != SPCONV_OK) return st;
  spconv::BuildOffsets offs;
  std::memset(&offs, 0, sizeof offs);
  for (int32_t a = 0; a < 27; ++a) {  // the lexicographic 3x3x3 list, (dz, dy, dx)
    offs.d[3 * a] = a / 9 - 1;
    offs.d[3 * a + 1] = (a / 3) % 3 - 1;
    offs.d[3 * a + 2] = a % 3 - 1;
  }
  void* ws_build = workspace_dev;
  void* ws_layout = static_cast<char*>(workspace_dev) + (spconv_build_nmap_workspace_size(N) + 255) / 256 * 256;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = spconv::launch_build_nmap(coords_dev, N, offs, 27, nmap_dev, ws_build, s, status_dev,
                                 spconv::xrun_raw_bits(ws_layout, N));
  if (st != SPCONV_OK) return st;
  st = spconv::launch_xrun_layout(coords_dev, nmap_dev, N, slots_dev, slots_capacity, slot_count_dev, ws_layout, s,
                                  spconv::xrun_flags_ready(ws_build));
  return st == SPCONV_OK ? spconv::ok() : st;
}

spconv_status spconv_submconv3d_xrun(const void* feats_dev, const int32_t* nmap_dev, const int32_t* slots_dev,
                                     int64_t slots_capacity, const int64_t* slot_count_dev, const void* w_dev,
                                     const void* bias_dev, void* out_dev, int64_t N, int32_t K, int32_t Ci,
                                     int32_t Co, spconv_dtype dtype, void* stream) {
  return spconv_submconv3d_xrun_ex(feats_dev, nmap_dev, slots_dev, slots_capacity, slot_count_dev, w_dev, bias_dev,
                                   nullptr, out_dev, N, K, Ci, Co, dtype, SPCONV_ACT_NONE, stream);
}

spconv_status spconv_submconv3d_xrun_ex(const void* feats_dev, const int32_t* nmap_dev, const int32_t* slots_dev,
                                        int64_t slots_capacity, const int64_t* slot_count_dev, const void* w_dev,
                                        const void* bias_dev, const void* residual_dev, void* out_dev, int64_t N,
                                        int32_t K, int32_t Ci, int32_t Co, spconv_dtype dtype,
                                        spconv_activation act, void* stream) {
  if (act != SPCONV_ACT_NONE && act != SPCONV_ACT_RELU && act != SPCONV_ACT_SILU)
    return fail(SPCONV_ERR_INVALID_ARG, "unknown activation");
  if (N < 1 || N >= (int64_t{1} << 30)) return fail(SPCONV_ERR_INVALID_ARG, "N must be in [1, 2^30)");
  if (dtype != SPCONV_BF16 || K != 27 || Ci != 128 || Co < 16 || Co > 128 || Co % 16 != 0)
    return fail(SPCONV_ERR_UNSUPPORTED, "the x-run conv takes bf16, K = 27, Ci = 128 and Co in [16, 128], a multiple of 16");
  if (feats_dev == nullptr || nmap_dev == nullptr || slots_dev == nullptr || slot_count_dev == nullptr ||
      w_dev == nullptr || out_dev == nullptr)
    return fail(SPCONV_ERR_INVALID_ARG, "feats, nmap, slots, slot_count, w and out must be non-NULL");
  if (!spconv::aligned(feats_dev, 16) || !spconv::aligned(w_dev, 16) || !spconv::aligned(out_dev, 16) ||
      !spconv::aligned(nmap_dev, 4) || !spconv::aligned(slots_dev, 4) || !spconv::aligned(slot_count_dev, 8) ||
      (bias_dev != nullptr && !spconv::aligned(bias_dev, 2)) ||
      (residual_dev != nullptr && !spconv::aligned(residual_dev, 16)))
    return fail(SPCONV_ERR_INVALID_ARG, "misaligned pointer");
  if (slots_capacity < 1) return fail(SPCONV_ERR_INVALID_ARG, "slots_capacity must be >= 1");
  spconv_status st = spconv::check_device();
  if (st != SPCONV_OK) return st;
  st = spconv::launch_conv_xrun(feats_dev, nmap_dev, slots_dev, slots_capacity, slot_count_dev, w_dev, bias_dev,
                                residual_dev, out_dev, N, Co, static_cast<int>(act), false,
                                static_cast<cudaStream_t>(stream));
  return st == SPCONV_OK ? spconv::ok() : st;
}

spconv_status spconv_submconv3d_dgrad_xrun(const void* dout_dev, const int32_t* nmap_dev, const int32_t* slots_dev,
                                           int64_t slots_capacity, const int64_t* slot_count_dev,
                                           const void* w_dev, void* dfeats_dev, int64_t N, int32_t K, int32_t Ci,
                                           int32_t Co, spconv_dtype dtype, void* stream) {
  if (N < 1 || N >= (int64_t{1} << 30)) return fail(SPCONV_ERR_INVALID_ARG, "N must be in [1, 2^30)");
  if (dtype != SPCONV_BF16 || K != 27 || Co != 128 || Ci < 16 || Ci > 128 || Ci % 16 != 0)
    return fail(SPCONV_ERR_UNSUPPORTED,
                "the x-run input gradient takes bf16, K = 27, Co = 128 and Ci in [16, 128], a multiple of 16");
  if (dout_dev == nullptr || nmap_dev == nullptr || slots_dev == nullptr || slot_count_dev == nullptr ||
      w_dev == nullptr || dfeats_dev == nullptr)
    return fail(SPCONV_ERR_INVALID_ARG, "dout, nmap, slots, slot_count, w and dfeats must be non-NULL");
  if (!spconv::aligned(dout_dev, 16) || !spconv::aligned(w_dev, 16) || !spconv::aligned(dfeats_dev, 16) ||
      !spconv::aligned(nmap_dev, 4) || !spconv::aligned(slots_dev, 4) || !spconv::aligned(slot_count_dev, 8))
    return fail(SPCONV_ERR_INVALID_ARG, "misaligned pointer");
  if (slots_capacity < 1) return fail(SPCONV_ERR_INVALID_ARG, "slots_capacity must be >= 1");
  spconv_status st = spconv::check_device();
  if (st != SPCONV_OK) return st;
  st = spconv::launch_conv_xrun(dout_dev, nmap_dev, slots_dev, slots_capacity, slot_count_dev, w_dev, nullptr,
                                nullptr, dfeats_dev, N, Ci, static_cast<int>(SPCONV_ACT_NONE), true,
                                static_cast<cudaStream_t>(stream));
  return st == SPCONV_OK ? spconv::ok() : st;
}

spconv_status spconv_submconv3d_ex(const void* feats_dev, const int32_t* nmap_dev,
                                   const void* w_dev, const void* bias_dev,
                                   const void* residual_dev, void* out_dev, int64_t N, int32_t K,
                                   int32_t Ci, int32_t Co, spconv_dtype dtype,
                                   spconv_activation act, void* stream) {
  return spconv::submconv3d_impl(feats_dev, nmap_dev, w_dev, bias_dev, residual_dev, out_dev, N, K, Ci,
                                 Co, dtype, act, false, stream);
}

spconv_status spconv_submconv3d_dgrad(const void* dout_dev, const int32_t* nmap_dev,
                                      const void* w_dev, void* dfeats_dev, int64_t N, int32_t K,
                                      int32_t Ci, int32_t Co, spconv_dtype dtype, void* stream) {
  // The same convolution over dout with the weights of offset k taken as
  // w[K-1-k] transposed: rows of width Co in, rows of width Ci out.
  return spconv::submconv3d_impl(dout_dev, nmap_dev, w_dev, nullptr, nullptr, dfeats_dev, N, K, Co, Ci,
                                 dtype, SPCONV_ACT_NONE, true, stream);
}

spconv_status spconv_submconv3d_wgrad(const void* feats_dev, const void* dout_dev,
                                      const int32_t* nmap_dev, float* dw_dev, float* dbias_dev,
                                      int64_t N, int32_t K, int32_t Ci, int32_t Co, spconv_dtype dtype,
                                      void* stream) {
  if (N < 0 || N >= INT32_MAX) return fail(SPCONV_ERR_INVALID_ARG, "N must satisfy 0 <= N < 2^31-1");
  if (K < 1 || Ci < 1 || Co < 1) return fail(SPCONV_ERR_INVALID_ARG, "K, Ci and Co must be >= 1");
  if (dtype != SPCONV_F32 && dtype != SPCONV_TF32 && dtype != SPCONV_BF16)
    return fail(SPCONV_ERR_INVALID_ARG, "unknown dtype");
  if (dw_dev == nullptr) return fail(SPCONV_ERR_INVALID_ARG, "dw must be non-NULL");
  if (N > 0 && (feats_dev == nullptr || dout_dev == nullptr || nmap_dev == nullptr))
    return fail(SPCONV_ERR_INVALID_ARG, "feats, dout and nmap must be non-NULL");
  const size_t elem = dtype == SPCONV_BF16 ? 2 : 4;
  if (!spconv::aligned(feats_dev, elem) || !spconv::aligned(dout_dev, elem) ||
      !spconv::aligned(nmap_dev, 4) || !spconv::aligned(dw_dev, 4) ||
      (dbias_dev != nullptr && !spconv::aligned(dbias_dev, 4)))
    return fail(SPCONV_ERR_INVALID_ARG, "misaligned array");
  if (static_cast<uint64_t>(N) * static_cast<uint64_t>(K) > (1ull << 40))
    return fail(SPCONV_ERR_UNSUPPORTED, "K * N too large");
  spconv_status st = spconv::check_device();
  if (st != SPCONV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    // no voxels: the gradients are zero
    if (!spconv::cuda_ok(cudaMemsetAsync(dw_dev, 0, static_cast<size_t>(K) * Ci * Co * sizeof(float), s),
                         "cudaMemsetAsync(dw)", &st))
      return st;
    if (dbias_dev != nullptr &&
        !spconv::cuda_ok(cudaMemsetAsync(dbias_dev, 0, static_cast<size_t>(Co) * sizeof(float), s),
                         "cudaMemsetAsync(dbias)", &st))
      return st;
    return spconv::ok();
  }
  // bf16 with tensor-core-friendly shapes runs on the tensor cores; every
  // other case on the exact CUDA-core kernel.
  const bool tc = dtype == SPCONV_BF16 && Ci % 16 == 0 && Co % 16 == 0 && spconv::aligned(feats_dev, 16) &&
                  spconv::aligned(dout_dev, 16);
  if (tc) {
    st = spconv::launch_wgrad_tc(feats_dev, dout_dev, nmap_dev, dw_dev, N, K, Ci, Co, s);
    if (st == SPCONV_OK && dbias_dev != nullptr) st = spconv::launch_dbias(dtype, dout_dev, dbias_dev, N, Co, s);
  } else {
    st = spconv::launch_wgrad_simt(dtype, feats_dev, dout_dev, nmap_dev, dw_dev, dbias_dev, N, K, Ci, Co, s);
  }
  return st == SPCONV_OK ? spconv::ok() : st;
}

spconv_status spconv_count_valid_pairs(const int32_t* nmap_dev, int64_t N, int32_t K,
                                       int64_t* count_dev, void* stream) {
  if (N < 0 || N >= INT32_MAX || K < 1) return fail(SPCONV_ERR_INVALID_ARG, "bad N or K");
  if (count_dev == nullptr || (N > 0 && nmap_dev == nullptr))
    return fail(SPCONV_ERR_INVALID_ARG, "nmap and count must be non-NULL");
  if (!spconv::aligned(count_dev, 8)) return fail(SPCONV_ERR_INVALID_ARG, "count must be 8-byte aligned");
  spconv_status st = spconv::check_device();
  if (st != SPCONV_OK) return st;
  st = spconv::launch_count_valid_pairs(nmap_dev, N, K, count_dev, static_cast<cudaStream_t>(stream));
  return st == SPCONV_OK ? spconv::ok() : st;
}

spconv_status spconv_device_status(void* stream) {
  unsigned int bits = 0;
  spconv_status st = spconv::read_and_clear_device_error(static_cast<cudaStream_t>(stream), &bits);
  if (st != SPCONV_OK) return st;
  st = spconv::read_and_clear_wgrad_device_error(static_cast<cudaStream_t>(stream), &bits);
  if (st != SPCONV_OK) return st;
  st = spconv::read_and_clear_xrun_device_error(static_cast<cudaStream_t>(stream), &bits);
  if (st != SPCONV_OK) return st;
  if (bits != 0) return fail(SPCONV_ERR_DEVICE, "device error bits 0x" + std::to_string(bits));
  return spconv::ok();
}

}  // extern "C"

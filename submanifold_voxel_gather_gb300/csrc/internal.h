// Internal launchers shared between the C ABI and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include <cuda_runtime.h>

#include "spconv.h"

namespace spconv {

// Records `msg` as the calling thread's last error and returns `code`.
spconv_status fail(spconv_status code, const std::string& msg);

// Checks a CUDA runtime result; on failure records it and returns false.
bool cuda_ok(cudaError_t err, const char* what, spconv_status* out);

// Number of SMs of the current device (cached per device).
int sm_count();

// ---- neighbour map (nmap_hash.cu)
struct BuildOffsets {
  int32_t d[3 * SPCONV_MAX_BUILD_OFFSETS];
};

size_t hash_capacity(int64_t n);
// With status_dev == nullptr the call waits for `stream` and returns the
// build's verdict; otherwise it writes the verdict (an spconv_status) to
// status_dev on the stream and returns without waiting.
// With xflags (lexicographic 3x3x3 offsets), the dense-row query also
// writes the x-run layout's per-voxel flags there and sets the word at
// xrun_flags_ready(workspace); the other build paths leave both alone.
spconv_status launch_build_nmap(const int32_t* coords, int64_t n, const BuildOffsets& offs,
                                int32_t k, int32_t* nmap, void* workspace, cudaStream_t stream,
                                int32_t* status_dev = nullptr, uint8_t* xflags = nullptr);
// The word of a build workspace that tells whether the x-run flags were written.
const int* xrun_flags_ready(const void* workspace);
// Device address of the allocation-free variant's static scratch on the
// current device (looked up on every call).
spconv_status noalloc_scratch(void** scratch);
spconv_status launch_count_valid_pairs(const int32_t* nmap, int64_t n, int32_t k, int64_t* count,
                                       cudaStream_t stream);

// ---- exact fp32 convolution on CUDA cores (conv_simt.cu)
spconv_status launch_conv_simt_f32(const float* feats, const int32_t* nmap, const float* w,
                                   const float* bias, const float* residual, float* out,
                                   int64_t n, int32_t k, int32_t ci, int32_t co,
                                   spconv_activation act, bool dgrad, cudaStream_t stream);

// ---- tensor-core convolution (conv_tc.cu); dtype is SPCONV_BF16.  With
// dgrad, ci/co are the dout/dfeats widths (forward Co/Ci), feats is dout and
// the weights of offset k are w[K-1-k] transposed (forward layout in place).
// `order`, if not null, is a permutation of 0..N-1: tile slot s gathers the
// map column order[s] and writes output row order[s] (forward only).
spconv_status launch_conv_tc(spconv_dtype dtype, const void* feats, const int32_t* nmap,
                             const void* w, const void* bias, const void* residual, void* out,
                             int64_t n, int32_t k, int32_t ci, int32_t co, spconv_activation act,
                             bool dgrad, cudaStream_t stream, const int32_t* order = nullptr);

// ---- tile order (nmap_hash.cu): order[s] for s in chunks of kTileOrderChunk
// consecutive voxels, each chunk's voxels sorted by neighbour mask
constexpr int kTileOrderChunk = 4096;
spconv_status launch_tile_order(const int32_t* nmap, int64_t n, int32_t k, int32_t* order,
                                cudaStream_t stream);

// ---- weight / bias gradients, exact fp32 on CUDA cores (wgrad_simt.cu)
spconv_status launch_wgrad_simt(spconv_dtype dtype, const void* feats, const void* dout,
                                const int32_t* nmap, float* dw, float* dbias, int64_t n, int32_t k,
                                int32_t ci, int32_t co, cudaStream_t stream);

spconv_status launch_dbias(spconv_dtype dtype, const void* dout, float* dbias, int64_t n, int32_t co,
                           cudaStream_t stream);

// ---- weight gradient on the tensor cores, bf16 (wgrad_tc.cu); needs Ci and
// Co multiples of 16 and 16-byte aligned feats and dout
spconv_status launch_wgrad_tc(const void* feats, const void* dout, const int32_t* nmap, float* dw,
                              int64_t n, int32_t k, int32_t ci, int32_t co, cudaStream_t stream);

// ---- device error words.  ptx.cuh gives each translation unit its own
// copy, so every unit whose kernels can set it reads back its own: the
// forward / input-gradient conv (conv_tc.cu) and the weight gradient
// (wgrad_tc.cu).  Each call waits for the stream and clears the unit's
// bits after reading them: the conv's call stores them in *bits, the weight
// gradient's ORs them in, so call the conv's first.
spconv_status read_and_clear_device_error(cudaStream_t stream, unsigned int* bits);
spconv_status read_and_clear_wgrad_device_error(cudaStream_t stream, unsigned int* bits);
spconv_status read_and_clear_xrun_device_error(cudaStream_t stream, unsigned int* bits);

// ---- x-run slot layout (xrun.cu) and the row-shifted conv (conv_xrun.cu)
size_t xrun_workspace_bytes(int64_t n);
int64_t xrun_slot_capacity(int64_t n);
// flags_ready (optional): a word that, when set on the device, says the map
// build's dense query wrote its per-voxel bits at xrun_raw_bits(workspace,
// n); the layout then decides the separators from those bits alone instead
// of reading the map and the coordinates.
spconv_status launch_xrun_layout(const int32_t* coords, const int32_t* nmap, int64_t n, int32_t* slots,
                                 int64_t cap, int64_t* slot_count, void* workspace, cudaStream_t stream,
                                 const int* flags_ready = nullptr);
uint8_t* xrun_raw_bits(void* workspace, int64_t n);
// bf16, lexicographic 3x3x3 offsets; 128 reduced channels (forward Ci, or
// forward Co for the input gradient) and co <= 128 output channels.
// residual (or null) and act: the fused epilogue act(conv + bias + residual).
spconv_status launch_conv_xrun(const void* feats, const int32_t* nmap, const int32_t* slots,
                               int64_t slots_capacity, const int64_t* slot_count, const void* w,
                               const void* bias, const void* residual, void* out, int64_t n, int32_t co,
                               int act, bool dgrad, cudaStream_t stream);

}  // namespace spconv

// Slot layout over x-runs for the row-shifted convolution (conv_xrun.cu).
//
// A run is a maximal sequence of consecutive voxels (consecutive indices)
// whose cells are consecutive in x on one (z, y) line.  The layout lists the
// voxels in index order as "slots" and puts separator slots between runs, so
// that for every voxel slot s and dx in {-1, 0, +1}, slot s + dx stands for the
// cell (z, y, x + dx): the next voxel of the run, or a separator that stands
// for the cell just outside the run.  For each (dz, dy) group of the 3x3x3
// offsets the convolution then gathers one operand over the slots and reads
// the three dx offsets as the same rows shifted by one.
//
// Slot codes (int32):
//   n >= 0        voxel n;
//   -2 - 2n       the cell just right of voxel n (a run end): (z, y, x + 1);
//   -3 - 2n       the cell just left of voxel n (a run start): (z, y, x - 1);
//   -1            empty.
// A separator's gathered row for group (dz, dy) is nmap[(dz, dy, +1), n] or
// nmap[(dz, dy, -1), n]: the neighbour map already holds it.
//
// Between two runs one separator is enough when the right cells of the first
// run's end and the left cells of the next run's start have the same map
// entries in all nine groups (both missing, mostly); else there are two.  The
// first voxel gets a left separator, and the last one a right separator, when
// one of its nine outer cells is active.  Any voxel order gives a correct
// layout; sorted (z, y, x) order gives long runs.
//
// Three launches: per-voxel slot counts and block sums; one block scans the
// block sums and writes the slot count S; each voxel writes its slots.
#include <cuda_runtime.h>

#include "internal.h"

namespace spconv {
namespace {

constexpr int kXrunBlock = 1024;
constexpr int kXrunPer = 4;  // voxels per thread in the count and the fill
constexpr int64_t kXrunSpan = static_cast<int64_t>(kXrunBlock) * kXrunPer;

// Normalised map entry: the row, or n for every kind of missing entry.
__device__ __forceinline__ int32_t map_row(const int32_t* nmap, int64_t n, int k, int64_t v) {
  const int32_t e = __ldg(nmap + static_cast<int64_t>(k) * n + v);
  return (e >= 0 && e < n) ? e : static_cast<int32_t>(n);
}

__device__ __forceinline__ bool same_run(const int32_t* coords, int64_t a) {
  // voxel a + 1 continues voxel a's run
  const int32_t* p = coords + 3 * a;
  return __ldg(p + 3) == __ldg(p) && __ldg(p + 4) == __ldg(p + 1) && __ldg(p + 5) == __ldg(p + 2) + 1;
}

// Flags of voxel i: bits 0-1 = separators after it (0..2), bit 2 = a
// separator before it (voxel 0 only).  From the map and the coordinates.
__device__ __noinline__ uint32_t voxel_flags_from_map(const int32_t* coords, const int32_t* nmap, int64_t n,
                                                         int64_t i) {
  uint32_t f = 0;
  const bool run_end = i + 1 >= n || !same_run(coords, i);
  if (run_end) {
    if (i + 1 >= n) {
      bool any = false;
      for (int g = 0; g < 9; ++g) any |= map_row(nmap, n, 3 * g + 2, i) != n;
      f = any ? 1u : 0u;
    } else {
      bool same = true;
      for (int g = 0; g < 9; ++g) same &= map_row(nmap, n, 3 * g + 2, i) == map_row(nmap, n, 3 * g, i + 1);
      f = same ? 1u : 2u;
    }
  }
  if (i == 0) {
    bool any = false;
    for (int g = 0; g < 9; ++g) any |= map_row(nmap, n, 3 * g, 0) != n;
    if (any) f |= 4u;
  }
  return f;
}

// The same flags from the bits the map build's dense query writes per voxel
// (sorted input only): bit 0 a run ends at the voxel, bit 1 one of its nine
// (dz, dy, +1) cells is active, bit 2 one of its nine (dz, dy, -1) cells is
// active, bit 3 it ends a run and the next voxel is two cells further on its
// line.  A run end's right cells and the next voxel's left cells have equal
// map entries in all nine groups exactly when they are the same cells or none
// of them is active.  `a` is the voxel's bits, `a_next` the next voxel's.
__device__ __forceinline__ uint32_t voxel_flags_from_bits(int64_t i, int64_t n, uint32_t a, uint32_t a_next) {
  uint32_t f = 0;
  if (a & 1u) {
    if (i + 1 >= n) f = (a & 2u) ? 1u : 0u;
    else f = ((a & 8u) != 0u || ((a & 2u) == 0u && (a_next & 4u) == 0u)) ? 1u : 2u;
  }
  if (i == 0 && (a & 4u)) f |= 4u;
  return f;
}

__device__ __forceinline__ uint32_t slot_count_of(uint32_t f) { return 1u + (f & 3u) + ((f >> 2) & 1u); }

// The flags of voxels i0 .. i0 + kXrunPer - 1, one byte each (0 past n).
// With the dense query's bits (`pre`), computed from them; else read from
// `flags`, which the count wrote.  Both buffers are padded to 256 bytes.
__device__ __forceinline__ uint32_t flags4(const uint8_t* flags, const uint8_t* raw, bool pre, int64_t n,
                                           int64_t i0) {
  if (!pre) return *reinterpret_cast<const uint32_t*>(flags + i0);
  const uint32_t a4 = *reinterpret_cast<const uint32_t*>(raw + i0);
  const uint32_t a_after = i0 + kXrunPer < n ? raw[i0 + kXrunPer] : 0u;
  uint32_t packed = 0;
#pragma unroll
  for (int j = 0; j < kXrunPer; ++j) {
    const uint32_t a = (a4 >> (8 * j)) & 0xffu;
    const uint32_t a_next = j + 1 < kXrunPer ? (a4 >> (8 * (j + 1))) & 0xffu : a_after;
    if (i0 + j < n) packed |= voxel_flags_from_bits(i0 + j, n, a, a_next) << (8 * j);
  }
  return packed;
}

__device__ __forceinline__ uint32_t slot_count4(uint32_t f4, int64_t n, int64_t i0) {
  uint32_t cnt = 0;
#pragma unroll
  for (int j = 0; j < kXrunPer; ++j)
    if (i0 + j < n) cnt += slot_count_of((f4 >> (8 * j)) & 0xffu);
  return cnt;
}

// Each thread takes kXrunPer consecutive voxels: block sums of the slot
// counts; without the dense query's bits also the flags (one 32-bit store).
// `ready` is the word the dense query sets when it wrote the bits.
__global__ void __launch_bounds__(kXrunBlock) xrun_count_kernel(const int32_t* __restrict__ coords,
                                                                const int32_t* __restrict__ nmap, int64_t n,
                                                                uint8_t* __restrict__ flags,
                                                                int64_t* __restrict__ block_sums,
                                                                const int* __restrict__ ready,
                                                                const uint8_t* __restrict__ raw) {
  __shared__ uint32_t warp_sums[kXrunBlock / 32];
  const int64_t i0 = (static_cast<int64_t>(blockIdx.x) * kXrunBlock + threadIdx.x) * kXrunPer;
  const bool pre = ready != nullptr && *ready != 0;
  uint32_t cnt = 0;
  if (i0 < n) {
    uint32_t packed = 0;
    if (pre) {
      packed = flags4(flags, raw, true, n, i0);
    } else {
#pragma unroll 1
      for (int j = 0; j < kXrunPer; ++j)
        if (i0 + j < n) packed |= voxel_flags_from_map(coords, nmap, n, i0 + j) << (8 * j);
      *reinterpret_cast<uint32_t*>(flags + i0) = packed;
    }
    cnt = slot_count4(packed, n, i0);
  }
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_down_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t s = warp_sums[threadIdx.x];
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) block_sums[blockIdx.x] = s;
  }
}

// Exclusive scan of one value per thread of the block; returns the block total.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* warp_sums, T* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T w = warp_sums[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const T before = (warp > 0 ? warp_sums[warp - 1] : T(0)) + x - v;
  const T total = warp_sums[31];
  __syncthreads();  // warp_sums is reused by the next call
  *out = before;
  return total;
}

// One block: exclusive scan of the block sums in place; writes S.
__global__ void __launch_bounds__(kXrunBlock) xrun_scan_kernel(int64_t* __restrict__ block_sums, int64_t nb,
                                                               int64_t* __restrict__ slot_count) {
  __shared__ int64_t warp_sums[32];
  int64_t carry = 0;
  for (int64_t base = 0; base < nb; base += kXrunBlock) {
    const int64_t j = base + threadIdx.x;
    const int64_t v = j < nb ? block_sums[j] : 0;
    int64_t ex;
    const int64_t total = block_exclusive_scan<int64_t>(v, warp_sums, &ex);
    if (j < nb) block_sums[j] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) *slot_count = carry;
}

// Each voxel writes its slot and the separators around it (kXrunPer
// consecutive voxels per thread, as in the count).  A block's slots number
// at most 4 * kXrunBlock * kXrunPer, so the in-block scan is 32-bit.  They
// are assembled in shared memory (dynamic, kFillSmem bytes) and written out
// in one coalesced pass: written straight from the threads, each store
// instruction of a warp touched 32 short runs a few slots apart.
constexpr uint32_t kFillSmem = 4u * kXrunBlock * kXrunPer * 4u;
__global__ void __launch_bounds__(kXrunBlock) xrun_fill_kernel(const uint8_t* __restrict__ flags, int64_t n,
                                                               const int64_t* __restrict__ block_offsets,
                                                               int32_t* __restrict__ slots, int64_t cap,
                                                               int32_t* __restrict__ overflow,
                                                               const int* __restrict__ ready,
                                                               const uint8_t* __restrict__ raw) {
  extern __shared__ int32_t block_slots[];
  __shared__ uint32_t warp_sums[32];
  const int64_t i0 = (static_cast<int64_t>(blockIdx.x) * kXrunBlock + threadIdx.x) * kXrunPer;
  const bool pre = ready != nullptr && *ready != 0;
  const uint32_t f4 = i0 < n ? flags4(flags, raw, pre, n, i0) : 0u;
  const uint32_t cnt = i0 < n ? slot_count4(f4, n, i0) : 0u;
  uint32_t ex;
  const uint32_t total = block_exclusive_scan<uint32_t>(cnt, warp_sums, &ex);
  const int64_t s0 = block_offsets[blockIdx.x];
  if (s0 + total > cap) {  // the same for every thread of the block
    if (threadIdx.x == 0) atomicExch(overflow, 1);
    return;
  }
  uint32_t s = ex;
#pragma unroll
  for (int j = 0; j < kXrunPer; ++j) {
    if (i0 + j >= n) break;
    const uint32_t f = (f4 >> (8 * j)) & 0xffu;
    const int32_t v = static_cast<int32_t>(i0 + j);
    if (f & 4u) block_slots[s++] = -3 - 2 * v;  // left of voxel 0
    block_slots[s++] = v;
    const uint32_t after = f & 3u;
    if (after >= 1u) block_slots[s++] = -2 - 2 * v;        // right of this run end (shared when one)
    if (after == 2u) block_slots[s++] = -3 - 2 * (v + 1);  // left of the next run's start
  }
  __syncthreads();
  for (uint32_t k = threadIdx.x; k < total; k += kXrunBlock) slots[s0 + k] = block_slots[k];
}

}  // namespace

size_t xrun_workspace_bytes(int64_t n) {
  const int64_t nb = (n + kXrunSpan - 1) / kXrunSpan;
  return 2 * static_cast<size_t>(((n + 255) / 256) * 256) + static_cast<size_t>(nb) * 8u + 256u;
}

int64_t xrun_slot_capacity(int64_t n) { return 3 * n + 1; }

// The per-voxel bits the map build's dense query writes (after the flags).
uint8_t* xrun_raw_bits(void* workspace, int64_t n) { return static_cast<uint8_t*>(workspace) + ((n + 255) / 256) * 256; }

// Workspace: per-voxel flags (N bytes, rounded up to 256), the map build's
// per-voxel bits (the same), the block sums,
// and an overflow word (set if the slots would pass `cap`; never with
// cap >= xrun_slot_capacity(n)).
spconv_status launch_xrun_layout(const int32_t* coords, const int32_t* nmap, int64_t n, int32_t* slots,
                                 int64_t cap, int64_t* slot_count, void* workspace, cudaStream_t stream,
                                 const int* flags_ready) {
  const int64_t nb = (n + kXrunSpan - 1) / kXrunSpan;
  uint8_t* flags = static_cast<uint8_t*>(workspace);
  uint8_t* raw = xrun_raw_bits(workspace, n);
  int64_t* block_sums = reinterpret_cast<int64_t*>(static_cast<uint8_t*>(workspace) + 2 * ((n + 255) / 256) * 256);
  int32_t* overflow = reinterpret_cast<int32_t*>(block_sums + nb);
  spconv_status st = SPCONV_OK;
  if (!cuda_ok(cudaMemsetAsync(overflow, 0, sizeof(int32_t), stream), "cudaMemsetAsync", &st)) return st;
  xrun_count_kernel<<<static_cast<unsigned>(nb), kXrunBlock, 0, stream>>>(coords, nmap, n, flags, block_sums,
                                                                         flags_ready, raw);
  if (!cuda_ok(cudaGetLastError(), "xrun_count_kernel", &st)) return st;
  xrun_scan_kernel<<<1, kXrunBlock, 0, stream>>>(block_sums, nb, slot_count);
  if (!cuda_ok(cudaGetLastError(), "xrun_scan_kernel", &st)) return st;
  if (!cuda_ok(cudaFuncSetAttribute(xrun_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kFillSmem)),
               "cudaFuncSetAttribute", &st))
    return st;
  xrun_fill_kernel<<<static_cast<unsigned>(nb), kXrunBlock, kFillSmem, stream>>>(flags, n, block_sums, slots, cap,
                                                                                   overflow, flags_ready, raw);
  if (!cuda_ok(cudaGetLastError(), "xrun_fill_kernel", &st)) return st;
  return SPCONV_OK;
}

}  // namespace spconv

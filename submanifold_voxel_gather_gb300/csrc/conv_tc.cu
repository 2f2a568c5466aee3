// Fused submanifold convolution on the 5th-generation tensor cores (sm_103a).
//
// Computes out[n, co] = bias[co] + sum_k sum_ci feats[nmap[k, n], ci] * w[k, ci, co]
// (page "sparse_conv_metal.py", trellis-2-mrp-mlx: module docstring formula,
// kernel-body sentinel skip, wrapper bias) as an implicit GEMM with
// M = 128 voxels per tile, N = output channels (<= 256 per launch) and a
// reduction over (k, ci).  The page's kernel runs one scalar thread per
// (n, co); here a persistent CTA per SM runs a warp-specialised pipeline:
//
//   warp 2     nmap loader: copies the tile's (K x 128) neighbour indices into
//              a shared-memory slot (coalesced 128-byte reads per offset) and
//              records, per offset, whether any of the 128 entries is valid
//              (warp ballot).  Offsets with no valid entry are skipped whole.
//   warps 8-11 A producers: for each kept offset k and each 128-byte Ci chunk,
//              gather the 128 neighbour rows with 16-byte cp.async (each warp
//              instruction moves four whole 128-byte row segments) straight
//              into the 128-byte-swizzled K-major operand layout; rows that
//              are not valid are zero-filled without a read.  Completion is
//              tracked by the stage's mbarrier (cp.async.mbarrier.arrive).
//   warp 0     B producer: loads the w[k] chunk (MN-major, 128-byte swizzle)
//              with tiled TMA and writes the stage's metadata.
//   warp 1     MMA issuer (one thread): tcgen05.mma M=128, N=Co, K=16 into an
//              fp32 accumulator in tensor memory; the accumulator is
//              double-buffered so the epilogue of one tile overlaps the main
//              loop of the next.
//   warps 4-7  epilogue: tcgen05.ld of the accumulator rows, + bias (fp32),
//              one rounding to bf16, 16-byte stores.
//
// The gathered (K, N, Ci) operand only ever exists one tile at a time in
// shared memory.  Every wait on an mbarrier is bounded in time; on timeout the
// kernel records an error bit, drains its own copies and MMAs, frees its
// tensor memory and returns.
//
// Row gathers use the LSU path rather than TMA tile::gather4: measured on
// GB300, a 4-row gather4 (or a 4-row tiled box) costs ~80 SM cycles of TMA
// time, so 32 of them per 16 KB stage starve the tensor core ~10x; TMA is
// kept for the weight tiles, which are large boxes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

#ifndef SPCONV_GATHER_L1
#define SPCONV_GATHER_L1 1
#endif

namespace spconv {
namespace {

constexpr int kTileM = 128;
constexpr int kThreads = 384;
constexpr int kProducerWarp0 = 8;       // first A-producer warp
constexpr int kProducerThreads = 128;   // warps 8-11
constexpr int kSlots = 2;               // neighbour-index slots (tiles in flight)
constexpr int kSlotRowsMax = 32;        // offsets per slot (more offsets use several slots)
constexpr uint32_t kABytes = kTileM * 128;
constexpr int kMaxStages = 8;
constexpr int kMaxSmem = 232448;        // 227 KB opt-in limit per block

struct Bf16Traits {
  using T = __nv_bfloat16;
  static constexpr int kElem = 2;
  static constexpr int kChunk = 64;     // elements per 128-byte row
  static constexpr int kKPerMma = 16;
  static constexpr uint32_t kFmt = 1;   // BF16 in the instruction descriptor
  static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};

struct Tf32Traits {
  using T = float;
  static constexpr int kElem = 4;
  static constexpr int kChunk = 32;
  static constexpr int kKPerMma = 8;
  static constexpr uint32_t kFmt = 2;   // TF32
  static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};

struct TcParams {
  const void* feats;
  const int32_t* nmap;
  const void* bias;
  void* out;
  int64_t n;
  int64_t num_tiles;
  int32_t k;
  int32_t ci;
  int32_t co;        // row stride of out
  int32_t co_base;   // first output channel of this launch
  int32_t co_count;  // channels of this launch (<= 256)
  int32_t n_mma;     // MMA N: co_count rounded up to a 128-byte row of B
  int32_t num_chunks;
  int32_t num_groups;  // slots per tile: ceil(k / 32)
  int32_t slot_rows;   // min(k, 32)
  uint32_t stages;
  uint32_t stage_bytes;
  uint32_t box_bytes;  // one TMA box of w: kChunk x kChunk elements
  uint32_t tmem_cols;
  uint32_t idesc;
  uint32_t off_slots;
  uint32_t off_bias;
  uint32_t off_meta;
  uint32_t off_bars;
};

enum : uint32_t { kMetaFirst = 1u, kMetaLast = 2u };

__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }

// Bias + one rounding + store of 16 consecutive accumulator columns.
__device__ __forceinline__ void store16(__nv_bfloat16* dst, const uint32_t* acc, const float* b) {
  uint32_t packed[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(acc[2 * j]) + b[2 * j],
                                             __uint_as_float(acc[2 * j + 1]) + b[2 * j + 1]);
    packed[j] = *reinterpret_cast<uint32_t*>(&h);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  d[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
}

__device__ __forceinline__ void store16(float* dst, const uint32_t* acc, const float* b) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    d[j] = make_float4(__uint_as_float(acc[4 * j]) + b[4 * j], __uint_as_float(acc[4 * j + 1]) + b[4 * j + 1],
                       __uint_as_float(acc[4 * j + 2]) + b[4 * j + 2],
                       __uint_as_float(acc[4 * j + 3]) + b[4 * j + 3]);
}

// Offsets of one slot that the tile issues, and which of them ends the tile.
// With one slot per tile the tile ends at its highest kept offset (offset 0 if
// the tile has no valid entry at all: its rows are zero-filled, so the
// accumulator becomes exactly zero); with several slots the final offset is
// always issued so the end is known when it is reached.
__device__ __forceinline__ uint32_t slot_schedule(uint32_t mask, int g, int num_groups, int krows,
                                                  int* last_r) {
  *last_r = -1;
  if (g == num_groups - 1) {
    if (num_groups == 1) {
      if (mask == 0u) mask = 1u;
    } else {
      mask |= 1u << (krows - 1);
    }
    *last_r = 31 - __clz(mask);
  }
  return mask;
}

template <class Tr>
__global__ void __launch_bounds__(kThreads, 1)
    submconv_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const TcParams p) {
  using T = typename Tr::T;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t S = p.stages;

  int32_t* slots = reinterpret_cast<int32_t*>(smem + p.off_slots);
  float* bias_s = reinterpret_cast<float*>(smem + p.off_bias);
  uint32_t* meta = reinterpret_cast<uint32_t*>(smem + p.off_meta);
  uint32_t* slot_mask = meta + S;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* slot_full = bars + 2 * S;
  uint64_t* slot_empty = slot_full + kSlots;
  uint64_t* tmem_full = slot_empty + kSlots;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain = tmem_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  uint32_t* consumed_holder = tmem_holder + 1;
  uint32_t* fills_holder = tmem_holder + 2;

  if (warp == 0 && lane == 0) {
    for (uint32_t s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full[s]), kProducerThreads + 1);
      mbar_init(smem_addr(&empty[s]), 1);
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_addr(&slot_full[i]), 32);
      mbar_init(smem_addr(&slot_empty[i]), 32 + kProducerThreads);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&tmem_full[i]), 1);
      mbar_init(smem_addr(&tmem_empty[i]), 4);
    }
    mbar_init(smem_addr(drain), 1);
    *consumed_holder = 0;
    *fills_holder = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_holder), p.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 3) {
    const T* bias = static_cast<const T*>(p.bias);
    for (int j = lane; j < 256; j += 32)
      bias_s[j] = (bias != nullptr && j < p.co_count) ? to_f32(bias[p.co_base + j]) : 0.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int64_t n_rows = p.n;
  if (warp == 2) {
    // ------------------------------------------------------ nmap loader
    uint32_t slot = 0, slot_phase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      const int64_t n0 = t * kTileM;
      for (int g = 0; g < p.num_groups; ++g) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&slot_empty[slot]), slot_phase ^ 1))) {
          ok = false;
          break;
        }
        int32_t* dst = slots + slot * p.slot_rows * kTileM;
        const int krows = min(kSlotRowsMax, p.k - g * kSlotRowsMax);
        uint32_t mask = 0;
        for (int r0 = 0; r0 < krows; r0 += 8) {
          int32_t v[8][4];
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) {
            const int r = r0 + rr;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int64_t n = n0 + lane + 32 * j;
              v[rr][j] = -1;
              if (r < krows && n < n_rows)
                v[rr][j] = __ldg(p.nmap + static_cast<int64_t>(g * kSlotRowsMax + r) * n_rows + n);
            }
          }
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) {
            const int r = r0 + rr;
            bool any = false;
#pragma unroll
            for (int j = 0; j < 4; ++j) any |= (v[rr][j] >= 0 && v[rr][j] < n_rows);
            const uint32_t ballot = __ballot_sync(0xffffffffu, any);
            if (r < krows) {
#pragma unroll
              for (int j = 0; j < 4; ++j) dst[r * kTileM + lane + 32 * j] = v[rr][j];
              mask |= (ballot != 0u ? 1u : 0u) << r;
            }
          }
        }
        if (lane == 0) slot_mask[slot] = mask;
        mbar_arrive(smem_addr(&slot_full[slot]));
        if (++slot == kSlots) {
          slot = 0;
          slot_phase ^= 1;
        }
      }
    }
  } else if (warp >= kProducerWarp0) {
    // ------------------------------------------------------ A producers
    const uint32_t aw = warp - kProducerWarp0;  // rows 32*aw .. 32*aw+31
    const int sub_row = static_cast<int>(lane >> 3);
    const int chunk16 = static_cast<int>(lane & 7);
    const char* feats = static_cast<const char*>(p.feats);
    const int64_t row_bytes = static_cast<int64_t>(p.ci) * Tr::kElem;
    uint32_t stage = 0, st_phase = 0, slot = 0, sl_phase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      for (int g = 0; g < p.num_groups && ok; ++g) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&slot_full[slot]), sl_phase))) {
          ok = false;
          break;
        }
        const int32_t* src = slots + slot * p.slot_rows * kTileM;
        const int krows = min(kSlotRowsMax, p.k - g * kSlotRowsMax);
        int last_r;
        uint32_t mask = slot_schedule(slot_mask[slot], g, p.num_groups, krows, &last_r);
        while (mask != 0u && ok) {
          const int r = __ffs(mask) - 1;
          mask &= mask - 1;
          int32_t idx[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) idx[j] = src[r * kTileM + 32 * aw + 4 * j + sub_row];
          for (int c = 0; c < p.num_chunks; ++c) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage]), st_phase ^ 1))) {
              ok = false;
              break;
            }
            const int64_t col_byte = static_cast<int64_t>(c) * 128 + chunk16 * 16;
            const bool col_ok = col_byte < row_bytes;
            const uint32_t a_dst = smem_addr(smem + stage * p.stage_bytes);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int row = 32 * static_cast<int>(aw) + 4 * j + sub_row;
              const int32_t v = idx[j];
              const bool valid = col_ok && v >= 0 && v < n_rows;
              const char* gsrc = valid ? feats + static_cast<int64_t>(v) * row_bytes + col_byte : feats;
              const uint32_t d = a_dst + static_cast<uint32_t>(row) * 128u +
                                 (static_cast<uint32_t>(chunk16 ^ (row & 7)) << 4);
              cp_async_16<SPCONV_GATHER_L1 != 0>(d, gsrc, valid ? 16u : 0u);
            }
            cp_async_arrive_noinc(smem_addr(&full[stage]));
            if (++stage == S) {
              stage = 0;
              st_phase ^= 1;
            }
          }
        }
        mbar_arrive(smem_addr(&slot_empty[slot]));
        if (++slot == kSlots) {
          slot = 0;
          sl_phase ^= 1;
        }
      }
    }
    cp_async_wait_all();
  } else if (warp == 0) {
    // ------------------------------------------------------ B producer
    uint32_t stage = 0, st_phase = 0, slot = 0, sl_phase = 0, fills = 0;
    const int nboxes = p.n_mma / Tr::kChunk;
    const uint32_t b_bytes = static_cast<uint32_t>(p.n_mma) * 128u;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      bool first = true;
      for (int g = 0; g < p.num_groups && ok; ++g) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&slot_full[slot]), sl_phase))) {
          ok = false;
          break;
        }
        const int krows = min(kSlotRowsMax, p.k - g * kSlotRowsMax);
        const bool final_group = (g == p.num_groups - 1);
        int last_r;
        uint32_t mask = slot_schedule(slot_mask[slot], g, p.num_groups, krows, &last_r);
        while (mask != 0u && ok) {
          const int r = __ffs(mask) - 1;
          mask &= mask - 1;
          const int32_t kk = g * kSlotRowsMax + r;
          for (int c = 0; c < p.num_chunks; ++c) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage]), st_phase ^ 1))) {
              ok = false;
              break;
            }
            const uint32_t fullb = smem_addr(&full[stage]);
            if (lane == 0) {
              const int steps = min(Tr::kChunk, p.ci - c * Tr::kChunk) / Tr::kKPerMma;
              uint32_t m = static_cast<uint32_t>(steps) << 8;
              if (first) m |= kMetaFirst;
              if (final_group && r == last_r && c == p.num_chunks - 1) m |= kMetaLast;
              meta[stage] = m;
              mbar_arrive_expect_tx(fullb, b_bytes);
            }
            __syncwarp();
            const uint32_t b_dst = smem_addr(smem + stage * p.stage_bytes) + kABytes;
            if (static_cast<int>(lane) < nboxes)
              tma_load_3d(b_dst + lane * p.box_bytes, &tm_w,
                          p.co_base + static_cast<int>(lane) * Tr::kChunk, c * Tr::kChunk, kk,
                          fullb);
            first = false;
            ++fills;
            if (++stage == S) {
              stage = 0;
              st_phase ^= 1;
            }
          }
        }
        __syncwarp();
        mbar_arrive(smem_addr(&slot_empty[slot]));
        if (++slot == kSlots) {
          slot = 0;
          sl_phase ^= 1;
        }
      }
    }
    if (lane == 0) *fills_holder = fills;
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, st_phase = 0, consumed = 0;
      uint32_t tile_i = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++tile_i) {
        const uint32_t buf = tile_i & 1u;
        const uint32_t use = tile_i >> 1;
        if (!mbar_wait(smem_addr(&tmem_empty[buf]), (use & 1u) ^ 1u)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * static_cast<uint32_t>(p.n_mma);
        bool last = false;
        while (!last) {
          if (!mbar_wait(smem_addr(&full[stage]), st_phase)) {
            ok = false;
            break;
          }
          // The A rows were written by cp.async (generic proxy); the MMA reads
          // them through the async proxy.
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t m = meta[stage];
          const int steps = static_cast<int>((m >> 8) & 0xFFu);
          const uint32_t a0 = smem_addr(smem + stage * p.stage_bytes);
          const uint32_t b0 = a0 + kABytes;
          for (int s = 0; s < steps; ++s) {
            const uint64_t adesc = sw128_desc(a0 + s * 32u, 16u, 1024u);
            const uint64_t bdesc = sw128_desc(b0 + s * (Tr::kKPerMma * 128u), p.box_bytes, 1024u);
            const uint32_t acc = (s > 0 || (m & kMetaFirst) == 0u) ? 1u : 0u;
            if constexpr (Tr::kFmt == 2)
              umma_tf32(d_tmem, adesc, bdesc, p.idesc, acc);
            else
              umma_f16(d_tmem, adesc, bdesc, p.idesc, acc);
          }
          umma_commit(smem_addr(&empty[stage]));
          ++consumed;
          if (++stage == S) {
            stage = 0;
            st_phase ^= 1;
          }
          last = (m & kMetaLast) != 0u;
        }
        if (!ok) break;
        umma_commit(smem_addr(&tmem_full[buf]));
      }
      *consumed_holder = consumed;
      umma_commit(smem_addr(drain));
      mbar_wait(smem_addr(drain), 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------ epilogue
    const uint32_t sub = warp & 3u;
    T* out = static_cast<T*>(p.out);
    uint32_t tile_i = 0;
    for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++tile_i) {
      const uint32_t buf = tile_i & 1u;
      const uint32_t use = tile_i >> 1;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&tmem_full[buf]), use & 1u))) break;
      tc_fence_after();
      const int64_t row = t * kTileM + sub * 32 + lane;
      const uint32_t taddr = tmem_base + ((sub * 32u) << 16) + buf * static_cast<uint32_t>(p.n_mma);
      T* orow = out + row * p.co + p.co_base;
      int c0 = 0;
      for (; c0 + 32 <= p.co_count; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c0, v);
        tmem_ld_wait();
        if (row < n_rows) {
          store16(orow + c0, v, bias_s + c0);
          store16(orow + c0 + 16, v + 16, bias_s + c0 + 16);
        }
      }
      if (c0 < p.co_count) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(taddr + c0, v);
        tmem_ld_wait();
        if (row < n_rows) store16(orow + c0, v, bias_s + c0);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tmem_empty[buf]));
    }
  }

  // ---------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // Weight loads issued but never consumed exist only after a timed-out
    // wait: wait (bounded) for them to land before the CTA's memory goes away.
    const uint32_t fills = *fills_holder;
    for (uint32_t i = *consumed_holder; i < fills; ++i)
      mbar_wait(smem_addr(&full[i % S]), (i / S) & 1u);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(spconv_status* st) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                       cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (fn == nullptr) *st = fail(SPCONV_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  return fn;
}

template <class Tr>
spconv_status launch_typed(const void* feats, const int32_t* nmap, const void* w, const void* bias,
                           void* out, int64_t n, int32_t k, int32_t ci, int32_t co,
                           cudaStream_t stream) {
  spconv_status st = SPCONV_OK;
  EncodeTiledFn encode = encode_fn(&st);
  if (encode == nullptr) return st;

  CUtensorMap tm_w;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(co), static_cast<cuuint64_t>(ci),
                          static_cast<cuuint64_t>(k)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(co) * Tr::kElem,
                             static_cast<cuuint64_t>(ci) * co * Tr::kElem};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(Tr::kChunk), static_cast<cuuint32_t>(Tr::kChunk), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(&tm_w, Tr::kTmaType, 3, const_cast<void*>(w), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(SPCONV_ERR_CUDA, "cuTensorMapEncodeTiled(w) failed: " + std::to_string(r));
  }

  const int64_t num_tiles = (n + kTileM - 1) / kTileM;
  const int sms = sm_count();
  if (sms <= 0) return fail(SPCONV_ERR_CUDA, "could not query the SM count");
  const int grid = static_cast<int>(num_tiles < sms ? num_tiles : sms);

  for (int32_t co_base = 0; co_base < co; co_base += 256) {
    TcParams p{};
    p.feats = feats;
    p.nmap = nmap;
    p.bias = bias;
    p.out = out;
    p.n = n;
    p.num_tiles = num_tiles;
    p.k = k;
    p.ci = ci;
    p.co = co;
    p.co_base = co_base;
    p.co_count = (co - co_base) < 256 ? (co - co_base) : 256;
    p.n_mma = (p.co_count + Tr::kChunk - 1) / Tr::kChunk * Tr::kChunk;
    p.num_chunks = (ci + Tr::kChunk - 1) / Tr::kChunk;
    p.num_groups = (k + kSlotRowsMax - 1) / kSlotRowsMax;
    p.slot_rows = k < kSlotRowsMax ? k : kSlotRowsMax;
    p.box_bytes = Tr::kChunk * 128u;
    p.stage_bytes = kABytes + static_cast<uint32_t>(p.n_mma) * 128u;
    uint32_t cols = 32;
    while (cols < 2u * static_cast<uint32_t>(p.n_mma)) cols <<= 1;
    p.tmem_cols = cols;
    p.idesc = (1u << 4) | (Tr::kFmt << 7) | (Tr::kFmt << 10) | (1u << 16) |
              ((static_cast<uint32_t>(p.n_mma) >> 3) << 17) | ((kTileM >> 4) << 24);

    const uint32_t slot_bytes = static_cast<uint32_t>(p.slot_rows) * kTileM * 4u;
    const uint32_t fixed = kSlots * slot_bytes + 256u * 4u + (kMaxStages + kSlots) * 4u +
                           (2u * kMaxStages + 2u * kSlots + 5u) * 8u + 16u + 1024u;
    uint32_t stages = (kMaxSmem - fixed) / p.stage_bytes;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return fail(SPCONV_ERR_UNSUPPORTED, "shared memory too small for the tile shape");
    p.stages = stages;
    uint32_t off = stages * p.stage_bytes;
    p.off_slots = off;
    off += kSlots * slot_bytes;
    p.off_bias = off;
    off += 256u * 4u;
    p.off_meta = off;
    off += (stages + kSlots) * 4u;
    off = (off + 7u) & ~7u;
    p.off_bars = off;
    off += (2u * stages + 2u * kSlots + 5u) * 8u + 16u;
    const uint32_t smem_bytes = off + 1024u;  // slack for the 1024-byte alignment

    auto kern = submconv_tc_kernel<Tr>;
    spconv_status cst = SPCONV_OK;
    if (!cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem_bytes)),
                 "cudaFuncSetAttribute", &cst))
      return cst;
    kern<<<grid, kThreads, smem_bytes, stream>>>(tm_w, p);
    if (!cuda_ok(cudaGetLastError(), "submconv_tc_kernel launch", &cst)) return cst;
  }
  return SPCONV_OK;
}

}  // namespace

spconv_status read_and_clear_device_error(cudaStream_t stream, unsigned int* bits) {
  spconv_status st = SPCONV_OK;
  if (!cuda_ok(cudaStreamSynchronize(stream), "cudaStreamSynchronize", &st)) return st;
  const unsigned int zero = 0;
  if (!cuda_ok(cudaMemcpyFromSymbol(bits, g_device_error, sizeof(unsigned int)),
               "cudaMemcpyFromSymbol", &st))
    return st;
  if (!cuda_ok(cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int)),
               "cudaMemcpyToSymbol", &st))
    return st;
  return SPCONV_OK;
}

spconv_status launch_conv_tc(spconv_dtype dtype, const void* feats, const int32_t* nmap,
                             const void* w, const void* bias, void* out, int64_t n, int32_t k,
                             int32_t ci, int32_t co, cudaStream_t stream) {
  if (dtype == SPCONV_BF16)
    return launch_typed<Bf16Traits>(feats, nmap, w, bias, out, n, k, ci, co, stream);
  if (dtype == SPCONV_TF32)
    return launch_typed<Tf32Traits>(feats, nmap, w, bias, out, n, k, ci, co, stream);
  return fail(SPCONV_ERR_UNSUPPORTED, "tensor-core path supports bf16 and tf32 only");
}

}  // namespace spconv

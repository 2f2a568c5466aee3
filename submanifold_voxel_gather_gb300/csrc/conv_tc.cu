// Fused submanifold convolution on the 5th-generation tensor cores (sm_103a).
//
// Computes out[n, co] = bias[co] + sum_k sum_ci feats[nmap[k, n], ci] * w[k, ci, co]
// (page "sparse_conv_metal.py", trellis-2-mrp-mlx: module docstring formula,
// kernel-body sentinel skip, wrapper bias).  The page's kernel runs one scalar
// thread per (n, co).  Here the per-offset products are tcgen05 MMAs in the
// transposed orientation
//
//     out^T[co, n] += w[k]^T[co, ci] * gathered_feats_k^T[ci, n]
//
// with M = 128 output channels (one or two M blocks), N = 256 voxels and K =
// 16 input channels per instruction.  A wide
// N keeps the tensor core fed: an M=128 x N=256 x K=16 bf16 MMA reads 12 KB of
// shared memory in 128 cycles, where the M=128 x N=128 shape reads 8 KB in 64.
// It also halves the weight traffic per voxel.  A persistent CTA per SM runs a
// warp-specialised pipeline:
//
//   warp 2     nmap loader: streams the neighbour indices of each (tile,
//              offset) pair into a ring of shared-memory rows (coalesced
//              reads) and flags, by warp ballot, rows with no valid entry;
//              offsets with no valid entry in the tile are skipped whole.
//   warps 8-11 gather producers: for each kept offset and each 128-byte Ci
//              chunk, copy the tile's neighbour rows with 16-byte cp.async
//              (each warp instruction moves four whole 128-byte row segments)
//              into the 128-byte-swizzled K-major operand; rows that are not
//              valid are zero-filled without a read.
//   warp 0     weight producer: loads w[k]'s chunk (channel-major, 128-byte
//              swizzle) with tiled TMA and writes the stage metadata.
//   warp 1     MMA issuer (one thread): fp32 accumulator in tensor memory,
//              double-buffered for Co <= 128 so one tile's epilogue overlaps
//              the next tile's main loop (two M blocks fill all 512 columns
//              with one buffer: measured faster than N = 128 with two, which
//              doubles the weight traffic per voxel).
//   warps 4-7  epilogue: tcgen05.ld (lane = channel, column = voxel), + bias
//              (+ residual row and activation for the fused-epilogue entry
//              point), one rounding to bf16, transpose through shared memory,
//              coalesced 16-byte stores.
//
// Pipeline stages.  With Ci a multiple of 128 and at most 128 output channels
// a stage holds both 64-channel chunks of one offset (2 x 16 KB of weights and
// 2 x 32 KB of rows; two stages fit), else one chunk.  The per-stage cost was
// measured to be near-constant, so larger stages run faster.  Where an offset
// spans several stages (Ci >= 256), each chunk of a stage is a part with its
// own full and empty barriers: the MMAs of chunk 0 start while chunk 1 is
// still landing, and chunk 0's buffers are refilled while chunk 1's MMAs run.
//
// The gathered (K, N, Ci) operand only ever exists one stage at a time in
// shared memory.  Every mbarrier wait is bounded in time; on timeout the
// kernel records an error bit, drains its own copies and MMAs, frees its
// tensor memory and returns.
//
// Row gathers use the LSU path, not TMA tile::gather4: measured on GB300, a
// 4-row gather4 costs ~80 SM cycles of TMA time, which starves the MMAs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace spconv {
namespace {

constexpr int kThreads = 384;
constexpr int kProducerWarp0 = 8;      // gather producers: warps 8-11
constexpr int kProducerThreads = 128;
constexpr int kEpilogueWarp0 = 4;      // epilogue: warps 4-7
constexpr int kRing = 16;              // neighbour-index ring rows
constexpr int kChunk = 64;             // bf16 elements per 128-byte row
constexpr int kKPerMma = 16;
constexpr uint32_t kWBlockBytes = 128 * 128;  // one M block of weights per stage (16 KB)
// Descriptor start-address steps, in 16-byte units: an M block of weights,
// one K step of the channel-major weights (16 rows x 128 B) and one K step of
// the K-major gathered rows (32 B within each 128-byte row).
constexpr uint64_t kWBlockUnits = kWBlockBytes >> 4;
constexpr uint64_t kAStepUnits = (kKPerMma * 128) >> 4;
constexpr uint64_t kBStepUnits = (kKPerMma * 2) >> 4;
constexpr int kMaxStages = 8;
constexpr int kMaxSmem = 232448;       // 227 KB opt-in limit per block
// bf16 epilogue with a residual: 16-row chunks, one 128-channel block at a
// time, staged in fp32 (8 KB) next to two 4 KB windows of residual rows.
constexpr uint32_t kResRows = 16;
constexpr uint32_t kResWindowOff = kResRows * 128u * 4u;
constexpr uint32_t kResWindowBytes = kResRows * 128u * 2u;
static_assert(kResWindowOff + 2u * kResWindowBytes <= 32u * 128u * 4u, "fits the 16 KB output staging");

enum : uint32_t { kMetaFirst = 1u, kMetaEnd = 2u };

struct TcParams {
  const void* feats;     // bf16, or fp32 for the tf32 instantiation (as are bias, residual, out)
  const int32_t* nmap;
  const void* bias;
  const void* residual;  // (N, co) or null; may alias out
  void* out;
  const int32_t* order;  // tile slot -> voxel (a permutation of 0..N-1), or null for identity
  int64_t n;
  int64_t num_tiles;
  int32_t k;
  int32_t ci;
  int32_t co;        // row stride of out
  int32_t co_base;   // first output channel of this launch
  int32_t co_count;  // channels of this launch (<= 256)
  int32_t act;       // spconv_activation
  int32_t dgrad;     // input gradient: selects the kDgrad instantiation
  int32_t tma_out;   // plain bf16 epilogue in voxel order: each 32-row block of out is written by one TMA store
  int32_t tma_res;   // bf16 epilogue with a residual: 16-row windows of the residual come by TMA (tm_out holds its map)
  int32_t num_chunks;
  int32_t cps;       // 64-channel chunks per stage: 2 when Ci % 128 == 0 and Co <= 128, else 1
  uint32_t stages;
  uint32_t stage_bytes;
  uint32_t w_bytes;  // weight bytes per stage (M blocks x 16 KB)
  uint32_t tmem_cols;
  uint32_t idesc;
  uint32_t off_ring;
  uint32_t off_stage_out;
  uint32_t off_bias;
  uint32_t off_meta;
  uint32_t off_bars;
  uint32_t off_raw;   // tf32 forward: ring of two channel-major weight chunks (TMA), transposed by warp 3
  uint32_t raw_bytes; // bytes of one raw slot (M blocks x 16 KB)
};

// Named barrier for the four epilogue warps only.
__device__ __forceinline__ void epilogue_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// AND of `v` over the four epilogue warps (a barrier, so their loop exits
// stay in step even when one of them sees a wait time out).
__device__ __forceinline__ bool epilogue_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0u;
}

// Voxel (map column, output row) of tile slot `slot`, or -1: the identity,
// or the caller's tile order.  Entries of the order outside [0, N) are
// treated as empty slots.
__device__ __forceinline__ int64_t slot_voxel(const int32_t* order, int64_t slot, int64_t n) {
  if (slot >= n) return -1;
  if (order == nullptr) return slot;
  const int32_t v = __ldg(order + slot);
  return (v >= 0 && v < n) ? v : -1;
}

// Kept offsets: every row with a valid entry, and the last offset of a tile
// none of whose rows has one (its rows are zero-filled, so the accumulator
// becomes exactly zero and the tile's output is the bias).
__device__ __forceinline__ bool issue_row(uint32_t flag, int kk, int k_count, bool issued) {
  return flag != 0u || (kk == k_count - 1 && !issued);
}

// One MMA of the stage's kind: bf16 products (kind::f16, K = 16) or tf32
// products of fp32 storage (kind::tf32, K = 8); 32 bytes of K either way.
template <bool kTf32>
__device__ __forceinline__ void umma_kind(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  if constexpr (kTf32)
    umma_tf32(d_tmem, a_desc, b_desc, idesc, accumulate);
  else
    umma_f16(d_tmem, a_desc, b_desc, idesc, accumulate);
}

// tf32 forward: the weight chunk of one stage arrives channel-major (TMA,
// 128-byte swizzle: per 32-channel box, row ci of 128 bytes holds output
// channels co, 16-byte piece j at j ^ (ci & 7)), but kind::tf32 reads its A
// operand K-major only (row co of 128 bytes holding 32 input channels,
// 16-byte piece q = ci / 4 at q ^ (co & 7)).  One warp transposes it in 4 x 4
// blocks: four 16-byte loads (ci rows 4a..4a+3, channels 4b..4b+3) and four
// 16-byte stores (co rows 4b..4b+3, channels 4a..4a+3).  Lane i of lane group
// g takes block a = i, j = (i + d) mod 8 of box beta, with (beta, d) from the
// group and the iteration: the eight lanes of each 16-byte phase then touch
// eight distinct bank groups on both sides.
template <int MBLK>
__device__ __forceinline__ void transpose_weight_chunk(const uint8_t* raw, uint8_t* a_tile, uint32_t lane) {
  const uint32_t i = lane & 7u, g = lane >> 3;
#pragma unroll
  for (uint32_t t = 0; t < 8u * MBLK; ++t) {
    const uint32_t c = t * 4u + g;             // (box, shift) pair, 0 .. 32 MBLK - 1
    const uint32_t beta = c >> 3, d = c & 7u;  // box of 32 output channels, shift
    const uint32_t a = i, j = (i + d) & 7u;
    const uint32_t b = beta * 8u + j;          // 4-channel group of the output channel
    float4 v[4];
#pragma unroll
    for (uint32_t r = 0; r < 4; ++r) {
      const uint32_t ci = 4u * a + r;
      v[r] = *reinterpret_cast<const float4*>(raw + beta * 4096u + ci * 128u + ((j ^ (ci & 7u)) << 4));
    }
    const float x[4][4] = {{v[0].x, v[1].x, v[2].x, v[3].x},
                           {v[0].y, v[1].y, v[2].y, v[3].y},
                           {v[0].z, v[1].z, v[2].z, v[3].z},
                           {v[0].w, v[1].w, v[2].w, v[3].w}};
#pragma unroll
    for (uint32_t cc = 0; cc < 4; ++cc) {
      const uint32_t co = 4u * b + cc;         // row of the K-major tile (M blocks stacked)
      *reinterpret_cast<float4*>(a_tile + co * 128u + ((a ^ (co & 7u)) << 4)) =
          make_float4(x[cc][0], x[cc][1], x[cc][2], x[cc][3]);
    }
  }
}

// kHoist: the per-row source index and byte count are computed once per
// offset instead of once per chunk (used when an offset has two or more
// 128-byte chunks; with one chunk the in-loop form is measured faster).
// kDgrad: input gradient; the weights of offset k are w[K-1-k] transposed,
// read from the forward layout as a K-major operand.
// kSplit: two-chunk stages with one full / empty barrier pair per chunk.
// kTf32: fp32 storage, tf32 products (kind::tf32), fp32 output; a 128-byte
// chunk is 32 channels, one chunk per stage; the forward's weights are
// transposed in shared memory by warp 3 (kind::tf32 reads K-major A only).
template <int TILE_N, int MBLK, bool kHoist, bool kDgrad, bool kSplit, bool kTf32>
__global__ void __launch_bounds__(kThreads, 1)
    submconv_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_out,
                       const TcParams p) {
  constexpr int kRowsPerWarp = TILE_N / 4;       // gathered rows per producer warp
  constexpr int kIdxPerLane = kRowsPerWarp / 4;  // 4 rows per warp instruction
  static_assert(kRowsPerWarp == 64, "ring layout: 64 rows per gather producer warp");
  static_assert(!kSplit || (MBLK == 1 && kHoist), "per-chunk barriers need two-chunk stages");
  static_assert(!(kSplit && kTf32), "tf32 stages hold one chunk");
  constexpr int kChunkE = kTf32 ? 32 : kChunk;           // elements per 128-byte row
  constexpr int kKPerMmaE = kTf32 ? 8 : kKPerMma;        // K per MMA instruction
  constexpr uint32_t kEsz = kTf32 ? 4u : 2u;             // element bytes
  constexpr bool kTranspose = kTf32 && !kDgrad;          // weights transposed by warp 3
  constexpr bool kKMajorA = kDgrad || kTf32;             // A operand K-major
  constexpr int kLoaderPerLane = TILE_N / 32;
  constexpr int kOutStride = MBLK * 128;         // staged output row, elements
  // Two accumulator buffers (the epilogue of one tile overlaps the next) when
  // they fit in the 512 tensor-memory columns, else one.
  constexpr uint32_t kAccBufs = (2 * MBLK * TILE_N <= 512) ? 2u : 1u;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t S = p.stages;

  int32_t* ring = reinterpret_cast<int32_t*>(smem + p.off_ring);
  __nv_bfloat16* stage_out = reinterpret_cast<__nv_bfloat16*>(smem + p.off_stage_out);
  float* bias_s = reinterpret_cast<float*>(smem + p.off_bias);
  uint32_t* meta = reinterpret_cast<uint32_t*>(smem + p.off_meta);
  uint32_t* ring_flag = meta + S;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bars);
  // One full / empty barrier pair per part of a stage.  With one part the
  // stage is filled and released whole; with one part per chunk (kSplit), a
  // chunk's weight block and row block are.
  constexpr uint32_t parts = kSplit ? 2u : 1u;
  uint64_t* full = bars;
  uint64_t* empty = bars + S * parts;
  uint64_t* ring_full = bars + 2 * S * parts;
  uint64_t* ring_empty = ring_full + kRing;
  uint64_t* tmem_full = ring_empty + kRing;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain = tmem_empty + 2;
  uint64_t* raw_full = drain + 1;    // tf32 forward: raw weight slots (two)
  uint64_t* raw_empty = raw_full + 2;
  uint64_t* res_full = raw_empty + 2;  // bf16 residual epilogue: the two windows
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(res_full + 2);
  uint32_t* consumed_holder = tmem_holder + 1;
  uint32_t* fills_holder = tmem_holder + 2;
  uint32_t* raw_consumed_holder = tmem_holder + 3;
  uint32_t* raw_meta = tmem_holder + 4;  // two words: the stage metadata of each raw slot

  if (warp == 0 && lane == 0) {
    for (uint32_t s = 0; s < S * parts; ++s) {
      mbar_init(smem_addr(&full[s]), kProducerThreads + 1);
      mbar_init(smem_addr(&empty[s]), 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(smem_addr(&ring_full[i]), 32);
      mbar_init(smem_addr(&ring_empty[i]), 32 + kProducerThreads);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&tmem_full[i]), 1);
      mbar_init(smem_addr(&tmem_empty[i]), 4);
    }
    mbar_init(smem_addr(drain), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&raw_full[i]), 1);
      mbar_init(smem_addr(&raw_empty[i]), 1);
      mbar_init(smem_addr(&res_full[i]), 1);
    }
    *consumed_holder = 0;
    *fills_holder = 0;
    *raw_consumed_holder = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    if (p.tma_out || p.tma_res) tma_prefetch_desc(&tm_out);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_holder), p.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 3) {
    for (int j = lane; j < MBLK * 128; j += 32) {
      float b = 0.0f;
      if (p.bias != nullptr && j < p.co_count) {
        if constexpr (kTf32)
          b = static_cast<const float*>(p.bias)[p.co_base + j];
        else
          b = __bfloat162float(static_cast<const __nv_bfloat16*>(p.bias)[p.co_base + j]);
      }
      bias_s[j] = b;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int64_t n_rows = p.n;
  const int k_count = p.k;

  if (warp == 2) {
    // ------------------------------------------------------ nmap loader
    // Four (tile, offset) rows per batch: their loads are in flight together.
    uint32_t e = 0, ephase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      const int64_t n0 = t * TILE_N;
      int64_t col[kLoaderPerLane];  // map column of each of this lane's slots, or -1
#pragma unroll
      for (int j = 0; j < kLoaderPerLane; ++j) col[j] = slot_voxel(p.order, n0 + lane + 32 * j, n_rows);
      for (int k0 = 0; k0 < k_count && ok; k0 += 4) {
        int32_t v[4][kLoaderPerLane];
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int j = 0; j < kLoaderPerLane; ++j) {
            v[b][j] = -1;
            if (k0 + b < k_count && col[j] >= 0)
              v[b][j] = __ldg(p.nmap + static_cast<int64_t>(k0 + b) * n_rows + col[j]);
          }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          if (k0 + b >= k_count) break;
          if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ring_empty[e]), ephase ^ 1))) {
            ok = false;
            break;
          }
          bool any = false;
#pragma unroll
          for (int j = 0; j < kLoaderPerLane; ++j) {
            // normalised: a valid index, or -1 for every kind of invalid entry
            const int32_t nv = (v[b][j] >= 0 && v[b][j] < n_rows) ? v[b][j] : -1;
            any |= nv >= 0;
            // Row r is stored where its gather lane reads it: producer warp
            // r / 64 takes rows 4 j + s (s = r % 4) as 16 consecutive words.
            const int r = static_cast<int>(lane) + 32 * j;
            ring[e * TILE_N + (r >> 6) * 64 + (r & 3) * 16 + ((r & 63) >> 2)] = nv;
          }
          const uint32_t ballot = __ballot_sync(0xffffffffu, any);
          if (lane == 0) ring_flag[e] = ballot != 0u ? 1u : 0u;
          mbar_arrive(smem_addr(&ring_full[e]));
          if (++e == kRing) {
            e = 0;
            ephase ^= 1;
          }
        }
      }
    }
  } else if (warp >= kProducerWarp0) {
    // ------------------------------------------------------ gather producers
    const uint32_t aw = warp - kProducerWarp0;
    const int sub_row = static_cast<int>(lane >> 3);
    const int chunk16 = static_cast<int>(lane & 7);
    const char* feats = reinterpret_cast<const char*>(p.feats);
    const uint32_t row_bytes = static_cast<uint32_t>(p.ci) * kEsz;
    // Row-independent part of the destination: this lane's row group and its
    // swizzled 16-byte slot (rows 4 j + sub_row alternate between two
    // swizzle phases).  The producer loop is issue-bound, so its per-row
    // work is kept to an address multiply-add and the copy itself.
    const uint32_t dst_lane = (aw * kRowsPerWarp + static_cast<uint32_t>(sub_row)) * 128u;
    const uint32_t sw_even = static_cast<uint32_t>(chunk16 ^ sub_row) << 4;
    const uint32_t sw_odd = static_cast<uint32_t>(chunk16 ^ (sub_row + 4)) << 4;
    uint32_t stage = 0, st_phase = 0, e = 0, ephase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      bool issued = false;
      for (int kk = 0; kk < k_count && ok; ++kk) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ring_full[e]), ephase))) {
          ok = false;
          break;
        }
        const bool go = issue_row(ring_flag[e], kk, k_count, issued);
        int32_t idx[kIdxPerLane];   // a valid index or -1
        uint32_t vi[kIdxPerLane];   // kHoist: index, 0 where invalid
        uint32_t valid_bits = 0;    // kHoist: bit j set where row j is valid
        if (go) {
          // this lane's 16 row indices are consecutive: four 16-byte loads
          const int4* ip =
              reinterpret_cast<const int4*>(ring + e * TILE_N + static_cast<int>(aw) * kRowsPerWarp + sub_row * 16);
#pragma unroll
          for (int q = 0; q < kIdxPerLane / 4; ++q) {
            const int4 v4 = ip[q];
            idx[4 * q] = v4.x;
            idx[4 * q + 1] = v4.y;
            idx[4 * q + 2] = v4.z;
            idx[4 * q + 3] = v4.w;
          }
#pragma unroll
          for (int j = 0; j < kIdxPerLane; ++j) {
            if constexpr (kHoist) {
              vi[j] = idx[j] >= 0 ? static_cast<uint32_t>(idx[j]) : 0u;
              valid_bits |= (idx[j] >= 0 ? 1u : 0u) << j;
            }
          }
        }
        mbar_arrive(smem_addr(&ring_empty[e]));
        if (++e == kRing) {
          e = 0;
          ephase ^= 1;
        }
        if (!go) continue;
        issued = true;
        for (int cg = 0; cg < p.num_chunks && ok; cg += p.cps) {
          if constexpr (!kSplit) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage]), st_phase ^ 1))) {
              ok = false;
              break;
            }
          }
          for (int sub = 0; sub < p.cps; ++sub) {  // the stage's chunks, one row block each
            if constexpr (kSplit) {
              if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage * 2u + sub]), st_phase ^ 1))) {
                ok = false;
                break;
              }
            }
            const int c = cg + sub;
            const uint32_t col_byte = static_cast<uint32_t>(c) * 128u + static_cast<uint32_t>(chunk16) * 16u;
            const bool col_ok = col_byte < row_bytes;
            const char* chunk_base = feats + col_byte;
            const uint32_t f_dst = smem_addr(smem + stage * p.stage_bytes) + p.w_bytes +
                                   static_cast<uint32_t>(sub) * (TILE_N * 128u) + dst_lane;
            if constexpr (kHoist) {
              const uint32_t live = col_ok ? valid_bits : 0u;
#pragma unroll
              for (int j = 0; j < kIdxPerLane; ++j)
                cp_async_16<false>(f_dst + 512u * j + ((j & 1) ? sw_odd : sw_even),
                                   chunk_base + static_cast<uint64_t>(vi[j]) * row_bytes, ((live >> j) & 1u) << 4);
            } else {
#pragma unroll
              for (int j = 0; j < kIdxPerLane; ++j) {
                const bool valid = col_ok && idx[j] >= 0;
                const uint32_t v = valid ? static_cast<uint32_t>(idx[j]) : 0u;
                cp_async_16<false>(f_dst + 512u * j + ((j & 1) ? sw_odd : sw_even),
                                   chunk_base + static_cast<uint64_t>(v) * row_bytes, valid ? 16u : 0u);
              }
            }
            if constexpr (kSplit) cp_async_arrive_noinc(smem_addr(&full[stage * 2u + sub]));
          }
          if constexpr (!kSplit) cp_async_arrive_noinc(smem_addr(&full[stage]));
          if (++stage == S) {
            stage = 0;
            st_phase ^= 1;
          }
        }
      }
    }
    // End-of-work stage: tells the MMA issuer to close the last tile.
    if (ok && __all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage * parts]), st_phase ^ 1)))
      cp_async_arrive_noinc(smem_addr(&full[stage * parts]));
    cp_async_wait_all();
  } else if (warp == 0) {
    // ------------------------------------------------------ weight producer
    uint32_t stage = 0, st_phase = 0, e = 0, ephase = 0, fills = 0;
    uint32_t rslot = 0, rphase = 0;  // tf32 forward: raw weight slot ring
    bool ok = true;
    for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      bool issued = false;
      for (int kk = 0; kk < k_count && ok; ++kk) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ring_full[e]), ephase))) {
          ok = false;
          break;
        }
        const bool go = issue_row(ring_flag[e], kk, k_count, issued);
        __syncwarp();
        mbar_arrive(smem_addr(&ring_empty[e]));
        if (++e == kRing) {
          e = 0;
          ephase ^= 1;
        }
        if (!go) continue;
        if constexpr (kTranspose) {
          // tf32 forward: each chunk's weights go to a raw slot, channel-major
          // (four 32 x 32 boxes per M block), with the stage metadata; warp 3
          // transposes them into the stage.
          for (int c = 0; c < p.num_chunks && ok; ++c) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&raw_empty[rslot]), rphase ^ 1))) {
              ok = false;
              break;
            }
            const uint32_t rfull = smem_addr(&raw_full[rslot]);
            if (lane == 0) {
              const int steps = min(kChunkE, p.ci - c * kChunkE) / kKPerMmaE;
              raw_meta[rslot] = (static_cast<uint32_t>(steps) << 8) | (issued ? 0u : kMetaFirst);
              mbar_arrive_expect_tx(rfull, p.raw_bytes);
            }
            ++fills;
            __syncwarp();
            if (static_cast<int>(lane) < 4 * MBLK) {
              const int mb = static_cast<int>(lane) >> 2, q = static_cast<int>(lane) & 3;
              tma_load_3d(smem_addr(smem + p.off_raw) + rslot * p.raw_bytes + mb * kWBlockBytes + q * 4096u,
                          &tm_w, p.co_base + mb * 128 + q * 32, c * kChunkE, kk, rfull);
            }
            issued = true;
            rslot ^= 1u;
            if (rslot == 0) rphase ^= 1u;
          }
        } else {
          for (int c = 0; c < p.num_chunks && ok; c += p.cps) {
            for (int sub = 0; sub < p.cps; ++sub) {  // the stage's chunks, one weight block each
              const uint32_t part = kSplit ? stage * 2u + static_cast<uint32_t>(sub) : stage;
              const uint32_t fullb = smem_addr(&full[part]);
              if (kSplit || sub == 0) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[part]), st_phase ^ 1))) {
                  ok = false;
                  break;
                }
                if (lane == 0) {
                  if (sub == 0) {
                    // MMAs per part
                    const int steps =
                        (p.cps / static_cast<int>(parts)) * (min(kChunkE, p.ci - c * kChunkE) / kKPerMmaE);
                    meta[stage] = (static_cast<uint32_t>(steps) << 8) | (issued ? 0u : kMetaFirst);
                  }
                  mbar_arrive_expect_tx(fullb, p.w_bytes / parts);
                }
                ++fills;
              }
              __syncwarp();
              // With two parts MBLK is 1, so the part's block is `sub`; with one
              // part, the M blocks are side by side.
              if constexpr (kTf32) {
                // tf32 input gradient: rows of w[K-1-k] (output channel =
                // forward ci) with 32 of their forward-co entries each, K-major
                if (static_cast<int>(lane) < MBLK) {
                  const int mb = static_cast<int>(lane);
                  tma_load_3d(smem_addr(smem + stage * p.stage_bytes) + mb * kWBlockBytes, &tm_w,
                              c * kChunkE, p.co_base + mb * 128, k_count - 1 - kk, fullb);
                }
              } else if constexpr (!kDgrad) {
                // forward: w[k] channel-major, two 64-channel boxes per M block
                if (static_cast<int>(lane) < 2 * MBLK) {
                  const int mb = static_cast<int>(lane) >> 1, half = static_cast<int>(lane) & 1;
                  tma_load_3d(smem_addr(smem + stage * p.stage_bytes) + (sub + mb) * kWBlockBytes + half * 8192u,
                              &tm_w, p.co_base + mb * 128 + half * 64, (c + sub) * kChunk, kk, fullb);
                }
              } else if (static_cast<int>(lane) < MBLK) {
                // input gradient: rows of w[K-1-k] (output channel = forward ci)
                // with 64 of their forward-co entries each, K-major
                const int mb = static_cast<int>(lane);
                tma_load_3d(smem_addr(smem + stage * p.stage_bytes) + (sub + mb) * kWBlockBytes, &tm_w,
                            (c + sub) * kChunk, p.co_base + mb * 128, k_count - 1 - kk, fullb);
              }
            }
            issued = true;
            if (++stage == S) {
              stage = 0;
              st_phase ^= 1;
            }
          }
        }
      }
    }
    if constexpr (kTranspose) {
      // end-of-work marker through the raw ring (no bytes)
      if (ok && __all_sync(0xffffffffu, mbar_wait(smem_addr(&raw_empty[rslot]), rphase ^ 1))) {
        if (lane == 0) {
          raw_meta[rslot] = kMetaEnd;
          mbar_arrive(smem_addr(&raw_full[rslot]));
        }
        ++fills;
      }
    } else if (ok && __all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage * parts]), st_phase ^ 1))) {
      if (lane == 0) {
        meta[stage] = kMetaEnd;
        mbar_arrive(smem_addr(&full[stage * parts]));
      }
      ++fills;
    }
    if (lane == 0) *fills_holder = fills;
  } else if (warp == 3 && kTranspose) {
    // ------------------------------------------------------ weight transposer (tf32 forward)
    uint32_t stage = 0, st_phase = 0, rslot = 0, rphase = 0, consumed = 0;
    const uint8_t* raw_base = smem + p.off_raw;
    while (true) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&raw_full[rslot]), rphase))) break;
      const uint32_t m = raw_meta[rslot];
      if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage]), st_phase ^ 1))) break;
      if ((m & kMetaEnd) == 0u) {
        transpose_weight_chunk<MBLK>(raw_base + rslot * p.raw_bytes, smem + stage * p.stage_bytes, lane);
        // the MMA reads the tile through the async proxy
        fence_proxy_async_smem();
      }
      __syncwarp();
      ++consumed;
      if (lane == 0) {
        meta[stage] = m;
        mbar_arrive(smem_addr(&raw_empty[rslot]));
        mbar_arrive(smem_addr(&full[stage]));
      }
      if ((m & kMetaEnd) != 0u) break;
      rslot ^= 1u;
      if (rslot == 0) rphase ^= 1u;
      if (++stage == S) {
        stage = 0;
        st_phase ^= 1;
      }
    }
    if (lane == 0) *raw_consumed_holder = consumed;
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Descriptors of stage 0; a stage or K step only moves the start
      // address (the low 14 bits, in 16-byte units), so advancing is one add.
      // Weights channel-major (bf16 forward) or K-major (input gradient, and
      // the tf32 forward after the transposer).
      const uint64_t adesc0 = sw128_desc(smem_addr(smem), kKMajorA ? 16u : 8192u, 1024u);
      constexpr uint64_t a_step = kKMajorA ? kBStepUnits : kAStepUnits;
      const uint64_t bdesc0 = sw128_desc(smem_addr(smem) + p.w_bytes, 16u, 1024u);
      const uint64_t stage_units = p.stage_bytes >> 4;
      const uint32_t idesc = p.idesc;
      uint32_t stage = 0, st_phase = 0, consumed = 0, tile_i = 0, buf = 0;
      uint32_t d_tmem = tmem_base;
      bool open = false;
      while (true) {
        if (!mbar_wait(smem_addr(&full[stage * parts]), st_phase)) break;
        // The gathered rows were written by cp.async (generic proxy); the MMA
        // reads them through the async proxy.
        fence_proxy_async_smem();
        tc_fence_after();
        const uint32_t m = meta[stage];
        if ((m & (kMetaFirst | kMetaEnd)) != 0u && open) {
          umma_commit(smem_addr(&tmem_full[buf]));
          ++tile_i;
          open = false;
        }
        if ((m & kMetaEnd) != 0u) {
          ++consumed;
          break;
        }
        if ((m & kMetaFirst) != 0u) {
          buf = tile_i % kAccBufs;
          if (!mbar_wait(smem_addr(&tmem_empty[buf]), ((tile_i / kAccBufs) & 1u) ^ 1u)) break;
          tc_fence_after();
          d_tmem = tmem_base + buf * static_cast<uint32_t>(MBLK * TILE_N);
          open = true;
        }
        const int steps = static_cast<int>((m >> 8) & 0xFFu);
        const uint64_t ad = adesc0 + stage * stage_units;
        const uint64_t bd = bdesc0 + stage * stage_units;
        const uint32_t acc0 = (m & kMetaFirst) == 0u ? 1u : 0u;
        if constexpr (kSplit) {
          // two chunks (MBLK == 1), each its own part: chunk 1's weight
          // block and row block follow those of chunk 0
#pragma unroll
          for (int s = 0; s < kChunkE / kKPerMmaE; ++s)
            umma_kind<kTf32>(d_tmem, ad + s * a_step, bd + s * kBStepUnits, idesc, s > 0 ? 1u : acc0);
          umma_commit(smem_addr(&empty[stage * 2u]));
          ++consumed;
          if (!mbar_wait(smem_addr(&full[stage * 2u + 1u]), st_phase)) break;
          fence_proxy_async_smem();
          tc_fence_after();
#pragma unroll
          for (int s = 0; s < kChunkE / kKPerMmaE; ++s)
            umma_kind<kTf32>(d_tmem, ad + kWBlockUnits + s * a_step, bd + ((TILE_N * 128u) >> 4) + s * kBStepUnits, idesc,
                     1u);
          umma_commit(smem_addr(&empty[stage * 2u + 1u]));
          ++consumed;
        } else {
          if (steps == 2 * kChunkE / kKPerMmaE) {
            // two chunks in one part (MBLK == 1): chunk 1's weight block and
            // row block follow those of chunk 0
#pragma unroll
            for (int s = 0; s < 2 * kChunkE / kKPerMmaE; ++s) {
              const int sub = s >> 2, ss = s & 3;
              umma_kind<kTf32>(d_tmem, ad + sub * kWBlockUnits + ss * a_step,
                       bd + sub * ((TILE_N * 128u) >> 4) + ss * kBStepUnits, idesc, s > 0 ? 1u : acc0);
            }
          } else if (steps == kChunkE / kKPerMmaE) {
#pragma unroll
            for (int s = 0; s < kChunkE / kKPerMmaE; ++s)
#pragma unroll
              for (int mb = 0; mb < MBLK; ++mb)
                umma_kind<kTf32>(d_tmem + mb * TILE_N, ad + mb * kWBlockUnits + s * a_step,
                         bd + s * kBStepUnits, idesc, s > 0 ? 1u : acc0);
          } else {
            for (int s = 0; s < steps; ++s)
#pragma unroll
              for (int mb = 0; mb < MBLK; ++mb)
                umma_kind<kTf32>(d_tmem + mb * TILE_N, ad + mb * kWBlockUnits + s * a_step,
                         bd + s * kBStepUnits, idesc, s > 0 ? 1u : acc0);
          }
          umma_commit(smem_addr(&empty[stage]));
          ++consumed;
        }
        if (++stage == S) {
          stage = 0;
          st_phase ^= 1;
        }
      }
      *consumed_holder = consumed;
      umma_commit(smem_addr(drain));
      mbar_wait(smem_addr(drain), 0);
    }
    __syncwarp();
  } else if (warp >= kEpilogueWarp0) {
    // ------------------------------------------------------ epilogue
    const uint32_t sub = warp & 3u;
    const int et = static_cast<int>(threadIdx.x) - kEpilogueWarp0 * 32;  // 0..127
    const int chunks_per_row = p.co_count / 8;                           // 16-byte chunks
    const bool fused = p.residual != nullptr || p.act != SPCONV_ACT_NONE;
    // bf16 with a residual (the tiles' rows are consecutive voxels, no
    // order): 16-row chunks, one 128-channel block at a time.  The channel
    // phase stages acc + bias in fp32; TMA brings the block's 16 residual
    // rows into one of two windows (window u & 1 for step u = chunk * MBLK +
    // block, step u + 1's loading while step u is stored); the store phase
    // adds them per 16-byte piece, applies the activation and rounds once.
    // Without a residual the activation is applied before the bf16 staging
    // of the plain paths.  Each (row, piece) is read and then written by the
    // same thread, so the residual may be the output.
    float* stage_f = reinterpret_cast<float*>(stage_out);
    __nv_bfloat16* out_bf = static_cast<__nv_bfloat16*>(p.out);
    const uint32_t stage_base = smem_addr(stage_out);
    auto issue_window = [&](int64_t n0, int u) {
      const int c = u / MBLK, mb = u - (u / MBLK) * MBLK;
      const uint32_t bar = smem_addr(&res_full[u & 1]);
      fence_proxy_async_smem();  // the window's previous contents were read through the generic proxy
      const int64_t row = n0 + static_cast<int64_t>(c) * kResRows;
      if (row >= n_rows) {
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, kResWindowBytes);
        tma_load_2d(stage_base + kResWindowOff + static_cast<uint32_t>(u & 1) * kResWindowBytes, &tm_out,
                    p.co_base + mb * 128, static_cast<int32_t>(row), bar);
      }
    };
    // This thread's 16-byte output pieces of a 16-row block of M block mb:
    // (row, 8-channel column), the same in every step, computed once.
    int prow[MBLK][2], pcol[MBLK][2], npieces[MBLK];
#pragma unroll
    for (int mb = 0; mb < MBLK; ++mb) {
      const int ppr = max(0, min(128, p.co_count - mb * 128) / 8);
      npieces[mb] = static_cast<int>(kResRows) * ppr;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int q = et + 128 * j;
        prow[mb][j] = ppr > 0 ? q / ppr : 0;
        pcol[mb][j] = (q - prow[mb][j] * ppr) * 8;
      }
    }
    uint32_t res_phase = 0;    // bit w: the phase window w's barrier waits for next
    uint32_t res_pending = 0;  // window loads issued and not yet waited for (bits)
    bool ok_res = true;
    uint32_t tile_i = 0;
    for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++tile_i) {
      const uint32_t buf = tile_i % kAccBufs;
      const bool got = __all_sync(0xffffffffu, mbar_wait(smem_addr(&tmem_full[buf]), (tile_i / kAccBufs) & 1u));
      if (!epilogue_all(got)) break;
      tc_fence_after();
      const int64_t n0 = t * TILE_N;
      const uint32_t tcol = tmem_base + ((sub * 32u) << 16) + buf * static_cast<uint32_t>(MBLK * TILE_N);
      if constexpr (kTf32) {
        // fp32 output: one 128-channel block at a time staged in fp32 (32
        // rows x 128), then stored as 16-byte pieces (4 channels) of the
        // rows; the fused epilogue adds the residual piece and applies the
        // activation before the store.  Each thread reads and writes the same
        // (row, piece) pairs, so the residual may be the output.
        const float* residual_f = static_cast<const float*>(p.residual);
        float* out_f = static_cast<float*>(p.out);
        for (int vc = 0; vc < TILE_N / 32; ++vc) {
#pragma unroll
          for (int mb = 0; mb < MBLK; ++mb) {
            const int ppr = min(128, p.co_count - mb * 128) / 4;
            const int co_s = static_cast<int>(sub) * 32 + static_cast<int>(lane);
            epilogue_bar();  // the staging buffer is free
            uint32_t v[32];
            tmem_ld_32x32b_x32(tcol + mb * TILE_N + vc * 32, v);
            tmem_ld_wait();
            const float b = bias_s[mb * 128 + co_s];  // zero beyond co_count
#pragma unroll
            for (int i = 0; i < 32; ++i) stage_f[i * 128 + co_s] = __uint_as_float(v[i]) + b;
            epilogue_bar();
            for (int q = et; q < 32 * ppr; q += 128) {
              const int r = q / ppr;
              const int c4 = q - r * ppr;
              const int64_t row = slot_voxel(p.order, n0 + vc * 32 + r, n_rows);
              if (row < 0) continue;
              float4 a = *reinterpret_cast<const float4*>(stage_f + r * 128 + c4 * 4);
              const int64_t o = row * p.co + p.co_base + mb * 128 + c4 * 4;
              if (fused) {
                if (residual_f != nullptr) {
                  const float4 rr = __ldg(reinterpret_cast<const float4*>(residual_f + o));
                  a.x += rr.x;
                  a.y += rr.y;
                  a.z += rr.z;
                  a.w += rr.w;
                }
                a.x = apply_activation(a.x, p.act);
                a.y = apply_activation(a.y, p.act);
                a.z = apply_activation(a.z, p.act);
                a.w = apply_activation(a.w, p.act);
              }
              *reinterpret_cast<float4*>(out_f + o) = a;
            }
          }
        }
      } else if (p.tma_out) {
        // The staged block (32 rows x MBLK * 128 channels, the rows of out
        // in voxel order) goes out as one TMA store: the thread stores would
        // queue on the load/store pipe behind the gathers (measured: with
        // two M blocks and one accumulator buffer the MMAs waited 41% of the
        // time for the epilogue).  Rows past N and channels past Co fall
        // outside the tensor and are not written.
        for (int vc = 0; vc < TILE_N / 32; ++vc) {
          if (et == 0) bulk_wait_read_all();  // the previous block's store has read the buffer
          epilogue_bar();
#pragma unroll
          for (int mb = 0; mb < MBLK; ++mb) {
            const int co_l = mb * 128 + static_cast<int>(sub) * 32 + static_cast<int>(lane);
            uint32_t v[32];
            tmem_ld_32x32b_x32(tcol + mb * TILE_N + vc * 32, v);
            tmem_ld_wait();
            if (co_l < p.co_count) {
              const float b = bias_s[co_l];
              if (p.act == SPCONV_ACT_NONE) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  stage_out[i * kOutStride + co_l] = __float2bfloat16_rn(__uint_as_float(v[i]) + b);
              } else {
                with_activation(p.act, [&](auto tag) {
                  constexpr int kA = decltype(tag)::value;
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    stage_out[i * kOutStride + co_l] =
                        __float2bfloat16_rn(activation_bf16<kA>(__uint_as_float(v[i]) + b));
                });
              }
            }
          }
          fence_proxy_async_smem();  // the store reads the block through the async proxy
          epilogue_bar();
          if (et == 0 && n0 + vc * 32 < n_rows) {
            tma_store_2d(&tm_out, smem_addr(stage_out), p.co_base, static_cast<int32_t>(n0 + vc * 32));
            bulk_commit_group();
          }
        }
      } else if (p.residual == nullptr) {
        for (int vc = 0; vc < TILE_N / 32; ++vc) {
          epilogue_bar();  // the previous chunk's staged rows have been stored
#pragma unroll
          for (int mb = 0; mb < MBLK; ++mb) {
            const int co_l = mb * 128 + static_cast<int>(sub) * 32 + static_cast<int>(lane);
            uint32_t v[32];
            tmem_ld_32x32b_x32(tcol + mb * TILE_N + vc * 32, v);
            tmem_ld_wait();
            if (co_l < p.co_count) {
              const float b = bias_s[co_l];
              if (p.act == SPCONV_ACT_NONE) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  stage_out[i * kOutStride + co_l] = __float2bfloat16_rn(__uint_as_float(v[i]) + b);
              } else {
                with_activation(p.act, [&](auto tag) {
                  constexpr int kA = decltype(tag)::value;
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    stage_out[i * kOutStride + co_l] =
                        __float2bfloat16_rn(activation_bf16<kA>(__uint_as_float(v[i]) + b));
                });
              }
            }
          }
          epilogue_bar();
          for (int q = et; q < 32 * chunks_per_row; q += 128) {
            const int r = q / chunks_per_row;
            const int c8 = q - r * chunks_per_row;
            const int64_t n = slot_voxel(p.order, n0 + vc * 32 + r, n_rows);
            if (n >= 0)
              *reinterpret_cast<uint4*>(out_bf + n * p.co + p.co_base + c8 * 8) =
                  *reinterpret_cast<const uint4*>(stage_out + r * kOutStride + c8 * 8);
          }
        }
      } else {
        // residual epilogue (bf16); window 0 is free (step nu - 2 of the
        // previous tile was stored before its step nu - 1 began)
        constexpr int nu = static_cast<int>(TILE_N / kResRows) * MBLK;
        if (et == 0) issue_window(n0, 0);
        res_pending |= 1u;
        for (int u = 0; u < nu; ++u) {
          const int c = u / MBLK, mb = u - (u / MBLK) * MBLK;
          epilogue_bar();  // step u - 1 is stored: its window and the staging are free
          if (u + 1 < nu) {
            if (et == 0) issue_window(n0, u + 1);
            res_pending |= 1u << ((u + 1) & 1);
          }
          const int co_s = static_cast<int>(sub) * 32 + static_cast<int>(lane);
          uint32_t v[16];
          tmem_ld_32x32b_x16(tcol + mb * TILE_N + c * kResRows, v);
          tmem_ld_wait();
          const float b = bias_s[mb * 128 + co_s];  // zero beyond co_count
#pragma unroll
          for (int i = 0; i < static_cast<int>(kResRows); ++i) stage_f[i * 128 + co_s] = __uint_as_float(v[i]) + b;
          const uint32_t w = static_cast<uint32_t>(u & 1);
          ok_res = __all_sync(0xffffffffu, mbar_wait(smem_addr(&res_full[w]), (res_phase >> w) & 1u)) && ok_res;
          res_phase ^= 1u << w;
          res_pending &= ~(1u << w);
          epilogue_bar();  // staged, and every thread saw the window land
          const __nv_bfloat16* win =
              reinterpret_cast<const __nv_bfloat16*>(smem + p.off_stage_out + kResWindowOff + w * kResWindowBytes);
          with_activation(p.act, [&](auto tag) {
            constexpr int kA = decltype(tag)::value;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              // (selects, not an index by the run-time block: registers)
              if (et + 128 * j >= (mb == 0 ? npieces[0] : npieces[MBLK - 1])) break;
              const int r = mb == 0 ? prow[0][j] : prow[MBLK - 1][j];
              const int col = mb == 0 ? pcol[0][j] : pcol[MBLK - 1][j];
              const int64_t row = n0 + c * static_cast<int>(kResRows) + r;
              if (row >= n_rows) continue;
              const uint4 rr = *reinterpret_cast<const uint4*>(win + r * 128 + col);
              const float4 a0 = *reinterpret_cast<const float4*>(stage_f + r * 128 + col);
              const float4 a1 = *reinterpret_cast<const float4*>(stage_f + r * 128 + col + 4);
              const float x[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
              const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
              uint32_t o[4];
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const float lo = activation_bf16<kA>(x[2 * h] + __uint_as_float(rw[h] << 16));
                const float hi = activation_bf16<kA>(x[2 * h + 1] + __uint_as_float(rw[h] & 0xFFFF0000u));
                const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
                o[h] = *reinterpret_cast<const uint32_t*>(&pr);
              }
              *reinterpret_cast<uint4*>(out_bf + row * p.co + p.co_base + mb * 128 + col) =
                  make_uint4(o[0], o[1], o[2], o[3]);
            }
          });
        }
        if (!epilogue_all(ok_res)) break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tmem_empty[buf]));
    }
    // Only after a timed-out wait can a window load still be in flight:
    // wait for it (bounded) before the CTA's memory goes away.
    for (int w2 = 0; w2 < 2; ++w2)
      if (res_pending & (1u << w2)) mbar_wait(smem_addr(&res_full[w2]), (res_phase >> w2) & 1u);
    if (p.tma_out && et == 0) bulk_wait_all();  // the last stores are complete
  }

  // ---------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // Weight loads issued but never consumed exist only after a timed-out
    // wait: wait (bounded) for them to land before the CTA's memory goes away.
    const uint32_t fills = *fills_holder;
    if constexpr (kTranspose) {
      for (uint32_t i = *raw_consumed_holder; i < fills; ++i)
        mbar_wait(smem_addr(&raw_full[i & 1u]), (i >> 1) & 1u);
    } else {
      const uint32_t np = S * (kSplit ? 2u : 1u);
      for (uint32_t i = *consumed_holder; i < fills; ++i)
        mbar_wait(smem_addr(&full[i % np]), (i / np) & 1u);
    }
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
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                                       cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  if (fn == nullptr) *st = fail(SPCONV_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  return fn;
}

template <int TILE_N, int MBLK, bool kHoist, bool kDgrad, bool kSplit, bool kTf32>
spconv_status launch_shape(const CUtensorMap& tm_w, const CUtensorMap& tm_out, TcParams p, cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return fail(SPCONV_ERR_CUDA, "could not query the SM count");
  p.num_tiles = (p.n + TILE_N - 1) / TILE_N;
  const int grid = static_cast<int>(p.num_tiles < sms ? p.num_tiles : sms);
  p.w_bytes = p.cps * MBLK * kWBlockBytes;
  p.stage_bytes = p.w_bytes + p.cps * TILE_N * 128u;
  p.tmem_cols = 512u;  // kAccBufs accumulator buffers of MBLK x TILE_N columns
  // D f32; A and B bf16 (format 1) or tf32 (format 2); B (gathered rows)
  // K-major; A (weights) channel-major for the bf16 forward pass, K-major for
  // the input gradient and for the tf32 forward (transposed in the kernel).
  constexpr bool kTranspose = kTf32 && !kDgrad;
  const uint32_t a_mn_major = (kDgrad || kTf32) ? 0u : 1u;
  const uint32_t fmt = kTf32 ? 2u : 1u;
  p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn_major << 15) |
            ((static_cast<uint32_t>(TILE_N) >> 3) << 17) | ((128u >> 4) << 24);
  p.raw_bytes = kTranspose ? MBLK * kWBlockBytes : 0u;

  const uint32_t ring_bytes = kRing * TILE_N * 4u;
  // 32 staged output rows: bf16 for all channels, or fp32 for one 128-channel
  // block (fused epilogue); the larger of the two.
  const uint32_t stage_out_bytes = (32u * MBLK * 128u * 2u > 32u * 128u * 4u) ? 32u * MBLK * 128u * 2u
                                                                              : 32u * 128u * 4u;
  const uint32_t fixed = 2u * p.raw_bytes + ring_bytes + stage_out_bytes + 256u * 4u +
                         (kMaxStages + kRing) * 4u + (2u * kMaxStages + 2u * kRing + 11u) * 8u + 32u + 1024u;
  uint32_t stages = (kMaxSmem - fixed) / p.stage_bytes;
  constexpr uint32_t parts = kSplit ? 2u : 1u;
  if (stages * parts > kMaxStages) stages = kMaxStages / parts;
  if (stages < 2) return fail(SPCONV_ERR_UNSUPPORTED, "shared memory too small for the tile shape");
  p.stages = stages;
  uint32_t off = stages * p.stage_bytes;
  p.off_raw = off;  // 1024-aligned (stage sizes are multiples of 1 KB)
  off += 2u * p.raw_bytes;
  p.off_ring = off;
  off += ring_bytes;
  p.off_stage_out = off;
  off += stage_out_bytes;
  p.off_bias = off;
  off += 256u * 4u;
  p.off_meta = off;
  off += (stages + kRing) * 4u;
  off = (off + 7u) & ~7u;
  p.off_bars = off;
  off += (2u * stages * parts + 2u * kRing + 11u) * 8u + 32u;
  const uint32_t smem_bytes = off + 1024u;  // slack for the 1024-byte alignment

  auto kern = submconv_tc_kernel<TILE_N, MBLK, kHoist, kDgrad, kSplit, kTf32>;
  spconv_status st = SPCONV_OK;
  if (!cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem_bytes)),
               "cudaFuncSetAttribute", &st))
    return st;
  kern<<<grid, kThreads, smem_bytes, stream>>>(tm_w, tm_out, p);
  if (!cuda_ok(cudaGetLastError(), "submconv_tc_kernel launch", &st)) return st;
  return SPCONV_OK;
}

template <int MBLK, bool kHoist, bool kSplit, bool kTf32 = false>
spconv_status launch_dir(const CUtensorMap& tm_w, const CUtensorMap& tm_out, const TcParams& p,
                         cudaStream_t stream) {
  return p.dgrad != 0 ? launch_shape<256, MBLK, kHoist, true, kSplit, kTf32>(tm_w, tm_out, p, stream)
                      : launch_shape<256, MBLK, kHoist, false, kSplit, kTf32>(tm_w, tm_out, p, stream);
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
                             const void* w, const void* bias, const void* residual, void* out,
                             int64_t n, int32_t k, int32_t ci, int32_t co, spconv_activation act,
                             bool dgrad, cudaStream_t stream, const int32_t* order) {
  if (dtype != SPCONV_BF16 && dtype != SPCONV_TF32)
    return fail(SPCONV_ERR_UNSUPPORTED, "tensor-core path supports bf16 and tf32 only");
  const bool tf32 = dtype == SPCONV_TF32;
  const uint32_t esz = tf32 ? 4u : 2u;
  const int chunk = tf32 ? 32 : kChunk;  // channels per 128-byte row
  spconv_status st = SPCONV_OK;
  EncodeTiledFn encode = encode_fn(&st);
  if (encode == nullptr) return st;

  // w viewed as its (K, Ci_fwd, Co_fwd) layout, innermost Co_fwd; boxes are
  // 128 bytes wide (64 bf16 or 32 fp32 elements), 128-byte swizzle.  bf16
  // forward: box = 64 output channels x 64 input channels of one offset (the
  // channel-major UMMA operand).  tf32 forward: 32 x 32 boxes, transposed in
  // the kernel.  Input gradient (ci = Co_fwd, co = Ci_fwd): box = one row
  // width of forward-co x 128 forward-ci, i.e. 128 output rows with 64 (32)
  // input channels each (the K-major operand).
  const cuuint64_t wi = static_cast<cuuint64_t>(dgrad ? co : ci);  // forward Ci
  const cuuint64_t wo = static_cast<cuuint64_t>(dgrad ? ci : co);  // forward Co
  CUtensorMap tm_w;
  cuuint64_t dims[3] = {wo, wi, static_cast<cuuint64_t>(k)};
  cuuint64_t strides[2] = {wo * esz, wi * wo * esz};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(chunk), dgrad ? 128u : static_cast<cuuint32_t>(chunk), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(&tm_w, tf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                      const_cast<void*>(w), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(SPCONV_ERR_CUDA, "cuTensorMapEncodeTiled(w) failed: " + std::to_string(r));

  // Output channels per launch: up to 256 (two M blocks sharing each
  // gathered stage).  With a residual, 128: the residual epilogue of two M
  // blocks, which cannot overlap the next tile's MMAs (one accumulator
  // buffer), cost more than gathering the rows twice (measured, 64 -> 256
  // channels, 1.92 M voxels: 1.85 ms against 2.23; without a residual the
  // 256-channel launch stays faster, 1.18 ms against 1.70).
  const int32_t co_step = (residual != nullptr && !tf32) ? 128 : 256;
  for (int32_t co_base = 0; co_base < co; co_base += co_step) {
    TcParams p{};
    p.feats = feats;
    p.nmap = nmap;
    p.bias = bias;
    p.residual = residual;
    p.act = static_cast<int32_t>(act);
    p.dgrad = dgrad ? 1 : 0;
    p.out = out;
    p.order = order;
    p.n = n;
    p.k = k;
    p.ci = ci;
    p.co = co;
    p.co_base = co_base;
    p.co_count = (co - co_base) < co_step ? (co - co_base) : co_step;
    p.num_chunks = (ci + chunk - 1) / chunk;
    // Two 64-channel chunks per stage where they fit (two 96 KB stages):
    // a stage's cost is mostly fixed, so fewer, larger stages are faster
    // (measured: decoder 8.3 -> 7.7 ms, medium 0.72 -> 0.64 ms).
    p.cps = (ci % (2 * kChunk) == 0 && p.co_count <= 128) ? 2 : 1;
    // Per-chunk barriers where an offset spans two or more stages (measured:
    // Ci = 256, Co = 128 2.27 -> 2.05 ms; with Ci = 128 they cost 1-4%).
    const bool split = p.cps == 2 && p.num_chunks > 2;
    const bool hoist = p.num_chunks >= 2;
    // Output by TMA stores (plain bf16 epilogue, voxel order): out viewed as
    // a (N, Co) tensor, boxes of 32 rows x one launch's M blocks of channels.
    CUtensorMap tm_out;
    std::memset(&tm_out, 0, sizeof tm_out);
    p.tma_out = 0;
    p.tma_res = 0;
    if (!tf32 && order == nullptr && residual == nullptr) {
      const cuuint32_t box_co = p.co_count <= 128 ? 128u : 256u;
      cuuint64_t odims[2] = {static_cast<cuuint64_t>(co), static_cast<cuuint64_t>(n)};
      cuuint64_t ostrides[1] = {static_cast<cuuint64_t>(co) * 2u};
      cuuint32_t obox[2] = {box_co, 32u};
      cuuint32_t oestr[2] = {1, 1};
      CUresult ro = encode(&tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, odims, ostrides, obox, oestr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (ro != CUDA_SUCCESS)
        return fail(SPCONV_ERR_CUDA, "cuTensorMapEncodeTiled(out) failed: " + std::to_string(ro));
      p.tma_out = 1;
    } else if (!tf32 && order == nullptr && residual != nullptr) {
      // The residual (N, Co) by 16-row windows of 128 channels (channels
      // past Co and rows past N read as zero).
      cuuint64_t rdims[2] = {static_cast<cuuint64_t>(co), static_cast<cuuint64_t>(n)};
      cuuint64_t rstrides[1] = {static_cast<cuuint64_t>(co) * 2u};
      cuuint32_t rbox[2] = {128u, kResRows};
      cuuint32_t restr[2] = {1, 1};
      CUresult rr = encode(&tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(residual), rdims,
                           rstrides, rbox, restr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (rr != CUDA_SUCCESS)
        return fail(SPCONV_ERR_CUDA, "cuTensorMapEncodeTiled(residual) failed: " + std::to_string(rr));
      p.tma_res = 1;
    }
    if (tf32) {
      // one 32-channel chunk per stage (48 KB, or 64 KB with two M blocks)
      p.cps = 1;
      if (p.co_count <= 128)
        st = hoist ? launch_dir<1, true, false, true>(tm_w, tm_out, p, stream)
                   : launch_dir<1, false, false, true>(tm_w, tm_out, p, stream);
      else
        st = hoist ? launch_dir<2, true, false, true>(tm_w, tm_out, p, stream)
                   : launch_dir<2, false, false, true>(tm_w, tm_out, p, stream);
    } else if (split)
      st = launch_dir<1, true, true>(tm_w, tm_out, p, stream);
    else if (p.co_count <= 128)
      st = hoist ? launch_dir<1, true, false>(tm_w, tm_out, p, stream) : launch_dir<1, false, false>(tm_w, tm_out, p, stream);
    else
      st = hoist ? launch_dir<2, true, false>(tm_w, tm_out, p, stream) : launch_dir<2, false, false>(tm_w, tm_out, p, stream);
    if (st != SPCONV_OK) return st;
  }
  return SPCONV_OK;
}

}  // namespace spconv

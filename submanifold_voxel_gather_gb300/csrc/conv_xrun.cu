// Row-shifted submanifold convolution over an x-run slot layout (xrun.cu).
//
// Computes the same sum as conv_tc.cu,
//
//     out[n, co] = bias[co] + sum_k sum_ci feats[nmap[k, n], ci] * w[k, ci, co]
//
// (page "sparse_conv_metal.py", trellis-2-mrp-mlx: module docstring formula,
// kernel-body sentinel skip, wrapper bias), for the lexicographic 3x3x3
// offsets, Ci = 128 and Co <= 128, in bf16 with fp32 accumulation.
//
// Tiles are 256 consecutive slots of the layout.  For each (dz, dy) group
// of offsets a tile gathers one operand G of 258 rows: the group's neighbour
// row of every slot from one before the tile to one after it (a voxel slot
// reads nmap[(dz, dy, 0), n]; a separator reads the cell just outside its
// run, nmap[(dz, dy, +-1), n]).  The three offsets (dz, dy, dx) of the group
// are then MMAs on G started 0, 1 or 2 rows in: slot s + dx always stands for
// the cell x + dx of slot s's line.  So a tile gathers 9 x 258 rows instead
// of 27 x 256, and the MMAs run on the same shared-memory rows three times.
// Separator slots cost MMA work, and their outputs are dropped.
//
// Warp roles as in conv_tc.cu (persistent CTA per SM, 384 threads):
//   warp 2     loader: per (tile, group) the 258 gathered row indices into a
//              shared-memory ring, with a ballot flag when any is valid
//              (groups with none are skipped);
//   warps 8-11 gather producers: cp.async of G's rows (two 64-channel chunks,
//              K-major, 128-byte swizzle) into two G stages;
//   warp 0     weight producer: w[k]'s chunks by tiled TMA into a ring of
//              four 16 KB slots, with the per-slot metadata;
//   warp 1     MMA issuer: per kept group, 3 offsets x 2 chunks x 4 MMAs of
//              M = 128 channels, N = 256 slots, K = 16, fp32 in tensor memory
//              (two accumulator buffers);
//   warps 4-7  epilogue: + bias (and, fused, + residual and ReLU/SiLU), one
//              rounding to bf16, rows of voxel slots stored, separator rows
//              dropped.
// Every mbarrier wait is bounded; on timeout the kernel records an error bit,
// drains its own loads and MMAs, frees its tensor memory and returns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace spconv {
namespace {

constexpr int kThreads = 384;
constexpr int kTileN = 256;                   // slots per tile (MMA N)
constexpr int kGRows = kTileN + 2;            // gathered rows: one halo row each side
constexpr int kGRowsAlloc = 264;              // rounded up to whole 8-row swizzle atoms
constexpr int kGroups = 9;                    // (dz, dy) groups of the 3x3x3 offsets
constexpr int kChunks = 2;                    // 64-channel chunks of Ci = 128
constexpr uint32_t kGChunkBytes = kGRowsAlloc * 128u;           // 33,792 B (33 x 1024)
// The G memory is a ring of kGBufs chunk buffers (one 64-channel chunk of a
// group's rows each), filled and released chunk by chunk: a buffer is
// refilled once the 12 MMAs (3 offsets x 4) that read it are done, not the
// group's 24 (measured: with two whole-group stages the fill of group g + 2
// waited for all of group g's MMAs).
constexpr int kGBufs = 4;
constexpr uint32_t kWSlotBytes = 128u * 128u;                   // one offset's chunk: 16 KB
constexpr int kWSlots = 4;
constexpr int kXRing = 8;                     // loader ring rows
constexpr int kRingRow = kGRowsAlloc;         // int32 entries per ring row
constexpr int kProducerWarp0 = 8;
constexpr int kProducerThreads = 128;
constexpr int kEpilogueWarp0 = 4;
// Epilogue staging, 16 KB.  The plain epilogue stages 32-slot chunks of
// bf16 output rows (8 KB).  With a residual the chunks are 16 slots: their
// acc + bias rows in fp32 (8 KB), and two 4 KB windows of 16 residual rows
// each, loaded by TMA, chunk c into window c & 1 while chunk c - 1 is
// stored from the other.
constexpr uint32_t kStageBytes = 16384u;
constexpr uint32_t kResChunk = 16;                             // slots per fused chunk
constexpr uint32_t kWindowBytes = kResChunk * 128u * 2u;        // 4 KB
constexpr uint32_t kWindowOff = kResChunk * 128u * 4u;          // after the fp32 rows
static_assert(kWindowOff + 2u * kWindowBytes <= kStageBytes, "the fused staging must fit the 16 KB");
constexpr uint32_t kRowOffNone = 0xffu;  // slot without a voxel
constexpr uint32_t kRowOffFar = 0xfeu;   // voxel outside its chunk's window (only with an invalid layout)
constexpr uint64_t kAStepUnits = (16 * 128) >> 4;   // one K step of channel-major weights
constexpr uint64_t kBStepUnits = (16 * 2) >> 4;     // one K step of K-major rows
// An operand shifted by dxi rows in its 1024-byte-aligned chunk is the
// same 128-byte-swizzled descriptor with the start address moved dxi * 128
// bytes and the base-offset field left at 0: the tensor core takes the
// swizzle phase from the absolute address bits (measured on GB300 against a
// host GEMM for shifts 0..8; the shifted MMAs also run at the full rate).

enum : uint32_t { kMetaFirst = 1u, kMetaEnd = 2u };

struct XrParams {
  const __nv_bfloat16* feats;
  const int32_t* nmap;
  const int32_t* slots;
  const int64_t* slot_count;
  int64_t slots_capacity;  // entries of slots: S is clamped to it
  const __nv_bfloat16* bias;
  const __nv_bfloat16* residual;  // (N, co) or null; may be `out` itself
  __nv_bfloat16* out;
  int64_t n;
  int32_t act;       // spconv_activation of the fused epilogue
  int32_t co;        // row stride of out and weights' Co
  int32_t co_count;  // channels computed (== co, <= 128)
  uint32_t idesc;
  uint32_t off_g;
  uint32_t off_w;
  uint32_t off_ring;
  uint32_t off_stage_out;
  uint32_t off_codes;  // the epilogue's copy of the current tile's 256 slot codes
  uint32_t off_rowoff; // per slot of the tile: its voxel's row in its chunk's window; per chunk its first voxel
  uint32_t off_bias;
  uint32_t off_meta;
  uint32_t off_bars;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool epi_all(bool v) {
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

// Slot code of slot s (xrun.cu), or -1 outside [0, S).
__device__ __forceinline__ int32_t slot_code(const int32_t* slots, int64_t s, int64_t S) {
  return (s >= 0 && s < S) ? __ldg(slots + s) : -1;
}

// Map entry that holds the gathered row of a slot code for group g (offsets
// 3g, 3g+1, 3g+2 are dx = -1, 0, +1): a voxel slot n reads nmap[3g+1, n], a
// run-end separator of voxel n the cell right of it, nmap[3g+2, n], and a
// run-start separator the cell left of it, nmap[3g, n].  Branch-free (the
// loader issues all its loads before it uses any): an empty slot gives
// entry 0 and valid = false.
__device__ __forceinline__ int64_t group_entry(int64_t n, int32_t code, int g, bool* valid) {
  const int32_t h = -2 - code;
  const bool vox = code >= 0, sep = code <= -2;
  const int64_t v = vox ? code : (h >> 1);
  const int k = vox ? 3 * g + 1 : ((h & 1) ? 3 * g : 3 * g + 2);
  *valid = (vox || sep) && v < n;
  return *valid ? static_cast<int64_t>(k) * n + v : 0;
}

// Ring position of gathered row r: producer warp r / 64 takes rows 4 j + s
// (s = r % 4) as 16 consecutive words; rows 256 and 257 follow.
__device__ __forceinline__ int ring_pos(int r) {
  return r < kTileN ? (r >> 6) * 64 + (r & 3) * 16 + ((r & 63) >> 2) : r;
}

// Kept groups: every group with a valid row, and the last group of a tile
// none of whose groups has one (a tile always has voxel slots, whose own
// rows are valid in the (0, 0) group, so this is only a safeguard).
__device__ __forceinline__ bool issue_group(uint32_t flag, int g, bool issued) {
  return flag != 0u || (g == kGroups - 1 && !issued);
}

// kDgrad: input gradient, dfeats[n] = sum_k dout[nmap[k, n]] . w[26 - k]^T
// (the map is symmetric); the gathered rows are dout's (Co = 128 reduced
// channels) and the weights of offset k are w[26 - k] read from the forward
// layout as a K-major operand, as in conv_tc.cu.
// kPair: CTA pairs (clusters of two) share the weight stream.  The two CTAs
// of a pair take tiles 2i and 2i + 1 of each step (an odd tile count leaves
// the second CTA an empty last tile) and keep every group, so both consume
// the same weight slots in the same order; each loads one half of every
// slot and multicasts it to both, and a slot is refilled once both CTAs'
// MMAs are done with it.  Each SM then streams half the weight bytes.
template <bool kDgrad, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    submconv_xrun_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_res,
                         const XrParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;

  int32_t* ring = reinterpret_cast<int32_t*>(smem + p.off_ring);
  __nv_bfloat16* stage_out = reinterpret_cast<__nv_bfloat16*>(smem + p.off_stage_out);
  // Fused residual: the voxel rows of a 32-slot chunk are consecutive (the
  // layout lists voxels in index order), so the chunk's residual rows come
  // as one 32-row window by TMA, which keeps the epilogue's loads off the
  // load/store pipe that the gathers use (residual rows loaded by the
  // threads slowed the whole kernel by 40%).
  const bool fused = p.residual != nullptr;
  int32_t* codes_s = reinterpret_cast<int32_t*>(smem + p.off_codes);
  uint8_t* rowoff_s = smem + p.off_rowoff;                                          // [256]
  int32_t* chunk_first = reinterpret_cast<int32_t*>(smem + p.off_rowoff + kTileN);  // [16]
  float* bias_s = reinterpret_cast<float*>(smem + p.off_bias);
  uint32_t* wmeta = reinterpret_cast<uint32_t*>(smem + p.off_meta);
  uint32_t* ring_flag = wmeta + kWSlots;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bars);
  uint64_t* gfull = bars;
  uint64_t* gempty = gfull + kGBufs;
  uint64_t* wfull = gempty + kGBufs;
  uint64_t* wempty = wfull + kWSlots;
  uint64_t* ring_full = wempty + kWSlots;
  uint64_t* ring_empty = ring_full + kXRing;
  uint64_t* tmem_full = ring_empty + kXRing;
  uint64_t* tmem_empty = tmem_full + 2;
  uint64_t* drain = tmem_empty + 2;
  uint64_t* res_full = drain + 1;  // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(res_full + 2);
  uint32_t* consumed_holder = tmem_holder + 1;
  uint32_t* fills_holder = tmem_holder + 2;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kGBufs; ++s) {
      mbar_init(smem_addr(&gfull[s]), kProducerThreads);
      mbar_init(smem_addr(&gempty[s]), 1);
    }
    for (int s = 0; s < kWSlots; ++s) {
      mbar_init(smem_addr(&wfull[s]), 1);
      mbar_init(smem_addr(&wempty[s]), kPair ? 2 : 1);
    }
    for (int i = 0; i < kXRing; ++i) {
      mbar_init(smem_addr(&ring_full[i]), 32);
      mbar_init(smem_addr(&ring_empty[i]), 32 + kProducerThreads);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&tmem_full[i]), 1);
      mbar_init(smem_addr(&tmem_empty[i]), 4);
    }
    mbar_init(smem_addr(drain), 1);
    mbar_init(smem_addr(&res_full[0]), 1);
    mbar_init(smem_addr(&res_full[1]), 1);
    *consumed_holder = 0;
    *fills_holder = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    if (p.residual != nullptr) tma_prefetch_desc(&tm_res);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_holder), 512);
    tmem_relinquish();
  }
  if (warp == 3) {
    for (int j = lane; j < 128; j += 32)
      bias_s[j] = (p.bias != nullptr && j < p.co_count) ? __bfloat162float(p.bias[j]) : 0.0f;
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();  // the peer's barriers exist before any multicast targets them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int64_t n_rows = p.n;
  const int64_t S = max(int64_t{0}, min(__ldg(p.slot_count), p.slots_capacity));
  const int64_t num_tiles = (S + kTileN - 1) / kTileN;
  // Tiles t = blockIdx.x, blockIdx.x + gridDim.x, ...; a pair steps over its
  // two tiles together, so the second CTA may get one tile past the end
  // (all of its slots empty: gathers zero-fill, nothing is stored).
  const uint32_t rank = kPair ? cluster_cta_rank() : 0u;
  const int64_t t_end = num_tiles + static_cast<int64_t>(rank);

  if (warp == 2) {
    // ------------------------------------------------------ loader
    uint32_t e = 0, ephase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < t_end && ok; t += gridDim.x) {
      const int64_t s0 = t * kTileN;
      int32_t code[9];  // gathered rows r = lane + 32 j of the tile (r < 258)
#pragma unroll
      for (int j = 0; j < 9; ++j) {
        const int r = static_cast<int>(lane) + 32 * j;
        code[j] = r < kGRows ? slot_code(p.slots, s0 - 1 + r, S) : -1;
      }
      // Three groups at a time: addresses first, then their 27 loads, then
      // the checks, so the loads are independent and in flight together
      // (each load waited for in turn starved the MMAs: 16.7 ms at decoder
      // scale against 7.7 ms with the loads taken out).
#pragma unroll
      for (int gb = 0; gb < kGroups; gb += 3) {
        int32_t v[3][9];
        uint32_t ok_bits[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          ok_bits[q] = 0;
#pragma unroll
          for (int j = 0; j < 9; ++j) {
            bool valid;
            const int64_t at = group_entry(n_rows, code[j], gb + q, &valid);
            ok_bits[q] |= (valid ? 1u : 0u) << j;
            v[q][j] = __ldg(p.nmap + at);
          }
        }
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          if (!ok) break;
          if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ring_empty[e]), ephase ^ 1))) {
            ok = false;
            break;
          }
          bool any = false;
#pragma unroll
          for (int j = 0; j < 9; ++j) {
            const int r = static_cast<int>(lane) + 32 * j;
            const int32_t x = (((ok_bits[q] >> j) & 1u) != 0u && v[q][j] >= 0 && v[q][j] < n_rows) ? v[q][j] : -1;
            if (r < kGRows) {
              ring[e * kRingRow + ring_pos(r)] = x;
              any |= x >= 0;
            }
          }
          const uint32_t ballot = __ballot_sync(0xffffffffu, any);
          if (lane == 0) ring_flag[e] = ballot != 0u ? 1u : 0u;
          mbar_arrive(smem_addr(&ring_full[e]));
          if (++e == kXRing) {
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
    const uint32_t dst_lane = (aw * 64u + static_cast<uint32_t>(sub_row)) * 128u;
    const uint32_t sw_even = static_cast<uint32_t>(chunk16 ^ sub_row) << 4;
    const uint32_t sw_odd = static_cast<uint32_t>(chunk16 ^ (sub_row + 4)) << 4;
    // warp 0 also gathers rows 256 + sub_row (rows 258 and 259 are padding,
    // zero-filled and never read); row & 7 == sub_row there
    const uint32_t dst_extra = 256u * 128u + static_cast<uint32_t>(sub_row) * 128u + sw_even;
    uint32_t stage = 0, st_phase = 0, e = 0, ephase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < t_end && ok; t += gridDim.x) {
      bool issued = false;
      for (int g = 0; g < kGroups && ok; ++g) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ring_full[e]), ephase))) {
          ok = false;
          break;
        }
        const bool go = kPair || issue_group(ring_flag[e], g, issued);
        uint32_t vi[16];
        uint32_t valid_bits = 0;
        uint32_t xi = 0;
        bool x_ok = false;
        if (go) {
          const int4* ip = reinterpret_cast<const int4*>(ring + e * kRingRow + static_cast<int>(aw) * 64 + sub_row * 16);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int4 v4 = ip[q];
            const int32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              vi[4 * q + h] = w4[h] >= 0 ? static_cast<uint32_t>(w4[h]) : 0u;
              valid_bits |= (w4[h] >= 0 ? 1u : 0u) << (4 * q + h);
            }
          }
          if (aw == 0 && sub_row < 2) {
            const int32_t xv = ring[e * kRingRow + kTileN + sub_row];
            x_ok = xv >= 0;
            xi = x_ok ? static_cast<uint32_t>(xv) : 0u;
          }
        }
        mbar_arrive(smem_addr(&ring_empty[e]));
        if (++e == kXRing) {
          e = 0;
          ephase ^= 1;
        }
        if (!go) continue;
        issued = true;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&gempty[stage]), st_phase ^ 1))) {
            ok = false;
            break;
          }
          const uint32_t g_base = smem_addr(smem + p.off_g) + stage * kGChunkBytes;
          const char* chunk_base = feats + c * 128 + chunk16 * 16;
          const uint32_t f_dst = g_base + dst_lane;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            cp_async_16<false>(f_dst + 512u * j + ((j & 1) ? sw_odd : sw_even),
                               chunk_base + static_cast<uint64_t>(vi[j]) * 256u, ((valid_bits >> j) & 1u) << 4);
          if (aw == 0)
            cp_async_16<false>(g_base + dst_extra, chunk_base + static_cast<uint64_t>(xi) * 256u,
                               x_ok ? 16u : 0u);
          cp_async_arrive_noinc(smem_addr(&gfull[stage]));
          if (++stage == kGBufs) {
            stage = 0;
            st_phase ^= 1;
          }
        }
      }
    }
    cp_async_wait_all();
  } else if (warp == 0) {
    // ------------------------------------------------------ weight producer
    uint32_t ws = 0, wphase = 0, e = 0, ephase = 0, fills = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < t_end && ok; t += gridDim.x) {
      bool issued = false;
      for (int g = 0; g < kGroups && ok; ++g) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ring_full[e]), ephase))) {
          ok = false;
          break;
        }
        const bool go = kPair || issue_group(ring_flag[e], g, issued);
        __syncwarp();
        mbar_arrive(smem_addr(&ring_empty[e]));
        if (++e == kXRing) {
          e = 0;
          ephase ^= 1;
        }
        if (!go) continue;
        // chunk by chunk, the group's three offsets (the order the MMAs use)
        for (int c = 0; c < kChunks && ok; ++c) {
          for (int dxi = 0; dxi < 3; ++dxi) {
            const int k = 3 * g + dxi;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&wempty[ws]), wphase ^ 1))) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_addr(&wfull[ws]);
            if (lane == 0) {
              wmeta[ws] = (dxi == 0 && c == 0 && !issued) ? kMetaFirst : 0u;
              mbar_arrive_expect_tx(fb, kWSlotBytes);
            }
            __syncwarp();
            if constexpr (kPair) {
              // this CTA's half of the slot, multicast to both CTAs: forward,
              // 64 output channels x 64 input channels; input gradient, 64
              // forward-ci rows with 64 forward-co entries (8 KB either way)
              if (lane == 0) {
                const uint32_t dst = smem_addr(smem + p.off_w) + ws * kWSlotBytes + rank * 8192u;
                if constexpr (!kDgrad)
                  tma_load_3d_multicast(dst, &tm_w, static_cast<int>(rank) * 64, c * 64, k, fb, 0x3);
                else
                  tma_load_3d_multicast(dst, &tm_w, c * 64, static_cast<int>(rank) * 64, 26 - k, fb, 0x3);
              }
            } else if constexpr (!kDgrad) {
              // w[k] channel-major: two boxes of 64 output channels x 64
              // input channels (128-byte swizzle)
              if (lane < 2)
                tma_load_3d(smem_addr(smem + p.off_w) + ws * kWSlotBytes + lane * 8192u, &tm_w,
                            static_cast<int>(lane) * 64, c * 64, k, fb);
            } else {
              // w[26 - k]: 128 forward-ci rows with 64 forward-co entries
              // each (K-major, 128-byte swizzle), one box
              if (lane == 0)
                tma_load_3d(smem_addr(smem + p.off_w) + ws * kWSlotBytes, &tm_w, c * 64, 0, 26 - k, fb);
            }
            ++fills;
            if (++ws == kWSlots) {
              ws = 0;
              wphase ^= 1;
            }
          }
        }
        issued = true;
      }
    }
    // End of work: tells the MMA issuer to close the last tile.
    if (ok && __all_sync(0xffffffffu, mbar_wait(smem_addr(&wempty[ws]), wphase ^ 1))) {
      if (lane == 0) {
        wmeta[ws] = kMetaEnd;
        mbar_arrive(smem_addr(&wfull[ws]));
      }
      ++fills;
    }
    if (lane == 0) *fills_holder = fills;
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // weights channel-major (forward) or K-major (input gradient)
      const uint64_t adesc0 = sw128_desc(smem_addr(smem + p.off_w), kDgrad ? 16u : 8192u, 1024u);
      constexpr uint64_t a_step = kDgrad ? kBStepUnits : kAStepUnits;
      const uint32_t g_base = smem_addr(smem + p.off_g);
      const uint32_t idesc = p.idesc;
      uint32_t ws = 0, wphase = 0, gs = 0, gphase = 0, consumed = 0, tile_i = 0, buf = 0, acc = 0;
      uint32_t d_tmem = tmem_base;
      bool open = false, ok = true;
      while (ok) {
        if (!mbar_wait(smem_addr(&wfull[ws]), wphase)) break;
        tc_fence_after();
        const uint32_t m = wmeta[ws];
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
          buf = tile_i & 1u;
          if (!mbar_wait(smem_addr(&tmem_empty[buf]), ((tile_i >> 1) & 1u) ^ 1u)) break;
          tc_fence_after();
          d_tmem = tmem_base + buf * static_cast<uint32_t>(kTileN);
          open = true;
          acc = 0;
        }
        // Chunk by chunk: the chunk's rows (one G buffer), then the
        // group's three offsets on them, the operand started 0, 1 or 2 rows
        // in; the buffer is released after its 12 MMAs.
        for (int c = 0; c < kChunks && ok; ++c) {
          // the gathered rows were written by cp.async (generic proxy); the
          // MMA reads them through the async proxy
          if (!mbar_wait(smem_addr(&gfull[gs]), gphase)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t gaddr = g_base + gs * kGChunkBytes;
          for (int dxi = 0; dxi < 3; ++dxi) {
            if (dxi != 0 || c != 0) {
              if (!mbar_wait(smem_addr(&wfull[ws]), wphase)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint64_t ad = adesc0 + ws * (kWSlotBytes >> 4);
            const uint64_t bd = sw128_desc(gaddr + static_cast<uint32_t>(dxi) * 128u, 16u, 1024u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              umma_f16(d_tmem, ad + ks * a_step, bd + ks * kBStepUnits, idesc, acc);
              acc = 1;
            }
            if constexpr (kPair)
              umma_commit_multicast(smem_addr(&wempty[ws]), 0x3);  // both CTAs' copies of the slot
            else
              umma_commit(smem_addr(&wempty[ws]));
            ++consumed;
            if (++ws == kWSlots) {
              ws = 0;
              wphase ^= 1;
            }
          }
          if (!ok) break;
          umma_commit(smem_addr(&gempty[gs]));
          if (++gs == kGBufs) {
            gs = 0;
            gphase ^= 1;
          }
        }
        if (!ok) break;
      }
      *consumed_holder = consumed;
      umma_commit(smem_addr(drain));
      mbar_wait(smem_addr(drain), 0);
    }
    __syncwarp();
  } else if (warp >= kEpilogueWarp0 && warp < kEpilogueWarp0 + 4) {
    // ------------------------------------------------------ epilogue
    const uint32_t sub = warp & 3u;
    const int et = static_cast<int>(threadIdx.x) - kEpilogueWarp0 * 32;  // 0..127
    const int chunks_per_row = p.co_count / 8;
    const int co_l = static_cast<int>(sub) * 32 + static_cast<int>(lane);
    // The residual window of fused chunk c (16 slots), into window c & 1:
    // 16 rows from the chunk's first voxel (rows past N read as zero); a
    // chunk without voxels only completes the barrier's phase.
    const uint32_t res_bytes = kResChunk * static_cast<uint32_t>(p.co) * 2u;
    const uint32_t stage_base = smem_addr(smem + p.off_stage_out);
    float* stage_f32 = reinterpret_cast<float*>(smem + p.off_stage_out);
    auto window = [&](int c) {
      return reinterpret_cast<const __nv_bfloat16*>(smem + p.off_stage_out + kWindowOff +
                                                     static_cast<uint32_t>(c & 1) * kWindowBytes);
    };
    auto issue_residual = [&](int c) {
      const int32_t first = chunk_first[c];
      const uint32_t bar = smem_addr(&res_full[c & 1]);
      fence_proxy_async_smem();  // the window's previous contents were read through the generic proxy
      if (first < 0) {
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, res_bytes);
        tma_load_2d(stage_base + kWindowOff + static_cast<uint32_t>(c & 1) * kWindowBytes, &tm_res, 0, first, bar);
      }
    };
    // The voxel a slot names or sits next to, for the L2 prefetch of the
    // next tile's residual rows.
    auto slot_voxel_near = [&](int64_t s) -> int64_t {
      const int32_t c = slot_code(p.slots, s, S);
      if (c >= 0) return c;
      if (c <= -2) return static_cast<int64_t>((-2 - c) >> 1);
      return -1;
    };
    // This thread's 16-byte output pieces: (row, 8-channel column) of a
    // 32-slot chunk (plain, up to four) or a 16-slot chunk (residual, up to
    // two); the same in every chunk, so computed once.
    int prow[4], pcol[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int q = et + 128 * j;
      prow[j] = q / chunks_per_row;
      pcol[j] = (q - prow[j] * chunks_per_row) * 8;
    }
    const int plain_pieces = 32 * chunks_per_row, res_pieces = static_cast<int>(kResChunk) * chunks_per_row;
    uint32_t res_phase = 0;  // bit b: the phase window b's barrier waits for next
    bool ok_res = true;
    uint32_t res_pending = 0;  // window loads issued and not yet waited for (bits)
    uint32_t tile_i = 0;
    for (int64_t t = blockIdx.x; t < t_end; t += gridDim.x, ++tile_i) {
      const uint32_t buf = tile_i & 1u;
      const int64_t s0 = t * kTileN;
      // The tile's slot codes (the output row of each slot), read once and
      // coalesced while the accumulator is still being computed: a row's
      // store then never waits on a load of its code.  Warp `sub` holds
      // slots 32 sub + lane and 128 + 32 sub + lane: 16-slot chunks 2 sub,
      // 2 sub + 1, 8 + 2 sub and 9 + 2 sub, one per half-warp.
      epi_bar();  // the previous tile's codes are no longer read
      const int32_t code0 = slot_code(p.slots, s0 + et, S);
      const int32_t code1 = slot_code(p.slots, s0 + et + 128, S);
      codes_s[et] = code0;
      codes_s[et + 128] = code1;
      if (fused) {
        const uint32_t half = lane < 16 ? 0x0000ffffu : 0xffff0000u;
        const bool v0 = code0 >= 0 && code0 < n_rows, v1 = code1 >= 0 && code1 < n_rows;
        const uint32_t f0 = __reduce_min_sync(half, v0 ? static_cast<uint32_t>(code0) : 0xffffffffu);
        const uint32_t f1 = __reduce_min_sync(half, v1 ? static_cast<uint32_t>(code1) : 0xffffffffu);
        const uint32_t d0 = static_cast<uint32_t>(code0) - f0, d1 = static_cast<uint32_t>(code1) - f1;
        rowoff_s[et] = static_cast<uint8_t>(!v0 ? kRowOffNone : (d0 < kResChunk ? d0 : kRowOffFar));
        rowoff_s[et + 128] = static_cast<uint8_t>(!v1 ? kRowOffNone : (d1 < kResChunk ? d1 : kRowOffFar));
        if ((lane & 15) == 0) {
          chunk_first[et / kResChunk] = f0 == 0xffffffffu ? -1 : static_cast<int32_t>(f0);
          chunk_first[(et + 128) / kResChunk] = f1 == 0xffffffffu ? -1 : static_cast<int32_t>(f1);
        }
      }
      epi_bar();  // the codes (and the chunks' windows) are in
      if (fused) {
        // Both windows are free here (the previous tile's stores are done):
        // chunks 0 and 1 now, and the next tile's residual rows into L2.
        if (et == 0) {
          issue_residual(0);
          issue_residual(1);
          const int64_t vn = slot_voxel_near(s0 + static_cast<int64_t>(gridDim.x) * kTileN);
          if (vn >= 0 && vn < n_rows) {
            const int64_t rows = n_rows - vn < kTileN ? n_rows - vn : static_cast<int64_t>(kTileN);
            bulk_prefetch_l2(p.residual + vn * p.co, static_cast<uint32_t>(rows * p.co * 2));
          }
        }
        res_pending = 3u;
      }
      const bool got = __all_sync(0xffffffffu, mbar_wait(smem_addr(&tmem_full[buf]), (tile_i >> 1) & 1u));
      if (!epi_all(got)) break;
      tc_fence_after();
      const uint32_t tcol = tmem_base + ((sub * 32u) << 16) + buf * static_cast<uint32_t>(kTileN);
      if (fused) {
        for (int c = 0; c < static_cast<int>(kTileN / kResChunk); ++c) {
          epi_bar();  // the previous chunk's rows have been stored
          if (c >= 1 && c + 1 < static_cast<int>(kTileN / kResChunk)) {
            // window (c + 1) & 1 held chunk c - 1, whose stores are done
            if (et == 0) issue_residual(c + 1);
            res_pending |= 1u << ((c + 1) & 1);
          }
          uint32_t v[16];
          tmem_ld_32x32b_x16(tcol + c * kResChunk, v);
          tmem_ld_wait();
          if (co_l < p.co_count) {
            const float b = bias_s[co_l];
#pragma unroll
            for (int i = 0; i < static_cast<int>(kResChunk); ++i) stage_f32[i * 128 + co_l] = __uint_as_float(v[i]) + b;
          }
          const uint32_t wb = static_cast<uint32_t>(c & 1);
          ok_res = __all_sync(0xffffffffu, mbar_wait(smem_addr(&res_full[wb]), (res_phase >> wb) & 1u)) && ok_res;
          res_phase ^= 1u << wb;
          res_pending &= ~(1u << wb);
          epi_bar();  // staged, and every thread saw the window land
          const __nv_bfloat16* win = window(c);
          with_activation(p.act, [&](auto tag) {
            constexpr int kA = decltype(tag)::value;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              if (et + 128 * j >= res_pieces) break;
              const int r = prow[j], col = pcol[j];
              const int32_t code = codes_s[c * kResChunk + r];
              if (code < 0 || code >= n_rows) continue;
              const uint32_t o = rowoff_s[c * kResChunk + r];
              const uint4 rr = o < kResChunk
                                   ? *reinterpret_cast<const uint4*>(win + o * static_cast<uint32_t>(p.co) + col)
                                   : *reinterpret_cast<const uint4*>(p.residual + static_cast<int64_t>(code) * p.co + col);
              const float4 a0 = *reinterpret_cast<const float4*>(stage_f32 + r * 128 + col);
              const float4 a1 = *reinterpret_cast<const float4*>(stage_f32 + r * 128 + col + 4);
              const float x[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
              const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
              uint32_t ow[4];
  #pragma unroll
              for (int h = 0; h < 4; ++h) {
                const float lo = activation_bf16<kA>(x[2 * h] + __uint_as_float(rw[h] << 16));
                const float hi = activation_bf16<kA>(x[2 * h + 1] + __uint_as_float(rw[h] & 0xffff0000u));
                const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
                ow[h] = *reinterpret_cast<const uint32_t*>(&pr);
              }
              *reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(code) * p.co + col) =
                  make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
          });
        }
      } else {
        for (int vc = 0; vc < kTileN / 32; ++vc) {
          epi_bar();  // the previous chunk's staged rows have been stored
          uint32_t v[32];
          tmem_ld_32x32b_x32(tcol + vc * 32, v);
          tmem_ld_wait();
          if (co_l < p.co_count) {
            const float b = bias_s[co_l];
            with_activation(p.act, [&](auto tag) {
              constexpr int kA = decltype(tag)::value;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                stage_out[i * 128 + co_l] = __float2bfloat16_rn(activation_bf16<kA>(__uint_as_float(v[i]) + b));
            });
          }
          epi_bar();  // staged
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (et + 128 * j >= plain_pieces) break;
            const int r = prow[j], col = pcol[j];
            const int32_t code = codes_s[vc * 32 + r];
            if (code >= 0 && code < n_rows)
              *reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(code) * p.co + col) =
                  *reinterpret_cast<const uint4*>(stage_out + r * 128 + col);
          }
        }
      }
      if (!epi_all(ok_res)) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&tmem_empty[buf]));
    }
    // Only after a timed-out wait can a window load still be in flight:
    // wait for it (bounded) before the CTA's memory goes away.
    for (int b2 = 0; b2 < 2; ++b2)
      if (res_pending & (1u << b2)) mbar_wait(smem_addr(&res_full[b2]), (res_phase >> b2) & 1u);
  }

  // ---------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // weight loads issued but never consumed exist only after a timed-out
    // wait: wait (bounded) for them to land before the CTA's memory goes away
    const uint32_t fills = *fills_holder;
    for (uint32_t i = *consumed_holder; i < fills; ++i)
      mbar_wait(smem_addr(&wfull[i % kWSlots]), (i / kWSlots) & 1u);
  }
  __syncthreads();
  // No load or commit of the peer targets this CTA's memory any more.
  if constexpr (kPair) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn xrun_encode_fn(spconv_status* st) {
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

}  // namespace

spconv_status read_and_clear_xrun_device_error(cudaStream_t stream, unsigned int* bits) {
  spconv_status st = SPCONV_OK;
  if (!cuda_ok(cudaStreamSynchronize(stream), "cudaStreamSynchronize", &st)) return st;
  unsigned int mine = 0;
  const unsigned int zero = 0;
  if (!cuda_ok(cudaMemcpyFromSymbol(&mine, g_device_error, sizeof(unsigned int)),
               "cudaMemcpyFromSymbol", &st))
    return st;
  if (!cuda_ok(cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int)),
               "cudaMemcpyToSymbol", &st))
    return st;
  *bits |= mine;
  return SPCONV_OK;
}

spconv_status launch_conv_xrun(const void* feats, const int32_t* nmap, const int32_t* slots,
                               int64_t slots_capacity, const int64_t* slot_count, const void* w,
                               const void* bias, const void* residual, void* out, int64_t n, int32_t co,
                               int act, bool dgrad, cudaStream_t stream) {
  spconv_status st = SPCONV_OK;
  EncodeTiledFn encode = xrun_encode_fn(&st);
  if (encode == nullptr) return st;
  CUtensorMap tm_w;
  // Weights in their forward (K, Ci_fwd, Co_fwd) layout as a 3-D tensor
  // (co_fwd, ci_fwd, k).  Forward: Ci_fwd = 128, boxes of 64 output x 64
  // input channels.  Input gradient: Co_fwd = 128 is reduced and `co` output
  // channels are Ci_fwd; boxes of 64 forward-co x 128 forward-ci.
  const cuuint64_t wo = dgrad ? 128u : static_cast<cuuint64_t>(co);  // forward Co
  const cuuint64_t wi = dgrad ? static_cast<cuuint64_t>(co) : 128u;  // forward Ci
  cuuint64_t dims[3] = {wo, wi, 27u};
  cuuint64_t strides[2] = {wo * 2u, wi * wo * 2u};
  // Paired CTAs load half a slot each: 64 x 64 boxes for the input gradient too.
  constexpr bool kPaired = true;
  cuuint32_t box[3] = {64u, (dgrad && !kPaired) ? 128u : 64u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, strides, box,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPCONV_ERR_CUDA, "cuTensorMapEncodeTiled(w) failed: " + std::to_string(r));
  // The residual (N, co) as 2-D rows; box = kResChunk rows of co channels,
  // no swizzle (rows past N read as zero).  Unused without a residual.
  CUtensorMap tm_res = tm_w;
  if (residual != nullptr) {
    cuuint64_t rdims[2] = {static_cast<cuuint64_t>(co), static_cast<cuuint64_t>(n)};
    cuuint64_t rstrides[1] = {static_cast<cuuint64_t>(co) * 2u};
    // one fused chunk's window: kResChunk rows (kWindowBytes at co = 128)
    cuuint32_t rbox[2] = {static_cast<cuuint32_t>(co), kResChunk};
    cuuint32_t restr[2] = {1u, 1u};
    r = encode(&tm_res, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(residual), rdims, rstrides, rbox,
               restr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(SPCONV_ERR_CUDA, "cuTensorMapEncodeTiled(residual) failed: " + std::to_string(r));
  }

  XrParams p{};
  p.feats = static_cast<const __nv_bfloat16*>(feats);
  p.nmap = nmap;
  p.slots = slots;
  p.slot_count = slot_count;
  p.slots_capacity = slots_capacity;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.residual = static_cast<const __nv_bfloat16*>(residual);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.n = n;
  p.act = act;
  p.co = co;
  p.co_count = co;
  // D f32, A and B bf16, A (weights) channel-major (forward) or K-major
  // (input gradient), B (rows) K-major, N = 256, M = 128
  const uint32_t a_mn_major = dgrad ? 0u : 1u;
  p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | (a_mn_major << 15) |
            ((static_cast<uint32_t>(kTileN) >> 3) << 17) | ((128u >> 4) << 24);
  uint32_t off = 0;
  p.off_g = off;
  off += kGBufs * kGChunkBytes;
  p.off_w = off;
  off += kWSlots * kWSlotBytes;
  p.off_ring = off;
  off += kXRing * kRingRow * 4u;
  p.off_stage_out = off;
  off += kStageBytes;  // 128-byte aligned, as are the windows in it (TMA destinations)
  p.off_codes = off;
  off += kTileN * 4u;
  p.off_rowoff = off;
  off += kTileN + (kTileN / kResChunk) * 4u;
  p.off_bias = off;
  off += 128u * 4u;
  p.off_meta = off;
  off += (kWSlots + kXRing) * 4u;
  off = (off + 7u) & ~7u;
  p.off_bars = off;
  off += (2u * kGBufs + 2u * kWSlots + 2u * kXRing + 7u) * 8u + 16u;
  const uint32_t smem_bytes = off + 1024u;  // slack for the 1024-byte alignment
  if (smem_bytes > 232448u) return fail(SPCONV_ERR_UNSUPPORTED, "x-run conv: shared memory layout too large");

  auto kern = dgrad ? submconv_xrun_kernel<true, kPaired> : submconv_xrun_kernel<false, kPaired>;
  if (!cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes)),
               "cudaFuncSetAttribute", &st))
    return st;
  const int sms = sm_count();
  if (sms <= 0) return fail(SPCONV_ERR_CUDA, "could not query the SM count");
  // Clusters of two CTAs, as many as fit at once (one CTA per SM).
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
  // co-resident pairs, looked up once per device and direction
  constexpr int kMaxDevices = 64;
  static int cached[kMaxDevices][2] = {};
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev), "cudaGetDevice", &st)) return st;
  int clusters = (dev >= 0 && dev < kMaxDevices) ? cached[dev][dgrad ? 1 : 0] : 0;
  if (clusters <= 0) {
    if (!cuda_ok(cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg), "cudaOccupancyMaxActiveClusters", &st))
      return st;
    if (dev >= 0 && dev < kMaxDevices) cached[dev][dgrad ? 1 : 0] = clusters;
  }
  if (clusters < 1) return fail(SPCONV_ERR_UNSUPPORTED, "x-run conv: no CTA pair fits on this device");
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (clusters < sms / 2 ? clusters : sms / 2)), 1, 1);
  if (!cuda_ok(cudaLaunchKernelEx(&cfg, kern, tm_w, tm_res, p), "submconv_xrun_kernel", &st)) return st;
  return SPCONV_OK;
}

}  // namespace spconv

// Weight gradient of the submanifold convolution on the tensor cores (bf16):
//
//     dw[k, ci, co] = sum over valid entries m = nmap[k, n] of feats[m, ci] * dout[n, co]
//
// (the chain rule applied to the formula of page "sparse_conv_metal.py",
// trellis-2-mrp-mlx: module docstring; the page computes the forward pass
// only).  Per offset this is a contraction over voxels.  It runs as
//
//     dw^T[co, (k, ci)] += dout^T[co, n] * gathered[n, (k, ci)]
//
// with M = 128 output channels (A = a tile of dout rows, loaded by tiled TMA:
// the rows of a voxel chunk are contiguous, channel-major operand), N = up to
// 256 columns made of four "atoms" of 64 input channels, each atom one
// (offset, 64-channel) slice of the gathered feature rows (channel-major
// operand written by cp.async), and K = 16 voxels per instruction; a stage is
// a chunk of 64 voxels.  One CTA accumulates one atom group over a long
// voxel range in tensor memory (two 256-column buffers, so one item's flush
// overlaps the next item's MMAs) and then adds its 128 x 256 partial tile to
// dw with fp32 reductions.  dw is zeroed before the launch.
//
// Warp roles mirror the forward kernel: warps 2 and 3 load the map entries
// of each (item, chunk) into a ring (alternate chunks) and flag atoms with
// any valid entry; warps 8-11
// gather the atoms' feature rows (zero rows for missing neighbours, and no
// stage at all for a chunk in which no atom has one); warp 0 loads the dout
// tile and writes the stage metadata; warp 1 issues the MMAs; warps 4-7 read
// the accumulator and reduce it into dw.  Every wait is bounded in time.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace spconv {
namespace {

constexpr int kThreads = 384;
constexpr int kProducerWarp0 = 8;
constexpr int kProducerThreads = 128;
constexpr int kEpilogueWarp0 = 4;
constexpr int kRing = 16;  // even: the two map loaders keep to alternate rows
static_assert(kRing % 2 == 0, "two loaders take alternate ring rows");
constexpr int kChunkVox = 64;              // voxels per stage (K of four MMAs)
constexpr int kAtoms = 4;                  // 64-channel atoms per item (N <= 256)
constexpr uint32_t kABytes = 128 * 128;    // dout tile: 128 channels x 64 voxels
constexpr uint32_t kAtomBytes = 64 * 128;  // one atom: 64 channels x 64 voxels
constexpr uint32_t kStageBytes = kABytes + kAtoms * kAtomBytes;
constexpr int kMaxStages = 8;
constexpr int kMaxSmem = 232448;
constexpr uint64_t kKStepUnits = (16 * 128) >> 4;  // 16 voxel rows of 128 B, 16-byte units

enum : uint32_t { kMetaFirst = 1u, kMetaEnd = 2u };

struct WgParams {
  const __nv_bfloat16* feats;
  const int32_t* nmap;
  float* dw;
  int64_t n;
  int64_t total_chunks;     // ceil(N / 64)
  int64_t chunks_per_item;  // voxel chunks of one item
  int64_t num_ranges;
  int64_t num_items;        // num_groups * num_ranges
  int32_t k;
  int32_t ci;
  int32_t co;
  int32_t co_base;          // first output channel of this launch
  int32_t co_count;         // channels of this launch (<= 128)
  int32_t atoms_per_k;      // ceil(Ci / 64)
  int32_t num_atoms;        // K * atoms_per_k
  int32_t num_groups;       // ceil(num_atoms / 4)
  uint32_t stages;
  uint32_t off_ring;
  uint32_t off_meta;
  uint32_t off_bars;
};

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

// Item i: atom group i % num_groups over voxel range i / num_groups (CTAs
// running at the same time share a range, so its dout tiles stay in L2).
__device__ __forceinline__ void item_coords(const WgParams& p, int64_t item, int32_t* group,
                                            int64_t* c0, int64_t* c_count) {
  *group = static_cast<int32_t>(item % p.num_groups);
  const int64_t range = item / p.num_groups;
  *c0 = range * p.chunks_per_item;
  const int64_t left = p.total_chunks - *c0;
  *c_count = left < p.chunks_per_item ? left : p.chunks_per_item;
}

// A chunk is issued when one of its atoms has a valid entry, and the last
// chunk of an item none of whose chunks had one is issued anyway (all its
// rows are zero, so the item's accumulator becomes exactly zero).
__device__ __forceinline__ bool issue_chunk(uint32_t mask, bool last, bool issued) {
  return mask != 0u || (last && !issued);
}

__global__ void __launch_bounds__(kThreads, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tm_dout, const WgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t S = p.stages;

  int32_t* ring = reinterpret_cast<int32_t*>(smem + p.off_ring);  // [kRing][kAtoms][64]
  uint32_t* meta = reinterpret_cast<uint32_t*>(smem + p.off_meta);
  uint32_t* ring_mask = meta + S;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* ring_full = bars + 2 * S;
  uint64_t* ring_empty = ring_full + kRing;
  uint64_t* tmem_full = ring_empty + kRing;
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
    for (int i = 0; i < kRing; ++i) {
      mbar_init(smem_addr(&ring_full[i]), 32);
      mbar_init(smem_addr(&ring_empty[i]), 32 + kProducerThreads);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&tmem_full[i]), 1);
      mbar_init(smem_addr(&tmem_empty[i]), 4);
    }
    mbar_init(smem_addr(drain), 1);
    *consumed_holder = 0;
    *fills_holder = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_dout);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int64_t n_rows = p.n;

  if (warp == 2 || warp == 3) {
    // ------------------------------------------------------ map loaders
    // One ring row per (item, chunk): the 64 entries of each atom's offset,
    // normalised to a valid index or -1, and a mask of atoms with any valid
    // entry.  The CTA's (item, chunk) sequence is split between two warps:
    // warp 2 fills the rows of even positions, warp 3 of odd ones (the ring
    // length is even, so each keeps to its own rows).  Two voxels per lane;
    // batches of four of the warp's chunks, the next batch's loads in flight
    // while this one is published.  The map is read from device memory
    // once, so a loader's pace is set by the load latency: two loaders
    // keep twice the chunks in flight.
    constexpr int kBatch = 4;
    const int64_t parity = warp - 2;
    struct Pos {
      int64_t item, c, c0, cnt;
      int32_t group;
    };
    auto advance = [&](Pos& q, int64_t steps) {
      q.c += steps;
      while (q.item < p.num_items && q.c >= q.cnt) {
        q.c -= q.cnt;
        q.item += gridDim.x;
        if (q.item < p.num_items) item_coords(p, q.item, &q.group, &q.c0, &q.cnt);
      }
    };
    auto load_batch = [&](int32_t (&vv)[kBatch][kAtoms][2], Pos q) {
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
#pragma unroll
        for (int j = 0; j < kAtoms; ++j) {
          const int32_t atom = q.group * kAtoms + j;
          const int32_t kk = atom / p.atoms_per_k;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int64_t vox = (q.c0 + q.c) * kChunkVox + lane + 32 * h;
            vv[b][j][h] = -1;
            if (q.item < p.num_items && atom < p.num_atoms && vox < n_rows)
              vv[b][j][h] = __ldg(p.nmap + static_cast<int64_t>(kk) * n_rows + vox);
          }
        }
        advance(q, 2);
      }
    };
    Pos pos{static_cast<int64_t>(blockIdx.x), 0, 0, 0, 0};
    if (pos.item < p.num_items) item_coords(p, pos.item, &pos.group, &pos.c0, &pos.cnt);
    advance(pos, parity);
    int64_t t = parity;  // position in the CTA's sequence: ring row t % kRing
    bool ok = true;
    int32_t cur[kBatch][kAtoms][2], nxt[kBatch][kAtoms][2];
    load_batch(cur, pos);
    while (pos.item < p.num_items && ok) {
      Pos npos = pos;
      advance(npos, 2 * kBatch);
      load_batch(nxt, npos);
      Pos q = pos;
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (q.item >= p.num_items) break;
        const uint32_t e = static_cast<uint32_t>(t % kRing);
        const uint32_t ephase = static_cast<uint32_t>((t / kRing) & 1);
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ring_empty[e]), ephase ^ 1))) {
          ok = false;
          break;
        }
        uint32_t mask = 0;
#pragma unroll
        for (int j = 0; j < kAtoms; ++j) {
          bool any = false;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int32_t nv = (cur[b][j][h] >= 0 && cur[b][j][h] < n_rows) ? cur[b][j][h] : -1;
            any |= nv >= 0;
            ring[(e * kAtoms + j) * kChunkVox + lane + 32 * h] = nv;
          }
          if (__ballot_sync(0xffffffffu, any) != 0u) mask |= 1u << j;
        }
        if (lane == 0) ring_mask[e] = mask;
        mbar_arrive(smem_addr(&ring_full[e]));
        t += 2;
        advance(q, 2);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
#pragma unroll
        for (int j = 0; j < kAtoms; ++j)
#pragma unroll
          for (int h = 0; h < 2; ++h) cur[b][j][h] = nxt[b][j][h];
      pos = npos;
    }
  } else if (warp >= kProducerWarp0) {
    // ------------------------------------------------------ gather producers
    // Warp aw gathers voxels aw*16 .. aw*16+15 of the chunk for all four
    // atoms; a warp instruction moves four 128-byte row pieces (8 lanes a
    // piece, 16 bytes a lane) into the channel-major, 128-byte-swizzled atom
    // (64 channels x 64 voxels: 8-voxel groups of 1024 bytes).
    const uint32_t aw = warp - kProducerWarp0;
    const int sub_row = static_cast<int>(lane >> 3);
    const int c16 = static_cast<int>(lane & 7);
    const char* feats = reinterpret_cast<const char*>(p.feats);
    const uint32_t row_bytes = static_cast<uint32_t>(p.ci) * 2u;
    uint32_t stage = 0, st_phase = 0, e = 0, ephase = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < p.num_items && ok; item += gridDim.x) {
      int32_t group;
      int64_t c0, c_count;
      item_coords(p, item, &group, &c0, &c_count);
      // Per atom: byte offset of this lane's 16 bytes in a feature row, and
      // whether they lie inside the row (the last atom may be partial).
      uint32_t col[kAtoms];
      bool col_ok[kAtoms];
#pragma unroll
      for (int j = 0; j < kAtoms; ++j) {
        const int32_t atom = group * kAtoms + j;
        col[j] = static_cast<uint32_t>(atom % p.atoms_per_k) * 128u + static_cast<uint32_t>(c16) * 16u;
        col_ok[j] = atom < p.num_atoms && col[j] < row_bytes;
      }
      bool issued = false;
      for (int64_t c = 0; c < c_count && ok; ++c) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ring_full[e]), ephase))) {
          ok = false;
          break;
        }
        const uint32_t mask = ring_mask[e];
        const bool go = issue_chunk(mask, c + 1 == c_count, issued);
        int32_t idx[kAtoms][4];
        if (go) {
#pragma unroll
          for (int j = 0; j < kAtoms; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
              idx[j][i] = ring[(e * kAtoms + j) * kChunkVox + static_cast<int>(aw) * 16 + 4 * i + sub_row];
        }
        mbar_arrive(smem_addr(&ring_empty[e]));
        if (++e == kRing) {
          e = 0;
          ephase ^= 1;
        }
        if (!go) continue;
        issued = true;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage]), st_phase ^ 1))) {
          ok = false;
          break;
        }
        const uint32_t b_base = smem_addr(smem + stage * kStageBytes) + kABytes;
#pragma unroll
        for (int j = 0; j < kAtoms; ++j) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int vrow = static_cast<int>(aw) * 16 + 4 * i + sub_row;  // voxel within the chunk
            const bool valid = col_ok[j] && ((mask >> j) & 1u) != 0u && idx[j][i] >= 0;
            const uint32_t vi = valid ? static_cast<uint32_t>(idx[j][i]) : 0u;
            const uint32_t d = b_base + static_cast<uint32_t>(j) * kAtomBytes +
                               static_cast<uint32_t>(vrow >> 3) * 1024u +
                               static_cast<uint32_t>(vrow & 7) * 128u +
                               (static_cast<uint32_t>(c16 ^ (vrow & 7)) << 4);
            cp_async_16<false>(d, feats + col[j] + static_cast<uint64_t>(vi) * row_bytes, valid ? 16u : 0u);
          }
        }
        cp_async_arrive_noinc(smem_addr(&full[stage]));
        if (++stage == S) {
          stage = 0;
          st_phase ^= 1;
        }
      }
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage]), st_phase ^ 1)))
      cp_async_arrive_noinc(smem_addr(&full[stage]));
    cp_async_wait_all();
  } else if (warp == 0) {
    // ------------------------------------------------------ dout tile + metadata
    uint32_t stage = 0, st_phase = 0, e = 0, ephase = 0, fills = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < p.num_items && ok; item += gridDim.x) {
      int32_t group;
      int64_t c0, c_count;
      item_coords(p, item, &group, &c0, &c_count);
      const uint32_t natoms = static_cast<uint32_t>(min(kAtoms, p.num_atoms - group * kAtoms));
      bool issued = false;
      for (int64_t c = 0; c < c_count && ok; ++c) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&ring_full[e]), ephase))) {
          ok = false;
          break;
        }
        const bool go = issue_chunk(ring_mask[e], c + 1 == c_count, issued);
        __syncwarp();
        mbar_arrive(smem_addr(&ring_empty[e]));
        if (++e == kRing) {
          e = 0;
          ephase ^= 1;
        }
        if (!go) continue;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage]), st_phase ^ 1))) {
          ok = false;
          break;
        }
        const uint32_t fullb = smem_addr(&full[stage]);
        if (lane == 0) {
          meta[stage] = (natoms << 8) | (issued ? 0u : kMetaFirst);
          mbar_arrive_expect_tx(fullb, kABytes);
        }
        __syncwarp();
        if (lane < 2)  // two 64-channel halves of the 64-voxel dout tile
          tma_load_2d(smem_addr(smem + stage * kStageBytes) + lane * 8192u, &tm_dout,
                      p.co_base + 64 * static_cast<int32_t>(lane), static_cast<int32_t>((c0 + c) * kChunkVox),
                      fullb);
        issued = true;
        ++fills;
        if (++stage == S) {
          stage = 0;
          st_phase ^= 1;
        }
      }
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[stage]), st_phase ^ 1))) {
      if (lane == 0) {
        meta[stage] = kMetaEnd;
        mbar_arrive(smem_addr(&full[stage]));
      }
      ++fills;
    }
    if (lane == 0) *fills_holder = fills;
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // A: dout tile, channel-major (two 64-channel halves 8 KB apart); B:
      // atoms, channel-major (8 KB apart); both with 8-voxel groups of 1 KB.
      const uint64_t adesc0 = sw128_desc(smem_addr(smem), 8192u, 1024u);
      const uint64_t bdesc0 = sw128_desc(smem_addr(smem) + kABytes, 8192u, 1024u);
      const uint64_t stage_units = kStageBytes >> 4;
      // D f32, A and B bf16, both MN-major, M = 128; N set per item.
      const uint32_t idesc_base = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
                                  ((128u >> 4) << 24);
      uint32_t stage = 0, st_phase = 0, consumed = 0, tile_i = 0, buf = 0;
      uint32_t d_tmem = tmem_base;
      bool open = false;
      while (true) {
        if (!mbar_wait(smem_addr(&full[stage]), st_phase)) break;
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
          buf = tile_i & 1u;
          if (!mbar_wait(smem_addr(&tmem_empty[buf]), ((tile_i >> 1) & 1u) ^ 1u)) break;
          tc_fence_after();
          d_tmem = tmem_base + buf * 256u;
          open = true;
        }
        const uint32_t natoms = (m >> 8) & 0xFu;
        const uint32_t idesc = idesc_base | (((natoms * 64u) >> 3) << 17);
        const uint64_t ad = adesc0 + stage * stage_units;
        const uint64_t bd = bdesc0 + stage * stage_units;
        const uint32_t acc0 = (m & kMetaFirst) == 0u ? 1u : 0u;
#pragma unroll
        for (int s = 0; s < kChunkVox / 16; ++s)
          umma_f16(d_tmem, ad + s * kKStepUnits, bd + s * kKStepUnits, idesc, s > 0 ? 1u : acc0);
        umma_commit(smem_addr(&empty[stage]));
        ++consumed;
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
    // ------------------------------------------------------ reduce into dw
    // Lane = output channel, column = (atom, input channel): for a fixed
    // column a warp's reductions hit 32 consecutive channels of one dw row.
    const uint32_t sub = warp & 3u;
    const int co_l = static_cast<int>(sub) * 32 + static_cast<int>(lane);
    uint32_t tile_i = 0;
    for (int64_t item = blockIdx.x; item < p.num_items; item += gridDim.x, ++tile_i) {
      int32_t group;
      int64_t c0, c_count;
      item_coords(p, item, &group, &c0, &c_count);
      const int natoms = min(kAtoms, p.num_atoms - group * kAtoms);
      const uint32_t buf = tile_i & 1u;
      const bool got = __all_sync(0xffffffffu, mbar_wait(smem_addr(&tmem_full[buf]), (tile_i >> 1) & 1u));
      if (!epilogue_all(got)) break;
      tc_fence_after();
      const uint32_t tcol = tmem_base + ((sub * 32u) << 16) + buf * 256u;
      for (int j = 0; j < natoms; ++j) {
        const int32_t atom = group * kAtoms + j;
        const int32_t kk = atom / p.atoms_per_k;
        for (int h = 0; h < 2; ++h) {
          const int32_t ci0 = (atom % p.atoms_per_k) * 64 + h * 32;
          if (ci0 >= p.ci) continue;  // warp-uniform
          uint32_t v[32];
          tmem_ld_32x32b_x32(tcol + static_cast<uint32_t>(j * 64 + h * 32), v);
          tmem_ld_wait();
          if (co_l < p.co_count) {
            float* dst = p.dw + (static_cast<int64_t>(kk) * p.ci + ci0) * p.co + p.co_base + co_l;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (ci0 + i < p.ci) atomicAdd(dst + static_cast<int64_t>(i) * p.co, __uint_as_float(v[i]));
          }
        }
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
    const uint32_t fills = *fills_holder;
    for (uint32_t i = *consumed_holder; i < fills; ++i) mbar_wait(smem_addr(&full[i % S]), (i / S) & 1u);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

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

}  // namespace

spconv_status read_and_clear_wgrad_device_error(cudaStream_t stream, unsigned int* bits) {
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

spconv_status launch_wgrad_tc(const void* feats, const void* dout, const int32_t* nmap, float* dw,
                              int64_t n, int32_t k, int32_t ci, int32_t co, cudaStream_t stream) {
  spconv_status st = SPCONV_OK;
  if (!cuda_ok(cudaMemsetAsync(dw, 0, static_cast<size_t>(k) * ci * co * sizeof(float), stream),
               "cudaMemsetAsync(dw)", &st))
    return st;
  EncodeTiledFn encode = encode_fn(&st);
  if (encode == nullptr) return st;
  // dout viewed as (N, Co), innermost Co: box = 64 channels x 64 voxels,
  // 128-byte swizzle (the channel-major operand); rows past N read as zero.
  CUtensorMap tm;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(co), static_cast<cuuint64_t>(n)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(co) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kChunkVox)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(dout), dims, strides, box,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPCONV_ERR_CUDA, "cuTensorMapEncodeTiled(dout) failed: " + std::to_string(r));
  const int sms = sm_count();
  if (sms <= 0) return fail(SPCONV_ERR_CUDA, "could not query the SM count");

  const uint32_t ring_bytes = kRing * kAtoms * kChunkVox * 4u;
  const uint32_t fixed = ring_bytes + (kMaxStages + kRing) * 4u + (2u * kMaxStages + 2u * kRing + 5u) * 8u +
                         16u + 1024u;
  uint32_t stages = (kMaxSmem - fixed) / kStageBytes;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return fail(SPCONV_ERR_UNSUPPORTED, "shared memory too small for the wgrad tile");

  for (int32_t co_base = 0; co_base < co; co_base += 128) {
    WgParams p{};
    p.feats = static_cast<const __nv_bfloat16*>(feats);
    p.nmap = nmap;
    p.dw = dw;
    p.n = n;
    p.k = k;
    p.ci = ci;
    p.co = co;
    p.co_base = co_base;
    p.co_count = (co - co_base) < 128 ? (co - co_base) : 128;
    p.atoms_per_k = (ci + 63) / 64;
    p.num_atoms = k * p.atoms_per_k;
    p.num_groups = (p.num_atoms + kAtoms - 1) / kAtoms;
    p.total_chunks = (n + kChunkVox - 1) / kChunkVox;
    // About four items per SM: long voxel ranges keep the reductions into dw
    // few (one 128 x 256 tile per item).  Among up to twice that many ranges
    // the count is taken whose items fill the last round over the CTAs best
    // (with 14 atom groups and 152 SMs: 76 ranges, 7 items per CTA, instead
    // of 44 ranges, where 8 CTAs ran a fifth item while the others waited).
    int64_t ranges = (4 * static_cast<int64_t>(sms) + p.num_groups - 1) / p.num_groups;
    if (ranges < 1) ranges = 1;
    {
      const int64_t r0 = ranges;
      double best = 1e30;
      for (int64_t r = r0; r <= 2 * r0 && r <= p.total_chunks; ++r) {
        const int64_t items = r * p.num_groups;
        const int64_t rounds = (items + sms - 1) / sms;
        const double waste = static_cast<double>(rounds * sms) / static_cast<double>(items);
        if (waste < best - 1e-9) {
          best = waste;
          ranges = r;
        }
      }
    }
    p.chunks_per_item = (p.total_chunks + ranges - 1) / ranges;
    p.num_ranges = (p.total_chunks + p.chunks_per_item - 1) / p.chunks_per_item;
    p.num_items = static_cast<int64_t>(p.num_groups) * p.num_ranges;
    p.stages = stages;
    uint32_t off = stages * kStageBytes;
    p.off_ring = off;
    off += ring_bytes;
    p.off_meta = off;
    off += (stages + kRing) * 4u;
    off = (off + 7u) & ~7u;
    p.off_bars = off;
    off += (2u * stages + 2u * kRing + 5u) * 8u + 16u;
    const uint32_t smem_bytes = off + 1024u;
    const int grid = static_cast<int>(p.num_items < sms ? p.num_items : sms);
    if (!cuda_ok(cudaFuncSetAttribute(wgrad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem_bytes)),
                 "cudaFuncSetAttribute", &st))
      return st;
    wgrad_tc_kernel<<<grid, kThreads, smem_bytes, stream>>>(tm, p);
    if (!cuda_ok(cudaGetLastError(), "wgrad_tc_kernel launch", &st)) return st;
  }
  return SPCONV_OK;
}

}  // namespace spconv

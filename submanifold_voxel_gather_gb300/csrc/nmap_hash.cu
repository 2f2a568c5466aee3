// GPU neighbour-map builder: open-addressing hash of voxel coordinates.
//
// The page "sparse_conv_metal.py" (trellis-2-mrp-mlx) consumes a (K, N) int32
// map whose entry [k, n] is the row of the voxel at coords[n] + offsets[k]
// and N where there is none (wrapper docstring, kernel body); it takes the
// map as given.  This file builds it.  A first pass checks the coordinate
// range and whether the coordinates are strictly increasing in (z, y, x)
// order, counts the (z, y) rows and finds the bounding box.  The rest of the
// build takes one of three paths, chosen on the device from that verdict
// (every kernel of the other paths returns at once):
//
// Sorted input whose bounding box is small enough (the usual case: a
// voxeliser emits sorted coordinates in a bounded grid).  The voxels of 32
// consecutive cells of a (z, y) row have consecutive indices, so the box's
// rows are laid out densely in the workspace as words of 32 cells: an
// occupancy bit per cell and the index of the word's first voxel.  A
// neighbour at x is then one word load: present if its bit is set, at index
// first + popcount of the lower bits.  No search and no probe:
//
//   clear   words := 0
//   insert  every voxel sets its bit (one atomic OR per word and warp); the
//           first voxel of each word writes its index
//   query   one thread per voxel: per (dz, dy) row one word load for x - 1,
//           x and x + 1 (two at a word edge)
//
// Sorted input with a larger box.  A hash of rows (row -> index of its first
// voxel, table sized from the row count) is enough:
//
//   clear   the row table's slots := EMPTY
//   insert  the first voxel of each row inserts the row with its length
//   query   one thread per voxel, per (dz, dy) group of offsets: one row
//           probe (first voxel and length), then a bisection over the row's
//           x values for x + dx (in ascending dx, each search starting where
//           the last one ended).  Consecutive voxels probe the same rows, so
//           the table and coordinate reads mostly hit in cache.
//
// Any other order (or duplicates, which are never strictly increasing):
//
//   clear   every slot's key := EMPTY
//   insert  one thread per voxel: linear probing with a 64-bit atomicCAS on
//           the packed key (21 bits per axis); an equal key already present
//           flags a duplicate coordinate
//   query   one thread per voxel, loop over the K offsets: probe for the
//           shifted key (one 16-byte load per probe), write nmap[k, n] with
//           coalesced stores across the warp
//
// The map is symmetric: if offsets k and k' are opposite, nmap[k, n] = m
// exactly when nmap[k', m] = n.  So only one offset of each opposite pair is
// probed; a hit writes both entries, and the rows of the unprobed offsets are
// filled with N beforehand (by the clear kernel).  A zero offset gives
// nmap[k, n] = n without a probe.  This halves the probes of a symmetric
// offset set such as {-1,0,1}^3.
//
// Capacity is the next power of two >= 2N (load factor <= 1/2), so probe
// sequences are short; every probe loop is still bounded by the capacity.
#include <cuda_runtime.h>

#include <climits>

#include <string>

#include "internal.h"

namespace spconv {

namespace {

constexpr int kThreads = 256;
constexpr unsigned long long kEmptyKey = ~0ull;
constexpr size_t kFlagBytes = 256;

enum : int { kFlagDuplicate = 1, kFlagRange = 2, kFlagFull = 4, kFlagUnsorted = 8 };

// Flag words: [0] error / order bits, [1] (z, y) row count, [2..7] the
// bounding box (z min, z max, y min, y max, x min, x max), [8] set when the
// dense query has written the x-run layout's per-voxel flags.
enum : int { kFlagBoxMin = 2, kFlagXrunReady = 8 };

enum : int8_t { kRoleProbe = 0, kRoleMirror = 1, kRoleSelf = 2 };

// Per-offset work of the query kernels (built on the host from the offsets).
struct QueryPlan {
  int32_t d[3 * SPCONV_MAX_BUILD_OFFSETS];   // offsets (dz, dy, dx)
  int16_t mirror[SPCONV_MAX_BUILD_OFFSETS];  // probed offset: its opposite's row, or -1
  int8_t role[SPCONV_MAX_BUILD_OFFSETS];     // kRoleProbe / kRoleMirror / kRoleSelf
  // Sorted-input path: the offsets grouped by (dz, dy); the members of group
  // g are mem_k/mem_dx[grp_first[g] .. grp_first[g] + grp_count[g]), in
  // ascending dx.
  int32_t groups;
  int32_t grp_dz[SPCONV_MAX_BUILD_OFFSETS];
  int32_t grp_dy[SPCONV_MAX_BUILD_OFFSETS];
  int16_t grp_first[SPCONV_MAX_BUILD_OFFSETS];
  int16_t grp_count[SPCONV_MAX_BUILD_OFFSETS];
  int16_t mem_k[SPCONV_MAX_BUILD_OFFSETS];
  int32_t mem_dx[SPCONV_MAX_BUILD_OFFSETS];
};

struct alignas(16) Slot {
  unsigned long long key;
  int32_t val;
  int32_t pad;
};

__device__ __forceinline__ unsigned long long pack_coord(int z, int y, int x) {
  return (static_cast<unsigned long long>(z) << 42) | (static_cast<unsigned long long>(y) << 21) |
         static_cast<unsigned long long>(x);
}

// 64-bit finaliser of MurmurHash3 (Austin Appleby, public domain).
__device__ __forceinline__ unsigned long long mix_hash(unsigned long long k) {
  k ^= k >> 33;
  k *= 0xff51afd7ed558ccdull;
  k ^= k >> 33;
  k *= 0xc4ceb9fe1a85ec53ull;
  k ^= k >> 33;
  return k;
}

__device__ __forceinline__ bool in_grid(int v) {
  return v >= 0 && v < SPCONV_COORD_LIMIT;
}

__device__ __forceinline__ unsigned long long row_key(int z, int y) {
  return (static_cast<unsigned long long>(z) << 21) | static_cast<unsigned long long>(y);
}

// Slots of the row table for `rows` rows: the next power of two >= 2 rows
// (at least 64).  Never more than hash_capacity(N), as rows <= N.
__device__ __forceinline__ unsigned long long row_capacity(unsigned int rows) {
  const unsigned long long want = 2ull * rows;
  if (want <= 64ull) return 64ull;
  return 1ull << (64 - __clzll(want - 1ull));
}

// Home slot of row (z, y): a 32-bit integer hash of the row (multiply,
// xor-shift rounds; the table never exceeds 2^32 slots as N < 2^31).
__device__ __forceinline__ uint32_t row_home(int z, int y, uint32_t rmask) {
  uint32_t h = static_cast<uint32_t>(z) * 0x9E3779B1u + static_cast<uint32_t>(y);
  h ^= h >> 16;
  h *= 0x7FEB352Du;
  h ^= h >> 15;
  h *= 0x846CA68Bu;
  h ^= h >> 16;
  return h & rmask;
}

// Row (zq, yq) of the row table: [start, end), or start = -1 if absent.
__device__ __forceinline__ void find_row(const Slot* __restrict__ table, uint32_t rmask, int zq, int yq,
                                         int32_t& start, int32_t& end) {
  start = -1;
  end = -1;
  const unsigned long long rk = row_key(zq, yq);
  uint32_t h = row_home(zq, yq, rmask);
  for (uint32_t probe = 0; probe <= rmask; ++probe) {
    const int4 sl = __ldg(reinterpret_cast<const int4*>(table + h));
    const unsigned long long sk =
        (static_cast<unsigned long long>(static_cast<uint32_t>(sl.y)) << 32) | static_cast<uint32_t>(sl.x);
    if (sk == rk) {
      start = sl.z;
      end = sl.z + sl.w;
      return;
    }
    if (sk == kEmptyKey) return;
    h = (h + 1u) & rmask;
  }
}

// First j in [lo, hi) whose x is >= t (hi if none); x values increase over
// the range (one row of sorted input).
__device__ __forceinline__ int32_t row_lower_bound(const int32_t* __restrict__ xs, int32_t lo, int32_t hi,
                                                   int t) {
  while (lo < hi) {
    const int32_t mid = static_cast<int32_t>((static_cast<uint32_t>(lo) + static_cast<uint32_t>(hi)) >> 1);
    if (__ldg(xs + 3 * static_cast<int64_t>(mid)) < t) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ unsigned long long voxel_key(const int32_t* __restrict__ coords, int64_t j) {
  return pack_coord(__ldg(coords + 3 * j), __ldg(coords + 3 * j + 1), __ldg(coords + 3 * j + 2));
}

// flags[0] := 0 (error and order bits), flags[1] := 0 (row count), the
// bounding box := empty.
__global__ void build_reset_kernel(int* flags) {
  if (threadIdx.x == 0) {
    flags[0] = 0;
    flags[1] = 0;
    flags[kFlagXrunReady] = 0;
    for (int a = 0; a < 3; ++a) {
      flags[kFlagBoxMin + 2 * a] = INT_MAX;
      flags[kFlagBoxMin + 2 * a + 1] = INT_MIN;
    }
  }
}

// The dense row layout of a sorted input's bounding box (see the header).
struct DenseRows {
  int32_t zmin, ymin, xmin;
  int32_t nz, ny, nx;  // box extents
  int32_t wpr;         // occupancy words per row
  uint32_t rows;       // nz * ny
  uint2* words;        // rows * wpr entries {occupancy bits, index of the word's first voxel}
};

// Whether the build takes the dense path (sorted, in range, and the box's
// rows fit in the workspace's table region of table_bytes), and its layout.
// Every kernel decides from the same flag words, so they all agree.
__device__ __forceinline__ bool dense_rows(const int* flags, void* table, unsigned long long table_bytes,
                                           DenseRows* d) {
  if (flags[0] & (kFlagRange | kFlagUnsorted)) return false;
  const int zmin = flags[kFlagBoxMin], zmax = flags[kFlagBoxMin + 1];
  const int ymin = flags[kFlagBoxMin + 2], ymax = flags[kFlagBoxMin + 3];
  const int xmin = flags[kFlagBoxMin + 4], xmax = flags[kFlagBoxMin + 5];
  if (zmax < zmin || ymax < ymin || xmax < xmin) return false;
  const unsigned long long nz = zmax - zmin + 1ull, ny = ymax - ymin + 1ull, nx = xmax - xmin + 1ull;
  const unsigned long long wpr = (nx + 31ull) >> 5;
  const unsigned long long rows = nz * ny;
  if (rows >= (1ull << 31) || rows * wpr >= (1ull << 31)) return false;
  if (rows * wpr * 8ull > table_bytes) return false;
  d->zmin = zmin;
  d->ymin = ymin;
  d->xmin = xmin;
  d->nz = static_cast<int32_t>(nz);
  d->ny = static_cast<int32_t>(ny);
  d->nx = static_cast<int32_t>(nx);
  d->wpr = static_cast<int32_t>(wpr);
  d->rows = static_cast<uint32_t>(rows);
  d->words = static_cast<uint2*>(table);
  return true;
}

// Coordinate range, strict (z, y, x) order and the number of (z, y) rows.
// Verdicts are gathered per block and published with one atomic each.
__global__ void __launch_bounds__(kThreads) order_check_kernel(const int32_t* __restrict__ coords, int64_t n,
                                                               int* flags) {
  __shared__ int bits;
  __shared__ unsigned int rows;
  if (threadIdx.x == 0) {
    bits = 0;
    rows = 0;
  }
  __syncthreads();
  __shared__ int box[6];
  if (threadIdx.x < 6) box[threadIdx.x] = (threadIdx.x & 1) ? INT_MIN : INT_MAX;
  __syncthreads();
  int my_bits = 0;
  unsigned int my_rows = 0;
  int lo[3] = {INT_MAX, INT_MAX, INT_MAX}, hi[3] = {INT_MIN, INT_MIN, INT_MIN};
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int z = __ldg(coords + 3 * i), y = __ldg(coords + 3 * i + 1), x = __ldg(coords + 3 * i + 2);
    if (!in_grid(z) || !in_grid(y) || !in_grid(x)) my_bits |= kFlagRange;
    if (i + 1 < n && !(pack_coord(z, y, x) < voxel_key(coords, i + 1))) my_bits |= kFlagUnsorted;
    if (i == 0 || __ldg(coords + 3 * (i - 1)) != z || __ldg(coords + 3 * (i - 1) + 1) != y) ++my_rows;
    lo[0] = min(lo[0], z);
    hi[0] = max(hi[0], z);
    lo[1] = min(lo[1], y);
    hi[1] = max(hi[1], y);
    lo[2] = min(lo[2], x);
    hi[2] = max(hi[2], x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    my_bits |= __shfl_xor_sync(0xffffffffu, my_bits, off);
    my_rows += __shfl_xor_sync(0xffffffffu, my_rows, off);
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      lo[a] = min(lo[a], __shfl_xor_sync(0xffffffffu, lo[a], off));
      hi[a] = max(hi[a], __shfl_xor_sync(0xffffffffu, hi[a], off));
    }
  }
  if ((threadIdx.x & 31) == 0) {
    if (my_bits) atomicOr(&bits, my_bits);
    if (my_rows) atomicAdd(&rows, my_rows);
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      atomicMin(&box[2 * a], lo[a]);
      atomicMax(&box[2 * a + 1], hi[a]);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (bits) atomicOr(flags, bits);
    if (rows) atomicAdd(reinterpret_cast<unsigned int*>(flags + 1), rows);
  }
  if (threadIdx.x < 6) {
    if (threadIdx.x & 1) {
      if (box[threadIdx.x] != INT_MIN) atomicMax(flags + kFlagBoxMin + threadIdx.x, box[threadIdx.x]);
    } else if (box[threadIdx.x] != INT_MAX) {
      atomicMin(flags + kFlagBoxMin + threadIdx.x, box[threadIdx.x]);
    }
  }
}

// Clears the table and flags, and writes N into the map rows of the offsets
// whose entries come from their opposite's hits (kRoleMirror).
__global__ void hash_clear_kernel(Slot* table, unsigned long long cap, int* flags, int32_t* nmap,
                                  int64_t n, int32_t fill_count, const __grid_constant__ QueryPlan plan) {
  const int f = flags[0];
  if (f & kFlagRange) return;
  const unsigned long long stride = static_cast<unsigned long long>(gridDim.x) * blockDim.x;
  const unsigned long long tid = static_cast<unsigned long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  // whole 16-byte slots (EMPTY key, value -1): full-sector stores
  int4* slots = reinterpret_cast<int4*>(table);
  DenseRows d;
  if (dense_rows(flags, table, cap * sizeof(Slot), &d)) {  // sorted, small box: the dense rows
    const unsigned long long nw = static_cast<unsigned long long>(d.rows) * d.wpr;
    for (unsigned long long i = tid; i < nw; i += stride) d.words[i] = make_uint2(0u, 0u);
    return;
  }
  if (!(f & kFlagUnsorted)) {  // sorted input: only the row table
    const unsigned long long cap_r = row_capacity(static_cast<unsigned int>(flags[1]));
    for (unsigned long long i = tid; i < cap_r; i += stride) slots[i] = make_int4(-1, -1, -1, -1);
    return;
  }
  for (unsigned long long i = tid; i < cap; i += stride) slots[i] = make_int4(-1, -1, -1, -1);
  if (fill_count > 0) {
    const int32_t missing = static_cast<int32_t>(n);
    for (int32_t r = 0, seen = 0; seen < fill_count; ++r) {
      if (plan.role[r] != kRoleMirror) continue;
      ++seen;
      int32_t* row = nmap + static_cast<int64_t>(r) * n;
      for (unsigned long long i = tid; i < static_cast<unsigned long long>(n); i += stride) row[i] = missing;
    }
  }
}

__global__ void hash_insert_kernel(const int32_t* __restrict__ coords, int64_t n, Slot* table,
                                   unsigned long long mask, int* flags) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int f = flags[0];
  if (f & kFlagRange) return;
  DenseRows d;
  if (dense_rows(flags, table, (mask + 1ull) * sizeof(Slot), &d)) {
    // dense rows: every voxel sets its occupancy bit (the voxels of one word
    // and warp combine their bits first: one atomic OR each); the first
    // voxel of each word (the input being sorted, the word's voxels have
    // consecutive indices) writes its index beside the bits
    const bool live = i < n;
    uint32_t word = 0xFFFFFFFFu, bit = 0u;
    if (live) {
      const int z = coords[3 * i], y = coords[3 * i + 1], x = coords[3 * i + 2];
      const uint32_t row = static_cast<uint32_t>(z - d.zmin) * static_cast<uint32_t>(d.ny) +
                           static_cast<uint32_t>(y - d.ymin);
      const uint32_t cx = static_cast<uint32_t>(x - d.xmin);
      word = row * static_cast<uint32_t>(d.wpr) + (cx >> 5);
      bit = 1u << (cx & 31u);
    }
    // the previous voxel's word: from the lane before, or loaded by lane 0
    uint32_t prev_word = __shfl_up_sync(0xffffffffu, word, 1);
    if ((threadIdx.x & 31u) == 0u && live) {
      prev_word = 0xFFFFFFFEu;
      if (i > 0) {
        const int pz = coords[3 * (i - 1)], py = coords[3 * (i - 1) + 1], px = coords[3 * (i - 1) + 2];
        prev_word = (static_cast<uint32_t>(pz - d.zmin) * static_cast<uint32_t>(d.ny) +
                     static_cast<uint32_t>(py - d.ymin)) * static_cast<uint32_t>(d.wpr) +
                    (static_cast<uint32_t>(px - d.xmin) >> 5);
      }
    }
    if (live && prev_word != word) d.words[word].y = static_cast<uint32_t>(i);
    const uint32_t peers = __match_any_sync(0xffffffffu, word);
    const uint32_t bits = __reduce_or_sync(peers, bit);
    if (live && (threadIdx.x & 31u) == static_cast<uint32_t>(__ffs(peers) - 1)) atomicOr(&d.words[word].x, bits);
    return;
  }
  if (i >= n) return;
  const int z = coords[3 * i], y = coords[3 * i + 1], x = coords[3 * i + 2];
  if (!(f & kFlagUnsorted)) {
    // sorted input: the first voxel of each (z, y) row inserts the row
    if (i > 0 && coords[3 * (i - 1)] == z && coords[3 * (i - 1) + 1] == y) return;
    const uint32_t rmask = static_cast<uint32_t>(row_capacity(static_cast<unsigned int>(flags[1])) - 1ull);
    const unsigned long long rk = row_key(z, y);
    uint32_t h = row_home(z, y, rmask);
    for (uint32_t probe = 0; probe <= rmask; ++probe) {
      const unsigned long long prev = atomicCAS(&table[h].key, kEmptyKey, rk);
      if (prev == kEmptyKey) {
        // The row's first voxel and its length: the first index past i whose
        // (z, y) differs, by doubling steps then bisection (once per row).
        int64_t lo = i, hi = n, step = 1;  // row(lo) == (z, y)
        while (true) {
          const int64_t probe = lo + step;
          if (probe >= n) break;
          if (coords[3 * probe] != z || coords[3 * probe + 1] != y) {
            hi = probe;
            break;
          }
          lo = probe;
          step <<= 1;
        }
        while (hi - lo > 1) {  // row(lo) == (z, y); hi == n or row(hi) != (z, y)
          const int64_t mid = lo + (hi - lo) / 2;
          if (coords[3 * mid] == z && coords[3 * mid + 1] == y) lo = mid;
          else hi = mid;
        }
        table[h].val = static_cast<int32_t>(i);
        table[h].pad = static_cast<int32_t>(hi - i);
        return;
      }
      if (prev == rk) {  // a row starting twice: the input was not sorted after all
        atomicOr(flags, kFlagDuplicate);
        return;
      }
      h = (h + 1u) & rmask;
    }
    atomicOr(flags, kFlagFull);
    return;
  }
  if (!in_grid(z) || !in_grid(y) || !in_grid(x)) {
    atomicOr(flags, kFlagRange);
    return;
  }
  const unsigned long long key = pack_coord(z, y, x);
  unsigned long long h = mix_hash(key) & mask;
  for (unsigned long long probe = 0; probe <= mask; ++probe) {
    const unsigned long long prev = atomicCAS(&table[h].key, kEmptyKey, key);
    if (prev == kEmptyKey) {
      table[h].val = static_cast<int32_t>(i);
      return;
    }
    if (prev == key) {
      atomicOr(flags, kFlagDuplicate);
      return;
    }
    h = (h + 1) & mask;
  }
  atomicOr(flags, kFlagFull);
}

// Dense rows: the voxel at (zq, yq, xq) of a row inside the box (`inbox`,
// its words from wbase), or `missing`.
__device__ __forceinline__ int32_t dense_lookup(const DenseRows& d, bool inbox, uint32_t wbase, int xq,
                                               int32_t missing) {
  const uint32_t cx = static_cast<uint32_t>(xq - d.xmin);
  if (!inbox || cx >= static_cast<uint32_t>(d.nx)) return missing;
  const uint2 e = __ldg(d.words + wbase + (cx >> 5));
  const uint32_t b = cx & 31u;
  if (((e.x >> b) & 1u) == 0u) return missing;
  return static_cast<int32_t>(e.y + __popc(e.x & ((1u << b) - 1u)));
}

// Dense rows: the voxels at x - 1, x and x + 1 of one row (cx = x - xmin,
// inside the box), from the occupancy word that holds cx; the word before or
// after it is read only when cx is its first or last bit.
__device__ __forceinline__ void dense_lookup3(const DenseRows& d, bool inbox, uint32_t wbase, uint32_t cx,
                                              int32_t missing, int32_t* left, int32_t* mid, int32_t* right) {
  *left = missing;
  *mid = missing;
  *right = missing;
  if (!inbox) return;
  const uint32_t wi = cx >> 5, b = cx & 31u;
  const uint2 e = __ldg(d.words + wbase + wi);
  const int32_t base = static_cast<int32_t>(e.y);
  const uint32_t own = (e.x >> b) & 1u;
  const int32_t rank = base + __popc(e.x & ((1u << b) - 1u));  // voxels of the row before cx
  if (own) *mid = rank;
  if (b > 0u) {
    if ((e.x >> (b - 1u)) & 1u) *left = rank - 1;
  } else if (wi > 0u) {
    const uint2 f = __ldg(d.words + wbase + wi - 1u);
    if (f.x >> 31) *left = static_cast<int32_t>(f.y) + __popc(f.x) - 1;
  }
  if (b < 31u) {
    if ((e.x >> (b + 1u)) & 1u) *right = rank + static_cast<int32_t>(own);
  } else if (cx + 1u < static_cast<uint32_t>(d.nx)) {
    const uint2 f = __ldg(d.words + wbase + wi + 1u);
    if (f.x & 1u) *right = static_cast<int32_t>(f.y);
  }
}

// Sorted input, dense rows: nmap[k, n] for every offset; for the
// lexicographic 3x3x3 list one occupancy-word load per (dz, dy) row (two at a
// word edge), else one per offset.
// kXFlags (lexicographic 3x3x3 list only): also what the x-run layout
// (xrun.cu) needs of each voxel, from the entries in registers: bit 0 the
// voxel ends a run (no voxel at x + 1), bit 1 one of its nine (dz, dy, +1)
// cells is active, bit 2 one of its nine (dz, dy, -1) cells is active, bit 3
// the voxel ends a run and the cell (z, y, x + 2) is active (then, the input
// being sorted, that cell is the next voxel's).
// Eight blocks per SM (32 registers): the query waits on its loads, so the
// extra warps pay (measured at decoder scale: build 0.606 -> 0.590 ms).
template <bool kStd27, bool kXFlags>
__global__ void __launch_bounds__(kThreads, 8)
    nmap_query_dense_kernel(const int32_t* __restrict__ coords, int64_t n, void* table,
                            unsigned long long table_bytes, int* flags,
                            const __grid_constant__ QueryPlan plan, int32_t* __restrict__ nmap,
                            uint8_t* __restrict__ xflags) {
  static_assert(!kXFlags || kStd27, "x-run flags need the lexicographic 3x3x3 offsets");
  DenseRows d;
  if (!dense_rows(flags, table, table_bytes, &d)) return;
  const int64_t i64 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i64 >= n) return;
  const int32_t i = static_cast<int32_t>(i64);
  const int32_t missing = static_cast<int32_t>(n);
  const int z = __ldg(coords + 3 * static_cast<int64_t>(i)), y = __ldg(coords + 3 * static_cast<int64_t>(i) + 1);
  const int x = __ldg(coords + 3 * static_cast<int64_t>(i) + 2);
  auto row_of = [&](int zq, int yq, bool* inbox, uint32_t* wbase) {
    const uint32_t rz = static_cast<uint32_t>(zq - d.zmin), ry = static_cast<uint32_t>(yq - d.ymin);
    *inbox = rz < static_cast<uint32_t>(d.nz) && ry < static_cast<uint32_t>(d.ny);
    *wbase = *inbox ? (rz * static_cast<uint32_t>(d.ny) + ry) * static_cast<uint32_t>(d.wpr) : 0u;
  };
  if constexpr (kStd27) {
    bool any_left = false, any_right = false, run_end = false, next_at_2 = false;  // kXFlags
#pragma unroll
    for (int dz = -1; dz <= 1; ++dz) {
#pragma unroll
      for (int dy = -1; dy <= 1; ++dy) {
        const int k0 = 9 * (dz + 1) + 3 * (dy + 1);  // offset (dz, dy, -1); +1, +2 follow
        bool in_box;
        uint32_t wbase;
        row_of(z + dz, y + dy, &in_box, &wbase);
        int32_t left, mid, right;
        dense_lookup3(d, in_box, wbase, static_cast<uint32_t>(x - d.xmin), missing, &left, &mid, &right);
        nmap[static_cast<int64_t>(k0) * n + i] = left;
        nmap[static_cast<int64_t>(k0 + 1) * n + i] = (dz == 0 && dy == 0) ? i : mid;
        nmap[static_cast<int64_t>(k0 + 2) * n + i] = right;
        if constexpr (kXFlags) {
          any_left |= left != missing;
          any_right |= right != missing;
          if (dz == 0 && dy == 0) {
            run_end = right == missing;
            // sorted input: after a run end, the next voxel is (z, y, x + 2) when that cell is active
            next_at_2 = run_end && dense_lookup(d, in_box, wbase, x + 2, missing) != missing;
          }
        }
      }
    }
    if constexpr (kXFlags) {
      xflags[i] = static_cast<uint8_t>((run_end ? 1u : 0u) | (any_right ? 2u : 0u) | (any_left ? 4u : 0u) |
                                       (next_at_2 ? 8u : 0u));
      if (blockIdx.x == 0 && threadIdx.x == 0) flags[kFlagXrunReady] = 1;
    }
  } else {
    for (int32_t g = 0; g < plan.groups; ++g) {
      bool in_box;
      uint32_t wbase;
      row_of(z + plan.grp_dz[g], y + plan.grp_dy[g], &in_box, &wbase);
      const int m0 = plan.grp_first[g], m1 = m0 + plan.grp_count[g];
      for (int m = m0; m < m1; ++m)
        nmap[static_cast<int64_t>(plan.mem_k[m]) * n + i] = dense_lookup(d, in_box, wbase, x + plan.mem_dx[m], missing);
    }
  }
}

// Sorted input: nmap[k, n] for every offset, by row probe + search.  The
// loop is short on instructions (this kernel is issue-bound): 32-bit
// indices, a 32-bit row hash, and for the lexicographic 3x3x3 offset list
// (kStd27) everything unrolled: per (dz, dy) row one probe, one bisection
// for x - 1, then direct checks for x and x + 1; the voxel's own row needs
// no probe (x - 1 and x + 1 can only be its neighbours in the array).
template <bool kStd27>
__global__ void __launch_bounds__(kThreads)
    nmap_query_rows_kernel(const int32_t* __restrict__ coords, int64_t n, const Slot* __restrict__ table,
                           unsigned long long table_bytes, const int* __restrict__ flags,
                           const __grid_constant__ QueryPlan plan, int32_t* __restrict__ nmap) {
  const int f = flags[0];
  if (f & (kFlagRange | kFlagUnsorted)) return;
  DenseRows dr;
  if (dense_rows(flags, const_cast<Slot*>(table), table_bytes, &dr)) return;  // the dense query runs
  // grid-stride over the voxels: a small grid, so that the launch costs
  // little on the builds that take another path
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i64 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i64 < n; i64 += stride) {
  const int32_t i = static_cast<int32_t>(i64);  // N < 2^31 - 1
  const int32_t n32 = static_cast<int32_t>(n);
  const uint32_t rmask = static_cast<uint32_t>(row_capacity(static_cast<unsigned int>(flags[1])) - 1ull);
  const int32_t* xs = coords + 2;
  const int z = __ldg(coords + 3 * static_cast<int64_t>(i)), y = __ldg(coords + 3 * static_cast<int64_t>(i) + 1);
  const int x = __ldg(xs + 3 * static_cast<int64_t>(i));
  const int32_t missing = n32;
  if constexpr (kStd27) {
#pragma unroll
    for (int dz = -1; dz <= 1; ++dz) {
#pragma unroll
      for (int dy = -1; dy <= 1; ++dy) {
        const int k0 = 9 * (dz + 1) + 3 * (dy + 1);  // offset (dz, dy, -1); +1, +2 follow
        int32_t r0 = missing, r1 = missing, r2 = missing;
        if (dz == 0 && dy == 0) {
          r1 = i;
          if (i > 0 && __ldg(xs + 3 * static_cast<int64_t>(i - 1)) == x - 1 &&
              __ldg(coords + 3 * static_cast<int64_t>(i - 1)) == z &&
              __ldg(coords + 3 * static_cast<int64_t>(i - 1) + 1) == y)
            r0 = i - 1;
          if (i + 1 < n32 && __ldg(xs + 3 * static_cast<int64_t>(i + 1)) == x + 1 &&
              __ldg(coords + 3 * static_cast<int64_t>(i + 1)) == z &&
              __ldg(coords + 3 * static_cast<int64_t>(i + 1) + 1) == y)
            r2 = i + 1;
        } else {
          const int zq = z + dz, yq = y + dy;
          int32_t start = -1, end = -1;
          if (in_grid(zq) && in_grid(yq)) find_row(table, rmask, zq, yq, start, end);
          if (start >= 0) {
            int32_t j = row_lower_bound(xs, start, end, x - 1);
            int xj = j < end ? __ldg(xs + 3 * static_cast<int64_t>(j)) : INT_MAX;
            if (xj == x - 1) {
              r0 = j++;
              xj = j < end ? __ldg(xs + 3 * static_cast<int64_t>(j)) : INT_MAX;
            }
            if (xj == x) {
              r1 = j++;
              xj = j < end ? __ldg(xs + 3 * static_cast<int64_t>(j)) : INT_MAX;
            }
            if (xj == x + 1) r2 = j;
          }
        }
        nmap[static_cast<int64_t>(k0) * n + i] = r0;
        nmap[static_cast<int64_t>(k0 + 1) * n + i] = r1;
        nmap[static_cast<int64_t>(k0 + 2) * n + i] = r2;
      }
    }
  } else {
    for (int32_t g = 0; g < plan.groups; ++g) {
      const int zq = z + plan.grp_dz[g], yq = y + plan.grp_dy[g];
      const int m0 = plan.grp_first[g], m1 = m0 + plan.grp_count[g];
      int32_t start = -1, end = -1;
      if (in_grid(zq) && in_grid(yq)) find_row(table, rmask, zq, yq, start, end);
      // Members come in ascending dx: each search starts where the last ended.
      int32_t cur = start;
      for (int m = m0; m < m1; ++m) {
        int32_t found = missing;
        if (start >= 0 && cur < end) {
          const int xq = x + plan.mem_dx[m];
          cur = row_lower_bound(xs, cur, end, xq);
          if (cur < end && __ldg(xs + 3 * static_cast<int64_t>(cur)) == xq) found = cur;
        }
        nmap[static_cast<int64_t>(plan.mem_k[m]) * n + i] = found;
      }
    }
  }
  }
}

// Any other input order: hash probes (one offset of each opposite pair).
__global__ void __launch_bounds__(kThreads)
    nmap_query_kernel(const int32_t* __restrict__ coords, int64_t n, const Slot* __restrict__ table,
                      unsigned long long mask, const int* __restrict__ flags,
                      const __grid_constant__ QueryPlan plan, int32_t k_count, int32_t* __restrict__ nmap) {
  const int f = flags[0];
  if ((f & kFlagRange) || !(f & kFlagUnsorted)) return;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;  // small grid, as above
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
  const int z = coords[3 * i], y = coords[3 * i + 1], x = coords[3 * i + 2];
  const int32_t missing = static_cast<int32_t>(n);
  for (int32_t k = 0; k < k_count; ++k) {
    const int8_t role = plan.role[k];
    if (role == kRoleMirror) continue;
    int32_t found = missing;
    if (role == kRoleSelf) {
      found = static_cast<int32_t>(i);
    } else {
      const int qz = z + plan.d[3 * k], qy = y + plan.d[3 * k + 1], qx = x + plan.d[3 * k + 2];
      if (in_grid(qz) && in_grid(qy) && in_grid(qx)) {
        const unsigned long long key = pack_coord(qz, qy, qx);
        unsigned long long h = mix_hash(key) & mask;
        for (unsigned long long probe = 0; probe <= mask; ++probe) {
          const int4 s = __ldg(reinterpret_cast<const int4*>(table + h));
          const unsigned long long sk =
              (static_cast<unsigned long long>(static_cast<uint32_t>(s.y)) << 32) |
              static_cast<uint32_t>(s.x);
          if (sk == key) {
            found = s.z;
            break;
          }
          if (sk == kEmptyKey) break;
          h = (h + 1) & mask;
        }
      }
      const int16_t mk = plan.mirror[k];
      if (mk >= 0 && found != missing) nmap[static_cast<int64_t>(mk) * n + found] = static_cast<int32_t>(i);
    }
    nmap[static_cast<int64_t>(k) * n + i] = found;
  }
  }
}

__global__ void count_valid_kernel(const int32_t* __restrict__ nmap, int64_t total, int64_t n,
                                   unsigned long long* count) {
  unsigned long long local = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int32_t v = nmap[i];
    local += (v >= 0 && v < n) ? 1u : 0u;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) local += __shfl_down_sync(0xffffffffu, local, off);
  if ((threadIdx.x & 31) == 0 && local != 0) atomicAdd(count, local);
}

__global__ void zero_u64_kernel(unsigned long long* p) { *p = 0; }

// Tile order: within each chunk of kTileOrderChunk consecutive voxels, the
// voxels sorted by their neighbour mask (bit k set when nmap[k, n] is a
// neighbour, for the first 32 offsets), ties by index.  Tiles then hold
// voxels with like masks, so fewer of a tile's gathered rows are empty;
// chunks keep the tiles spatially local.  One block per chunk: the keys
// (mask, index) are sorted in shared memory with a bitonic network.
constexpr int kOrderThreads = 1024;

__global__ void __launch_bounds__(kOrderThreads)
    tile_order_kernel(const int32_t* __restrict__ nmap, int64_t n, int32_t k, int32_t* __restrict__ order) {
  __shared__ unsigned long long keys[kTileOrderChunk];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kTileOrderChunk;
  const int count = static_cast<int>(n - base < kTileOrderChunk ? n - base : kTileOrderChunk);
  const int kk = k < 32 ? k : 32;
  for (int t = threadIdx.x; t < kTileOrderChunk; t += kOrderThreads) {
    unsigned long long key = ~0ull;  // padding sorts last
    if (t < count) {
      uint32_t mask = 0;
      for (int j = 0; j < kk; ++j) {
        const int32_t v = __ldg(nmap + static_cast<int64_t>(j) * n + base + t);
        mask |= (v >= 0 && v < n ? 1u : 0u) << j;
      }
      key = (static_cast<unsigned long long>(mask) << 32) | static_cast<unsigned int>(t);
    }
    keys[t] = key;
  }
  __syncthreads();
  for (int size = 2; size <= kTileOrderChunk; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < kTileOrderChunk / 2; t += kOrderThreads) {
        const int i = 2 * t - (t & (stride - 1));  // first element of pair t
        const int j = i + stride;
        const unsigned long long a = keys[i], b = keys[j];
        if ((a > b) == ((i & size) == 0)) {  // ascending where bit `size` of i is 0
          keys[i] = b;
          keys[j] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int t = threadIdx.x; t < count; t += kOrderThreads)
    order[base + t] = static_cast<int32_t>(base + static_cast<int64_t>(keys[t] & 0xFFFFFFFFull));
}

}  // namespace

const int* xrun_flags_ready(const void* workspace) {
  return static_cast<const int*>(workspace) + kFlagXrunReady;
}

size_t hash_capacity(int64_t n) {
  size_t cap = 64;
  while (cap < static_cast<size_t>(2 * n)) cap <<= 1;
  return cap;
}

namespace {
// The build's error flags as a status code (the precedence of the host-side
// check: coordinate range, then duplicates, then table overflow).
__global__ void flags_to_status_kernel(const int* flags, int32_t* status) {
  if (threadIdx.x != 0) return;
  const int f = *flags;
  *status = (f & kFlagRange) ? SPCONV_ERR_INVALID_ARG
            : (f & kFlagDuplicate) ? SPCONV_ERR_DUPLICATE_COORD
            : (f & kFlagFull) ? SPCONV_ERR_DEVICE
                              : SPCONV_OK;
}
}  // namespace

spconv_status launch_build_nmap(const int32_t* coords, int64_t n, const BuildOffsets& offs,
                                int32_t k, int32_t* nmap, void* workspace, cudaStream_t stream,
                                int32_t* status_dev, uint8_t* xflags) {
  const size_t cap = hash_capacity(n);
  int* flags = static_cast<int*>(workspace);
  Slot* table = reinterpret_cast<Slot*>(static_cast<char*>(workspace) + kFlagBytes);
  const int sms = sm_count();
  if (sms <= 0) return fail(SPCONV_ERR_CUDA, "could not query the SM count");
  spconv_status st = SPCONV_OK;

  const unsigned long long clear_blocks = (cap + kThreads - 1) / kThreads;
  const unsigned clear_grid =
      static_cast<unsigned>(clear_blocks < 16ull * sms ? clear_blocks : 16ull * sms);
  QueryPlan plan;
  int32_t fill_count = 0;
  for (int32_t a = 0; a < k; ++a) {
    plan.d[3 * a] = offs.d[3 * a];
    plan.d[3 * a + 1] = offs.d[3 * a + 1];
    plan.d[3 * a + 2] = offs.d[3 * a + 2];
    plan.mirror[a] = -1;
    plan.role[a] = -1;
  }
  for (int32_t a = 0; a < k; ++a) {
    if (plan.role[a] >= 0) continue;  // already the mirror of an earlier offset
    const int32_t* da = plan.d + 3 * a;
    if (da[0] == 0 && da[1] == 0 && da[2] == 0) {
      plan.role[a] = kRoleSelf;
      continue;
    }
    plan.role[a] = kRoleProbe;
    for (int32_t b = a + 1; b < k; ++b) {
      const int32_t* db = plan.d + 3 * b;
      if (plan.role[b] < 0 && db[0] == -da[0] && db[1] == -da[1] && db[2] == -da[2]) {
        plan.mirror[a] = static_cast<int16_t>(b);
        plan.role[b] = kRoleMirror;
        ++fill_count;
        break;
      }
    }
  }
  // Sorted-input path: offsets grouped by (dz, dy), members by ascending dx.
  plan.groups = 0;
  {
    int32_t grp_of[SPCONV_MAX_BUILD_OFFSETS];
    int32_t counts[SPCONV_MAX_BUILD_OFFSETS] = {};
    for (int32_t a = 0; a < k; ++a) {
      int32_t g = 0;
      while (g < plan.groups && !(plan.grp_dz[g] == offs.d[3 * a] && plan.grp_dy[g] == offs.d[3 * a + 1])) ++g;
      if (g == plan.groups) {
        plan.grp_dz[g] = offs.d[3 * a];
        plan.grp_dy[g] = offs.d[3 * a + 1];
        ++plan.groups;
      }
      grp_of[a] = g;
      ++counts[g];
    }
    int32_t first = 0;
    for (int32_t g = 0; g < plan.groups; ++g) {
      plan.grp_first[g] = static_cast<int16_t>(first);
      plan.grp_count[g] = 0;
      first += counts[g];
    }
    for (int32_t a = 0; a < k; ++a) {  // insertion in ascending dx within the group
      const int32_t g = grp_of[a];
      int32_t pos = plan.grp_first[g] + plan.grp_count[g];
      const int32_t dx = offs.d[3 * a + 2];
      while (pos > plan.grp_first[g] && plan.mem_dx[pos - 1] > dx) {
        plan.mem_dx[pos] = plan.mem_dx[pos - 1];
        plan.mem_k[pos] = plan.mem_k[pos - 1];
        --pos;
      }
      plan.mem_dx[pos] = dx;
      plan.mem_k[pos] = static_cast<int16_t>(a);
      ++plan.grp_count[g];
    }
  }

  const unsigned grid = static_cast<unsigned>((n + kThreads - 1) / kThreads);
  const unsigned check_grid = grid < 16u * static_cast<unsigned>(sms) ? grid : 16u * static_cast<unsigned>(sms);
  build_reset_kernel<<<1, 32, 0, stream>>>(flags);
  if (!cuda_ok(cudaGetLastError(), "build_reset_kernel launch", &st)) return st;
  order_check_kernel<<<check_grid, kThreads, 0, stream>>>(coords, n, flags);
  if (!cuda_ok(cudaGetLastError(), "order_check_kernel launch", &st)) return st;

  hash_clear_kernel<<<clear_grid, kThreads, 0, stream>>>(table, cap, flags, nmap, n, fill_count,
                                                         plan);
  if (!cuda_ok(cudaGetLastError(), "hash_clear_kernel launch", &st)) return st;

  hash_insert_kernel<<<grid, kThreads, 0, stream>>>(coords, n, table, cap - 1, flags);
  if (!cuda_ok(cudaGetLastError(), "hash_insert_kernel launch", &st)) return st;

  // Dense-row path (sorted input, small box): the query; it returns at
  // once on the other paths.
  const unsigned long long table_bytes = static_cast<unsigned long long>(cap) * sizeof(Slot);
  bool std27 = k == 27;
  for (int32_t a = 0; a < k && std27; ++a)
    std27 = offs.d[3 * a] == a / 9 - 1 && offs.d[3 * a + 1] == (a / 3) % 3 - 1 && offs.d[3 * a + 2] == a % 3 - 1;
  if (std27 && xflags != nullptr)
    nmap_query_dense_kernel<true, true><<<grid, kThreads, 0, stream>>>(coords, n, table, table_bytes, flags, plan,
                                                                       nmap, xflags);
  else if (std27)
    nmap_query_dense_kernel<true, false><<<grid, kThreads, 0, stream>>>(coords, n, table, table_bytes, flags, plan,
                                                                        nmap, nullptr);
  else
    nmap_query_dense_kernel<false, false><<<grid, kThreads, 0, stream>>>(coords, n, table, table_bytes, flags,
                                                                         plan, nmap, nullptr);
  if (!cuda_ok(cudaGetLastError(), "nmap_query_dense_kernel launch", &st)) return st;

  // the row-hash and voxel-hash queries: grid-stride kernels on at most 16
  // blocks per SM (cheap when their path is not taken)
  const unsigned small_grid = grid < 16u * static_cast<unsigned>(sms) ? grid : 16u * static_cast<unsigned>(sms);
  if (std27)
    nmap_query_rows_kernel<true><<<small_grid, kThreads, 0, stream>>>(coords, n, table, table_bytes, flags, plan, nmap);
  else
    nmap_query_rows_kernel<false><<<small_grid, kThreads, 0, stream>>>(coords, n, table, table_bytes, flags, plan, nmap);
  if (!cuda_ok(cudaGetLastError(), "nmap_query_rows_kernel launch", &st)) return st;
  nmap_query_kernel<<<small_grid, kThreads, 0, stream>>>(coords, n, table, cap - 1, flags, plan, k, nmap);
  if (!cuda_ok(cudaGetLastError(), "nmap_query_kernel launch", &st)) return st;

  if (status_dev != nullptr) {
    // Asynchronous form: the verdict goes to device memory, no host wait.
    flags_to_status_kernel<<<1, 32, 0, stream>>>(flags, status_dev);
    if (!cuda_ok(cudaGetLastError(), "flags_to_status_kernel launch", &st)) return st;
    return SPCONV_OK;
  }
  int host_flags = 0;
  if (!cuda_ok(cudaMemcpyAsync(&host_flags, flags, sizeof(int), cudaMemcpyDeviceToHost, stream),
               "flag readback", &st))
    return st;
  if (!cuda_ok(cudaStreamSynchronize(stream), "cudaStreamSynchronize", &st)) return st;
  if (host_flags & kFlagRange)
    return fail(SPCONV_ERR_INVALID_ARG, "a coordinate lies outside [0, 2^20)");
  if (host_flags & kFlagDuplicate)
    return fail(SPCONV_ERR_DUPLICATE_COORD, "two voxels share a coordinate");
  if (host_flags & kFlagFull) return fail(SPCONV_ERR_DEVICE, "hash table overflow");
  return SPCONV_OK;
}

spconv_status launch_tile_order(const int32_t* nmap, int64_t n, int32_t k, int32_t* order,
                                cudaStream_t stream) {
  spconv_status st = SPCONV_OK;
  if (n == 0) return SPCONV_OK;
  const int64_t chunks = (n + kTileOrderChunk - 1) / kTileOrderChunk;
  tile_order_kernel<<<static_cast<unsigned>(chunks), kOrderThreads, 0, stream>>>(nmap, n, k, order);
  if (!cuda_ok(cudaGetLastError(), "tile_order_kernel launch", &st)) return st;
  return SPCONV_OK;
}

spconv_status launch_count_valid_pairs(const int32_t* nmap, int64_t n, int32_t k, int64_t* count,
                                       cudaStream_t stream) {
  spconv_status st = SPCONV_OK;
  unsigned long long* c = reinterpret_cast<unsigned long long*>(count);
  zero_u64_kernel<<<1, 1, 0, stream>>>(c);
  if (!cuda_ok(cudaGetLastError(), "zero kernel launch", &st)) return st;
  const int64_t total = static_cast<int64_t>(k) * n;
  if (total == 0) return SPCONV_OK;
  const int sms = sm_count();
  if (sms <= 0) return fail(SPCONV_ERR_CUDA, "could not query the SM count");
  const int64_t blocks = (total + kThreads - 1) / kThreads;
  const unsigned grid = static_cast<unsigned>(blocks < 8ll * sms ? blocks : 8ll * sms);
  count_valid_kernel<<<grid, kThreads, 0, stream>>>(nmap, total, n, c);
  if (!cuda_ok(cudaGetLastError(), "count_valid_kernel launch", &st)) return st;
  return SPCONV_OK;
}

// ------------------------------------------------------------------------
// Allocation-free variant.  Some callers cannot allocate device memory at
// the point where they need a neighbour map (for example code running inside
// a host framework that owns every device allocation, or a fixed-budget
// deployment that forbids allocations after start-up).  For them the hash
// table lives in one file-scope device array of fixed size instead of a
// caller-provided workspace.  The array takes 32 MiB + 256 B on each device
// where this library's module is loaded, until the process exits.
namespace {

constexpr size_t kNoAllocBytes = kFlagBytes + 2 * static_cast<size_t>(SPCONV_NOALLOC_MAX_VOXELS) * 16;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

}  // namespace

spconv_status noalloc_scratch(void** scratch) {
  // Host code only has a stand-in for the array's name; its device address
  // comes from the runtime, for the current device.  It is looked up on
  // every call (cheap next to the build, which waits for its stream): a
  // cached address would go stale if the device's context were reset and
  // the module loaded again elsewhere.
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess)
    return fail(SPCONV_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
  *scratch = p;
  return SPCONV_OK;
}

}  // namespace spconv

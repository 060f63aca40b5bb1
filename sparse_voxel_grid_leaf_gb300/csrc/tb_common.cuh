// Shared definitions of the batched topology pass (host + device).
//
// The pass follows fVDB PR #757 ("Batched leaf-mask topology construction for
// generated conv grids", Summary item 1): an emission kernel over all source
// leaves of all grids writes candidate output-leaf slots, a segmented radix
// sort puts them in canonical node order, a head-flag scan dedups them and
// derives per-grid counts and parent linkage, one readback sizes the outputs,
// and batched writers emit the leaf records.
//
// Slots carry a 64-bit canonical key and a 32-bit source reference only; the
// 512-bit output masks are recomputed from the source masks by the writer,
// which keeps the sort payload at 12 bytes per slot.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace tb {

// Pass kinds.  kIjk and kLeaves are the front ends (one slot per input voxel
// or input leaf); the other three are the topology ops of the chain.
enum PassOp : int32_t { kIjk = 0, kLeaves = 1, kRefine = 2, kCoarsen = 3, kDilate = 4 };

constexpr int kBins = 256;            // 8-bit radix digits
constexpr int kMaxDigitPasses = 8;    // 64-bit key
constexpr int kSrcShift = 5;          // slot value = source index << 5 | target code

// Error bits reported through the readback header.
constexpr uint32_t kErrTimeout = 1u;       // a bounded look-back wait gave up
constexpr uint32_t kErrBadOffsets = 2u;    // jagged offsets not monotone / not covering
constexpr uint32_t kErrNotAligned = 4u;    // a leaf origin is not a multiple of 8
constexpr uint32_t kErrNotCanonical = 8u;  // tb_validate: order or mask violation
constexpr uint32_t kErrSlotOverflow = 16u; // emission exceeded the host's bound (bug guard)

// Look-back status words: two flag bits on top of the value.
constexpr uint32_t kFlagA32 = 1u << 30, kFlagP32 = 2u << 30, kVal32 = (1u << 30) - 1;
constexpr uint64_t kFlagA64 = 1ull << 62, kFlagP64 = 2ull << 62, kSeg64 = 1ull << 61,
                   kVal64 = (1ull << 61) - 1;
constexpr uint32_t kSpinLimit = 1u << 22;  // about 0.1-1 s of polling

// Compressed canonical sort key.  Field order from the most significant bit:
// grid | tile x | tile y | tile z | upper x | upper y | upper z | lower x |
// lower y | lower z, where for leaf coordinate lc = origin >> 3 the tile is
// lc >> 9 (offset by the batch minimum), the upper child offset is
// (lc >> 4) & 31 and the lower child offset is lc & 15.  Bits that are
// constant over the batch's coordinate range are dropped; the order of the
// remaining fields is the canonical order.
struct KeyLayout {
  int32_t W;             // total key width in bits (<= 64)
  int32_t gw, gshift;    // grid field
  int32_t tile_base[3];  // minimum tile coordinate per axis
  int32_t tw[3];         // tile field widths
  int32_t uw[3];         // upper-offset field widths (0..5)
  int32_t lwl[3];        // lower-offset field widths (0..4)
  int32_t tshift[3], ushift[3], lshift[3];
  int32_t lc_const[3];   // leaf-coordinate bits 0..8 that are constant and dropped
  int32_t lower_bits;    // key >> lower_bits                 == (grid, tile, upper offset)
  int32_t node_bits;     // key >> (lower_bits + upper bits)  == (grid, tile)
};

// Host-visible part of a pass's control block (read back in one copy,
// followed by leaf/lower/upper offsets [B+1] each).
struct ReadbackHeader {
  unsigned long long num_slots;
  unsigned long long num_leaves;
  unsigned long long num_lowers;
  unsigned long long num_uppers;
  unsigned int err;
  unsigned int pad;
  unsigned int bbox_enc[6];  // order-preserving encodings (see enc_min / enc_max)
};
static_assert(sizeof(ReadbackHeader) == 64, "readback header layout");

// Device-only counters and histograms of one pass (zeroed at call start).
struct PassCtl {
  unsigned int emit_ticket;
  unsigned int dedup_tile_ctr;
  unsigned int dedup_ticket;
  unsigned int write_tile_ctr;
  unsigned int write_ticket;
  unsigned int pad[3];
  unsigned int sort_tile_ctr[kMaxDigitPasses];
  unsigned long long head_totals[4];
  unsigned int hist[kMaxDigitPasses][kBins];
  unsigned int bin_base[kMaxDigitPasses][kBins];
};

// Order-preserving encodings for atomicMax-based min/max on zero-initialised
// memory: enc_max(x) orders like x and enc_max(INT32_MIN) == 0; enc_min(x)
// orders like -x and enc_min(INT32_MAX) == 0.
__host__ __device__ inline unsigned int enc_max(int32_t x) { return (unsigned int)x ^ 0x80000000u; }
__host__ __device__ inline unsigned int enc_min(int32_t x) { return ~((unsigned int)x ^ 0x80000000u); }
__host__ __device__ inline int32_t dec_max(unsigned int e) { return (int32_t)(e ^ 0x80000000u); }
__host__ __device__ inline int32_t dec_min(unsigned int e) { return (int32_t)(~e ^ 0x80000000u); }

// ---------------------------------------------------------------- pass arguments

struct PassArgs {
  KeyLayout K;
  int32_t B;
  int32_t P;              // digit passes
  int32_t lo[3], hi[3];   // box of a dilation pass
  // source
  const int32_t* ijk;            // kIjk: [N,3]
  const int64_t* in_offsets;     // kIjk / kLeaves without leaf_grid: [B+1]
  const int32_t* src_origins;    // [L,3]
  const uint64_t* src_masks;     // [L,8]
  const int32_t* src_grid;       // [L] or null
  const unsigned long long* src_count_dev;  // device count (chained pass) or null
  long long src_count;                      // host count when src_count_dev is null
  // control
  ReadbackHeader* rb;
  int64_t* leaf_off;   // [B+1]
  int64_t* lower_off;  // [B+1]
  int64_t* upper_off;  // [B+1]
  PassCtl* ctl;
  long long slot_cap;
  // sort buffers
  uint64_t* keys[2];
  uint32_t* vals[2];
  uint32_t* sort_status;   // [P][sort_tiles_cap][256]
  long long sort_tiles_cap;
  unsigned long long* dedup_status;  // [dedup_tiles_cap][3]
  unsigned long long* write_status;  // [write_tiles_cap]
  uint32_t* first;       // [3][B]: 1 + first leaf / lower / upper index of each grid
  uint32_t* run_start;   // [slot_cap + 1]
  uint32_t* leaf_lower;  // [slot_cap]
  uint32_t* leaf_upper;  // [slot_cap]
  unsigned int* gbox;    // [B][6] encoded grid bbox accumulators
  int32_t sorted;        // which keys/vals buffer holds the sorted slots
};

// Outputs of a writer: the final batch arrays, or the next pass's source.
struct WriteOut {
  int32_t* origins;
  uint64_t* masks;
  int32_t* leaf_grid;
  // final only
  int64_t* voxel_offset;
  uint64_t* word_prefix;
  int32_t* leaf_bbox;
  int32_t* leaf_parent;
  int64_t* voxel_counts;
  int32_t* grid_bbox;
  int32_t* node_counts;
  int64_t* leaf_offsets;
  int64_t* lower_offsets;
  int64_t* upper_offsets;
  int32_t* lower_origins;
  int32_t* lower_parent;
  int32_t* upper_origins;
};

#ifdef __CUDACC__

// ---------------------------------------------------------------- memory helpers

__device__ __forceinline__ uint64_t ld_relaxed(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void load_mask(const uint64_t* masks, long long i, uint64_t m[8]) {
  const uint4* p = reinterpret_cast<const uint4*>(masks + 8 * i);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 v = __ldg(p + q);
    m[2 * q] = (uint64_t)v.x | ((uint64_t)v.y << 32);
    m[2 * q + 1] = (uint64_t)v.z | ((uint64_t)v.w << 32);
  }
}

// ---------------------------------------------------------------- keys

__device__ __forceinline__ uint64_t shr64(uint64_t x, int s) { return s >= 64 ? 0ull : (x >> s); }

__device__ __forceinline__ uint64_t encode_key(const KeyLayout& K, uint32_t g, int32_t lcx, int32_t lcy,
                                               int32_t lcz) {
  const int32_t lc[3] = {lcx, lcy, lcz};
  uint64_t key = K.gw ? ((uint64_t)g << K.gshift) : 0ull;
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    const uint32_t t = (uint32_t)((lc[a] >> 9) - K.tile_base[a]);
    if (K.tw[a]) key |= (uint64_t)t << K.tshift[a];
    key |= (uint64_t)(((uint32_t)lc[a] >> 4) & ((1u << K.uw[a]) - 1u)) << K.ushift[a];
    key |= (uint64_t)((uint32_t)lc[a] & ((1u << K.lwl[a]) - 1u)) << K.lshift[a];
  }
  return key;
}

__device__ __forceinline__ void decode_key(const KeyLayout& K, uint64_t key, uint32_t& g, int32_t lc[3]) {
  g = K.gw ? (uint32_t)(key >> K.gshift) : 0u;
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    const uint32_t t = K.tw[a] ? (uint32_t)((key >> K.tshift[a]) & ((1ull << K.tw[a]) - 1ull)) : 0u;
    const uint32_t u = (uint32_t)(key >> K.ushift[a]) & ((1u << K.uw[a]) - 1u);
    const uint32_t l = (uint32_t)(key >> K.lshift[a]) & ((1u << K.lwl[a]) - 1u);
    const uint32_t tile = (uint32_t)K.tile_base[a] + t;
    lc[a] = (int32_t)((tile << 9) | (uint32_t)K.lc_const[a] | (u << 4) | l);
  }
}

// ---------------------------------------------------------------- leaf mask arithmetic
// Mask word w holds the voxels with local x == w; bit 8*y + z.

// Refinement by 2: word w of child c = (cx, cy, cz) of a leaf is built from
// parent word 4*cx + (w >> 1): parent rows 4*cy .. 4*cy+3, bits 4*cz .. 4*cz+3,
// each parent bit doubled in z and each row doubled in y.
__device__ __forceinline__ uint64_t refine_word(uint64_t parent_word, int cy, int cz) {
  uint64_t out = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    uint32_t x = (uint32_t)(parent_word >> (8 * (4 * cy + r) + 4 * cz)) & 0xFu;
    x = (x | (x << 2)) & 0x33u;
    x = (x | (x << 1)) & 0x55u;
    x = x | (x << 1);
    const uint64_t row = (uint64_t)x;
    out |= (row | (row << 8)) << (16 * r);
  }
  return out;
}

// Coarsening by 2: t = OR of the two source words 2X', 2X'+1 that fall into
// coarse x (X' in 0..3).  Rows and bits are OR-ed pairwise and compacted into
// coarse rows 4*qy .. 4*qy+3, bits 4*qz .. 4*qz+3 (q = source leaf's octant
// inside the coarse leaf).
__device__ __forceinline__ uint64_t coarsen_word(uint64_t t, int qy, int qz) {
  uint64_t r = t | (t >> 8);
  r = r | (r >> 1);
  r &= 0x0055005500550055ull;
  r = (r | (r >> 1)) & 0x0033003300330033ull;
  r = (r | (r >> 2)) & 0x000F000F000F000Full;
  uint64_t out = 0;
#pragma unroll
  for (int Y = 0; Y < 4; ++Y) out |= ((r >> (16 * Y)) & 0xFull) << (8 * (4 * qy + Y) + 4 * qz);
  return out;
}

// Box dilation restricted to one target leaf offset: the z part (bits within
// a row) and the y part (rows within a word) for target offset t in {-1,0,1}.
__device__ __forceinline__ uint64_t dilate_z(uint64_t s, int tz, int lo, int hi) {
  if (tz == 0) {
    uint64_t r = s;
    if (hi > 0) r |= (s << 1) & 0xFEFEFEFEFEFEFEFEull;
    if (lo < 0) r |= (s >> 1) & 0x7F7F7F7F7F7F7F7Full;
    return r;
  }
  if (tz > 0) return (s >> 7) & 0x0101010101010101ull;  // z = 7 moves to z = 0 of the next leaf
  return (s << 7) & 0x8080808080808080ull;              // z = 0 moves to z = 7 of the previous leaf
}
__device__ __forceinline__ uint64_t dilate_y(uint64_t s, int ty, int lo, int hi) {
  if (ty == 0) {
    uint64_t r = s;
    if (hi > 0) r |= s << 8;
    if (lo < 0) r |= s >> 8;
    return r;
  }
  if (ty > 0) return s >> 56;  // row 7 moves to row 0 of the next leaf
  return s << 56;              // row 0 moves to row 7 of the previous leaf
}

// ---------------------------------------------------------------- scans and look-back

// Exclusive scan over a 256-thread block; returns the thread's exclusive
// prefix and writes the block total to *total.  `scratch` holds 8 words.
template <typename T>
__device__ __forceinline__ T block_excl_scan_256(T v, T* scratch, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  T warp_base = 0, all = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const T s = scratch[w];
    if (w < warp) warp_base += s;
    all += s;
  }
  __syncthreads();
  *total = all;
  return warp_base + incl - v;
}

// Decoupled look-back over 32-bit status words (one per tile).  Publishes
// the tile's aggregate, accumulates predecessors until an inclusive prefix is
// found, then publishes the tile's inclusive prefix.  Returns the exclusive
// prefix.  A wait on a tile that never publishes ends after kSpinLimit polls
// with kErrTimeout set.
__device__ __forceinline__ uint32_t lookback32(uint32_t* status, long long stride, long long tile,
                                               uint32_t agg, unsigned int* err) {
  if (tile == 0) {
    st_relaxed(status, kFlagP32 | agg);
    return 0;
  }
  st_relaxed(status + tile * stride, kFlagA32 | agg);
  uint32_t excl = 0;
  long long t = tile - 1;
  uint32_t spins = 0;
  while (t >= 0) {
    const uint32_t w = ld_relaxed(status + t * stride);
    const uint32_t f = w & ~kVal32;
    if (f == 0) {
      if (++spins > kSpinLimit) {
        atomicOr(err, kErrTimeout);
        break;
      }
      __nanosleep(32);
      continue;
    }
    excl += w & kVal32;
    if (f == kFlagP32) break;
    --t;
  }
  st_relaxed(status + tile * stride, kFlagP32 | (excl + agg));
  return excl;
}

// Same on 64-bit words; with `seg` the scan is segmented: an aggregate that
// contains a segment head stops the walk (its value is the sum since that head).
__device__ __forceinline__ uint64_t lookback64(unsigned long long* status, long long stride, long long tile,
                                               uint64_t agg, bool has_head, unsigned int* err) {
  const uint64_t seg = has_head ? kSeg64 : 0ull;
  if (tile == 0) {
    st_relaxed(status, kFlagP64 | agg);
    return 0;
  }
  st_relaxed(status + tile * stride, kFlagA64 | seg | agg);
  uint64_t excl = 0;
  long long t = tile - 1;
  uint32_t spins = 0;
  while (t >= 0) {
    const uint64_t w = ld_relaxed(status + t * stride);
    const uint64_t f = w & (3ull << 62);
    if (f == 0) {
      if (++spins > kSpinLimit) {
        atomicOr(err, kErrTimeout);
        break;
      }
      __nanosleep(32);
      continue;
    }
    excl += w & kVal64;
    if (f == kFlagP64 || (w & kSeg64)) break;
    --t;
  }
  st_relaxed(status + tile * stride, kFlagP64 | (has_head ? agg : excl + agg));
  return excl;
}

// "Last block done": returns true in exactly one block, after every other
// block of the grid has passed this point (its prior writes made visible).
__device__ __forceinline__ bool last_block_done(unsigned int* ticket) {
  __shared__ unsigned int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
  __syncthreads();
  if (s_last) __threadfence();
  return s_last != 0;
}

#endif  // __CUDACC__

}  // namespace tb

// Shared definitions of the batched topology pass (host + device).
//
// The pass follows fVDB PR #757 ("Batched leaf-mask topology construction for
// generated conv grids", Summary item 1): an emission step over all source
// leaves of all grids writes candidate output-leaf slots, a radix sort puts
// them in canonical node order, a head-flag scan dedups them and derives
// per-grid counts and parent linkage, one readback sizes the outputs, and a
// batched writer emits the leaf records.
//
// Slots carry a 64-bit canonical key and a 32-bit source reference only; the
// 512-bit output masks are recomputed from the source masks where needed,
// which keeps the sort payload at 12 bytes per slot.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace tb {

// Pass kinds.  kIjk and kLeaves are the front ends (one slot per input voxel
// or input leaf); the others are the topology ops of a chain: refine and
// coarsen by a factor 2, 4 or 8 in one pass, a box dilation, and refinement
// by 2 followed by a box within [-1, 1]^3 (the k3s2 transpose) in one pass.
enum PassOp : int32_t { kIjk = 0, kLeaves = 1, kRefine = 2, kCoarsen = 3, kDilate = 4, kRefineDilate = 5 };
constexpr int kNumOps = 6;

constexpr int kNodeCap = 16384;       // most lower nodes (and tiles) of a node-path pass
constexpr int kBins = 256;            // 8-bit radix digits
constexpr int kMaxDigitPasses = 8;    // 64-bit key
// slot value = source index << code_bits | target code; code_bits per pass
// kind (pass_code_bits): 0 for the leaf front end, 3 log2(f) for refine and
// coarsen by f, 5 for a box dilation, 6 for refine-then-dilate.  The ijk
// front end's slot value is the voxel's bit in its leaf, 64 x + 8 y + z.

// Error bits reported through the readback header.
constexpr uint32_t kErrTimeout = 1u;       // a bounded wait (look-back or grid barrier) gave up
constexpr uint32_t kErrBadOffsets = 2u;    // jagged offsets not monotone / not covering
constexpr uint32_t kErrNotAligned = 4u;    // a leaf origin is not a multiple of 8
constexpr uint32_t kErrNotCanonical = 8u;  // tb_validate: order or mask violation
constexpr uint32_t kErrSlotOverflow = 16u; // emission exceeded the host's bound (bug guard)
constexpr uint32_t kErrLayout = 32u;       // a front end's input needs a key wider than 64 bits

// Look-back status words: two flag bits on top of the value.
constexpr uint32_t kFlagA32 = 1u << 30, kFlagP32 = 2u << 30, kVal32 = (1u << 30) - 1;
constexpr uint64_t kFlagA64 = 1ull << 62, kFlagP64 = 2ull << 62, kSeg64 = 1ull << 61,
                   kVal64 = (1ull << 61) - 1;
constexpr uint32_t kSpinLimit = 1u << 24;  // polls (with a short sleep) before a wait gives up

// Compressed canonical sort key.  Canonical order is lexicographic over
// (grid, T.x, T.y, T.z, U.x, U.y, U.z, V.x, V.y, V.z) where, for leaf
// coordinate lc = origin >> 3 on an axis, T = lc >> 9 (root tile),
// U = (lc >> 4) & 31 (child of the upper node), V = lc & 15 (child of the
// lower node).  Given the batch's range [Lo, Hi] of lc per axis, each field is
// stored relative to the smallest value it takes in its enclosing node:
//   T' = T - T(Lo);   U' = U - (T == T(Lo) ? U(Lo) : 0);
//   V' = V - (lc >> 4 == Lo >> 4 ? V(Lo) : 0).
// U is only ever compared between keys with equal T (and V between keys with
// equal T and U), so these per-node shifts keep the order while letting the
// fields shrink to the bits the range needs.
struct KeyLayout {
  int32_t W;             // total key width in bits (<= 64)
  int32_t gw, gshift;    // grid field
  int32_t t_lo[3];       // T(Lo) per axis
  int32_t u_lo[3];       // U(Lo)
  int32_t v_lo[3];       // V(Lo)
  int32_t tw[3], uw[3], vw[3];  // field widths
  int32_t tshift[3], ushift[3], vshift[3];
  int32_t lower_bits;    // key >> lower_bits == (grid, tile, upper child)
  int32_t node_bits;     // key >> node_bits  == (grid, tile)
};

// Host-visible block of a pass (read back in one copy):
// header | leaf_off[B+1] | lower_off[B+1] | upper_off[B+1] | voxels[B] | gbox[B*6]
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
  unsigned int dedup_tile_ctr;
  unsigned int dedup_ticket;
  unsigned int n_nodes;  // node path: lower nodes made by the emission
  unsigned int n_tiles;  // node path: root tiles (upper nodes) made by the emission
  unsigned int pad[4];
  unsigned int sort_tile_ctr[kMaxDigitPasses];
  unsigned long long head_totals[4];
  unsigned int hist[kMaxDigitPasses][kBins];
};

struct GridBarrier {
  unsigned int count;
  unsigned int gen;
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
  int32_t op;             // PassOp, or -1: no pass at this stage of the chain
  int32_t B;
  int32_t P;              // digit passes
  int32_t last;           // 1: final pass (count phase), 0: intermediate (hands leaves on)
  int32_t tchunk;         // targets per emission thread (1 .. targets per source)
  int32_t lo[3], hi[3];   // box of a dilation pass
  int32_t factor;         // refine / coarsen factor (2, 4, 8)
  int32_t code_bits;      // width of the target code in a slot value
  // source
  const int32_t* ijk;            // kIjk: [N,3]
  const int64_t* in_offsets;     // kIjk / kLeaves without src_grid: [B+1]
  const int32_t* src_origins;    // [L,3]
  const uint64_t* src_masks;     // [L,8]
  const int32_t* src_grid;       // [L] or null
  const unsigned long long* src_count_dev;  // device count (chained pass) or null
  long long src_count;                      // host count when src_count_dev is null
  // control (zeroed region)
  unsigned int* err;   // the call's device error word
  ReadbackHeader* rb;
  int64_t* leaf_off;   // [B+1]
  int64_t* lower_off;  // [B+1]
  int64_t* upper_off;  // [B+1]
  int64_t* grid_vox;   // [B] voxels per grid
  unsigned int* gbox;  // [B][6] encoded grid bbox accumulators
  PassCtl* ctl;
  uint32_t* sort_status;             // [P][sort_tiles_cap][256]
  long long sort_tiles_cap;
  unsigned long long* dedup_status;  // [dedup_tiles_cap][3]: leaves, lower nodes, upper nodes
  uint32_t* first;                   // [3][B]: 1 + first leaf / lower / upper index of each grid
  long long slot_cap;
  // slot buffers (not zeroed)
  uint64_t* keys[2];
  uint32_t* vals[2];
  int32_t sorted;        // which keys/vals buffer holds the sorted slots
  uint32_t* run_start;   // [slot_cap + 1]
  uint32_t* leaf_lower;  // [slot_cap]
  uint32_t* leaf_upper;  // [slot_cap]
  int64_t* leaf_voff;    // [slot_cap] voxel offset of each unique leaf (last pass)
  uint32_t* leaf_pop;    // [slot_cap] voxels of each unique leaf (last pass)
  uint32_t* leaf_g;      // [slot_cap] grid of each unique leaf (last pass)
  unsigned long long* blk_agg;  // [gridDim.x] segmented voxel aggregate per block (last pass)
  unsigned long long* grp_agg;  // [gridDim.x * 32] segmented voxel aggregate per 8-lane group (last pass)
  unsigned long long* phase_ts;  // optional [8] globaltimer stamps (profiling), else null
  // merged leaves: the next pass's source (intermediate pass), or the staged
  // masks and origins the final writer copies (last pass; null: the writer
  // merges the runs itself, and out_grid is unused)
  int32_t* out_origins;
  uint64_t* out_masks;
  int32_t* out_grid;
  // Node path (whole-grid launches whose output lower nodes are few): the
  // emission records every target leaf as a bit of its lower node's 4096-bit
  // child mask (NanoVDB's lower-node child mask, x-major bit order = the
  // canonical order of the leaves inside the node) in a hash table of lower
  // nodes; the nodes phase ranks the nodes by their canonical keys and takes
  // the masks' popcount prefixes; the place phase gives every leaf its index
  // (leaves before its node + set bits before it in its node's mask), writes
  // its record and merges every slot's contribution into it.  No sort.
  int32_t node;           // 1: this pass takes the node path
  int32_t node_zero;      // staged masks cleared: 0 never (one slot per leaf), 1 in the nodes phase, 2 in a phase of their own
  int32_t mid;            // phases between emission and leaves: P digit passes (and the index), or nodes [, clear], place
  int32_t node_cap;       // most lower nodes (the host's bound)
  uint32_t node_hmask;    // hash slots - 1 (a power of two): node and tile ids are slots
  int32_t node_pad;
  unsigned long long* nh_key;  // [hslots] lower-node key + 1, 0 = free (zeroed)
  unsigned long long* th_key;  // [hslots] tile key + 1, 0 = free (zeroed)
  uint64_t* node_mask;         // [hslots][64] child masks (zeroed)
  uint32_t* gmin;              // [2][B] ~(rank of the first lower node), ~(rank of the first tile) per grid (zeroed)
  uint64_t* node_key;          // [hslots] key >> lower_bits
  int32_t* node_lc;            // [hslots][4] lower-node coordinate (leaf coordinate >> 4) per axis, grid
  uint32_t* node_tile;         // [hslots] tile id
  uint32_t* node_rank;         // [hslots] canonical rank within the batch
  uint32_t* node_wpre;         // [hslots][64] set bits of the child mask before each word
  uint32_t* rank_cnt;          // [node_cap] leaves of the node of each rank
  uint32_t* tile_rank;         // [hslots]
  uint32_t* node_list;         // [node_cap] the nodes' ids in order of making
  uint32_t* tile_list;         // [node_cap] the tiles' ids in order of making
  uint32_t* nref;              // [slot_cap] node id << 12 | child bit of each slot
  // member launches (k_member): every grid of a chain runs as its own batch of
  // one grid on its share of the chain's buffers.  In a member template the
  // buffer pointers above are the chain's bases, and B, rb and the per-grid
  // arrays are the chain's; the kernel derives each member's arguments.
  int32_t member;            // 1: a member template
  int32_t cl;                // CTAs per member (one cluster)
  const int64_t* unit_off;   // [B+1] first stage-0 source (leaf or voxel) of each grid
  long long m_stage;         // slots of this stage per stage-0 source (capacity)
  long long m_slots;         // slot-array capacity of the chain per stage-0 source
  long long m_out;           // out-array capacity of this stage per stage-0 source
  char* unit_ctl;            // this stage's member control blocks, ctl_stride bytes apart
  long long ctl_stride;      // readback part | PassCtl (P histogram rows) | first[3]
  long long ctl_rb_bytes;    // bytes of the readback part
};

// Arguments of one cooperative launch: n_chain chains of up to n_stage
// passes over the same input; pass[c * n_stage + k] is stage k of chain c
// (op < 0 where chain c is shorter).  The array lives in device memory.
// With `front` set, pass 0 of chain 0 (the only pass) is a front end whose
// key layout every block plans itself from the input's bbox (its K, P and
// `sorted` in the pass's arguments are placeholders).
struct ChainArgs {
  const PassArgs* pass;  // [n_chain * n_stage], device memory
  int32_t n_chain;
  int32_t n_stage;
  GridBarrier* bar;
  unsigned int* err;
  int32_t front;
  // member launches: B grids per chain, cl CTAs per member, and the
  // finished members of each chain (zeroed)
  int32_t B;
  int32_t cl;
  unsigned int* done;  // [n_chain]
  // the readback without a stream synchronisation: the last CTA out copies
  // the readback span (span_bytes, a multiple of 16, from dev_span) to pinned
  // host memory and then stores `seq` to the host flag; null host_span: off
  char* host_span;
  const char* dev_span;
  long long span_bytes;
  unsigned int* exit_ctr;  // zeroed
  unsigned int* host_flag;
  unsigned int seq;
};


// Outputs of the final writer.
struct WriteOut {
  int32_t* origins;
  uint64_t* masks;
  int32_t* leaf_grid;
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
  // the arrays' room: a writer whose counts exceed it writes nothing (the
  // host sized it from an earlier call of the same shape and writes again)
  long long L_cap, NL_cap, NU_cap;
};

// ---------------------------------------------------------------- keys

__host__ __device__ inline uint64_t shr64(uint64_t x, int s) { return s >= 64 ? 0ull : (x >> s); }

__host__ __device__ inline uint64_t encode_key(const KeyLayout& K, uint32_t g, int32_t lcx, int32_t lcy,
                                               int32_t lcz) {
  const int32_t lc[3] = {lcx, lcy, lcz};
  uint64_t key = K.gw ? ((uint64_t)g << K.gshift) : 0ull;
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    const int32_t T = lc[a] >> 9;
    const uint32_t U = ((uint32_t)lc[a] >> 4) & 31u, V = (uint32_t)lc[a] & 15u;
    const bool t0 = (T == K.t_lo[a]);
    const bool b0 = t0 && (U == (uint32_t)K.u_lo[a]);
    const uint32_t t = (uint32_t)(T - K.t_lo[a]);
    const uint32_t u = U - (t0 ? (uint32_t)K.u_lo[a] : 0u);
    const uint32_t v = V - (b0 ? (uint32_t)K.v_lo[a] : 0u);
    if (K.tw[a]) key |= (uint64_t)t << K.tshift[a];
    if (K.uw[a]) key |= (uint64_t)u << K.ushift[a];
    if (K.vw[a]) key |= (uint64_t)v << K.vshift[a];
  }
  return key;
}

__host__ __device__ inline void decode_key(const KeyLayout& K, uint64_t key, uint32_t& g, int32_t lc[3]) {
  g = K.gw ? (uint32_t)(key >> K.gshift) : 0u;
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    const uint32_t t = K.tw[a] ? (uint32_t)((key >> K.tshift[a]) & ((1ull << K.tw[a]) - 1ull)) : 0u;
    const uint32_t u = K.uw[a] ? (uint32_t)(key >> K.ushift[a]) & ((1u << K.uw[a]) - 1u) : 0u;
    const uint32_t v = K.vw[a] ? (uint32_t)(key >> K.vshift[a]) & ((1u << K.vw[a]) - 1u) : 0u;
    const int32_t T = K.t_lo[a] + (int32_t)t;
    const bool t0 = (t == 0);
    const uint32_t U = u + (t0 ? (uint32_t)K.u_lo[a] : 0u);
    const bool b0 = t0 && (U == (uint32_t)K.u_lo[a]);
    const uint32_t V = v + (b0 ? (uint32_t)K.v_lo[a] : 0u);
    lc[a] = (int32_t)(((uint32_t)T << 9) | (U << 4) | V);
  }
}

// One chain's share of a multi-chain writer launch.
constexpr int kMaxWriteTasks = 16;
struct WriteTask {
  PassArgs a;
  WriteOut o;
};
// The tasks of one writer launch, passed by value as its kernel parameter.
struct WriteTasks {
  WriteTask t[kMaxWriteTasks];
  int32_t n;
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
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void load_mask(const uint64_t* masks, long long i, uint64_t m[8]) {
  const uint4* p = reinterpret_cast<const uint4*>(masks + 8 * i);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 v = __ldcg(p + q);
    m[2 * q] = (uint64_t)v.x | ((uint64_t)v.y << 32);
    m[2 * q + 1] = (uint64_t)v.z | ((uint64_t)v.w << 32);
  }
}

// ---------------------------------------------------------------- leaf mask arithmetic
// Mask word w holds the voxels with local x == w; bit 8*y + z.

// Refinement by 2: word w of child c = (cx, cy, cz) of a leaf is built from
// parent word 4*cx + (w >> 1): parent rows 4*cy .. 4*cy+3, bits 4*cz .. 4*cz+3,
// each parent bit doubled in z and each row doubled in y.
__device__ __forceinline__ uint64_t refine_word(uint64_t parent_word, int cy, int cz) {
  // every row's nibble 4 cz .. 4 cz + 3 at once, each bit doubled in its byte
  uint64_t x = (parent_word >> (4 * cz)) & 0x0F0F0F0F0F0F0F0Full;
  x = (x | (x << 2)) & 0x3333333333333333ull;
  x = (x | (x << 1)) & 0x5555555555555555ull;
  x |= x << 1;
  // rows 4 cy .. 4 cy + 3, each doubled
  uint64_t v = (x >> (32 * cy)) & 0xFFFFFFFFull;
  v = (v | (v << 16)) & 0x0000FFFF0000FFFFull;
  v = (v | (v << 8)) & 0x00FF00FF00FF00FFull;
  return v | (v << 8);
}

// Refinement by f = 4 or 8: word w of child c = (cx, cy, cz) of a leaf comes
// from parent word (8 cx + w) / f; child row y from parent row (8 cy + y) / f
// and child bit z from parent bit (8 cz + z) / f.  parent_word is that word.
__device__ __forceinline__ uint64_t refine_word_f(uint64_t parent_word, int cy, int cz, int f) {
  const int bs = 8 / f;  // parent rows (and bits) per child along an axis
  uint64_t out = 0;
#pragma unroll
  for (int y = 0; y < 8; ++y) {
    const uint32_t sb = (uint32_t)(parent_word >> (8 * (cy * bs + y / f))) & 0xFFu;
    uint32_t tb = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < bs && ((sb >> (cz * bs + j)) & 1u)) tb |= ((1u << f) - 1u) << (j * f);
    out |= (uint64_t)(tb & 0xFFu) << (8 * y);
  }
  return out;
}

// Coarsening by f = 4 or 8 of the rows and bits of t (the OR of the f source
// words that fall into one coarse word): source row y goes to coarse row
// qy * 8/f + y / f, bit z to coarse bit qz * 8/f + z / f, where (qy, qz) is
// the source leaf's position inside the coarse leaf.
__device__ __forceinline__ uint64_t coarsen_word_f(uint64_t t, int qy, int qz, int f) {
  if (f == 8) return t ? 1ull << (8 * qy + qz) : 0ull;  // the whole source leaf is one coarse voxel
  // f == 4: rows 0-3 and 4-7 fold into coarse rows 2 qy and 2 qy + 1; within
  // a row, bits 0-3 and 4-7 into coarse bits 2 qz and 2 qz + 1
  uint64_t r = t | (t >> 8);
  r |= r >> 16;  // byte 0: OR of rows 0-3, byte 4: OR of rows 4-7
  uint64_t out = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t b = (uint32_t)(r >> (32 * h)) & 0xFFu;
    const uint32_t c = ((b & 0x0Fu) ? 1u : 0u) | ((b & 0xF0u) ? 2u : 0u);
    out |= (uint64_t)c << (8 * (2 * qy + h) + 2 * qz);
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

// Box dilation by [lo, hi] (lo in -7..0, hi in 0..7 per axis) restricted to
// one target leaf at offset t in {-1, 0, 1} along an axis: a voxel at local
// coordinate c reaches local coordinate c + d - 8 t of the target for every d
// in [lo, hi] that keeps it inside 0..7.  Per axis that is an OR of shifts by
// k = d - 8 t, |k| <= 7.
//   z: bits within each row (byte) of a word;
//   y: rows within a word;
//   x: words of the mask (see dilate_x).
__device__ __forceinline__ uint64_t dilate_z(uint64_t s, int tz, int lo, int hi) {
  uint64_t r = 0;
  for (int d = lo; d <= hi; ++d) {
    const int k = d - 8 * tz;
    if (k >= 8 || k <= -8) continue;
    r |= k >= 0 ? (s << k) & (0x0101010101010101ull * ((0xFFu << k) & 0xFFu))
                : (s >> -k) & (0x0101010101010101ull * (0xFFu >> -k));
  }
  return r;
}
__device__ __forceinline__ uint64_t dilate_y(uint64_t s, int ty, int lo, int hi) {
  uint64_t r = 0;
  for (int d = lo; d <= hi; ++d) {
    const int k = d - 8 * ty;
    if (k >= 8 || k <= -8) continue;
    r |= k >= 0 ? s << (8 * k) : s >> (-8 * k);
  }
  return r;
}
// The same three parts for a box within [-1, 1] per axis, with constant
// masks: the common conv-grid case (k3s1, the pads, the k3s2 transpose).
__device__ __forceinline__ uint64_t dilate_z1(uint64_t s, int tz, int lo, int hi) {
  if (tz == 0) {
    uint64_t r = s;
    if (hi > 0) r |= (s << 1) & 0xFEFEFEFEFEFEFEFEull;
    if (lo < 0) r |= (s >> 1) & 0x7F7F7F7F7F7F7F7Full;
    return r;
  }
  if (tz > 0) return (s >> 7) & 0x0101010101010101ull;  // z = 7 moves to z = 0 of the next leaf
  return (s << 7) & 0x8080808080808080ull;              // z = 0 moves to z = 7 of the previous leaf
}
__device__ __forceinline__ uint64_t dilate_y1(uint64_t s, int ty, int lo, int hi) {
  if (ty == 0) {
    uint64_t r = s;
    if (hi > 0) r |= s << 8;
    if (lo < 0) r |= s >> 8;
    return r;
  }
  if (ty > 0) return s >> 56;  // row 7 moves to row 0 of the next leaf
  return s << 56;              // row 0 moves to row 7 of the previous leaf
}
__device__ __forceinline__ uint64_t dilate_x1(const uint64_t m[8], int k, int tx, int lo, int hi) {
  if (tx == 0) {
    uint64_t r = m[k];
    if (hi > 0 && k >= 1) r |= m[k - 1];
    if (lo < 0 && k <= 6) r |= m[k + 1];
    return r;
  }
  if (tx > 0) return k == 0 ? m[7] : 0ull;
  return k == 7 ? m[0] : 0ull;
}

// Word k of the x part for target offset tx: the OR of source words k - k'
// for the shifts k' = d - 8 tx that land inside the target.
__device__ __forceinline__ uint64_t dilate_x(const uint64_t m[8], int k, int tx, int lo, int hi) {
  uint64_t r = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int sh = k - j + 8 * tx;  // the d that carries word j to word k
    if (sh >= lo && sh <= hi) r |= m[j];
  }
  return r;
}
// The voxels of a source leaf that reach target offset t along an axis lie in
// local coordinates [8t - hi, 8t + 7 - lo] within 0..7; the bits of that zone
// as a mask over the 8 positions (bit c = coordinate c).
__device__ __forceinline__ uint32_t dilate_zone(int t, int lo, int hi) {
  const int a = 8 * t - hi < 0 ? 0 : 8 * t - hi, b = 8 * t + 7 - lo > 7 ? 7 : 8 * t + 7 - lo;
  return a > b ? 0u : ((0xFFu >> (7 - b)) & (0xFFu << a)) & 0xFFu;
}

// OR-reduce-scatter over an aligned group of 8 lanes: lane w of the group
// returns the OR over the group's lanes of c[w].
__device__ __forceinline__ uint64_t reduce_scatter8(const uint64_t c[8], int w) {
  uint64_t k4[4], k2[2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint64_t send = (w & 4) ? c[k] : c[k + 4];
    const uint64_t recv = __shfl_xor_sync(0xffffffffu, send, 4);
    k4[k] = ((w & 4) ? c[k + 4] : c[k]) | recv;
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint64_t send = (w & 2) ? k4[k] : k4[k + 2];
    const uint64_t recv = __shfl_xor_sync(0xffffffffu, send, 2);
    k2[k] = ((w & 2) ? k4[k + 2] : k4[k]) | recv;
  }
  const uint64_t send = (w & 1) ? k2[0] : k2[1];
  const uint64_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
  return ((w & 1) ? k2[1] : k2[0]) | recv;
}

// ---------------------------------------------------------------- scans, look-back, barrier

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

// Decoupled look-back over 32-bit status words (one thread per digit): publish
// the tile's aggregate, add predecessors until an inclusive prefix is found,
// publish the inclusive prefix.  Returns the exclusive prefix.  Predecessors
// are read eight at a time (independent loads), nearest first, so tiles that
// run at the same time resolve in about one load latency per window.  A wait
// on a tile that never publishes ends after kSpinLimit polls with kErrTimeout
// set.
__device__ __forceinline__ uint32_t lookback32(uint32_t* status, long long stride, long long tile,
                                               uint32_t agg, unsigned int* err) {
  constexpr int kWin = 8;
  if (tile == 0) {
    st_relaxed(status, kFlagP32 | agg);
    return 0;
  }
  st_relaxed(status + tile * stride, kFlagA32 | agg);
  uint32_t excl = 0;
  long long t = tile - 1;
  uint32_t spins = 0;
  while (t >= 0) {
    uint32_t w[kWin];
#pragma unroll
    for (int j = 0; j < kWin; ++j) w[j] = t - j >= 0 ? ld_relaxed(status + (t - j) * stride) : kFlagP32;
    int used = 0;
    bool done = false;
#pragma unroll
    for (int j = 0; j < kWin; ++j) {
      if (done || used < j) continue;  // stop at the first unpublished predecessor
      const uint32_t f = w[j] & ~kVal32;
      if (f == 0) continue;
      excl += w[j] & kVal32;
      used = j + 1;
      done = f == kFlagP32;
    }
    if (done) break;
    t -= used;
    if (used == 0) {
      if (++spins > kSpinLimit) {
        atomicOr(err, kErrTimeout);
        break;
      }
      __nanosleep(32);
    }
  }
  st_relaxed(status + tile * stride, kFlagP32 | (excl + agg));
  return excl;
}

// Warp-wide decoupled look-back over 64-bit status words, in two steps so a
// tile can publish its aggregate early and resolve its prefix later.
// lb64_publish: lane 0 stores the tile's aggregate (with the segment flag when
// the tile holds a segment head).  lb64_resolve (a whole warp; lanes inspect
// 32 predecessors at once) adds predecessor values until an inclusive prefix
// -- or, for a segmented scan, an aggregate holding a segment head -- ends the
// walk, publishes the tile's inclusive prefix and returns the exclusive prefix
// in every lane.  A wait on a tile that never publishes ends after kSpinLimit
// polls with kErrTimeout set.
__device__ __forceinline__ void lb64_publish(unsigned long long* status, long long stride, long long tile,
                                             uint64_t agg, bool has_head) {
  if ((threadIdx.x & 31) == 0)
    st_relaxed(status + tile * stride, (tile == 0 ? kFlagP64 : (kFlagA64 | (has_head ? kSeg64 : 0ull))) | agg);
}

__device__ __forceinline__ uint64_t lb64_resolve(unsigned long long* status, long long stride, long long tile,
                                                 uint64_t agg, bool has_head, unsigned int* err) {
  const int lane = threadIdx.x & 31;
  if (tile == 0) return 0;
  uint64_t excl = 0;
  long long base = tile - 1;  // window covers tiles base, base-1, ..., base-31
  uint32_t spins = 0;
  while (base >= 0) {
    const long long t = base - lane;
    const uint64_t w = t >= 0 ? ld_relaxed(status + t * stride) : kFlagP64;  // before tile 0: an empty prefix
    const bool ready = (w >> 62) != 0;
    const bool stop = ((w >> 62) == 2) || (w & kSeg64);
    const uint32_t stop_mask = __ballot_sync(0xffffffffu, ready && stop);
    const uint32_t ready_mask = __ballot_sync(0xffffffffu, ready);
    const int first_stop = stop_mask ? __ffs(stop_mask) - 1 : 32;
    const uint32_t need = first_stop == 32 ? 0xffffffffu : ((2u << first_stop) - 1u);
    if ((ready_mask & need) != need) {
      if (++spins > kSpinLimit) {
        if (lane == 0) atomicOr(err, kErrTimeout);
        break;
      }
      __nanosleep(32);
      continue;
    }
    uint64_t v = (lane <= first_stop && t >= 0) ? (w & kVal64) : 0ull;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    excl += v;
    if (first_stop < 32) break;
    base -= 32;
  }
  if (lane == 0) st_relaxed(status + tile * stride, kFlagP64 | (has_head ? agg : excl + agg));
  return excl;
}

// Segmented exclusive scan over a 256-thread block of (head flag f, value v)
// pairs in thread order; a set flag starts a new segment.  Returns the
// thread's exclusive (flag, sum since the last head) and the block aggregate.
// `scratch_f` / `scratch_v` hold 8 entries.
__device__ __forceinline__ void block_seg_scan_256(uint32_t f, unsigned long long v, uint32_t* scratch_f,
                                                   unsigned long long* scratch_v, uint32_t& ef,
                                                   unsigned long long& ev, uint32_t& tf, unsigned long long& tv) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t F = f;
  unsigned long long V = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t F2 = __shfl_up_sync(0xffffffffu, F, off);
    const unsigned long long V2 = __shfl_up_sync(0xffffffffu, V, off);
    if (lane >= off) {
      if (!F) V += V2;
      F |= F2;
    }
  }
  uint32_t lf = __shfl_up_sync(0xffffffffu, F, 1);
  unsigned long long lv = __shfl_up_sync(0xffffffffu, V, 1);
  if (lane == 0) {
    lf = 0;
    lv = 0;
  }
  if (lane == 31) {
    scratch_f[warp] = F;
    scratch_v[warp] = V;
  }
  __syncthreads();
  uint32_t pf = 0;
  unsigned long long pv = 0;
  tf = 0;
  tv = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t wf = scratch_f[w];
    const unsigned long long wv = scratch_v[w];
    if (w < warp) {
      pv = wf ? wv : pv + wv;
      pf |= wf;
    }
    tv = wf ? wv : tv + wv;
    tf |= wf;
  }
  __syncthreads();
  ef = pf | lf;
  ev = lf ? lv : pv + lv;
}

// ---------------------------------------------------------------- front-end bounds

// Block reduction of encoded bounds, then one atomic per bound per block.
__device__ __forceinline__ void reduce_bbox(const int32_t mn[3], const int32_t mx[3], unsigned int* enc) {
  __shared__ unsigned int s_enc[6];
  if (threadIdx.x < 6) s_enc[threadIdx.x] = 0;
  __syncthreads();
  unsigned int e[6] = {enc_min(mn[0]), enc_min(mn[1]), enc_min(mn[2]), enc_max(mx[0]), enc_max(mx[1]),
                       enc_max(mx[2])};
#pragma unroll
  for (int k = 0; k < 6; ++k) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) e[k] = max(e[k], __shfl_xor_sync(0xffffffffu, e[k], off));
  }
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int k = 0; k < 6; ++k) atomicMax(&s_enc[k], e[k]);
  __syncthreads();
  if (threadIdx.x < 6 && s_enc[threadIdx.x]) atomicMax(&enc[threadIdx.x], s_enc[threadIdx.x]);
}

// Jagged offsets: offsets[0] == 0, non-decreasing, offsets[B] == n.
__device__ __forceinline__ void check_offsets(const int64_t* off, int32_t B, long long n, unsigned int* err) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g <= B; g += stride) {
    const int64_t v = off[g];
    bool bad = (g == 0 && v != 0) || (g == B && v != n) || v < 0 || v > n;
    if (g > 0 && off[g - 1] > v) bad = true;
    if (bad) atomicOr(err, kErrBadOffsets);
  }
}

// This thread's share (stride over the vg blocks of a virtual grid) of the
// bounds of N voxel coordinates.
__device__ __forceinline__ void ijk_bounds(const int32_t* ijk, long long N, int32_t mn[3], int32_t mx[3], int vb,
                                           int vg) {
  for (int a = 0; a < 3; ++a) {
    mn[a] = INT32_MAX;
    mx[a] = INT32_MIN;
  }
  const long long stride = (long long)vg * blockDim.x;
  for (long long i = (long long)vb * blockDim.x + threadIdx.x; i < N; i += stride)
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      const int32_t v = __ldg(ijk + 3 * i + a);
      mn[a] = min(mn[a], v);
      mx[a] = max(mx[a], v);
    }
}

// This thread's share (over a virtual grid, as ijk_bounds) of the exact voxel
// bounds of L leaves (from their set bits); flags origins that are not
// multiples of 8.
__device__ __forceinline__ void leaves_bounds(const int32_t* origins, const uint64_t* masks, long long L,
                                              int32_t mn[3], int32_t mx[3], unsigned int* err, int vb, int vg) {
  for (int a = 0; a < 3; ++a) {
    mn[a] = INT32_MAX;
    mx[a] = INT32_MIN;
  }
  const long long stride = (long long)vg * blockDim.x;
  for (long long i = (long long)vb * blockDim.x + threadIdx.x; i < L; i += stride) {
    uint64_t m[8];
    load_mask(masks, i, m);
    uint64_t all = 0;
    uint32_t xbits = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      all |= m[w];
      if (m[w]) xbits |= 1u << w;
    }
    const int32_t o[3] = {__ldg(origins + 3 * i), __ldg(origins + 3 * i + 1), __ldg(origins + 3 * i + 2)};
    if ((o[0] | o[1] | o[2]) & 7) atomicOr(err, kErrNotAligned);
    if (!all) continue;
    uint32_t ybits = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if ((all >> (8 * r)) & 0xFFull) ybits |= 1u << r;
    uint64_t z = all | (all >> 32);
    z |= z >> 16;
    z |= z >> 8;
    const uint32_t zbits = (uint32_t)(z & 0xFFull);
    const uint32_t b[3] = {xbits, ybits, zbits};
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      mn[a] = min(mn[a], o[a] + (__ffs(b[a]) - 1));
      mx[a] = max(mx[a], o[a] + (31 - __clz(b[a])));
    }
  }
}

// Software grid barrier for a cooperative launch (all blocks co-resident):
// a monotone arrival counter; barrier n completes when the counter reaches
// n * gridDim.x.  The wait gives up after kSpinLimit polls with kErrTimeout
// set, so a broken barrier ends the kernel instead of hanging it.
// Waits until *p reaches `target` (a wrap-safe difference) or `limit` polls
// have passed; then sets kErrTimeout in *err and returns false.  Every
// spin-wait on another block's progress in this library goes through a
// bounded wait like this one.
__device__ __forceinline__ bool wait_reach(const uint32_t* p, uint32_t target, uint32_t limit, unsigned int* err) {
  uint32_t spins = 0;
  while ((int)(ld_relaxed(p) - target) < 0) {
    if (++spins > limit) {
      atomicOr(err, kErrTimeout);
      return false;
    }
    if (spins > 256) __nanosleep(32);
  }
  return true;
}

__device__ __forceinline__ void grid_sync(GridBarrier* bar, unsigned int* err) {
  __syncthreads();  // the block's writes before thread 0's release below
  if (threadIdx.x == 0) {
    unsigned int old;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(&bar->count) : "memory");
    const unsigned int target = (old / gridDim.x + 1) * gridDim.x;
    wait_reach(&bar->count, target, kSpinLimit, err);
    asm volatile("fence.acq_rel.gpu;" ::: "memory");  // with the relaxed poll: an acquire
  }
  __syncthreads();
}

#endif  // __CUDACC__

}  // namespace tb
